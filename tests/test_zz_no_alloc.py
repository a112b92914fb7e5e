"""fs_dispatch_noalloc: the dispatch for callers that cannot give the library
device scratch memory (a plugin interface that passes only inputs and outputs,
or a code path that must not call cudaMalloc/cudaFree).  It must produce
exactly what fs_dispatch produces with a caller workspace -- counts, offsets,
positions, permutation and permuted rows are integer/byte results, so the
comparison is bit for bit -- on consecutive calls that reuse the library's one
static scratch array.  The file name makes pytest collect it last."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_expert_gb300 import configs, fs, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _topk(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.rand((T, E), generator=g).argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def _outputs(T, E, k, d, dt):
    i32 = dict(dtype=torch.int32, device=DEV)
    return [torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32), torch.full((T * k,), -7, **i32),
            torch.full((T * k,), -7, **i32), torch.zeros((T * k, d), dtype=dt, device=DEV)]


@pytest.mark.parametrize("T,E,k,d", [(3000, 64, 6, 256), (65536, 256, 8, 128)])
def test_noalloc_matches_workspace_dispatch_twice(T, E, k, d):
    cfg = configs.LayerConfig("na", T=T, d=d, E=E, k=k, c=64, n_shared=0, c_shared=0, L=1, gate="softmax",
                              dtype="bf16")
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    u = synth.make_x(cfg, DEV)
    for call, seed in enumerate((101, 202)):       # two calls in a row, different routings
        idx = _topk(T, E, k, seed + T).to(DEV)
        ref = _outputs(T, E, k, d, u.dtype)
        got = _outputs(T, E, k, d, u.dtype)
        fs.fs_dispatch(desc, idx, u, *ref, ws)
        fs.fs_dispatch_noalloc(desc, idx, u, *got)
        torch.cuda.synchronize()
        assert fs.fs_get_error() == (0, 0)
        for name, a, b in zip(("counts", "offsets", "pos", "perm_src", "x_perm"), ref, got):
            assert torch.equal(a, b), "call %d: %s differs" % (call, name)
        assert int(ref[1][-1]) == T * k


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # ceil(T / 1024) * E = 300 * 256 = 76,800 ints > 65,536: rejected before any launch
    cfg = configs.LayerConfig("big", T=300 * 1024, d=64, E=256, k=1, c=64, n_shared=0, c_shared=0, L=1,
                              gate="softmax", dtype="bf16")
    desc = fs.make_desc(cfg)
    fake = torch.empty(16, dtype=torch.int32, device=DEV)   # never touched
    n0 = fs.fs_launch_count()
    with pytest.raises(fs.FsError) as e:
        fs.fs_dispatch_noalloc(desc, fake, fake, fake, fake, fake, fake, fake)
    assert e.value.status == 3 and "static maximum" in str(e.value)
    assert fs.fs_launch_count() == n0
