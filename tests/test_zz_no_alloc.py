"""fs_dispatch_noalloc: the dispatch for callers that cannot give the library
device scratch memory (a plugin interface that passes only inputs and outputs,
or a code path that must not call cudaMalloc/cudaFree).  It must produce
exactly what fs_dispatch produces with a caller workspace -- counts, offsets,
positions, permutation and permuted rows (bf16 rows, or FP8 codes and row
scales) are integer/byte results, so the comparison is bit for bit -- on
consecutive calls that reuse the library's one static scratch array.  The
largest accepted shape sits exactly at the array's size (ceil(T / 1024) * E =
65,536 ints); one token more is rejected.  The file name makes pytest collect
it last."""
import pytest
import torch

from mixture_experts_layer_expert_gb300 import configs, fs, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT_INTS = 65536       # the static scratch holds this many ints


def _topk(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.rand((T, E), generator=g).argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def _outputs(T, E, k, d, dt, fp8=False, copy=True):
    i32 = dict(dtype=torch.int32, device=DEV)
    if not copy:
        xp = None
    elif fp8:
        xp = torch.zeros(fs.fs_fp8_rows_bytes(T * k, d), dtype=torch.uint8, device=DEV)
    else:
        xp = torch.zeros((T * k, d), dtype=dt, device=DEV)
    return [torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32), torch.full((T * k,), -7, **i32),
            torch.full((T * k,), -7, **i32), xp]


@pytest.mark.parametrize("T,E,k,d,dtype,copy", [(3000, 64, 6, 256, "bf16", True),
                                                (65536, 256, 8, 128, "bf16", True),
                                                (131072, 512, 1, 64, "bf16", True),     # exactly at the limit
                                                (2500, 32, 4, 256, "fp8", True),        # quantising copy
                                                (5000, 128, 8, 128, "bf16", False)])    # no row copy
def test_noalloc_matches_workspace_dispatch_twice(T, E, k, d, dtype, copy):
    cfg = configs.LayerConfig("na", T=T, d=d if dtype == "bf16" else max(d, 128), E=E, k=k, c=128, n_shared=0,
                              c_shared=0, L=1, gate="softmax", dtype=dtype)
    if T == 131072:
        assert -(-T // 1024) * E == LIMIT_INTS
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    u = synth.make_x(cfg, DEV)
    fp8 = dtype == "fp8"
    for call, seed in enumerate((101, 202)):       # two calls in a row, different routings
        idx = _topk(T, E, k, seed + T).to(DEV)
        ref = _outputs(T, E, k, cfg.d, u.dtype, fp8, copy)
        got = _outputs(T, E, k, cfg.d, u.dtype, fp8, copy)
        fs.fs_dispatch(desc, idx, u, *ref, ws)
        fs.fs_dispatch_noalloc(desc, idx, u, *got)
        torch.cuda.synchronize()
        assert fs.fs_get_error() == (0, 0)
        for name, a, b in zip(("counts", "offsets", "pos", "perm_src", "x_perm"), ref, got):
            if a is None:
                assert b is None
                continue
            assert torch.equal(a, b), "call %d: %s differs" % (call, name)
        assert int(ref[1][-1]) == T * k


@pytest.mark.parametrize("T,E", [(300 * 1024, 256), (131073, 512)])
def test_noalloc_rejects_shapes_beyond_its_scratch(T, E):
    # ceil(T / 1024) * E = 76,800 or 66,048 ints > 65,536: rejected before any launch
    assert -(-T // 1024) * E > LIMIT_INTS
    cfg = configs.LayerConfig("big", T=T, d=64, E=E, k=1, c=64, n_shared=0, c_shared=0, L=1,
                              gate="softmax", dtype="bf16")
    desc = fs.make_desc(cfg)
    fake = torch.empty(16, dtype=torch.int32, device=DEV)   # never touched
    n0 = fs.fs_launch_count()
    with pytest.raises(fs.FsError) as e:
        fs.fs_dispatch_noalloc(desc, fake, fake, fake, fake, fake, fake, fake)
    assert e.value.status == 3 and "static maximum" in str(e.value)
    assert fs.fs_launch_count() == n0
