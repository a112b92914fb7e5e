"""GPU parity of the FP8 expert path (FS_FP8) against the oracle's FP8 form.

Integer and byte results are compared bit for bit: the E4M3 codes and the
power-of-two row scales of fs_quantize_rows_fp8, of the FP8 weight packing and
of the FP8 Dispatch copy, since both sides quantise the same bf16 values with
the same rule (smallest e with max |x| 2^-e <= 448, nearest-even E4M3).
Floating-point results (the expert outputs, the shared expert, the stack)
meet the bf16 bounds: relative Frobenius <= 5e-3, max-abs <= 2e-2 rms.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_expert_gb300 import configs, fs, synth
from parity import compare, oracle_cfg, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _no_dev_error():
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    assert st == 0, "device error word = %d" % code


def small(**kw):
    base = dict(name="f8", T=300, d=256, E=8, k=2, c=256, n_shared=1, c_shared=128, L=1,
                gate="softmax_renorm", dtype="fp8")
    base.update(kw)
    return configs.LayerConfig(**base)


def _bf16_rows(rows, cols, seed):
    """bf16 rows with assorted magnitudes: zero rows, a row whose largest
    element is exactly 448 * 2^j (a scale boundary), tiny and large rows."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, cols), generator=g)
    mag = torch.exp2(torch.randint(-20, 12, (rows, 1), generator=g).float())
    x = x * mag
    if rows > 4:
        x[1] = 0.0
        x[2, 5] = 448.0 * 2.0 ** -3
        x[2] = x[2].clamp(-448.0 * 2.0 ** -3, 448.0 * 2.0 ** -3)
        x[3] = x[3] * 1e-30
    return x.to(torch.bfloat16)


def _codes_equal(got, want, what):
    """E4M3 codes bit for bit; the two zeros are equal values (0x00 / 0x80)."""
    g = got.astype(np.uint8)
    w = want.astype(np.uint8)
    zero = ((g & 0x7F) == 0) & ((w & 0x7F) == 0)
    bad = (g != w) & ~zero
    assert not bad.any(), "%s: %d codes differ, first at %s (got %#x want %#x)" % (
        what, int(bad.sum()), np.argwhere(bad)[0], g[bad][0], w[bad][0])


@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 256), (1000, 384), (4099, 2048), (64, 8192)])
def test_quantize_rows_bit_exact(fs, rows, cols):
    x = _bf16_rows(rows, cols, rows + cols)
    xd = x.to(DEV)
    q = fs.fp8_rows_empty(rows, cols, DEV)
    q.fill_(0xAB)
    fs.fs_quantize_rows_fp8(rows, cols, xd, q)
    _no_dev_error()
    codes, scales = fs.fp8_rows_split(q, rows, cols)
    rc, re, _ = oracle.quant_rows(synth.to_numpy(x), "bf16")
    _codes_equal(codes.cpu().numpy(), rc, "codes")
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.float64), np.exp2(re.astype(np.float64)))


def _unpack(buf, G, N, K):
    """Codes [G, N, K] and scales [G, N] of an FP8 weight pack (tiled layout)."""
    NB = (N + 255) // 256
    KB = K // 128
    nc = G * NB * KB * 32768
    c = buf[:nc].cpu().numpy().reshape(G, NB, KB, 256, 128).transpose(0, 1, 3, 2, 4).reshape(G, NB * 256, K)
    pad = c[:, N:, :]
    s = buf[nc:nc + 4 * G * N].view(torch.float32).cpu().numpy().reshape(G, N)
    return c[:, :N, :], s, pad


def _oracle_rows(w_rows_bf16):
    codes, exps, _ = oracle.quant_rows(synth.to_numpy(w_rows_bf16.reshape(-1, w_rows_bf16.shape[-1])), "bf16")
    return codes, np.exp2(exps.astype(np.float64))


@pytest.mark.parametrize("E,c,d", [(3, 128, 256), (2, 384, 384), (5, 256, 128)])
def test_pack_fp8_bit_exact(fs, E, c, d):
    cfg = small(E=E, c=c, d=d, n_shared=2, c_shared=128)
    w = synth.make_block_weights(cfg, 0, DEV)
    p = fs.pack_block(cfg, w)
    _no_dev_error()
    # gate/up: packed row n of expert e is W2 (gate) row 64 (n // 128) + n % 128 for
    # n % 128 < 64, else W1 (up) row 64 (n // 128) + n % 128 - 64
    n = np.arange(2 * c)
    blk, within = n // 128, n % 128
    src = 64 * blk + np.where(within < 64, within, within - 64)
    is_gate = within < 64
    w1, w2 = w["w1"].cpu(), w["w2"].cpu()
    ref13 = torch.where(torch.from_numpy(is_gate)[None, :, None], w2[:, src], w1[:, src])      # [E, 2c, d]
    codes, scales, pad = _unpack(p["w13"], E, 2 * c, d)
    rc, rs = _oracle_rows(ref13)
    _codes_equal(codes.reshape(-1, d), rc, "w13 codes")
    np.testing.assert_array_equal(scales.reshape(-1), rs)
    assert not pad.any()
    codes, scales, pad = _unpack(p["w3"], E, d, c)
    rc, rs = _oracle_rows(w["w3"].cpu())
    _codes_equal(codes.reshape(-1, c), rc, "w3 codes")
    np.testing.assert_array_equal(scales.reshape(-1), rs)
    assert not pad.any()
    # shared experts: the concatenated down projection [d, ns cs]
    w3cat = torch.cat([w["w3s"][s].cpu() for s in range(cfg.n_shared)], dim=1)
    codes, scales, _ = _unpack(p["w3_shared"], 1, d, cfg.n_shared * cfg.c_shared)
    rc, rs = _oracle_rows(w3cat)
    _codes_equal(codes.reshape(-1, w3cat.shape[1]), rc, "w3_shared codes")
    np.testing.assert_array_equal(scales.reshape(-1), rs)


def _rand_topk(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.rand((T, E), generator=g).argsort(dim=1)[:, :k].to(torch.int32).contiguous()


@pytest.mark.parametrize("T,E,k,d", [(1, 8, 2, 128), (300, 8, 2, 256), (2049, 64, 6, 384), (1000, 256, 8, 7168),
                                     (257, 512, 16, 128)])     # the largest E and k the library takes
def test_dispatch_fp8_bit_exact(fs, T, E, k, d):
    cfg = small(T=T, E=E, k=k, d=d)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    u = synth.make_x(cfg, DEV)
    u[0, :] = 0.0
    idx = _rand_topk(T, E, k, T + E).to(DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    pos, perm = torch.empty(T * k, **i32), torch.empty(T * k, **i32)
    xq = fs.fp8_rows_empty(T * k, d, DEV)
    fs.fs_dispatch(desc, idx, u, counts, offsets, pos, perm, xq, ws)
    _no_dev_error()
    rc_, ro, rp, rperm = oracle.dispatch(T, k, E, idx.cpu().numpy())
    np.testing.assert_array_equal(counts.cpu().numpy(), rc_)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(pos.cpu().numpy(), rp)
    np.testing.assert_array_equal(perm.cpu().numpy(), rperm)
    codes, scales = fs.fp8_rows_split(xq, T * k, d)
    uc, ue, _ = oracle.quant_rows(synth.to_numpy(u), "bf16")
    _codes_equal(codes.cpu().numpy(), uc[rperm], "x_perm codes")
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.float64), np.exp2(ue[rperm].astype(np.float64)))


def _segments(counts):
    offs = np.zeros(len(counts) + 1, np.int32)
    offs[1:] = np.cumsum(counts)
    return offs


@pytest.mark.parametrize("counts,d,c", [
    ([130, 0, 1, 127, 128, 300, 5, 256], 256, 128),
    ([0, 0, 0, 1], 128, 128),
    ([700], 384, 384),                    # N = d = 384: a half tile at the end of the down GEMM's N
    ([64] * 40 + [129], 128, 256),
    ([600, 900], 1024, 512),              # 8 K-blocks of 128 on the gate/up GEMM
])
def test_grouped_swiglu_fp8(fs, counts, d, c):
    E = len(counts)
    rows = int(sum(counts))
    cfg = small(T=rows, E=E, k=1, d=d, c=c)
    g = torch.Generator(device=DEV).manual_seed(11)
    x = torch.randn((rows, d), generator=g, device=DEV).to(torch.bfloat16)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    xq = fs.fp8_rows_empty(rows, d, DEV)
    fs.fs_quantize_rows_fp8(rows, d, x, xq)
    offs = torch.from_numpy(_segments(counts)).to(DEV)
    y = torch.full((rows, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    fs.fs_grouped_swiglu(desc, xq, offs, packed["w13"], packed["w3"], y, ws)
    _no_dev_error()
    expert = np.repeat(np.arange(E, dtype=np.int32), counts)
    _, ry = oracle.expert_rows(oracle_cfg(cfg), synth.to_numpy(x), expert, synth.to_numpy(w["w1"]),
                               synth.to_numpy(w["w2"]), synth.to_numpy(w["w3"]))
    compare(to64(y), ry, "fp8", "y_perm")


@pytest.mark.parametrize("ns,cs,T", [(1, 128, 300), (2, 256, 129), (1, 512, 1000)])
def test_shared_expert_fp8(fs, ns, cs, T):
    cfg = small(T=T, n_shared=ns, c_shared=cs, d=256)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    u = synth.make_x(cfg, DEV)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    s = torch.full((T, cfg.d), float("nan"), dtype=torch.float32, device=DEV)
    fs.fs_shared_expert(desc, u, packed["w13_shared"], packed["w3_shared"], s, ws)
    _no_dev_error()
    # the oracle's shared path: one FP8 MLP over the concatenated width (block S at fp32)
    oc = oracle_cfg(cfg)
    bw = oracle.Weights(w_r=synth.to_numpy(w["w_r"]), w1=synth.to_numpy(w["w1"]), w2=synth.to_numpy(w["w2"]),
                        w3=synth.to_numpy(w["w3"]), w1s=synth.to_numpy(w["w1s"]), w2s=synth.to_numpy(w["w2s"]),
                        w3s=synth.to_numpy(w["w3s"]))
    ref = oracle.stack(oc, [bw], "partial", synth.to_numpy(u), want_rs=True)
    compare(to64(s), ref["S"][0], "fp8", "S")


def test_gather_is_unsupported_for_fp8(fs):
    cfg = small()
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    t = torch.empty(64, dtype=torch.int32, device=DEV)
    n0 = fs.fs_launch_count()
    with pytest.raises(fs.FsError) as e:
        fs.fs_grouped_swiglu_gather(desc, t, t, t, t, t, t, ws)
    assert e.value.status == 2 and fs.fs_launch_count() == n0


# ------------------------------------------------------------ FP8 stacks

from test_gpu_stack import _check_stack, parity_rows   # noqa: E402


@pytest.mark.parametrize("wiring,L", [("partial", 3), ("outdated", 3), ("disabled", 2)])
def test_small_stack_fp8(fs, wiring, L):
    cfg = small(T=333, L=L, n_shared=2, c_shared=128)
    _check_stack(cfg, synth.make_problem(cfg, DEV), wiring)


@pytest.mark.parametrize("gate,E,k,ns", [("sigmoid_norm", 32, 8, 1), ("softmax", 16, 4, 0), ("sigmoid", 4, 1, 1)])
def test_small_stack_fp8_gates(fs, gate, E, k, ns):
    cfg = small(T=520, E=E, k=k, gate=gate, n_shared=ns, c_shared=128 if ns else 0, L=2, d=384, c=128)
    _check_stack(cfg, synth.make_problem(cfg, DEV), "partial")


@pytest.mark.parametrize("wiring,L", [("partial", 3), ("outdated", 2)])
def test_overlap_stack_fp8_matches_sequential(fs, wiring, L):
    cfg = small(T=700, E=16, k=4, gate="sigmoid_norm", L=L)
    prob = synth.make_problem(cfg, DEV)
    stack = fs.FarSkipStack(cfg, prob["blocks"], wiring=wiring)
    o, o_star = stack.forward(prob["x"])
    o, o_star = o.clone(), o_star.clone()
    o2, o2_star = stack.forward_overlap(prob["x"])
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    assert torch.equal(o2, o) and torch.equal(o2_star, o_star)


FULL_FP8 = ["v2lite_fp8", "qwen3_fp8", "scout_fp8", "v3_fp8", "v3_decode_fp8"]
# tokens the oracle's FP8 form follows (None = every token); at least 1,000, so
# the < 0.1% rules resolve single tokens
ROWS_FP8 = {"v2lite_fp8": 1024, "qwen3_fp8": 2048, "scout_fp8": 1024, "v3_fp8": 1024, "v3_decode_fp8": None}


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL_FP8)
def test_full_size_fp8_sampled(fs, name):
    """Full-size FP8 workloads in the benchmark's launch configuration; the
    oracle's FP8 form follows a seeded sample of tokens (every token of the V3
    decode batch), blockwise and end to end."""
    cfg = configs.CONFIGS[name]
    prob = synth.make_problem(cfg, DEV)
    _check_stack(cfg, prob, cfg.wiring, parity_rows(cfg, ROWS_FP8[name]))


def test_dispatch_noalloc_fp8_matches_dispatch(fs):
    """The no-allocation Dispatch with FS_FP8 writes the same codes, scales and
    permutation as fs_dispatch with a workspace."""
    T, E, k, d = 2049, 64, 6, 384
    cfg = small(T=T, E=E, k=k, d=d)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    u = synth.make_x(cfg, DEV)
    idx = _rand_topk(T, E, k, 77).to(DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    outs = []
    for noalloc in (False, True):
        c, o = torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32)
        p, pm = torch.full((T * k,), -7, **i32), torch.full((T * k,), -7, **i32)
        xq = fs.fp8_rows_empty(T * k, d, DEV)
        xq.fill_(0xAB)
        if noalloc:
            fs.fs_dispatch_noalloc(desc, idx, u, c, o, p, pm, xq)
        else:
            fs.fs_dispatch(desc, idx, u, c, o, p, pm, xq, ws)
        outs.append((c, o, p, pm, xq))
    _no_dev_error()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
