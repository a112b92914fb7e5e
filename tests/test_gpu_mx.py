"""GPU parity of the block-scaled FP8 expert path (FS_MXFP8) against the oracle's
MX form (one power-of-two scale per 32 elements along the contraction).

Integer and byte results are compared bit for bit: the E4M3 codes and UE8M0
block scales of fs_quantize_rows_mx, of the MX weight packs and of the MX
Dispatch copy, and Dispatch's counts, 128-row-padded offsets, positions and
permutation.  Floating-point results (the expert outputs, the shared expert,
the stack) meet the bf16 bounds, with the one-flip allowance of the stacks.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_expert_gb300 import configs, fs, synth
from parity import compare, oracle_cfg, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
MX = 32


def _no_dev_error():
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    assert st == 0, "device error word = %d" % code


def small(**kw):
    base = dict(name="mx", T=300, d=256, E=8, k=2, c=256, n_shared=1, c_shared=128, L=1,
                gate="softmax_renorm", dtype="mxfp8")
    base.update(kw)
    return configs.LayerConfig(**base)


def _codes_equal(got, want, what):
    g = got.astype(np.uint8)
    w = want.astype(np.uint8)
    zero = ((g & 0x7F) == 0) & ((w & 0x7F) == 0)
    bad = (g != w) & ~zero
    assert not bad.any(), "%s: %d codes differ, first at %s (got %#x want %#x)" % (
        what, int(bad.sum()), np.argwhere(bad)[0], g[bad][0], w[bad][0])


def _chunk_index(r, b):
    """Byte of row r's scale of block b inside its 512-byte chunk."""
    return (r % 32) * 16 + ((r % 128) // 32) * 4 + (b % 4)


def _mx_matrix(buf, rows, cols):
    """Codes [rows128, cols] and block exponents [rows128, cols / 32] of an MX matrix."""
    codes, sf = fs.mx_rows_split(buf, rows, cols)
    codes = codes.cpu().numpy()
    sf = sf.cpu().numpy()
    r128 = codes.shape[0]
    r = np.arange(r128)[:, None]
    b = np.arange(cols // MX)[None, :]
    exps = sf[r // 128, b // 4, _chunk_index(r, b)].astype(np.int64) - 127
    return codes, exps


def _mx_weights(buf, G, N, K):
    """Codes [G, NB 256, K] and block exponents [G, NB 256, K / 32] of an MX weight pack."""
    NB, KB = (N + 255) // 256, K // 128
    nc = G * NB * KB * 32768
    host = buf.cpu().numpy()
    codes = host[:nc].reshape(G, NB, KB, 256, 128).transpose(0, 1, 3, 2, 4).reshape(G, NB * 256, K)
    sf = host[nc:nc + G * NB * KB * 1024].reshape(G, NB, KB, 1024)
    rr = np.arange(NB * 256)[:, None]
    b = np.arange(K // MX)[None, :]
    byte = (rr % 256 // 128) * 512 + _chunk_index(rr % 256, b)
    exps = sf[:, rr // 256, b // 4, byte].astype(np.int64) - 127
    return codes, exps


def _oracle_blocks(x_bf16):
    codes, exps, _ = oracle.quant_blocks(synth.to_numpy(x_bf16.reshape(-1, x_bf16.shape[-1])), MX, "bf16")
    return codes, exps


def _bf16_rows(rows, cols, seed):
    """bf16 rows whose 32-element blocks have assorted magnitudes (2^-20 .. 2^11),
    zero blocks and a block whose largest element is exactly 448 2^-3."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, cols), generator=g)
    mag = torch.exp2(torch.randint(-20, 12, (rows, cols // MX), generator=g).float()).repeat_interleave(MX, dim=1)
    x = x * mag
    if rows > 3:
        x[1, :MX] = 0.0
        x[2, MX:2 * MX] = x[2, MX:2 * MX].clamp(-448.0 * 2.0 ** -3, 448.0 * 2.0 ** -3)
        x[2, MX + 5] = 448.0 * 2.0 ** -3
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 256), (1000, 384), (4099, 2048)])
def test_quantize_rows_mx_bit_exact(fs, rows, cols):
    x = _bf16_rows(rows, cols, rows + cols)
    q = fs.mx_rows_empty(rows, cols, DEV)
    q.fill_(0xAB)
    fs.fs_quantize_rows_mx(rows, cols, x.to(DEV), q)
    _no_dev_error()
    codes, exps = _mx_matrix(q, rows, cols)
    rc, re = _oracle_blocks(x)
    _codes_equal(codes[:rows], rc, "codes")
    np.testing.assert_array_equal(exps[:rows], re)
    # rows up to the next multiple of 128: zero codes, unit scales
    assert not codes[rows:].any() and not exps[rows:].any()


@pytest.mark.parametrize("E,c,d", [(3, 128, 256), (2, 384, 384), (5, 256, 128)])
def test_pack_mx_bit_exact(fs, E, c, d):
    cfg = small(E=E, c=c, d=d, n_shared=2, c_shared=128)
    w = synth.make_block_weights(cfg, 0, DEV)
    p = fs.pack_block(cfg, w)
    _no_dev_error()
    n = np.arange(2 * c)
    blk, within = n // 128, n % 128
    src = 64 * blk + np.where(within < 64, within, within - 64)
    w1, w2 = w["w1"].cpu(), w["w2"].cpu()
    ref13 = torch.where(torch.from_numpy(within < 64)[None, :, None], w2[:, src], w1[:, src])
    for name, ref, N, K, G in (("w13", ref13, 2 * c, d, E), ("w3", w["w3"].cpu(), d, c, E),
                               ("w3_shared", torch.cat([w["w3s"][s].cpu() for s in range(cfg.n_shared)], 1)[None],
                                d, cfg.n_shared * cfg.c_shared, 1)):
        codes, exps = _mx_weights(p[name], G, N, K)
        rc, re = _oracle_blocks(ref)
        _codes_equal(codes[:, :N].reshape(-1, K), rc, name + " codes")
        np.testing.assert_array_equal(exps[:, :N].reshape(-1, K // MX), re)
        assert not codes[:, N:].any() and not exps[:, N:].any()


def _rand_topk(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.rand((T, E), generator=g).argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def _padded(counts):
    seg = (np.asarray(counts) + 127) // 128 * 128
    offs = np.zeros(len(counts) + 1, np.int64)
    offs[1:] = np.cumsum(seg)
    return offs


@pytest.mark.parametrize("T,E,k,d", [(1, 8, 2, 128), (300, 8, 2, 256), (2049, 64, 6, 384), (1000, 256, 8, 7168),
                                     (257, 512, 16, 128)])     # the largest E and k the library takes
def test_dispatch_mx_bit_exact(fs, T, E, k, d):
    """Counts as the counting sort gives them; offsets the exclusive prefix of the
    counts rounded up to 128; each (token, slot) at its padded segment start plus
    its stable rank; the rows' codes and block scales those of the token."""
    cfg = small(T=T, E=E, k=k, d=d)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    u = synth.make_x(cfg, DEV)
    u[0, :MX] = 0.0
    idx = _rand_topk(T, E, k, T + E).to(DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    prow = fs.fs_dispatch_rows(desc)
    assert prow == (T * k + 127 * E + 127) // 128 * 128
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    pos, perm = torch.empty(T * k, **i32), torch.full((prow,), -7, **i32)
    xq = fs.mx_rows_empty(prow, d, DEV)
    fs.fs_dispatch(desc, idx, u, counts, offsets, pos, perm, xq, ws)
    _no_dev_error()
    rc_, ro, rp, rperm = oracle.dispatch(T, k, E, idx.cpu().numpy())
    np.testing.assert_array_equal(counts.cpu().numpy(), rc_)
    po = _padded(rc_)
    np.testing.assert_array_equal(offsets.cpu().numpy(), po)
    # the oracle's unpadded position p of expert e moves to po[e] + (p - ro[e])
    e_of = idx.cpu().numpy().reshape(-1)
    want_pos = po[e_of] + (rp - ro[e_of])
    np.testing.assert_array_equal(pos.cpu().numpy(), want_pos)
    got_perm = perm.cpu().numpy()
    np.testing.assert_array_equal(got_perm[want_pos], rperm[rp])
    codes, exps = _mx_matrix(xq, prow, d)
    uc, ue = _oracle_blocks(u.cpu())
    tok = np.arange(T).repeat(k)
    _codes_equal(codes[want_pos], uc[tok], "x_perm codes")
    np.testing.assert_array_equal(exps[want_pos], ue[tok])


@pytest.mark.parametrize("counts,d,c", [
    ([130, 0, 1, 127, 128, 300, 5, 256], 256, 128),
    ([0, 0, 0, 1], 128, 128),
    ([700], 384, 384),                    # N = d = 384: a half tile at the end of the down GEMM's N
    ([64] * 40 + [129], 128, 256),
    ([600, 900], 1024, 512),              # 8 K-blocks of 128 on the gate/up GEMM
])
def test_grouped_swiglu_mx(fs, counts, d, c):
    """The routed experts on 128-row-aligned segments (the MX Dispatch layout):
    every valid row's output against the oracle's MX expert."""
    E = len(counts)
    rows = int(sum(counts))
    cfg = small(T=rows, E=E, k=1, d=d, c=c)
    desc = fs.make_desc(cfg)
    prow = fs.fs_dispatch_rows(desc)
    po = _padded(counts)
    assert po[-1] <= prow
    g = torch.Generator(device=DEV).manual_seed(11)
    x = torch.randn((rows, d), generator=g, device=DEV).to(torch.bfloat16)
    where = np.concatenate([po[e] + np.arange(n) for e, n in enumerate(counts)]).astype(np.int64)
    xp = torch.zeros((prow, d), dtype=torch.bfloat16, device=DEV)
    xp[torch.from_numpy(where).to(DEV)] = x
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    ws = fs.alloc_workspace(desc, 0)
    xq = fs.mx_rows_empty(prow, d, DEV)
    fs.fs_quantize_rows_mx(prow, d, xp, xq)
    offs = torch.from_numpy(po.astype(np.int32)).to(DEV)
    y = torch.full((prow, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    fs.fs_grouped_swiglu(desc, xq, offs, packed["w13"], packed["w3"], y, ws)
    _no_dev_error()
    expert = np.repeat(np.arange(E, dtype=np.int32), counts)
    _, ry = oracle.expert_rows(oracle_cfg(cfg), synth.to_numpy(x), expert, synth.to_numpy(w["w1"]),
                               synth.to_numpy(w["w2"]), synth.to_numpy(w["w3"]))
    compare(to64(y[torch.from_numpy(where).to(DEV)]), ry, "mxfp8", "y_perm")


@pytest.mark.parametrize("ns,cs,T", [(1, 128, 300), (2, 256, 129), (1, 512, 1000)])
def test_shared_expert_mx(fs, ns, cs, T):
    cfg = small(T=T, n_shared=ns, c_shared=cs, d=256)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    u = synth.make_x(cfg, DEV)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    s = torch.full((T, cfg.d), float("nan"), dtype=torch.float32, device=DEV)
    fs.fs_shared_expert(desc, u, packed["w13_shared"], packed["w3_shared"], s, ws)
    _no_dev_error()
    bw = oracle.Weights(w_r=synth.to_numpy(w["w_r"]), w1=synth.to_numpy(w["w1"]), w2=synth.to_numpy(w["w2"]),
                        w3=synth.to_numpy(w["w3"]), w1s=synth.to_numpy(w["w1s"]), w2s=synth.to_numpy(w["w2s"]),
                        w3s=synth.to_numpy(w["w3s"]))
    ref = oracle.stack(oracle_cfg(cfg), [bw], "partial", synth.to_numpy(u), want_rs=True)
    compare(to64(s), ref["S"][0], "mxfp8", "S")


# ------------------------------------------------------------ MX stacks

from test_gpu_stack import _check_stack, parity_rows   # noqa: E402


@pytest.mark.parametrize("wiring,L", [("partial", 3), ("outdated", 3), ("disabled", 3)])
def test_small_stack_mx(fs, wiring, L):
    cfg = small(T=333, L=L, n_shared=2, c_shared=128)
    _check_stack(cfg, synth.make_problem(cfg, DEV), wiring)


@pytest.mark.parametrize("gate,E,k,ns", [("sigmoid_norm", 32, 8, 1), ("softmax", 16, 4, 0), ("sigmoid", 4, 1, 1)])
def test_small_stack_mx_gates(fs, gate, E, k, ns):
    cfg = small(T=520, E=E, k=k, gate=gate, n_shared=ns, c_shared=128 if ns else 0, L=2, d=384, c=128)
    _check_stack(cfg, synth.make_problem(cfg, DEV), "partial")


@pytest.mark.parametrize("wiring,L,ns", [("partial", 3, 1), ("outdated", 2, 1), ("partial", 2, 0)])
def test_overlap_stack_mx_matches_sequential(fs, wiring, L, ns):
    """The two-stream schedule on the MX path (stream2's Dispatch also quantising
    u_k for the shared experts; padded expert segments in both slots) against
    the one-stream stack, which the tests above check against the oracle."""
    cfg = small(T=700, E=16, k=4, gate="sigmoid_norm", L=L, n_shared=ns, c_shared=128 if ns else 0)
    prob = synth.make_problem(cfg, DEV)
    stack = fs.FarSkipStack(cfg, prob["blocks"], wiring=wiring)
    o, o_star = stack.forward(prob["x"])
    o, o_star = o.clone(), o_star.clone()
    o2, o2_star = stack.forward_overlap(prob["x"])
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    assert torch.equal(o2, o) and torch.equal(o2_star, o_star)


# V2-Lite: L = 4, c = 1408 (11 stages of 128 along the down projection's
# contraction; weight rows of 176 16-byte vectors, not a multiple of 32)
ROWS_MX = {"v3_mxfp8": 1024, "v3_decode_mxfp8": None, "qwen3_mxfp8": 2048, "v2lite_mxfp8": 1024}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(ROWS_MX))
def test_full_size_mx_sampled(fs, name):
    """Full-size MX workloads in the benchmark's launch configuration; the oracle's
    MX form follows a seeded sample of tokens (every token of the V3 decode batch)."""
    cfg = configs.CONFIGS[name]
    prob = synth.make_problem(cfg, DEV)
    _check_stack(cfg, prob, cfg.wiring, parity_rows(cfg, ROWS_MX[name]))
