"""GPU parity of each C-ABI entry point against the CPU oracle, at sizes the
oracle finishes in seconds that still span several tiles and ragged tails,
plus edge cases (empty experts, one token, k = E, E = 512, k = 16)."""
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_expert_gb300 import configs, fs, synth
from parity import compare, oracle_cfg, oracle_weights, to64, topk_mismatch

pytestmark = pytest.mark.gpu

DEV = "cuda"


def small(dtype="bf16", **kw):
    base = dict(name="small", T=300, d=256, E=8, k=2, c=128, n_shared=1, c_shared=128, L=1,
                gate="softmax_renorm", dtype=dtype)
    base.update(kw)
    return configs.LayerConfig(**base)


def _no_dev_error():
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    assert st == 0, "device error word = %d" % code


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("dtype,E,k,gate,T,d", [
    ("f32", 8, 2, "softmax_renorm", 256, 128),
    ("bf16", 8, 2, "softmax_renorm", 300, 256),
    ("bf16", 64, 6, "softmax", 1000, 512),
    ("bf16", 128, 8, "softmax_renorm", 777, 256),
    ("bf16", 16, 1, "sigmoid", 513, 320),
    ("bf16", 256, 8, "sigmoid_norm", 1200, 448),
    ("bf16", 512, 16, "sigmoid_norm", 130, 256),
    ("bf16", 4, 4, "softmax", 70, 64),
])
def test_router_topk(fs, dtype, E, k, gate, T, d):
    cfg = small(dtype, E=E, k=k, gate=gate, T=T, d=d, zipf_s=1.2 if E == 128 else None)
    x = synth.make_x(cfg, DEV)
    w = synth.make_block_weights(cfg, 0, DEV)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    fs.fs_router_topk(desc, x, w["w_r"], w["bias"], idx, tw, logits, ws)
    _no_dev_error()
    oc = oracle_cfg(cfg)
    bias = synth.to_numpy(w["bias"])
    z, ridx, rw = oracle.router(oc, synth.to_numpy(x), synth.to_numpy(w["w_r"]), bias)
    zg = to64(logits)
    zref = z - (bias.astype(np.float64)[None, :] if bias is not None else 0.0)
    rel = np.linalg.norm(zg - zref) / np.linalg.norm(zref)
    assert rel < (1e-6 if dtype == "f32" else 2e-6), rel
    bad = topk_mismatch(idx.cpu().numpy(), ridx, zref, k, bias)
    ok = ~bad
    # gate weights on the tokens whose sets agree (slot order agrees too away from ties)
    gi = idx.cpu().numpy()[ok]
    order_ok = np.all(gi == ridx[ok], axis=1)
    np.testing.assert_allclose(tw.cpu().numpy()[ok][order_ok], rw[ok][order_ok], rtol=2e-5, atol=1e-6)


# ---------------------------------------------------------------- dispatch

def _rand_topk(T, E, k, seed, skew=False):
    g = torch.Generator().manual_seed(seed)
    if skew:   # experts 0..k-1 for most tokens: many empty experts
        idx = torch.arange(k, dtype=torch.int32).repeat(T, 1)
        some = torch.randperm(T, generator=g)[: T // 10]
        for t in some.tolist():
            idx[t] = torch.randperm(E, generator=g)[:k].to(torch.int32)
        return idx
    keys = torch.rand((T, E), generator=g)
    return keys.argsort(dim=1)[:, :k].to(torch.int32).contiguous()


@pytest.mark.parametrize("T,E,k,d,dtype,skew", [
    (1, 8, 2, 64, "bf16", False),
    (300, 8, 2, 256, "bf16", False),
    (1500, 64, 6, 128, "bf16", False),
    (2049, 256, 8, 192, "bf16", True),
    (4100, 512, 16, 64, "bf16", False),
    (257, 8, 8, 128, "f32", False),
    (1024, 16, 1, 64, "f32", True),
])
def test_dispatch_bit_exact(fs, T, E, k, d, dtype, skew):
    cfg = small(dtype, T=T, E=E, k=k, d=d)
    idx = _rand_topk(T, E, k, seed=T + E, skew=skew)
    u = synth.make_x(cfg, DEV)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    pos = torch.empty(T * k, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    x_perm = torch.empty((T * k, d), dtype=u.dtype, device=DEV)
    fs.fs_dispatch(desc, idx.to(DEV), u, counts, offsets, pos, perm, x_perm, ws)
    _no_dev_error()
    rc, ro, rp, rperm = oracle.dispatch(T, k, E, idx.numpy())
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(pos.cpu().numpy(), rp)
    np.testing.assert_array_equal(perm.cpu().numpy(), rperm)
    # rows are byte copies
    xp = x_perm.cpu()
    assert torch.equal(xp, u.cpu()[torch.from_numpy(rperm).long()])


def test_dispatch_bad_index_sets_error(fs):
    cfg = small(T=64, E=8, k=2, d=64)
    idx = _rand_topk(64, 8, 2, seed=1)
    idx[5, 1] = 8          # out of range
    u = synth.make_x(cfg, DEV)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    z = lambda n: torch.empty(n, dtype=torch.int32, device=DEV)
    x_perm = torch.zeros((128, 64), dtype=u.dtype, device=DEV)
    fs.fs_dispatch(desc, idx.to(DEV), u, z(8), z(9), z(128), z(128), x_perm, ws)
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    assert st == 5 and code == 1
    assert fs.fs_get_error() == (0, 0)   # read clears it


def test_bounded_wait_times_out_and_the_context_survives(fs):
    """A pipeline wait on a barrier nothing signals gives up after its limit,
    records the timeout in the device error word and returns; the GPU keeps
    working (a Dispatch afterwards is correct)."""
    import time
    t0 = time.perf_counter()
    fs.fs_selftest_wait_timeout(50_000)             # 50 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert fs.fs_get_error() == (5, 3)
    assert 0.04 < elapsed < 5.0, elapsed
    assert fs.fs_get_error() == (0, 0)
    T, E, k = 300, 8, 2
    idx = _rand_topk(T, E, k, seed=3)
    counts, offs, pos, perm = oracle.dispatch(T, k, E, idx.numpy())
    cfg = small(T=T, E=E, k=k, d=64)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    z = lambda n: torch.empty(n, dtype=torch.int32, device=DEV)
    got = [z(E), z(E + 1), z(T * k), z(T * k)]
    u = synth.make_x(cfg, DEV)
    fs.fs_dispatch(desc, idx.to(DEV), u, *got, None, ws)
    _no_dev_error()
    for a, b in zip(got, (counts, offs, pos, perm)):
        np.testing.assert_array_equal(a.cpu().numpy(), b)


# ----------------------------------------------------------- grouped SwiGLU

def _segments(counts):
    offs = np.zeros(len(counts) + 1, np.int32)
    offs[1:] = np.cumsum(counts)
    return offs


@pytest.mark.parametrize("dtype,counts,d,c", [
    ("bf16", [130, 0, 1, 127, 128, 300, 5, 256], 256, 128),
    ("bf16", [0, 0, 0, 1], 128, 64),
    ("bf16", [700], 192, 192),            # 2c = 384: a half tile at the end of N
    ("bf16", [64] * 40 + [129], 128, 256),
    ("f32", [130, 0, 1, 63, 64, 65, 200, 7], 128, 128),
])
def test_grouped_swiglu(fs, dtype, counts, d, c):
    E = len(counts)
    rows = int(sum(counts))
    cfg = small(dtype, T=rows, E=E, k=1, d=d, c=c)
    g = torch.Generator(device=DEV).manual_seed(7)
    sdt = synth.storage_dtype(cfg)
    x = torch.randn((rows, d), generator=g, device=DEV).to(sdt)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    offs = torch.from_numpy(_segments(counts)).to(DEV)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    y = torch.full((rows, d), float("nan"), dtype=sdt, device=DEV)
    fs.fs_grouped_swiglu(desc, x, offs, packed["w13"], packed["w3"], y, ws)
    _no_dev_error()
    expert = np.repeat(np.arange(E, dtype=np.int32), counts)
    _, ry = oracle.expert_rows(oracle_cfg(cfg), synth.to_numpy(x), expert, synth.to_numpy(w["w1"]),
                               synth.to_numpy(w["w2"]), synth.to_numpy(w["w3"]))
    compare(to64(y), ry, dtype, "y_perm")


def test_grouped_swiglu_bad_offsets_sets_error(fs):
    """Offsets that decrease (made on the host; nothing faults): the plan records
    DEV_ERR_OFFSETS (code 2) and yields no tiles, so y_perm is left untouched; a
    consistent call afterwards matches the oracle."""
    counts = [100, 50, 50]
    cfg = small("bf16", T=200, E=3, k=1, d=128, c=128)
    g = torch.Generator(device=DEV).manual_seed(8)
    x = torch.randn((200, 128), generator=g, device=DEV).to(torch.bfloat16)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    y = torch.full((200, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    bad = torch.tensor([0, 100, 50, 200], dtype=torch.int32, device=DEV)
    fs.fs_grouped_swiglu(desc, x, bad, packed["w13"], packed["w3"], y, ws)
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (5, 2)
    assert torch.isnan(y.float()).all(), "rows written from an inconsistent plan"
    offs = torch.from_numpy(_segments(counts)).to(DEV)
    fs.fs_grouped_swiglu(desc, x, offs, packed["w13"], packed["w3"], y, ws)
    _no_dev_error()
    expert = np.repeat(np.arange(3, dtype=np.int32), counts)
    _, ry = oracle.expert_rows(oracle_cfg(cfg), synth.to_numpy(x), expert, synth.to_numpy(w["w1"]),
                               synth.to_numpy(w["w2"]), synth.to_numpy(w["w3"]))
    compare(to64(y), ry, "bf16", "y_perm")


@pytest.mark.parametrize("dtype,T,E,k,d,c,skew", [
    ("bf16", 300, 8, 2, 256, 128, False), ("bf16", 1000, 64, 6, 128, 192, True), ("bf16", 1, 8, 2, 64, 64, False),
    ("bf16", 4097, 16, 4, 192, 128, False), ("f32", 257, 8, 2, 128, 128, False),
])
def test_grouped_swiglu_gather(fs, dtype, T, E, k, d, c, skew):
    """Routed experts reading their rows straight from u through the Dispatch
    permutation: equal to the oracle on u[perm_src], and bit-identical to the
    copy-then-GEMM path."""
    cfg = small(dtype, T=T, E=E, k=k, d=d, c=c)
    idx = _rand_topk(T, E, k, seed=T + 7, skew=skew)
    counts, offs, pos, perm = oracle.dispatch(T, k, E, idx.numpy())
    u = synth.make_x(cfg, DEV)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    y = torch.full((T * k, d), float("nan"), dtype=u.dtype, device=DEV)
    perm_t = torch.from_numpy(perm).to(DEV)
    offs_t = torch.from_numpy(offs).to(DEV)
    if os.environ.get("FS_TC_VARIANT") == "pair" and dtype != "f32":
        # the CTA-pair GEMM has no gathered-row loads: the call says so and launches nothing
        with pytest.raises(fs.FsError) as err:
            fs.fs_grouped_swiglu_gather(desc, u, perm_t, offs_t, packed["w13"], packed["w3"], y, ws)
        assert fs.STATUS[err.value.status] == "FS_ERR_UNSUPPORTED"
        _no_dev_error()
        pytest.skip("gathered loads are not available with the CTA-pair GEMM variant")
    fs.fs_grouped_swiglu_gather(desc, u, perm_t, offs_t, packed["w13"], packed["w3"], y, ws)
    _no_dev_error()
    x_perm = u[perm_t.long()].contiguous()
    y2 = torch.empty_like(y)
    fs.fs_grouped_swiglu(desc, x_perm, offs_t, packed["w13"], packed["w3"], y2, ws)
    _no_dev_error()
    assert torch.equal(y, y2)
    expert = np.repeat(np.arange(E, dtype=np.int32), counts)
    _, ry = oracle.expert_rows(oracle_cfg(cfg), synth.to_numpy(u)[perm], expert, synth.to_numpy(w["w1"]),
                               synth.to_numpy(w["w2"]), synth.to_numpy(w["w3"]))
    compare(to64(y), ry, dtype, "y_perm (gathered)")


@pytest.mark.parametrize("dtype,ns,cs,T", [("bf16", 1, 128, 300), ("bf16", 2, 192, 129), ("f32", 1, 256, 100)])
def test_shared_expert(fs, dtype, ns, cs, T):
    cfg = small(dtype, T=T, n_shared=ns, c_shared=cs, d=256)
    x = synth.make_x(cfg, DEV)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    s = torch.empty((T, cfg.d), dtype=torch.float32, device=DEV)
    fs.fs_shared_expert(desc, x, packed["w13_shared"], packed["w3_shared"], s, ws)
    _no_dev_error()
    out = oracle.stack(oracle_cfg(cfg), oracle_weights([w]), "partial", synth.to_numpy(x), want_rs=True)
    compare(to64(s), out["S"][0], dtype, "shared")


@pytest.mark.parametrize("dtype,T,k,d,ns,cs,resid,partial", [
    ("bf16", 300, 2, 256, 1, 128, "act", True),
    ("bf16", 1000, 8, 320, 2, 128, "f32", True),       # ragged M tile, half N tile (d = 320)
    ("bf16", 77, 6, 512, 1, 192, "f32_in", False),
    ("bf16", 1, 1, 64, 1, 64, "act", True),
    ("fp8", 700, 8, 384, 1, 256, "act", True),
    ("fp8", 333, 4, 256, 2, 128, "f32", False),
])
def test_shared_expert_combine_matches_unfused(fs, dtype, T, k, d, ns, cs, resid, partial):
    """fs_shared_expert_combine (Combine in the shared down projection's epilogue)
    gives the same bits as fs_shared_expert followed by fs_combine, for every
    wiring's next input and residual precision."""
    E = max(k, 8)
    cfg = small(dtype, T=T, E=E, k=k, d=d, n_shared=ns, c_shared=cs)
    x = synth.make_x(cfg, DEV)
    w = synth.make_block_weights(cfg, 0, DEV)
    packed = fs.pack_block(cfg, w)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    g = torch.Generator(device=DEV).manual_seed(12)
    idx = _rand_topk(T, E, k, seed=6)
    _, _, pos, _ = oracle.dispatch(T, k, E, idx.numpy())
    pos = torch.from_numpy(pos).to(DEV)
    y = torch.randn((T * k, d), generator=g, device=DEV).to(torch.bfloat16)
    tw = torch.rand((T, k), generator=g, device=DEV)
    pdt = torch.bfloat16 if resid == "act" else torch.float32
    odt = torch.float32 if resid == "f32" else torch.bfloat16
    op = torch.randn((T, d), generator=g, device=DEV).to(pdt)
    s = torch.empty((T, d), dtype=torch.float32, device=DEV)
    fs.fs_shared_expert(desc, x, packed["w13_shared"], packed["w3_shared"], s, ws)
    for wi in ("partial", "outdated", "disabled"):
        outs = []
        for fused in (False, True):
            o_star = torch.full((T, d), 7.0, dtype=odt, device=DEV) if partial else None
            o = torch.full((T, d), 7.0, dtype=odt, device=DEV)
            un = torch.full((T, d), 7.0, dtype=torch.bfloat16, device=DEV)
            if fused:
                fs.fs_shared_expert_combine(desc, x, packed["w13_shared"], packed["w3_shared"], y, pos, tw, op,
                                            o_star, o, un, wi, ws)
            else:
                fs.fs_combine(desc, y, pos, tw, op, s, o_star, o, un, wi)
            outs.append((o_star, o, un))
        _no_dev_error()
        for name, a, b in zip(("o*", "o", "u_next"), *outs):
            if a is not None:
                assert torch.equal(a, b), "%s: %s differs from the unfused path" % (wi, name)


# ----------------------------------------------------------------- combine

@pytest.mark.parametrize("dtype,T,k,d,shared,partial,resid", [
    ("bf16", 300, 2, 256, True, True, "act"), ("bf16", 77, 8, 512, False, True, "act"),
    ("bf16", 1, 1, 64, True, False, "act"), ("f32", 256, 2, 128, True, True, "act"),
    ("bf16", 1000, 16, 128, True, True, "act"), ("bf16", 300, 8, 256, True, True, "f32"),
    ("bf16", 200, 4, 192, True, True, "f32_in"),
])
def test_combine(fs, dtype, T, k, d, shared, partial, resid):
    """resid: 'act' = residual in the activation type; 'f32' = fp32 in and out;
    'f32_in' = fp32 in, activation type out (the last block of a stack)."""
    E = max(k, 8)
    cfg = small(dtype, T=T, E=E, k=k, d=d)
    sdt = synth.storage_dtype(cfg)
    g = torch.Generator(device=DEV).manual_seed(11)
    idx = _rand_topk(T, E, k, seed=5)
    _, _, pos, _ = oracle.dispatch(T, k, E, idx.numpy())
    y = torch.randn((T * k, d), generator=g, device=DEV).to(sdt)
    w = torch.rand((T, k), generator=g, device=DEV)
    pdt = sdt if resid == "act" else torch.float32
    odt = torch.float32 if resid == "f32" else sdt
    op = torch.randn((T, d), generator=g, device=DEV).to(pdt)
    s = torch.randn((T, d), generator=g, device=DEV) if shared else None     # fp32
    o_star = torch.empty((T, d), dtype=odt, device=DEV) if partial else None
    o = torch.empty((T, d), dtype=odt, device=DEV)
    u_next = {wi: torch.empty((T, d), dtype=sdt, device=DEV) for wi in ("partial", "outdated", "disabled")}
    for wi, un in u_next.items():
        fs.fs_combine(fs.make_desc(cfg), y, torch.from_numpy(pos).to(DEV), w, op, s, o_star, o, un, wi)
    _no_dev_error()
    ost = oracle.STORE_BF16 if odt == torch.bfloat16 else oracle.STORE_F32
    # the oracle combine takes one element type: widen everything to fp64 (exact)
    f64 = lambda t: None if t is None else t.double().cpu().numpy()
    y_in, sn, opn = f64(y), f64(s), f64(op)
    r_star, r = oracle.combine(T, k, d, y_in, pos, w.cpu().numpy(), opn, sn, storage=ost)
    # fp32 sums vs fp64 sums, each rounded once: equal but for 1-ulp rounding flips
    # plus the fp32 accumulation error, bounded by a few fp32 ulps of the term magnitudes
    ulp = 2.0 ** -7 if odt == torch.bfloat16 else 2.0 ** -23
    yv = np.abs(to64(y))[pos.reshape(T, k)]                      # [T, k, d]
    mag = np.abs(to64(op)) + (np.abs(to64(s)) if shared else 0.0) + np.einsum("tk,tkd->td", w.cpu().numpy(), yv)
    diff = np.abs(to64(o) - r)
    assert np.all(diff <= ulp * np.abs(r) + k * 2.0 ** -22 * mag + 1e-30), diff.max()
    if partial:
        d_star = np.abs(to64(o_star) - r_star)
        assert np.all(d_star <= ulp * np.abs(r_star) + 2.0 ** -23 * mag + 1e-30), d_star.max()
    # next-block inputs: the chosen residual rounded to the activation type
    act = oracle.STORE_BF16 if dtype == "bf16" else oracle.STORE_F32
    r_star_u, r_u = oracle.combine(T, k, d, y_in, pos, w.cpu().numpy(), opn, sn, storage=act)
    ulp_u = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -23
    for wi, want in (("partial", r_star_u), ("disabled", r_u)):
        du = np.abs(to64(u_next[wi]) - want)
        assert np.all(du <= ulp_u * np.abs(want) + k * 2.0 ** -22 * mag + 1e-30), (wi, du.max())
    assert torch.equal(u_next["outdated"], op.to(sdt))
