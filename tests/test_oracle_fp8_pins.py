"""Pins for the oracle's FP8 expert path (the pages' inference setting: FP8
quantisation with fused MoE forward kernels, "FarSkip-Collective" summary,
experimental setup, software configuration; the format and the scaling are a
reading of this build, stated in oracle.c).

What fixes each function, and the mistake each pin catches:
  E4M3 values       -- every finite code of the library's float8_e4m3fn type is a
                       fixed point with the same code (wrong exponent bias,
                       missing subnormals, wrong code packing)
  E4M3 rounding     -- random values and every midpoint between neighbouring
                       codes agree with the library conversion (ties to even,
                       not away); beyond 448 the reading saturates
  row scales        -- brute-force search for the smallest power-of-two scale
                       that fits the row into +-448 (off-by-one exponent,
                       boundary rows with max exactly 448 2^j)
  gate/up reduction -- with FP8-representable operands the FP8 hidden equals
                       the exact one (a scale applied to the wrong operand, a
                       weight row quantised with another matrix's exponent)
  down reduction    -- with W3 = 2^s I the FP8 output is the quantised hidden
                       times 2^s (hidden not quantised, scale off)
  block consistency -- a block's routed and shared sums equal the per-row FP8
                       experts (token row not quantised, shared experts not
                       treated as one concatenated MLP)
  error size        -- FP8 vs bf16 layer: nonzero and within the E4M3 bound
"""
import math

import numpy as np
import pytest
import torch

import oracle

F8 = torch.float8_e4m3fn


def lib_e4m3(x):
    """Library routine: torch's float8_e4m3fn conversion (round to nearest even)."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(F8).float().numpy().astype(np.float64)


def lib_codes(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(F8).view(torch.uint8).numpy()


def finite_codes():
    c = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    v = c.view(F8).float().numpy().astype(np.float64)
    keep = ~np.isnan(v)
    return c.numpy()[keep], v[keep]


def test_every_e4m3_code_is_a_fixed_point():
    codes, vals = finite_codes()
    assert len(codes) == 254 and vals.max() == 448.0 and vals[vals > 0].min() == 2.0 ** -9
    out, oc = oracle.e4m3(vals)
    np.testing.assert_array_equal(out, vals)
    np.testing.assert_array_equal(oc, codes)


def test_e4m3_rounding_matches_the_library():
    r = np.random.default_rng(81)
    mag = np.exp2(r.uniform(-13.0, math.log2(460.0), 200_000))
    x = (mag * r.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    # every midpoint between neighbouring finite non-negative codes (the ties)
    _, vals = finite_codes()
    pos = np.unique(vals[vals >= 0])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)   # exact in fp32
    x = np.concatenate([x, mids, -mids, np.float32([0.0, 2.0 ** -10, 3 * 2.0 ** -11, 464.0])])
    out, oc = oracle.e4m3(x.astype(np.float64))
    np.testing.assert_array_equal(out, lib_e4m3(x))
    nz = out != 0                      # signed zeros: compare codes only off zero
    np.testing.assert_array_equal(oc[nz], lib_codes(x)[nz])


def test_e4m3_saturates_beyond_the_largest_value():
    x = np.array([464.0001, 480.0, 1e6, np.inf, -500.0, -np.inf])
    out, oc = oracle.e4m3(x)
    np.testing.assert_array_equal(out, [448, 448, 448, 448, -448, -448])
    np.testing.assert_array_equal(oc, [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE])


def _brute_exp(row):
    amax = np.abs(row).max()
    if amax == 0:
        return 0
    for e in range(-200, 200):
        if amax * 2.0 ** -e <= 448.0:
            return e
    raise AssertionError


def test_row_scales_brute_force():
    r = np.random.default_rng(82)
    rows = [r.standard_normal(40) * s for s in (1e-6, 0.01, 1.0, 3.0, 1e4)]
    rows += [np.r_[448.0 * 2.0 ** j, r.uniform(-1, 1, 39)] for j in (-9, 0, 3)]      # max exactly 448 2^j
    rows += [np.r_[-224.0 * 2.0 ** j, r.uniform(-1, 1, 39) * 2.0 ** j] for j in (-2, 5)]  # max 224 2^j
    rows += [np.zeros(40), np.r_[np.zeros(39), 1e-3]]
    x = np.stack(rows).astype(np.float32)
    codes, exps, deq = oracle.quant_rows(x)
    for i, row in enumerate(x.astype(np.float64)):
        e = _brute_exp(row)
        assert exps[i] == e, (i, exps[i], e)
        s = 2.0 ** -e
        np.testing.assert_array_equal(deq[i], lib_e4m3(row * s) / s)
        nz = deq[i] != 0
        np.testing.assert_array_equal(codes[i][nz], lib_codes(row * s)[nz])
        if np.abs(row).max() > 0:
            assert 224.0 < np.abs(row).max() * s <= 448.0
        # E4M3 error bound: half a quantum (2^-4 relative for normals, 2^-10 scaled for subnormals)
        assert np.all(np.abs(deq[i] - row) <= np.maximum(2.0 ** -4 * np.abs(row), 2.0 ** (e - 10)) + 0)


def _representable_rows(r, shape, exps):
    """Rows of E4M3 values times 2^e_row whose largest magnitude lies in
    (224, 448] 2^e_row, so the oracle's row scale is exactly 2^e_row."""
    _, vals = finite_codes()
    v = r.choice(vals[np.abs(vals) <= 224.0], size=shape)
    v[..., 0] = r.choice(vals[(np.abs(vals) > 224.0)], size=shape[:-1])
    return v * np.exp2(exps)[..., None]


def test_gate_up_reduces_to_exact_on_representable_operands():
    r = np.random.default_rng(83)
    T, d, E, c = 12, 32, 3, 16
    a = _representable_rows(r, (T, d), r.integers(-12, -6, T).astype(float))
    w1 = _representable_rows(r, (E, c, d), r.integers(-14, -9, (E, c)).astype(float))
    w2 = _representable_rows(r, (E, c, d), r.integers(-11, -6, (E, c)).astype(float))
    w3 = r.standard_normal((E, d, c)) / 4
    ex = r.integers(0, E, T).astype(np.int32)
    kw = dict(in_dtype=oracle.F64, storage=oracle.STORE_BF16)
    h8, _ = oracle.expert_rows(oracle.make_cfg(d, E, 1, c, fp8=True, **kw), a, ex, w1, w2, w3)
    h, _ = oracle.expert_rows(oracle.make_cfg(d, E, 1, c, fp8=False, **kw), a, ex, w1, w2, w3)
    np.testing.assert_array_equal(h8, h)
    assert np.abs(h).max() > 0


def test_down_projection_reduces_to_the_quantised_hidden():
    r = np.random.default_rng(84)
    T, d, E = 10, 32, 2
    c = d
    a = r.standard_normal((T, d))
    w1 = r.standard_normal((E, c, d)) / math.sqrt(d)
    w2 = r.standard_normal((E, c, d)) / math.sqrt(d) * 3
    s = np.array([-3.0, 2.0])
    w3 = np.stack([np.eye(d) * 2.0 ** s[e] for e in range(E)])
    ex = np.arange(T, dtype=np.int32) % E
    cfg = oracle.make_cfg(d, E, 1, c, in_dtype=oracle.F64, storage=oracle.STORE_BF16, fp8=True)
    h, y = oracle.expert_rows(cfg, a, ex, w1, w2, w3)
    _, _, hq = oracle.quant_rows(h)
    want = hq * np.exp2(s[ex])[:, None]
    bf = torch.from_numpy(want).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(y, bf)
    assert not np.array_equal(hq, h)      # the quantisation is not the identity here


def test_down_projection_with_representable_weights_is_a_matmul_of_the_quantised_hidden():
    r = np.random.default_rng(87)
    T, d, E, c = 10, 32, 3, 16
    a = r.standard_normal((T, d))
    w1 = r.standard_normal((E, c, d)) / math.sqrt(d)
    w2 = r.standard_normal((E, c, d)) / math.sqrt(d)
    w3 = _representable_rows(r, (E, d, c), r.integers(-16, -8, (E, d)).astype(float))
    ex = r.integers(0, E, T).astype(np.int32)
    cfg = oracle.make_cfg(d, E, 1, c, in_dtype=oracle.F64, storage=oracle.STORE_BF16, fp8=True)
    h, y = oracle.expert_rows(cfg, a, ex, w1, w2, w3)
    _, _, hq = oracle.quant_rows(h)
    want = np.einsum("tj,tij->ti", hq, w3[ex])          # library matmul over the exact weights
    bf = torch.from_numpy(want).to(torch.bfloat16).double().numpy()
    close = np.abs(y - bf) <= 2.0 ** -8 * np.abs(bf)    # at most one bf16 ulp from summation order
    assert close.all() and (y == bf).mean() > 0.95


def _fp8_block_problem(seed, T=16, d=32, E=5, k=2, c=16, ns=2, cs=16):
    r = np.random.default_rng(seed)
    w = dict(w_r=r.standard_normal((E, d)) / math.sqrt(d),
             w1=r.standard_normal((E, c, d)) / math.sqrt(d),
             w2=r.standard_normal((E, c, d)) / math.sqrt(d),
             w3=r.standard_normal((E, d, c)) / math.sqrt(c),
             w1s=r.standard_normal((ns, cs, d)) / math.sqrt(d),
             w2s=r.standard_normal((ns, cs, d)) / math.sqrt(d),
             w3s=r.standard_normal((ns, d, cs)) / math.sqrt(cs) * np.array([1.0, 5.0])[:ns, None, None])
    x = r.standard_normal((T, d))
    return w, x


def test_block_sums_are_the_per_row_fp8_experts():
    T, d, E, k, c, ns, cs = 16, 32, 5, 2, 16, 2, 16
    w, x = _fp8_block_problem(85, T, d, E, k, c, ns, cs)
    cfg = oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", oracle.F64, oracle.STORE_BF16, fp8=True)
    out = oracle.stack(cfg, [oracle.Weights(**w)], "partial", x, want_rs=True)
    # routed: R[t] = sum_s w_s y_{e_s}(x[t]) with the FP8 per-row expert
    rows = np.repeat(x, k, axis=0)
    ex = out["topk_idx"][0].reshape(-1)
    _, y = oracle.expert_rows(cfg, rows, ex, w["w1"], w["w2"], w["w3"])
    R = (out["topk_w"][0].reshape(-1, 1) * y).reshape(T, k, d).sum(1)
    np.testing.assert_allclose(out["R"][0], R, rtol=1e-13, atol=1e-13)
    # shared: one expert of width ns cs over the concatenated weights
    w3cat = np.concatenate([w["w3s"][s] for s in range(ns)], axis=1)            # [d, ns cs]
    cfg1 = oracle.make_cfg(d, 1, 1, ns * cs, 0, 0, "softmax_renorm", oracle.F64, oracle.STORE_BF16, fp8=True)
    _, ys = oracle.expert_rows(cfg1, x, np.zeros(T, np.int32), w["w1s"].reshape(1, ns * cs, d),
                               w["w2s"].reshape(1, ns * cs, d), w3cat[None])
    # S is the unrounded shared output at residual (fp32) precision; ys went through bf16 storage
    s32 = out["S"][0]
    np.testing.assert_allclose(torch.from_numpy(s32).to(torch.bfloat16).double().numpy(), ys, rtol=0, atol=0)


def test_fp8_layer_error_is_within_the_e4m3_bound():
    T, d, E, k, c, ns, cs = 24, 64, 6, 2, 32, 1, 32
    w, x = _fp8_block_problem(86, T, d, E, k, c, ns, cs)
    kw = dict(in_dtype=oracle.F64, storage=oracle.STORE_BF16)
    o8 = oracle.stack(oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", fp8=True, **kw),
                      [oracle.Weights(**w)], "partial", x, want_rs=True)
    ob = oracle.stack(oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", fp8=False, **kw),
                      [oracle.Weights(**w)], "partial", x, want_rs=True)
    np.testing.assert_array_equal(o8["topk_idx"], ob["topk_idx"])   # the router is not quantised
    for key in ("R", "S"):
        rel = np.linalg.norm(o8[key] - ob[key]) / np.linalg.norm(ob[key])
        # each E4M3 rounding has relative rms about 2^-4 / sqrt(3) = 3.6%; a product path
        # goes through about five of them (token, gate/up row, hidden, down row), about 8% in
        # quadrature: nonzero, and well under 15%
        assert 0.02 < rel < 0.15, (key, rel)


# ------------------------------------------------ block scales (the MX form)
# One power-of-two scale per block of 32 consecutive elements along the
# contraction, chosen per block by the row rule above.

MX = 32


def test_mx_block_scales_brute_force():
    """Block exponents equal a brute-force search per 32-element block, codes the
    library's conversion of each block scaled by its own 2^-e, and each block is
    quantised on its own (changing one block changes no other block)."""
    r = np.random.default_rng(91)
    rows, cols = 9, 4 * MX
    x = r.standard_normal((rows, cols))
    x *= np.exp2(r.integers(-12, 12, (rows, cols // MX))).repeat(MX, axis=1)      # a magnitude per block
    x[0, :MX] = 0.0                                                                # an all-zero block
    x[1, MX:2 * MX] = 0.0
    x[1, MX + 3] = 448.0 * 2.0 ** -5                                               # max exactly 448 2^j
    x[2, 2 * MX + 7] = -224.0 * 2.0 ** 3                                           # max exactly 224 2^j
    x = x.astype(np.float32)
    codes, exps, deq = oracle.quant_blocks(x, MX)
    assert exps.shape == (rows, cols // MX)
    for i in range(rows):
        for b in range(cols // MX):
            blk = x[i, b * MX:(b + 1) * MX].astype(np.float64)
            e = _brute_exp(blk)
            assert exps[i, b] == e, (i, b, exps[i, b], e)
            s = 2.0 ** -e
            np.testing.assert_array_equal(deq[i, b * MX:(b + 1) * MX], lib_e4m3(blk * s) / s)
            nz = deq[i, b * MX:(b + 1) * MX] != 0
            np.testing.assert_array_equal(codes[i, b * MX:(b + 1) * MX][nz], lib_codes(blk * s)[nz])
            assert np.all(np.abs(deq[i, b * MX:(b + 1) * MX] - blk) <=
                          np.maximum(2.0 ** -4 * np.abs(blk), 2.0 ** (e - 10)))
    # locality: rescaling block 2 of every row leaves blocks 0, 1, 3 untouched
    y = x.copy()
    y[:, 2 * MX:3 * MX] *= 37.0
    c2, e2, d2 = oracle.quant_blocks(y, MX)
    keep = np.r_[0:2 * MX, 3 * MX:4 * MX]
    np.testing.assert_array_equal(c2[:, keep], codes[:, keep])
    np.testing.assert_array_equal(e2[:, [0, 1, 3]], exps[:, [0, 1, 3]])
    assert not np.array_equal(e2[:, 2], exps[:, 2])
    # a block as long as the row is the row scale
    cr, er, dr = oracle.quant_blocks(x, cols)
    c1, e1, d1 = oracle.quant_rows(x)
    np.testing.assert_array_equal(dr, d1)
    np.testing.assert_array_equal(er[:, 0], e1)


def _mx_representable(r, shape, exps):
    """Rows whose every 32-element block is E4M3 values times 2^e_block with the
    block's largest magnitude in (224, 448] 2^e_block, so the oracle's block
    scale is exactly 2^e_block (exps: [..., n_blocks])."""
    _, vals = finite_codes()
    nb = shape[-1] // MX
    v = r.choice(vals[np.abs(vals) <= 224.0], size=shape)
    for b in range(nb):
        v[..., b * MX] = r.choice(vals[np.abs(vals) > 224.0], size=shape[:-1])
    return v * np.repeat(np.exp2(exps), MX, axis=-1)


def test_mx_gate_up_reduces_to_exact_on_representable_operands():
    """With every activation and weight block exactly representable at its own
    block scale, the MX hidden equals the exact (unquantised) hidden; with the
    row form the same operands (blocks of different scales in one row) are not
    representable, so the MX form is not the row form in disguise."""
    r = np.random.default_rng(92)
    T, d, E, c = 10, 4 * MX, 3, 2 * MX
    a = _mx_representable(r, (T, d), r.integers(-12, -4, (T, d // MX)).astype(float))
    w1 = _mx_representable(r, (E, c, d), r.integers(-16, -8, (E, c, d // MX)).astype(float))
    w2 = _mx_representable(r, (E, c, d), r.integers(-13, -6, (E, c, d // MX)).astype(float))
    w3 = r.standard_normal((E, d, c)) / 4
    ex = r.integers(0, E, T).astype(np.int32)
    kw = dict(in_dtype=oracle.F64, storage=oracle.STORE_BF16)
    hm, _ = oracle.expert_rows(oracle.make_cfg(d, E, 1, c, fp8="mx", **kw), a, ex, w1, w2, w3)
    h, _ = oracle.expert_rows(oracle.make_cfg(d, E, 1, c, fp8=False, **kw), a, ex, w1, w2, w3)
    hr, _ = oracle.expert_rows(oracle.make_cfg(d, E, 1, c, fp8="row", **kw), a, ex, w1, w2, w3)
    np.testing.assert_array_equal(hm, h)
    assert np.abs(h).max() > 0 and not np.array_equal(hr, h)


def test_mx_down_projection_is_a_matmul_of_the_block_quantised_hidden():
    """With representable W3 blocks the MX output is a library matmul of the
    hidden quantised in 32-element blocks (and not of the row-quantised one)."""
    r = np.random.default_rng(93)
    T, d, E, c = 10, 2 * MX, 3, 4 * MX
    a = r.standard_normal((T, d))
    w1 = r.standard_normal((E, c, d)) / math.sqrt(d)
    w2 = r.standard_normal((E, c, d)) / math.sqrt(d) * np.exp2(r.integers(-3, 4, (E, c, 1)))
    w3 = _mx_representable(r, (E, d, c), r.integers(-16, -8, (E, d, c // MX)).astype(float))
    ex = r.integers(0, E, T).astype(np.int32)
    cfg = oracle.make_cfg(d, E, 1, c, in_dtype=oracle.F64, storage=oracle.STORE_BF16, fp8="mx")
    h, y = oracle.expert_rows(cfg, a, ex, w1, w2, w3)
    _, _, hq = oracle.quant_blocks(h, MX)
    want = np.einsum("tj,tij->ti", hq, w3[ex])
    bf = torch.from_numpy(want).to(torch.bfloat16).double().numpy()
    close = np.abs(y - bf) <= 2.0 ** -8 * np.abs(bf)
    assert close.all() and (y == bf).mean() > 0.95
    _, _, hq_row = oracle.quant_rows(h)
    assert not np.array_equal(hq_row, hq)


def test_mx_equals_row_scaling_when_every_block_shares_the_row_scale():
    """Operands whose every 32-element block has the same power-of-two scale as
    its whole row quantise identically in both forms, so the MX layer equals the
    pinned row-scaled FP8 layer exactly."""
    r = np.random.default_rng(94)
    T, d, E, k, c, ns, cs = 8, 2 * MX, 4, 2, 2 * MX, 1, MX

    def same_scale(shape, e_rows):
        v = _mx_representable(r, shape, np.repeat(e_rows[..., None], shape[-1] // MX, axis=-1))
        return v

    w = dict(w_r=r.standard_normal((E, d)) / math.sqrt(d),
             w1=same_scale((E, c, d), r.integers(-16, -8, (E, c)).astype(float)),
             w2=same_scale((E, c, d), r.integers(-14, -8, (E, c)).astype(float)),
             w3=same_scale((E, d, c), r.integers(-16, -8, (E, d)).astype(float)),
             w1s=same_scale((ns, cs, d), r.integers(-16, -8, (ns, cs)).astype(float)),
             w2s=same_scale((ns, cs, d), r.integers(-14, -8, (ns, cs)).astype(float)),
             w3s=same_scale((ns, d, cs), r.integers(-16, -8, (ns, d)).astype(float)))
    x = same_scale((T, d), r.integers(-6, -2, T).astype(float))
    kw = dict(in_dtype=oracle.F64, storage=oracle.EXACT)
    om = oracle.stack(oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", fp8="mx", **kw), [oracle.Weights(**w)],
                      "partial", x, want_rs=True)
    orow = oracle.stack(oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", fp8="row", **kw),
                        [oracle.Weights(**w)], "partial", x, want_rs=True)
    # the hidden is formed inside the layer, so its blocks need not share a scale:
    # compare the routed/shared sums only where the hidden is exactly representable,
    # i.e. check the gate/up stage through the exact form instead
    ob = oracle.stack(oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", fp8=False, **kw), [oracle.Weights(**w)],
                      "partial", x, want_rs=True)
    np.testing.assert_array_equal(om["topk_idx"], orow["topk_idx"])
    for key in ("R", "S"):
        em = np.linalg.norm(om[key] - ob[key]) / np.linalg.norm(ob[key])
        er = np.linalg.norm(orow[key] - ob[key]) / np.linalg.norm(ob[key])
        # only the hidden's quantisation differs: MX blocks follow the hidden's
        # local magnitude, so the MX error is no larger than the row form's
        assert 0 < em <= er * 1.05, (key, em, er)


@pytest.mark.parametrize("wide", [False, True])
def test_mx_block_sums_are_the_per_row_mx_experts(wide):
    """A block's routed and shared sums equal the per-row MX experts (the token
    row quantised once, in blocks, for all its experts); wide: token blocks
    alternate magnitudes 1 and 2^16 (weights compensating), where quantising the
    token row with one scale would flush every other block."""
    T, d, E, k, c, ns, cs = 16, 2 * MX, 5, 2, 2 * MX, 2, MX
    w, x = _fp8_block_problem(95, T, d, E, k, c, ns, cs)
    if wide:
        s = np.exp2(16.0 * ((np.arange(d) // MX) % 2))
        x = (x * s).astype(np.float32).astype(np.float64)
        for key in ("w1", "w2", "w1s", "w2s"):
            w[key] = w[key] / s
    cfg = oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", oracle.F64, oracle.STORE_BF16, fp8="mx")
    out = oracle.stack(cfg, [oracle.Weights(**w)], "partial", x, want_rs=True)
    rows = np.repeat(x, k, axis=0)
    ex = out["topk_idx"][0].reshape(-1)
    _, y = oracle.expert_rows(cfg, rows, ex, w["w1"], w["w2"], w["w3"])
    R = (out["topk_w"][0].reshape(-1, 1) * y).reshape(T, k, d).sum(1)
    np.testing.assert_allclose(out["R"][0], R, rtol=1e-13, atol=1e-13)
    w3cat = np.concatenate([w["w3s"][s] for s in range(ns)], axis=1)
    cfg1 = oracle.make_cfg(d, 1, 1, ns * cs, 0, 0, "softmax_renorm", oracle.F64, oracle.STORE_BF16, fp8="mx")
    _, ys = oracle.expert_rows(cfg1, x, np.zeros(T, np.int32), w["w1s"].reshape(1, ns * cs, d),
                               w["w2s"].reshape(1, ns * cs, d), w3cat[None])
    np.testing.assert_allclose(torch.from_numpy(out["S"][0]).to(torch.bfloat16).double().numpy(), ys, rtol=0, atol=0)


def test_mx_layer_error_is_within_the_e4m3_bound_and_below_row_scaling():
    """The MX layer's error against the unquantised layer is nonzero and within the
    E4M3 bound; and block scales follow local magnitudes: on rows with one large
    outlier the row form's scale (set by the outlier) flushes the small elements
    of the row towards zero, while the MX form keeps them at E4M3 precision
    outside the outlier's block."""
    T, d, E, k, c, ns, cs = 24, 4 * MX, 6, 2, 2 * MX, 1, MX
    w, x = _fp8_block_problem(96, T, d, E, k, c, ns, cs)
    kw = dict(in_dtype=oracle.F64, storage=oracle.STORE_BF16)
    res = {}
    for mode in ("mx", False):
        res[mode] = oracle.stack(oracle.make_cfg(d, E, k, c, ns, cs, "softmax_renorm", fp8=mode, **kw),
                                 [oracle.Weights(**w)], "partial", x, want_rs=True)
    for key in ("R", "S"):
        ref = res[False][key]
        em = np.linalg.norm(res["mx"][key] - ref) / np.linalg.norm(ref)
        assert 0.02 < em < 0.15, (key, em)
    xo = x.copy()
    xo[:, 5] = 1e6                                            # an outlier in block 0 of every row
    _, _, dm = oracle.quant_blocks(xo, MX)
    _, _, dr = oracle.quant_rows(xo)
    rest = np.r_[MX:d]                                        # the blocks without the outlier
    em = np.abs(dm[:, rest] - xo[:, rest]).max() / np.abs(xo[:, rest]).max()
    er = np.abs(dr[:, rest] - xo[:, rest]).max() / np.abs(xo[:, rest]).max()
    assert em <= 2.0 ** -4 and er > 10 * em, (em, er)


def _lib_mx(x, blk=MX):
    """Library form of the MX quantisation: per block, the brute-force exponent
    and torch's float8_e4m3fn conversion of the block times 2^-e (x float32
    values, so the scaled block is exact in float32)."""
    x = np.asarray(x, np.float64)
    out = np.empty_like(x)
    flat = x.reshape(-1, x.shape[-1])
    o = out.reshape(-1, x.shape[-1])
    for r in range(flat.shape[0]):
        for b in range(flat.shape[1] // blk):
            v = flat[r, b * blk:(b + 1) * blk]
            e = _brute_exp(v)
            o[r, b * blk:(b + 1) * blk] = lib_e4m3(v * 2.0 ** -e) * 2.0 ** e
    return out


def _lib_mx_expert(a, w1, w2, w3):
    """One MX expert by library routines: operands quantised per 32-block, numpy
    matmuls, bf16 storage of the hidden (torch) before its own block quantisation."""
    aq, w1q, w2q, w3q = _lib_mx(a), _lib_mx(w1), _lib_mx(w2), _lib_mx(w3)
    g, u = aq @ w2q.T, aq @ w1q.T
    h = torch.from_numpy(g / (1.0 + np.exp(-g)) * u).float().to(torch.bfloat16).double().numpy()
    return h, _lib_mx(h.astype(np.float32)) @ w3q.T


@pytest.mark.parametrize("layout", ["across_blocks", "within_blocks"])
def test_mx_expert_matches_a_library_form_on_a_wide_dynamic_range(layout):
    """Operands whose magnitudes differ by 2^16 -- more than E4M3's range -- from
    one 32-element block to the next (across_blocks: the activation's and the
    hidden's blocks alternate 1 and 2^16, the weights compensate so every block
    contributes alike) or between the two halves of each block (within_blocks).
    There the scale granularity decides the result: rows scales flush whole
    blocks, 16-element blocks keep halves that 32-element blocks flush.  The
    oracle's MX expert must match the library form."""
    r = np.random.default_rng(97)
    T, d, c = 6, 4 * MX, 4 * MX
    f32 = lambda v: v.astype(np.float32).astype(np.float64)
    if layout == "across_blocks":
        sx = 16.0 * ((np.arange(d) // MX) % 2)                # activation block magnitudes 2^0, 2^16, ...
        sh = 16.0 * ((np.arange(c) // MX) % 2)                # hidden block magnitudes, set through W1's rows
    else:
        sx = 16.0 * ((np.arange(d) // (MX // 2)) % 2)         # the two halves of every block differ by 2^16
        sh = np.zeros(c)
    a = f32(r.standard_normal((T, d)) * np.exp2(sx))
    w1 = f32(r.standard_normal((1, c, d)) / math.sqrt(d) * np.exp2(-sx)[None, None, :] * np.exp2(sh)[None, :, None])
    w2 = f32(r.standard_normal((1, c, d)) / math.sqrt(d) * np.exp2(-sx)[None, None, :])
    w3 = f32(r.standard_normal((1, d, c)) / math.sqrt(c) * np.exp2(-sh)[None, None, :])
    cfg = oracle.make_cfg(d, 1, 1, c, in_dtype=oracle.F64, storage=oracle.STORE_BF16, fp8="mx")
    h, y = oracle.expert_rows(cfg, a, np.zeros(T, np.int32), w1, w2, w3)
    hl, yl = _lib_mx_expert(a, w1[0], w2[0], w3[0])
    # the hidden: the same bf16 values except rare one-ulp flips (fp64 sums in a
    # different order); the output: within one E4M3 step of the library's
    assert (h == hl).mean() > 0.97
    np.testing.assert_allclose(h, hl, rtol=2.0 ** -7, atol=0)
    scale = np.abs(yl).max()
    assert np.abs(y - yl).max() <= 2.0 ** -3 * scale, (np.abs(y - yl).max(), scale)
    assert np.abs(yl).max() > 0
