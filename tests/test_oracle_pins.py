"""Pins for the CPU oracle: it is checked against what the page and mathematics
fix, never against itself or the CUDA path.

Source: "FarSkip-Collective: Unhobbling Blocking Communication in Mixture of
Experts Models" (papercache.org summary), §2.1 (MLP, TP slicing, MoE, router,
Dispatch/Combine, shared expert) and §3 (FarSkip equation, eq. 8a/8b).

Pins, and the mistake each one catches:
  golden gates      -- gate rules, top-k order, tie rule, bias (wrong normaliser, wrong order)
  golden MLP        -- SiLU on the wrong projection, transposed W3, SiLU special values
  golden dispatch   -- counting sort: counts, offsets, stability, pos/perm_src
  golden rounding   -- bf16 / fp32 round-to-nearest-even at storage points
  golden storage    -- the stored hidden h and each stored routed output y are
                       rounded where the layer stores them (dropped roundings)
  library routines  -- logits vs a matmul, top-k vs a stable argsort, softmax/expit,
                       counts vs bincount, permutation vs a stable argsort
  brute force       -- dense sum_j G_j MLP^j over all experts (tiny shapes)
  reductions        -- identical experts + normalised gate = one dense MLP;
                       TP-slice identity (c split into slices, partial MLPs summed)
  stack identities  -- telescoping sum, partial/outdated/disabled input wiring
                       (block logits recomputed from the telescoped residual),
                       disabled = plain residual recurrence, L=1 wiring-independent
  equivariance      -- token permutation, expert relabelling
  round trip        -- dispatch then combine with an identity expert returns u
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def rng(seed):
    return np.random.default_rng(seed)


def np_silu(v):
    return v / (1.0 + np.exp(-v))


def dense_mlp(a, w1, w2, w3):
    """Library-routine form of one expert (numpy matmuls), used only in
    brute-force / reduction identities, never as a stand-in for a pin."""
    return (np_silu(a @ w2.T) * (a @ w1.T)) @ w3.T


def rand_weights(r, d, E, c, ns=0, cs=0, bias=False):
    w = dict(w_r=r.standard_normal((E, d)) / math.sqrt(d),
             w1=r.standard_normal((E, c, d)) / math.sqrt(d),
             w2=r.standard_normal((E, c, d)) / math.sqrt(d),
             w3=r.standard_normal((E, d, c)) / math.sqrt(c))
    if bias:
        w["bias"] = r.standard_normal(E).astype(np.float32) * 0.3
    if ns:
        w["w1s"] = r.standard_normal((ns, cs, d)) / math.sqrt(d)
        w["w2s"] = r.standard_normal((ns, cs, d)) / math.sqrt(d)
        w["w3s"] = r.standard_normal((ns, d, cs)) / math.sqrt(cs)
    return w


def W(w):
    return oracle.Weights(**w)


def cfg_of(d, E, k, c, ns=0, cs=0, gate="softmax_renorm", storage=oracle.EXACT):
    return oracle.make_cfg(d, E, k, c, ns, cs, gate, oracle.F64, storage)


# ----------------------------------------------------------------- golden values

@pytest.mark.parametrize("gate", ["softmax", "softmax_renorm", "sigmoid", "sigmoid_norm"])
def test_golden_gates(gate):
    g = gold("gates.json")
    d, E, k = g["d"], g["E"], g["k"]
    w_r = np.zeros((E, d))
    w_r[:, 0] = np.log(g["w_r_col0_is_ln"])
    cfg = cfg_of(d, E, k, 8, gate=gate)
    _, idx, w = oracle.router(cfg, np.array(g["u"], np.float64), w_r)
    assert idx[0].tolist() == g["expect_idx"]
    np.testing.assert_allclose(w[0], g["expect_w"][gate], rtol=1e-14)


def test_golden_tie_and_bias():
    g = gold("gates.json")
    E, d = g["E"], g["d"]
    u = np.ones((1, d))
    t = g["tie_case"]
    cfg = cfg_of(d, E, t["k"], 8, gate="softmax_renorm")
    _, idx, w = oracle.router(cfg, u, np.zeros((E, d)), np.array(t["logits_via_bias"], np.float32))
    assert idx[0].tolist() == t["expect_idx"]
    np.testing.assert_allclose(w[0], t["expect_softmax_renorm"], rtol=1e-14)
    b = g["bias_case"]
    _, idx, _ = oracle.router(cfg_of(d, E, b["k"], 8), u, np.zeros((E, d)), np.array(b["bias"], np.float32))
    assert idx[0].tolist() == b["expect_idx"]


def test_golden_mlp():
    for case in gold("mlp_small.json")["cases"]:
        d, c = case["d"], case["c"]
        cfg = cfg_of(d, 1, 1, c)
        a = np.array([case["a"]], np.float64)
        h, y = oracle.expert_rows(cfg, a, np.zeros(1, np.int32), np.array([case["w1"]], np.float64),
                                  np.array([case["w2"]], np.float64), np.array([case["w3"]], np.float64))
        np.testing.assert_allclose(h[0], case["expect_h"], rtol=1e-12, atol=0)
        np.testing.assert_allclose(y[0], case["expect_y"], rtol=1e-12, atol=0)


def test_golden_storage_roundings():
    """The two bf16 storage points inside a block (tests/golden/storage_rounding.json):
    the expert hidden h between the projections and each routed output y before
    the gate-weighted sum, with values that fall strictly between bf16 neighbours,
    so storage mode and exact mode differ by the hand-derived amounts."""
    g = gold("storage_rounding.json")
    m = g["mlp"]
    for mode, st in (("exact", oracle.EXACT), ("bf16", oracle.STORE_BF16)):
        cfg = cfg_of(m["d"], 1, 1, m["c"], storage=st)
        h, y = oracle.expert_rows(cfg, np.array([m["a"]], np.float64), np.zeros(1, np.int32),
                                  np.array([m["w1"]], np.float64), np.array([m["w2"]], np.float64),
                                  np.array([m["w3"]], np.float64))
        assert h[0].tolist() == m[mode]["h"], (mode, h[0])
        assert y[0].tolist() == m[mode]["y"], (mode, y[0])
    b = g["block"]
    w = W(dict(w_r=np.array(b["w_r"], np.float64), w1=np.array(b["w1"], np.float64),
               w2=np.array(b["w2"], np.float64), w3=np.array(b["w3"], np.float64)))
    for mode, st in (("exact", oracle.EXACT), ("bf16", oracle.STORE_BF16)):
        cfg = cfg_of(b["d"], b["E"], b["k"], b["c"], storage=st)
        out = oracle.stack(cfg, [w], "partial", np.array([b["x"]], np.float64), want_rs=True)
        assert out["topk_idx"][0, 0].tolist() == [0, 1]
        assert out["topk_w"][0, 0].tolist() == [0.5, 0.5]
        assert out["o"][0].tolist() == b[mode]["o"], (mode, out["o"][0])
        assert out["o_star"][0].tolist() == b[mode]["o_star"], (mode, out["o_star"][0])
        assert out["R"][0, 0].tolist() == b[mode]["R"], (mode, out["R"][0, 0])


def test_golden_dispatch():
    g = gold("dispatch.json")
    counts, offsets, pos, perm = oracle.dispatch(g["T"], g["k"], g["E"], np.array(g["topk_idx"], np.int32))
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert perm.tolist() == g["perm_src"]
    assert pos.tolist() == g["pos"]


def test_golden_rounding():
    g = gold("rounding.json")
    for x, want in g["bf16"]:
        got = oracle.round_storage(x, oracle.STORE_BF16)
        assert got == (math.inf if want == "inf" else want), (x, got, want)
    for x, want in g["f32"]:
        assert oracle.round_storage(x, oracle.STORE_F32) == want
    # library cross-check on binary32-exact values: torch's fp32 -> bf16 conversion
    xs = rng(5).standard_normal(2000).astype(np.float32) * 10.0
    ref = torch.from_numpy(xs).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_storage(float(v), oracle.STORE_BF16) for v in xs])
    np.testing.assert_array_equal(got, ref)
    xs64 = rng(6).standard_normal(2000) * 3.0
    ref32 = xs64.astype(np.float32).astype(np.float64)
    got32 = np.array([oracle.round_storage(float(v), oracle.STORE_F32) for v in xs64])
    np.testing.assert_array_equal(got32, ref32)


# ------------------------------------------------------------ library routines

@pytest.mark.parametrize("gate", ["softmax", "softmax_renorm", "sigmoid", "sigmoid_norm"])
def test_router_vs_library(gate):
    from scipy.special import expit, softmax
    r = rng(1)
    T, d, E, k = 37, 24, 11, 3
    u = r.standard_normal((T, d))
    w_r = r.standard_normal((E, d)) / math.sqrt(d)
    b = (np.round(r.standard_normal(E) * 512) / 1024).astype(np.float32)  # b + 0.75 stays exact
    logits, idx, w = oracle.router(cfg_of(d, E, k, 8, gate=gate), u, w_r, b)
    z = u @ w_r.T + b.astype(np.float64)
    np.testing.assert_allclose(logits, z, rtol=1e-12, atol=1e-12)
    want_idx = np.argsort(-z, axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(idx, want_idx)
    zk = np.take_along_axis(z, want_idx, 1)
    if gate == "softmax":
        want = np.take_along_axis(softmax(z, axis=1), want_idx, 1)
    elif gate == "softmax_renorm":
        want = softmax(zk, axis=1)
    elif gate == "sigmoid":
        want = expit(zk)
    else:
        want = expit(zk) / expit(zk).sum(1, keepdims=True)
    np.testing.assert_allclose(w, want, rtol=1e-12)
    # P8 invariants
    if gate in ("softmax_renorm", "sigmoid_norm"):
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-13)
    if gate.startswith("softmax"):
        _, idx2, w2 = oracle.router(cfg_of(d, E, k, 8, gate=gate), u, w_r, b + np.float32(0.75))
        np.testing.assert_array_equal(idx2, idx)
        np.testing.assert_allclose(w2, w, rtol=1e-12)


def test_dispatch_vs_library():
    r = rng(2)
    T, k, E = 500, 4, 13
    idx = np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, pos, perm = oracle.dispatch(T, k, E, idx)
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) == counts)
    # stable sort of (t, s) pairs by expert == the permutation
    order = np.argsort(idx.ravel(), kind="stable")          # flat (t*k+s) in permuted order
    np.testing.assert_array_equal(perm, order // k)
    inv = np.empty_like(order)
    inv[order] = np.arange(T * k)
    np.testing.assert_array_equal(pos, inv)
    # P7: every segment is increasing in token, and perm_src o pos = identity on tokens
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
    np.testing.assert_array_equal(perm[pos], np.repeat(np.arange(T), k))


def test_dispatch_rejects_bad_index():
    with pytest.raises(RuntimeError):
        oracle.dispatch(2, 1, 3, np.array([[0], [3]], np.int32))


# ------------------------------------------------------------------ brute force

@pytest.mark.parametrize("gate", ["softmax", "softmax_renorm", "sigmoid", "sigmoid_norm"])
def test_brute_force_dense_moe(gate):
    """P5: R = sum_{j<E} G_j MLP^j(u), G zero off the top-k (dense over every expert)."""
    from scipy.special import expit, softmax
    r = rng(3)
    T, d, E, k, c = 12, 16, 6, 2, 8
    w = rand_weights(r, d, E, c, bias=True)
    u = r.standard_normal((T, d))
    cfg = cfg_of(d, E, k, c, gate=gate)
    out = oracle.stack(cfg, [W(w)], "partial", u, want_rs=True)
    z = u @ w["w_r"].T + w["bias"].astype(np.float64)
    R = np.zeros((T, d))
    for t in range(T):
        order = sorted(range(E), key=lambda j: (-z[t, j], j))  # enumerate all E, sort
        top = order[:k]
        G = np.zeros(E)
        if gate == "softmax":
            p = softmax(z[t])
            G[top] = p[top]
        elif gate == "softmax_renorm":
            G[top] = softmax(z[t, top])
        elif gate == "sigmoid":
            G[top] = expit(z[t, top])
        else:
            G[top] = expit(z[t, top]) / expit(z[t, top]).sum()
        for j in range(E):
            R[t] += G[j] * dense_mlp(u[t:t + 1], w["w1"][j], w["w2"][j], w["w3"][j])[0]
    np.testing.assert_allclose(out["R"][0], R, rtol=1e-11, atol=1e-12)
    # no shared expert: o* = x and o = x + R
    np.testing.assert_allclose(out["o_star"], u, rtol=0, atol=0)
    np.testing.assert_allclose(out["o"], u + R, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------- reductions

@pytest.mark.parametrize("gate,scale", [("softmax_renorm", None), ("sigmoid_norm", None),
                                        ("softmax", "sum"), ("sigmoid", "sum")])
def test_identical_experts_reduce_to_dense_mlp(gate, scale):
    """P3: identical experts: normalised gates give R = MLP(u); otherwise (sum_s w_s) MLP(u)."""
    r = rng(4)
    T, d, E, k, c = 20, 16, 5, 3, 12
    w = rand_weights(r, d, E, c)
    for key in ("w1", "w2", "w3"):
        w[key] = np.repeat(w[key][:1], E, axis=0).copy()
    u = r.standard_normal((T, d))
    out = oracle.stack(cfg_of(d, E, k, c, gate=gate), [W(w)], "partial", u, want_rs=True)
    m = dense_mlp(u, w["w1"][0], w["w2"][0], w["w3"][0])
    if scale == "sum":
        m = m * out["topk_w"][0].sum(1, keepdims=True)
    np.testing.assert_allclose(out["R"][0], m, rtol=1e-11, atol=1e-12)


def test_tp_slice_identity():
    """P6 (§2.1 TP slicing): W1/W2 row slices and W3 column slices; the sum of the
    partial MLPs equals the full MLP.  Run through the shared-expert path with
    n_shared slices versus one shared expert of the full width."""
    r = rng(7)
    T, d, c, parts = 9, 16, 24, 3
    w1 = r.standard_normal((c, d)) / 4
    w2 = r.standard_normal((c, d)) / 4
    w3 = r.standard_normal((d, c)) / 5
    base = rand_weights(r, d, 2, 8)
    u = r.standard_normal((T, d))
    full = dict(base, w1s=w1[None], w2s=w2[None], w3s=w3[None])
    cs = c // parts
    sl = dict(base,
              w1s=np.stack([w1[i * cs:(i + 1) * cs] for i in range(parts)]),
              w2s=np.stack([w2[i * cs:(i + 1) * cs] for i in range(parts)]),
              w3s=np.stack([np.ascontiguousarray(w3[:, i * cs:(i + 1) * cs]) for i in range(parts)]))
    o_full = oracle.stack(cfg_of(d, 2, 1, 8, 1, c), [W(full)], "partial", u, want_rs=True)
    o_sl = oracle.stack(cfg_of(d, 2, 1, 8, parts, cs), [W(sl)], "partial", u, want_rs=True)
    np.testing.assert_allclose(o_sl["S"], o_full["S"], rtol=1e-12, atol=1e-13)
    # and the shared output is the dense MLP of the full width
    np.testing.assert_allclose(o_full["S"][0], dense_mlp(u, w1, w2, w3), rtol=1e-11, atol=1e-12)
    # partial wiring: o* = x + S
    np.testing.assert_allclose(o_full["o_star"], u + o_full["S"][0], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------- stack identities

def _stack_problem(seed, L, T=10, d=16, E=6, k=2, c=8, ns=1, cs=8):
    r = rng(seed)
    ws = [rand_weights(r, d, E, c, ns, cs, bias=True) for _ in range(L)]
    x = r.standard_normal((T, d))
    return cfg_of(d, E, k, c, ns, cs, gate="softmax_renorm"), ws, x


@pytest.mark.parametrize("wiring", ["partial", "outdated", "disabled"])
def test_telescoping_and_wiring(wiring):
    """P1 (§3 FarSkip equation, eq. 8a/8b): o_L = x + sum_k (S_k + R_k), o_L - o_L* = R_L,
    and each block's logits are those of the input the wiring prescribes."""
    L = 4
    cfg, ws, x = _stack_problem(11, L)
    out = oracle.stack(cfg, [W(w) for w in ws], wiring, x, want_rs=True)
    R, S = out["R"], out["S"]
    o = [x]
    for b in range(L):
        o.append(o[-1] + S[b] + R[b])
    np.testing.assert_allclose(out["o"], o[L], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["o"] - out["o_star"], R[L - 1], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["o_star"], o[L - 1] + S[L - 1], rtol=1e-12, atol=1e-12)
    for b in range(L):          # block b+1 (1-based) input u_{b+1}
        if b == 0:
            u = x
        elif wiring == "partial":
            u = o[b - 1] + S[b - 1]          # o_b* = o_{b-1} + S_b
        elif wiring == "outdated":
            u = o[b - 1]                     # o_b* = o_{b-1}
        else:
            u = o[b]                         # o_b
        z = u @ ws[b]["w_r"].T + ws[b]["bias"].astype(np.float64)
        np.testing.assert_allclose(out["logits"][b], z, rtol=1e-10, atol=1e-11)
        # and R_b, S_b are the MoE / shared MLP of that input
        np.testing.assert_allclose(S[b], dense_mlp(u, ws[b]["w1s"][0], ws[b]["w2s"][0], ws[b]["w3s"][0]),
                                   rtol=1e-10, atol=1e-11)


def test_disabled_is_plain_recurrence_and_L1_agrees():
    """P2: with FarSkip disabled, L blocks = L applications of o_k = o_{k-1} + f_k(o_{k-1});
    with L = 1 all wirings agree."""
    L = 3
    cfg, ws, x = _stack_problem(12, L)
    full = oracle.stack(cfg, [W(w) for w in ws], "disabled", x)
    o = x
    for b in range(L):
        o = oracle.stack(cfg, [W(ws[b])], "disabled", o)["o"]
    np.testing.assert_allclose(full["o"], o, rtol=1e-13, atol=1e-13)
    one = [oracle.stack(cfg, [W(ws[0])], wi, x)["o"] for wi in ("partial", "outdated", "disabled")]
    np.testing.assert_array_equal(one[0], one[1])
    np.testing.assert_array_equal(one[0], one[2])


def test_partial_sees_every_block_once():
    """§3: every f_k enters o_L exactly once, and f_{k+1} sees all of o_k but R_k;
    zeroing the routed experts of the last block leaves o_L = o_L*."""
    cfg, ws, x = _stack_problem(13, 2)
    ws[1]["w3"] = np.zeros_like(ws[1]["w3"])
    out = oracle.stack(cfg, [W(w) for w in ws], "partial", x, want_rs=True)
    np.testing.assert_allclose(out["o"], out["o_star"], rtol=0, atol=0)


# ------------------------------------------------------------------ equivariance

def test_token_and_expert_equivariance():
    r = rng(14)
    L = 2
    cfg, ws, x = _stack_problem(15, L, T=14, E=7, k=3)
    base = oracle.stack(cfg, [W(w) for w in ws], "partial", x)
    perm_t = r.permutation(x.shape[0])
    pt = oracle.stack(cfg, [W(w) for w in ws], "partial", np.ascontiguousarray(x[perm_t]))
    np.testing.assert_allclose(pt["o"], base["o"][perm_t], rtol=1e-13, atol=1e-13)
    perm_e = r.permutation(cfg.E)          # relabel experts: new j holds old perm_e[j]
    ws2 = []
    for w in ws:
        w2 = dict(w)
        for key in ("w_r", "w1", "w2", "w3"):
            w2[key] = np.ascontiguousarray(w[key][perm_e])
        w2["bias"] = np.ascontiguousarray(w["bias"][perm_e])
        ws2.append(w2)
    pe = oracle.stack(cfg, [W(w) for w in ws2], "partial", x)
    np.testing.assert_allclose(pe["o"], base["o"], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(perm_e[pe["topk_idx"]], base["topk_idx"])


# -------------------------------------------------------------------- round trip

@pytest.mark.parametrize("k,wval", [(1, 1.0), (2, 0.5), (4, 0.25)])
def test_dispatch_combine_round_trip(k, wval):
    """P4: permute with Dispatch, identity expert, Combine with weights summing to 1
    (powers of two: exact) returns u bit for bit; o* = o_prev + S."""
    r = rng(16)
    T, d, E = 40, 8, 9
    idx = np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    u = r.standard_normal((T, d))
    counts, offsets, pos, perm = oracle.dispatch(T, k, E, idx)
    x_perm = np.ascontiguousarray(u[perm])
    w = np.full((T, k), wval, np.float32)
    o_star, o = oracle.combine(T, k, d, x_perm, pos, w, np.zeros((T, d)))
    np.testing.assert_array_equal(o, u)
    np.testing.assert_array_equal(o_star, np.zeros((T, d)))
    S = r.standard_normal((T, d))
    op = r.standard_normal((T, d))
    o_star, o = oracle.combine(T, k, d, x_perm, pos, w, op, S)
    np.testing.assert_array_equal(o_star, op + S)
    np.testing.assert_allclose(o, op + S + u, rtol=1e-15, atol=1e-15)


# --------------------------------------------------------------- storage modes

def test_bf16_storage_outputs_are_fp32_and_close():
    """With bf16 storage the stack returns the fp32 residual stream; the block
    inputs in between are bf16 values (checked through block 2's logits)."""
    cfg, ws, x = _stack_problem(17, 2)
    ex = oracle.stack(cfg, [W(w) for w in ws], "partial", x, want_rs=True)
    cfg_b = cfg_of(cfg.d, cfg.E, cfg.k, cfg.c, cfg.n_shared, cfg.c_shared, storage=oracle.STORE_BF16)
    bf = oracle.stack(cfg_b, [W(w) for w in ws], "partial", x, want_rs=True)
    for key in ("o", "o_star"):
        v = bf[key]
        np.testing.assert_array_equal(v, v.astype(np.float32).astype(np.float64))   # fp32 values
        rel = np.linalg.norm(v - ex[key]) / np.linalg.norm(ex[key])
        assert rel < 1e-2, rel
    # S feeds only the fp32 residual: fp32 values
    s1 = bf["S"][0]
    np.testing.assert_array_equal(s1, s1.astype(np.float32).astype(np.float64))
    # block 2 sees u_2 = bf16(o_1*) with o_1* = fp32(x + S_1)
    o1s = (x + s1).astype(np.float32)
    u2 = torch.from_numpy(o1s).to(torch.bfloat16).double().numpy()
    z2 = u2 @ ws[1]["w_r"].T + ws[1]["bias"].astype(np.float64)
    np.testing.assert_allclose(bf["logits"][1], z2, rtol=1e-12, atol=1e-12)


def test_bf16_inputs_widen_exactly():
    """bf16 inputs (raw uint16) are widened exactly: same result as the fp64 copy."""
    r = rng(18)
    T, d, E, k = 6, 16, 5, 2
    u = torch.from_numpy(r.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    w_r = torch.from_numpy(r.standard_normal((E, d)).astype(np.float32)).to(torch.bfloat16)
    u16 = u.view(torch.int16).numpy().view(np.uint16)
    w16 = w_r.view(torch.int16).numpy().view(np.uint16)
    cfg16 = oracle.make_cfg(d, E, k, 8, 0, 0, "softmax_renorm", oracle.BF16)
    z16, i16, w16o = oracle.router(cfg16, u16, w16)
    z64, i64, w64 = oracle.router(cfg_of(d, E, k, 8), u.double().numpy(), w_r.double().numpy())
    np.testing.assert_array_equal(z16, z64)
    np.testing.assert_array_equal(i16, i64)


# ---------------------------------------------- attention/MoE wiring (FarSkip §3)

def _attn_problem(seed, L, zero_att=False, **kw):
    cfg, ws, x = _stack_problem(seed, L, **kw)
    r = rng(seed + 100)
    d = x.shape[1]
    for w in ws:
        w["w_att"] = np.zeros((d, d)) if zero_att else r.standard_normal((d, d)) / math.sqrt(d)
    return cfg, ws, x


def test_attn_farskip_wiring_identities():
    """FarSkip §3 attention/MoE wiring: mlp-in_k = attn-in_k + routed-out_{k-1} (the page's
    decomposition), attn-in_k = o_{k-2} + attn-out_{k-1} + shared-out_{k-1}, and
    o_k = o_{k-1} + attn-out_k + shared-out_k + routed-out_k (telescoping)."""
    L = 4
    cfg, ws, x = _attn_problem(21, L)
    out = oracle.stack(cfg, [W(w) for w in ws], "attn_farskip", x, want_rs=True, want_inputs=True)
    A, U, P, O, R, S = out["A"], out["U"], out["P"], out["O"], out["R"], out["S"]
    att = [A[b] @ ws[b]["w_att"].T for b in range(L)]                # library matmul
    np.testing.assert_array_equal(A[0], x)
    np.testing.assert_array_equal(U[0], x)
    for b in range(1, L):
        np.testing.assert_allclose(U[b], A[b] + R[b - 1], rtol=1e-12, atol=1e-12)
        o_km2 = x if b == 1 else O[b - 2]
        np.testing.assert_allclose(A[b], o_km2 + att[b - 1] + S[b - 1], rtol=1e-12, atol=1e-12)
    o = x
    for b in range(L):
        np.testing.assert_allclose(P[b], o, rtol=1e-12, atol=1e-12)
        o = o + att[b] + S[b] + R[b]
        np.testing.assert_allclose(O[b], o, rtol=1e-11, atol=1e-11)
    # the MoE sees o_{k-1}: its routing is the router of mlp-in
    for b in range(L):
        z = U[b] @ ws[b]["w_r"].T + ws[b]["bias"].astype(np.float64)
        np.testing.assert_allclose(out["logits"][b], z, rtol=1e-10, atol=1e-10)


def test_attn_plain_is_the_ordinary_layer():
    """h_k = o_{k-1} + A_k(o_{k-1}); o_k = h_k + S_k(h_k) + R_k(h_k)."""
    L = 3
    cfg, ws, x = _attn_problem(22, L)
    out = oracle.stack(cfg, [W(w) for w in ws], "attn_plain", x, want_rs=True, want_inputs=True)
    o = x
    for b in range(L):
        np.testing.assert_allclose(out["A"][b], o, rtol=1e-12, atol=1e-12)
        h = o + o @ ws[b]["w_att"].T
        np.testing.assert_allclose(out["U"][b], h, rtol=1e-12, atol=1e-12)
        o = h + out["S"][b] + out["R"][b]
        np.testing.assert_allclose(out["O"][b], o, rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(out["OS"][b], h + out["S"][b], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("wiring", ["attn_farskip", "attn_plain"])
def test_zero_attention_reduces_to_the_moe_recurrence(wiring):
    """With A = 0 both attention wirings feed the MoE o_{k-1}: the disabled (plain) MoE stack."""
    cfg, ws, x = _attn_problem(23, 3, zero_att=True)
    a = oracle.stack(cfg, [W(w) for w in ws], wiring, x)
    ref = oracle.stack(cfg, [W({k: v for k, v in w.items() if k != "w_att"}) for w in ws], "disabled", x)
    np.testing.assert_allclose(a["o"], ref["o"], rtol=1e-13, atol=1e-13)


def test_attn_standin_is_a_matmul():
    r = rng(24)
    a = r.standard_normal((5, 16))
    w = r.standard_normal((16, 16))
    cfg = cfg_of(16, 2, 1, 8)
    np.testing.assert_allclose(oracle.attn_standin(cfg, a, w), a @ w.T, rtol=1e-13, atol=1e-13)
