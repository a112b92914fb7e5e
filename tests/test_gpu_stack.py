"""GPU parity of the FarSkip stack against the CPU oracle.

Two kinds of check, for small multi-tile shapes (every token) and for the
full-size workloads (in the launch configuration the benchmark times: the
stack runs over all T tokens, and the oracle follows every token of V2-Lite,
Qwen3 and the V3 decode batch, a seeded sample of 2,048 tokens of Scout and V3
prefill; token rows are independent through the whole stack):

blockwise   every block k is run on the GPU on the oracle's own inputs u_k
            (bf16) and o_{k-1} (fp32), spliced into the checked rows of a
            full-size GPU input, so both sides route identical inputs: the
            routing rule (top-k sets equal unless the k-th/(k+1)-th gap
            < 1e-4, such tokens < 0.1%) and the output tolerance (relative
            Frobenius <= 5e-3, max-abs <= 2e-2 rms plus the one-flip allowance
            of a stored bf16 value whose rounding flipped, tokens beyond it
            < 0.1%) hold per block: the tolerance is stated for a layer's outputs.
end-to-end  fs_farskip_stack as a whole vs the oracle stack.  After block 1
            the two sides' bf16 block inputs differ by rounding flips of the
            residual, so a later block may route a near-tie differently: every
            such token must be explained by that input difference (its oracle
            gap is below twice the logit change the GPU's input causes,
            explained_drift); they are left out of the output comparison.  An
            L-block stack composes L layers' errors through the residual, so the
            end-to-end bound is L x 5e-3 relative Frobenius (the per-layer bound
            added over the layers); the max-abs bound is a per-layer property and
            is checked blockwise.
The stack driver is also checked bit-for-bit against the same stack driven
step by step through the single-step entry points (which also gives the
GPU's routing and block inputs).  Observed statistics go to $FS_PARITY_LOG.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_expert_gb300 import configs, fs, synth
from parity import (GpuBlockRunner, HiddenFlips, TOL, compare, compare_flips, explained_drift, gpu_attn_layer,
                    gpu_attn_stepwise, gpu_stack_stepwise, oracle_cfg, oracle_weights, record, to64, topk_mismatch)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_gpu(cfg, prob, wiring):
    stack = fs.FarSkipStack(cfg, prob["blocks"], wiring=wiring)
    o, o_star = stack.forward(prob["x"])
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    assert st == 0, "device error word %d" % code
    return stack, o, o_star


_REF_CACHE = {}


def _fingerprint(prob):
    """A checksum of a problem's input and weights (position-weighted sums)."""
    ts = [prob["x"]]
    for b in prob["blocks"]:
        ts += [v for v in b.values() if v is not None]
    out = []
    for t in ts:
        f = t.detach().reshape(-1)[:1 << 20].float()
        out.append(float((f * torch.arange(1, f.numel() + 1, device=f.device, dtype=torch.float32)).sum()))
    return tuple(out)


def oracle_ref(cfg, prob, wiring, rows):
    """The oracle stack on the rows of x (with its per-block inputs and outputs);
    the last result is kept for a following test on the same problem."""
    key = (cfg, wiring, rows.tobytes(), _fingerprint(prob))
    if key not in _REF_CACHE:
        _REF_CACHE.clear()
        x = prob["x"][torch.as_tensor(rows, device=DEV)]
        _REF_CACHE[key] = oracle.stack(oracle_cfg(cfg), oracle_weights(prob["blocks"]), wiring, synth.to_numpy(x),
                                       want_inputs=True)
    return _REF_CACHE[key]


def _ref_logits(ref, b):
    """Oracle logits of block b including the router bias (the oracle adds it)."""
    return ref["logits"][b]


def blockwise(cfg, prob, blocks, wiring, rows, ref, gpu_inputs, tag=""):
    """Per-block parity on identical inputs (see module docstring).  gpu_inputs:
    the full-size GPU stack's (u_k, o_{k-1}) per block."""
    T = cfg.T
    rows_t = torch.as_tensor(rows, device=DEV)
    run = GpuBlockRunner(cfg, T)
    out = []
    for b, pw in enumerate(blocks):
        u, o_prev = gpu_inputs[b]
        u = u.clone()
        o_prev = o_prev.clone()
        if b > 0:   # splice the oracle's inputs into the checked rows
            u[rows_t] = torch.from_numpy(ref["U"][b]).to(DEV, u.dtype)
            o_prev[rows_t] = torch.from_numpy(ref["P"][b]).to(DEV, o_prev.dtype)
        o_k, o_star, _, idx = run.run(pw, u, o_prev, b == cfg.L - 1, wiring)
        bias = pw["bias"]
        bnp = None if bias is None else bias.cpu().numpy()
        z = _ref_logits(ref, b) - (0 if bnp is None else bnp.astype(np.float64)[None, :])
        bad = topk_mismatch(idx[rows], ref["topk_idx"][b], z, cfg.k, bnp)
        keep = ~bad
        st = {"block": b + 1, "tokens": int(len(rows)), "routing_near_ties": int(bad.sum())}
        if cfg.dtype == "f32":
            compare(to64(o_k[rows_t])[keep], ref["O"][b][keep], cfg.dtype, "block %d o_k" % (b + 1))
            compare(to64(o_star[rows_t])[keep], ref["OS"][b][keep], cfg.dtype, "block %d o_k*" % (b + 1))
        else:
            u16 = synth.to_numpy(torch.from_numpy(ref["U"][b]).to(torch.bfloat16))
            flips = HiddenFlips(cfg, {k_: synth.to_numpy(v) for k_, v in prob["blocks"][b].items()},
                                u16, ref["topk_idx"][b], ref["topk_w"][b])
            kept = np.nonzero(keep)[0]
            last = b == cfg.L - 1          # the last block's outputs are stored in bf16
            st["o"] = compare_flips(to64(o_k[rows_t])[keep], ref["O"][b][keep], flips, kept,
                                    "block %d o_k" % (b + 1), cfg.dtype, out_bf16=last)
            st["o_star"] = compare_flips(to64(o_star[rows_t])[keep], ref["OS"][b][keep], flips, kept,
                                         "block %d o_k*" % (b + 1), cfg.dtype, out_bf16=last)
        record("blockwise", workload=cfg.name + tag, wiring=wiring, **st)
        out.append(st)
    return out


def end_to_end(cfg, prob, o, o_star, wiring, rows, ref, routing, gpu_inputs, tag=""):
    """o, o_star: the stack's outputs over all T tokens; routing and gpu_inputs:
    the GPU's per-block routing and inputs (the stack's, through the single-step
    calls, checked bit-identical)."""
    rows_t = torch.as_tensor(rows, device=DEV)
    bad_any = np.zeros(len(rows), bool)
    drift = []
    for b in range(cfg.L):
        bias = prob["blocks"][b]["bias"]
        bnp = None if bias is None else synth.to_numpy(bias)
        z = _ref_logits(ref, b) - (0 if bnp is None else bnp.astype(np.float64)[None, :])
        if b == 0:       # identical inputs: the strict rule
            bad = topk_mismatch(routing[0][rows], ref["topk_idx"][0], z, cfg.k, bnp)
        else:
            u_g = synth.to_numpy(gpu_inputs[b][0][rows_t])
            n_bad, gmax, dmax = explained_drift(cfg, synth.to_numpy(prob["blocks"][b]["w_r"]), bnp, u_g,
                                                routing[b][rows], ref["topk_idx"][b], _ref_logits(ref, b),
                                                "block %d" % (b + 1))
            bad = np.any(np.sort(routing[b][rows], 1) != np.sort(ref["topk_idx"][b], 1), axis=1)
            drift.append({"block": b + 1, "tokens": int(bad.sum()), "max_gap": gmax, "max_delta": dmax})
        bad_any |= bad
    keep = ~bad_any
    got, got_s = to64(o[rows_t])[keep], to64(o_star[rows_t])[keep]
    st = {"tokens": int(len(rows)), "excluded": int(bad_any.sum()), "drift": drift}
    if cfg.L == 1:
        if cfg.dtype == "f32":
            compare(got, ref["o"][keep], cfg.dtype, "o_L")
            compare(got_s, ref["o_star"][keep], cfg.dtype, "o_L*")
        else:
            flips = HiddenFlips(cfg, {k_: synth.to_numpy(v) for k_, v in prob["blocks"][0].items()},
                                synth.to_numpy(prob["x"][rows_t]), ref["topk_idx"][0], ref["topk_w"][0])
            kept = np.nonzero(keep)[0]
            st["o"] = compare_flips(got, ref["o"][keep], flips, kept, "o_L", cfg.dtype, out_bf16=True)
            st["o_star"] = compare_flips(got_s, ref["o_star"][keep], flips, kept, "o_L*", cfg.dtype, out_bf16=True)
    else:
        tol = TOL[cfg.dtype]
        for g, r, what in ((got, ref["o"][keep], "o_L"), (got_s, ref["o_star"][keep], "o_L*")):
            rel = np.linalg.norm(g - r) / np.linalg.norm(r)
            st[what] = {"rel": float(rel), "max_abs_rms": float(np.abs(g - r).max() / np.sqrt(np.mean(r ** 2)))}
            assert rel <= tol["rel_fro"] * cfg.L, "%s: relative Frobenius %.3e > L x %.1e" % (
                what, rel, tol["rel_fro"])
    record("end_to_end", workload=cfg.name + tag, wiring=wiring, L=cfg.L, **st)
    return st


def _check_stack(cfg, prob, wiring, rows=None):
    stack, o, o_star = _run_gpu(cfg, prob, wiring)
    so, so_star, routing, inputs = gpu_stack_stepwise(cfg, stack.blocks, prob["x"], wiring, keep_inputs=True)
    assert torch.equal(so, o) and torch.equal(so_star, o_star), "stack driver != single-step calls"
    rows = np.arange(cfg.T) if rows is None else rows
    ref = oracle_ref(cfg, prob, wiring, rows)
    blockwise(cfg, prob, stack.blocks, wiring, rows, ref, inputs)
    end_to_end(cfg, prob, o, o_star, wiring, rows, ref, routing, inputs)
    return stack, o, o_star, ref


@pytest.mark.parametrize("wiring,L", [("partial", 3), ("outdated", 3), ("disabled", 3)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_stack_wirings(fs, wiring, L, dtype):
    # The disabled wiring feeds the whole residual back in; with random weights and
    # no normalisation the SwiGLU hidden grows like |u|^2 from block to block, and
    # its heavy tail makes a single flipped bf16 rounding of one hidden unit large
    # against the output's rms by the third block: the one-flip allowance covers
    # exactly that, and nothing else is allowed past the max-abs bound.
    cfg = configs.LayerConfig("s", T=333, d=256, E=8, k=2, c=192, n_shared=1, c_shared=128, L=L,
                              gate="softmax_renorm", dtype=dtype)
    _check_stack(cfg, synth.make_problem(cfg, DEV), wiring)


@pytest.mark.parametrize("gate,E,k,ns,zipf", [("softmax", 16, 4, 2, None), ("sigmoid", 4, 1, 1, None),
                                            ("sigmoid_norm", 32, 8, 1, None), ("softmax_renorm", 16, 4, 0, 1.2)])
def test_small_stack_gates(fs, gate, E, k, ns, zipf):
    cfg = configs.LayerConfig("g", T=520, d=192, E=E, k=k, c=128, n_shared=ns, c_shared=128 if ns else 0, L=2,
                              gate=gate, dtype="bf16", zipf_s=zipf)
    _check_stack(cfg, synth.make_problem(cfg, DEV), "partial")


def test_config_tiny_f32(fs):
    """The fp32 workload in full: L=2, T=256, d=128, E=8, top-2 renormalised softmax."""
    cfg = configs.CONFIGS["tiny_f32"]
    _check_stack(cfg, synth.make_problem(cfg, DEV), cfg.wiring)


def test_l1_wirings_agree(fs):
    cfg = configs.LayerConfig("l1", T=200, d=128, E=8, k=2, c=64, n_shared=1, c_shared=64, L=1,
                              gate="softmax_renorm", dtype="bf16")
    prob = synth.make_problem(cfg, DEV)
    outs = [_run_gpu(cfg, prob, w)[1].clone() for w in ("partial", "outdated", "disabled")]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_stack_is_deterministic(fs):
    cfg = configs.LayerConfig("det", T=1000, d=256, E=16, k=4, c=128, n_shared=1, c_shared=128, L=2,
                              gate="sigmoid_norm", dtype="bf16")
    prob = synth.make_problem(cfg, DEV)
    stack = fs.FarSkipStack(cfg, prob["blocks"])
    a = stack.forward(prob["x"])[0].clone()
    b = stack.forward(prob["x"])[0].clone()
    assert torch.equal(a, b)


# ------------------------------------------------------ full-size workloads

FULL = ["v2lite", "qwen3", "scout", "v3", "v3_decode"]
# tokens the oracle follows: None = every token, else a seeded sample
ROWS = {"v2lite": None, "qwen3": None, "scout": 2048, "v3": 2048, "v3_decode": None}
_CAP = int(os.environ.get("FS_PARITY_CAP", "0"))      # > 0: fewer rows, for quick local runs only


def parity_rows(cfg, n):
    n = cfg.T if n is None else min(n, cfg.T)
    if _CAP:
        n = min(n, _CAP)
    if n >= cfg.T:
        return np.arange(cfg.T)
    return np.sort(np.random.default_rng(0).choice(cfg.T, size=n, replace=False))


# the two-stream schedule is checked right after the one-stream run of the same
# workload, so both use one oracle computation
FULL_CASES = [("v2lite", "one_stream"), ("v2lite", "two_streams"), ("qwen3", "one_stream"), ("scout", "one_stream"),
              ("scout", "two_streams"), ("v3", "one_stream"), ("v3_decode", "one_stream")]


@pytest.mark.slow
@pytest.mark.parametrize("name,schedule", FULL_CASES)
def test_full_size_sampled(fs, name, schedule):
    """Full-size workload, one stack call over all T tokens (the benchmark's
    launch configuration); the oracle follows every token (V2-Lite, Qwen3, V3
    decode) or 2,048 sampled tokens (Scout, V3) through all L blocks.
    one_stream: fs_farskip_stack, blockwise and end to end.  two_streams: the
    FarSkip overlap schedule (fs_farskip_stack_overlap) at the shapes its overlap
    is measured on (V2-Lite L = 4, Scout L = 2), end to end against the oracle
    stack, and bit for bit against the one-stream stack."""
    cfg = configs.CONFIGS[name]
    prob = synth.make_problem(cfg, DEV)
    rows = parity_rows(cfg, ROWS[name])
    if schedule == "one_stream":
        _check_stack(cfg, prob, cfg.wiring, rows)
        return
    stack, o, o_star = _run_gpu(cfg, prob, cfg.wiring)
    o, o_star = o.clone(), o_star.clone()
    o2, o2_star = stack.forward_overlap(prob["x"])
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    _, _, routing, inputs = gpu_stack_stepwise(cfg, stack.blocks, prob["x"], cfg.wiring, keep_inputs=True)
    ref = oracle_ref(cfg, prob, cfg.wiring, rows)
    end_to_end(cfg, prob, o2, o2_star, cfg.wiring, rows, ref, routing, inputs, tag=" overlap")
    assert torch.equal(o2, o) and torch.equal(o2_star, o_star), "two-stream stack != one-stream stack"


@pytest.mark.slow
@pytest.mark.parametrize("name", ["v3", "qwen3", "v2lite", "scout"])
def test_full_size_routing_all_tokens(fs, name):
    """Block-1 routing of EVERY token at full size against the oracle's router:
    top-k sets equal except near-ties (< 1e-4), and those are < 0.1% of tokens."""
    cfg = configs.CONFIGS[name]
    x = synth.make_x(cfg, DEV)
    w = synth.make_block_weights(cfg, 0, DEV)
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    tw = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    fs.fs_router_topk(desc, x, w["w_r"], w["bias"], idx, tw, None, ws)
    torch.cuda.synchronize()
    bias = synth.to_numpy(w["bias"])
    z, ridx, rw = oracle.router(oracle_cfg(cfg), synth.to_numpy(x), synth.to_numpy(w["w_r"]), bias)
    zref = z - (0 if bias is None else bias.astype(np.float64)[None, :])
    bad = topk_mismatch(idx.cpu().numpy(), ridx, zref, cfg.k, bias)
    keep = ~bad
    gw = tw.cpu().numpy().astype(np.float64)[keep]
    # gate weights of the agreeing tokens, slot for slot (slot order = descending z)
    same_order = np.all(idx.cpu().numpy()[keep] == ridx[keep], axis=1)
    werr = float(np.abs(gw[same_order] - rw[keep][same_order]).max()) if same_order.any() else 0.0
    assert werr < 1e-5, werr
    record("routing_all_tokens", workload=name, tokens=cfg.T, near_ties=int(bad.sum()),
           slot_order_differs=int((~same_order).sum()), max_gate_weight_err=werr)


@pytest.mark.parametrize("wiring,L,dtype", [("partial", 1, "bf16"), ("partial", 3, "bf16"), ("outdated", 3, "bf16"),
                                           ("partial", 2, "f32"), ("outdated", 4, "bf16")])
def test_overlap_stack_vs_oracle(fs, wiring, L, dtype):
    """The two-stream FarSkip schedule against the oracle stack (end to end), and
    bit for bit against the one-stream stack."""
    cfg = configs.LayerConfig("ov", T=700, d=256, E=16, k=4, c=192, n_shared=1, c_shared=128, L=L,
                              gate="sigmoid_norm", dtype=dtype)
    prob = synth.make_problem(cfg, DEV)
    stack, o, o_star = _run_gpu(cfg, prob, wiring)
    o, o_star = o.clone(), o_star.clone()
    _, _, routing, inputs = gpu_stack_stepwise(cfg, stack.blocks, prob["x"], wiring, keep_inputs=True)
    rows = np.arange(cfg.T)
    ref = oracle_ref(cfg, prob, wiring, rows)
    for _ in range(2):       # twice: the second call reuses the library's events and slots
        o2, o2_star = stack.forward_overlap(prob["x"])
        torch.cuda.synchronize()
        assert fs.fs_get_error() == (0, 0)
        end_to_end(cfg, prob, o2, o2_star, wiring, rows, ref, routing, inputs, tag=" overlap")
        assert torch.equal(o2, o) and torch.equal(o2_star, o_star)


def test_overlap_stack_rejects_disabled_wiring(fs):
    cfg = configs.LayerConfig("ov", T=64, d=64, E=4, k=1, c=64, n_shared=0, c_shared=0, L=1, gate="sigmoid",
                              dtype="bf16")
    prob = synth.make_problem(cfg, DEV)
    stack = fs.FarSkipStack(cfg, prob["blocks"], wiring="disabled")
    with pytest.raises(fs.FsError):
        stack.forward_overlap(prob["x"])


# ------------------------------------------- attention/MoE wiring (FarSkip §3)

def test_attn_standin_gemm(fs):
    cfg = configs.LayerConfig("at", T=333, d=256, E=8, k=2, c=128, n_shared=0, c_shared=0, L=1, gate="softmax",
                              dtype="bf16")
    a = synth.make_x(cfg, DEV)
    w = synth.add_attention_standin([{}], cfg, DEV)[0]["w_att"]
    desc = fs.make_desc(cfg)
    ws = fs.alloc_workspace(desc, 0)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device=DEV)
    fs.fs_attn_standin(desc, a, w, out, ws)
    torch.cuda.synchronize()
    ref = oracle.attn_standin(oracle_cfg(cfg), to64(a), synth.to_numpy(w))
    rel = np.linalg.norm(to64(out) - ref) / np.linalg.norm(ref)
    assert rel < 2e-6, rel


@pytest.mark.parametrize("wiring,L,dtype", [("attn_farskip", 1, "bf16"), ("attn_farskip", 3, "bf16"),
                                           ("attn_plain", 2, "bf16"), ("attn_plain", 3, "bf16"),
                                           ("attn_farskip", 2, "f32"), ("attn_plain", 2, "f32"),
                                           ("attn_farskip", 2, "fp8"), ("attn_plain", 2, "fp8"),
                                           ("attn_farskip", 2, "mxfp8"), ("attn_plain", 2, "mxfp8")])
def test_attention_wirings_stack(fs, wiring, L, dtype):
    """fs_farskip_stack with a stand-in attention sub-block per layer vs the oracle.
    The stack is first checked bit for bit against the same layers driven through
    the single-step entry points (which gives the GPU's routing and MoE inputs).
    Per layer, on the oracle's own layer inputs (attention input, residual and
    MoE input -- for the plain layer the oracle's bf16(o_{k-1} + A_k) replaces the
    one the layer would form), routing meets the strict rule and the outputs the
    per-layer tolerance (with the one-flip allowance for bf16).  End to end: every
    routing difference explained by the input difference, L x the per-layer
    relative Frobenius bound."""
    cfg = configs.LayerConfig("aw", T=400, d=256, E=8, k=2, c=128, n_shared=1, c_shared=128, L=L,
                              gate="softmax_renorm", dtype=dtype)
    prob = synth.make_problem(cfg, DEV)
    synth.add_attention_standin(prob["blocks"], cfg, DEV)
    stack = fs.FarSkipStack(cfg, prob["blocks"], wiring=wiring)
    o, o_star = stack.forward(prob["x"])
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    so, so_star, routing, inputs = gpu_attn_stepwise(cfg, stack.blocks, prob["x"], wiring)
    assert torch.equal(so, o) and torch.equal(so_star, o_star), "stack driver != single-step calls"
    ref = oracle.stack(oracle_cfg(cfg), oracle_weights(prob["blocks"]), wiring, synth.to_numpy(prob["x"]),
                       want_inputs=True)
    wnp = [{k_: synth.to_numpy(v) for k_, v in b.items()} for b in prob["blocks"]]
    act = synth.storage_dtype(cfg)
    rtol = TOL[dtype]["rel_fro"]

    def routing_rule(b, idx, u_gpu, strict):
        if strict:
            return topk_mismatch(idx, ref["topk_idx"][b], ref["logits"][b], cfg.k)
        n_bad, gmax, dmax = explained_drift(cfg, wnp[b]["w_r"], None, synth.to_numpy(u_gpu), idx,
                                            ref["topk_idx"][b], ref["logits"][b], "layer %d" % (b + 1))
        return np.any(np.sort(idx, 1) != np.sort(ref["topk_idx"][b], 1), axis=1)

    # per layer on the oracle's layer inputs
    run = GpuBlockRunner(cfg, cfg.T)
    for b, pw in enumerate(stack.blocks):
        a_in = torch.from_numpy(ref["A"][b]).to(DEV, act)
        u_in = torch.from_numpy(ref["U"][b]).to(DEV, act)
        o_prev = torch.from_numpy(ref["P"][b]).to(DEV, act if b == 0 else torch.float32)
        o_k, o_s, idx, u_used, _, _ = gpu_attn_layer(run, pw, wiring, a_in, u_in, o_prev, b == L - 1,
                                                     u_plain=u_in if wiring == "attn_plain" else None)
        bad = routing_rule(b, idx, u_used, True)
        keep = ~bad
        if dtype == "f32":
            compare(to64(o_k)[keep], ref["O"][b][keep], dtype, "layer %d o_k" % (b + 1))
            compare(to64(o_s)[keep], ref["OS"][b][keep], dtype, "layer %d o_k*" % (b + 1))
            continue
        flips = HiddenFlips(cfg, wnp[b], synth.to_numpy(torch.from_numpy(ref["U"][b]).to(torch.bfloat16)),
                            ref["topk_idx"][b], ref["topk_w"][b])
        kept = np.nonzero(keep)[0]
        st = {"layer": b + 1, "drifted": int(bad.sum())}
        last = b == L - 1
        st["o"] = compare_flips(to64(o_k)[keep], ref["O"][b][keep], flips, kept, "layer %d o_k" % (b + 1),
                                out_bf16=last)
        st["o_star"] = compare_flips(to64(o_s)[keep], ref["OS"][b][keep], flips, kept, "layer %d o_k*" % (b + 1),
                                     out_bf16=last)
        record("attention_layer", wiring=wiring, L=L, **st)

    # end to end
    bad_any = np.zeros(cfg.T, bool)
    for b in range(L):
        bad_any |= routing_rule(b, routing[b], inputs[b], b == 0 and wiring == "attn_farskip")
    keep = ~bad_any
    st = {"excluded": int(bad_any.sum())}
    for got, want, what in ((o, ref["o"], "o_L"), (o_star, ref["o_star"], "o_L*")):
        g = to64(got)[keep]
        r = want[keep]
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        st[what] = float(rel)
        assert rel <= rtol * L, "%s: relative Frobenius %.3e" % (what, rel)
    record("attention_end_to_end", wiring=wiring, L=L, dtype=dtype, **st)


@pytest.mark.parametrize("dtype,overlap", [("bf16", False), ("bf16", True), ("fp8", False), ("fp8", True),
                                           ("mxfp8", False), ("mxfp8", True)])
def test_graph_replay_matches_eager(fs, dtype, overlap):
    """The stack captured once as a CUDA graph and replayed gives the same bits as
    the eager call, also after the input buffer is refilled."""
    cfg = configs.LayerConfig("gr", T=700, d=256, E=16, k=4, c=256, n_shared=1, c_shared=128, L=3,
                              gate="sigmoid_norm", dtype=dtype)
    prob = synth.make_problem(cfg, DEV)
    stack = fs.FarSkipStack(cfg, prob["blocks"], wiring="partial")
    x = prob["x"].clone()
    run = stack.forward_overlap if overlap else stack.forward
    run(x)
    o, o_star = (t.clone() for t in run(x))
    stack.capture(x, overlap=overlap)
    for _ in range(2):
        go, go_star = stack.replay()
        torch.cuda.synchronize()
        assert torch.equal(go, o) and torch.equal(go_star, o_star)
    x.copy_(synth.make_x(cfg.with_(seed=3), DEV))
    want = [t.clone() for t in run(x)]
    go, go_star = stack.replay()
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    assert torch.equal(go, want[0]) and torch.equal(go_star, want[1])
