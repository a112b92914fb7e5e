"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare within the tolerances
of the workload definition:
  bf16 storage / fp32 accumulate : relative Frobenius <= 5e-3 and
                                   max-abs <= 2e-2 * rms(reference), per element
                                   plus the one-flip allowance where a stored
                                   value's rounding flipped (see the rounding-flips
                                   note below)
  fp32                           : relative Frobenius <= 1e-5
  FP8 experts                    : the bf16 bounds with the E4M3 flip step.  Both
                                   sides quantise the same bf16 values with the
                                   same rule, the E4M3 products are exact in fp32,
                                   so what is left is accumulation order plus
                                   rare one-quantum flips.
  routing                        : top-k sets equal except where the k-th and
                                   (k+1)-th oracle logits differ by < 1e-4;
                                   such tokens must be < 0.1% and are left
                                   out of the output comparison.  In a later
                                   block of a stack, where the two sides' inputs
                                   differ by rounding, every differing token must
                                   be explained by that input difference
                                   (explained_drift).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from mixture_experts_layer_expert_gb300 import synth

TOL = {"bf16": dict(rel_fro=5e-3, max_abs_rms=2e-2), "f32": dict(rel_fro=1e-5, max_abs_rms=1e-4)}
TOL["fp8"] = TOL["bf16"]
TOL["mxfp8"] = TOL["bf16"]
GAP = 1e-4
MISMATCH_FRAC = 1e-3


def oracle_cfg(cfg, storage=True):
    dt = oracle.F32 if cfg.dtype == "f32" else oracle.BF16
    st = (oracle.STORE_F32 if cfg.dtype == "f32" else oracle.STORE_BF16) if storage else oracle.EXACT
    return oracle.make_cfg(cfg.d, cfg.E, cfg.k, cfg.c, cfg.n_shared, cfg.c_shared, cfg.gate, dt, st,
                           fp8={"fp8": "row", "mxfp8": "mx"}.get(cfg.dtype, False))


def oracle_weights(blocks):
    return [oracle.Weights(**{k: synth.to_numpy(v) for k, v in b.items()}) for b in blocks]



def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    tol = TOL[dtype]
    err = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / max(nref, 1e-300)
    rms = nref / np.sqrt(max(ref.size, 1))
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= tol["rel_fro"], "%s: relative Frobenius %.3e > %.1e" % (what, rel, tol["rel_fro"])
    assert mx <= tol["max_abs_rms"] * rms + 1e-30, "%s: max-abs %.3e > %.1e * rms (%.3e)" % (
        what, mx, tol["max_abs_rms"], rms)
    return rel, mx / max(rms, 1e-300)


# -------------------------------------------------------- rounding flips
# Both sides round the stored hidden h (bf16; FP8: then quantised to E4M3 per
# row) and each stored routed output y (bf16) with the same rule, but they round
# different pre-rounding values: fp32 sums (tensor cores) against fp64 sums
# (oracle).  Where the two straddle a rounding boundary the stored values differ
# by one step -- the storage analogue of a routing near-tie.  One step is at most
# 2^-7 of the value for bf16 (8 significant bits) and 2^-3 for E4M3 (3 mantissa
# bits), so one flipped hidden unit j changes output element i by at most
# w_s step |h_j| |W3[i, j]| and one flipped routed output by w_s 2^-7 |y_i|.  An
# outlier h_j (SwiGLU products are heavy-tailed, and grow with the block input)
# can make that exceed 2e-2 rms by itself.  Outputs therefore meet: relative
# Frobenius <= 5e-3 overall, and per element max-abs <= 2e-2 rms plus the
# largest such one-flip change feeding that element; elements beyond that
# (several flips at once, or an FP8 row whose scale exponent flipped) are
# counted per token and must be < 0.1% of tokens (one token in samples under
# 1,000).
BF16_STEP = 2.0 ** -7
FP8_STEP = 2.0 ** -3
W3_Q = 1.0 + 2.0 ** -4          # |W3| dequantised is within one half-step of the bf16 weight


def _bf16_to_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def allowed_tokens(n: int) -> int:
    """Tokens allowed past a < 0.1% rule: one in samples under 1,000."""
    return max(1, int(MISMATCH_FRAC * n))


class HiddenFlips:
    """One-flip allowances of a block's outputs for its token rows u (bf16 as
    uint16), routing (topk_idx, topk_w) and numpy weights `w` (page layout)."""

    def __init__(self, cfg, w: dict, u: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray):
        self.cfg, self.w, self.u, self.idx, self.tw = cfg, w, u, topk_idx, topk_w
        self.fp8 = cfg.dtype in ("fp8", "mxfp8")
        self.step = FP8_STEP if self.fp8 else BF16_STEP
        self.q = W3_Q if self.fp8 else 1.0
        self.oc = oracle_cfg(cfg)
        self._w3 = _bf16_to_f64(w["w3"])
        if cfg.n_shared:
            ns, cs, d = cfg.n_shared, cfg.c_shared, cfg.d
            self._w3cat_raw = np.ascontiguousarray(np.concatenate([w["w3s"][s] for s in range(ns)], axis=1))
            self._w3cat = _bf16_to_f64(self._w3cat_raw)
            self._w13s = (w["w1s"].reshape(1, ns * cs, d), w["w2s"].reshape(1, ns * cs, d))
            self._oc1 = oracle.make_cfg(d, 1, 1, ns * cs, 0, 0, cfg.gate, self.oc.in_dtype, self.oc.storage,
                                        fp8=self.oc.fp8)
        self._cache = {}

    def _token(self, t):
        if t not in self._cache:
            k = self.cfg.k
            rows = np.ascontiguousarray(np.repeat(self.u[t:t + 1], k, axis=0))
            h, y = oracle.expert_rows(self.oc, rows, self.idx[t].astype(np.int32), self.w["w1"], self.w["w2"],
                                      self.w["w3"])
            hs = None
            if self.cfg.n_shared:
                hs, _ = oracle.expert_rows(self._oc1, np.ascontiguousarray(self.u[t:t + 1]), np.zeros(1, np.int32),
                                           self._w13s[0], self._w13s[1], self._w3cat_raw[None])
            self._cache[t] = (np.abs(h), np.abs(y), None if hs is None else np.abs(hs[0]))
        return self._cache[t]

    def allowance(self, t: int, i: int) -> float:
        h, y, hs = self._token(t)
        a = 0.0
        for s in range(self.cfg.k):
            e = int(self.idx[t, s])
            ws = abs(float(self.tw[t, s]))
            a = max(a, ws * self.step * self.q * float(np.max(h[s] * np.abs(self._w3[e, i]))),
                    ws * BF16_STEP * float(y[s, i]))
        if hs is not None:
            a = max(a, self.step * self.q * float(np.max(hs * np.abs(self._w3cat[i]))))
        return a


Fp8Flips = HiddenFlips


def compare_flips(got: np.ndarray, ref: np.ndarray, flips: HiddenFlips, tokens: np.ndarray, what: str = "",
                  dtype: str = "bf16", out_bf16: bool = False):
    """Outputs [n, d] against the oracle with the one-flip allowance (see the
    rounding-flips note above); tokens[r] = the token of row r in the flips'
    inputs.  out_bf16: the GPU's output is itself stored in bf16 (a stack's last
    block) while the oracle returns it at residual precision, so each element
    also carries its own rounding, half a bf16 step: 2^-9 |ref| (for a
    heavy-tailed residual an element 10x the rms rounds by 0.02 rms on its own).
    Returns a dict of what was seen."""
    tol = TOL[dtype]
    err = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / max(nref, 1e-300)
    rms = nref / np.sqrt(max(ref.size, 1))
    assert rel <= tol["rel_fro"], "%s: relative Frobenius %.3e > %.1e" % (what, rel, tol["rel_fro"])
    base = tol["max_abs_rms"] * rms + (2.0 ** -9 * np.abs(ref) if out_bf16 else 0.0)
    over = np.argwhere(np.abs(err) > base)
    unexplained = set()
    for r, i in over:
        if r in unexplained:
            continue
        b = base[r, i] if out_bf16 else base
        if abs(err[r, i]) > b + flips.allowance(int(tokens[r]), int(i)):
            unexplained.add(int(r))
    n = got.shape[0]
    assert len(unexplained) <= allowed_tokens(n), (
        "%s: %d of %d tokens beyond max-abs + one-flip allowance" % (what, len(unexplained), n))
    mx = float(np.abs(err).max() / max(rms, 1e-300)) if err.size else 0.0
    return dict(rel=float(rel), max_abs_rms=mx, elems_over=int(len(over)),
                tokens_over=int(len(set(int(r) for r, _ in over))), unexplained=len(unexplained))


def compare_fp8(got, ref, flips, tokens, what=""):
    st = compare_flips(got, ref, flips, tokens, what, "fp8")
    return st["rel"], st["elems_over"], st["unexplained"]


# ------------------------------------------------------------- parity log
def record(kind: str, **fields):
    """Append one JSON line of observed parity statistics to $FS_PARITY_LOG
    (when set): the numbers behind the tolerances' headroom."""
    path = os.environ.get("FS_PARITY_LOG")
    if not path:
        return
    entry = {"kind": kind}
    for k_, v in fields.items():
        if isinstance(v, (np.floating, np.integer)):
            v = v.item()
        entry[k_] = v
    with open(path, "a") as f:
        f.write(json.dumps(entry) + "\n")


def kth_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Gap between the k-th and (k+1)-th largest logits per row (inf when k = E)."""
    E = logits.shape[1]
    if k >= E:
        return np.full(logits.shape[0], np.inf)
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]


def topk_mismatch(gpu_idx: np.ndarray, ref_idx: np.ndarray, ref_logits: np.ndarray, k: int, bias=None):
    """Tokens whose top-k SET differs.  Asserts every such token has an oracle
    k-th/(k+1)-th gap < 1e-4 and that they are < 0.1% of tokens.  Returns the
    boolean mask of mismatched tokens."""
    z = ref_logits if bias is None else ref_logits + bias[None, :].astype(np.float64)
    a = np.sort(gpu_idx, axis=1)
    b = np.sort(ref_idx, axis=1)
    bad = np.any(a != b, axis=1)
    if bad.any():
        gaps = kth_gap(z[bad], k)
        assert np.all(gaps < GAP), "top-k differs on tokens with gap >= 1e-4: %s" % gaps[gaps >= GAP][:5]
        assert bad.sum() <= allowed_tokens(len(bad)), "top-k mismatch on %d of %d tokens" % (
            int(bad.sum()), len(bad))
    return bad


class GpuBlockRunner:
    """One FarSkip block driven through the single-step C-ABI entry points
    (router, dispatch, routed experts, shared expert, combine) with buffers
    for T tokens; the same launch sequence fs_farskip_stack issues."""

    def __init__(self, cfg, T, DEV="cuda"):
        from mixture_experts_layer_expert_gb300 import fs
        self.fs, self.cfg, self.T, self.dev = fs, cfg, T, DEV
        d, k, E = cfg.d, cfg.k, cfg.E
        self.desc = fs.make_desc(cfg, T)
        self.ws = fs.alloc_workspace(self.desc, 0)
        self.dt = synth.storage_dtype(cfg)
        i32 = dict(dtype=torch.int32, device=DEV)
        self.idx = torch.empty((T, k), **i32)
        self.w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        self.counts, self.offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
        self.pos, self.perm = torch.empty(T * k, **i32), torch.empty(fs.fs_dispatch_rows(self.desc), **i32)
        prow = fs.fs_dispatch_rows(self.desc)          # T k, or the MX path's padded capacity
        if cfg.dtype == "fp8":
            self.x_perm = fs.fp8_rows_empty(T * k, d, DEV)
        elif cfg.dtype == "mxfp8":
            self.x_perm = fs.mx_rows_empty(prow, d, DEV)
        else:
            self.x_perm = torch.empty((T * k, d), dtype=self.dt, device=DEV)
        self.y_perm = torch.empty((prow, d), dtype=self.dt, device=DEV)
        self.s = torch.empty((T, d), dtype=torch.float32, device=DEV) if cfg.n_shared else None

    def run(self, pw, u, o_prev, last, wiring):
        """Returns (o_k, o_k*, u_next or None, topk_idx numpy)."""
        fs, T, d = self.fs, self.T, self.cfg.d
        fs.fs_router_topk(self.desc, u, pw["w_r"], pw["bias"], self.idx, self.w, None, self.ws)
        idx = self.idx.cpu().numpy().copy()
        fs.fs_dispatch(self.desc, self.idx, u, self.counts, self.offsets, self.pos, self.perm, self.x_perm, self.ws)
        fs.fs_grouped_swiglu(self.desc, self.x_perm, self.offsets, pw["w13"], pw["w3"], self.y_perm, self.ws)
        if self.s is not None:
            fs.fs_shared_expert(self.desc, u, pw["w13_shared"], pw["w3_shared"], self.s, self.ws)
        rdt = self.dt if last else torch.float32          # fp32 residual stream between blocks
        o_k = torch.empty((T, d), dtype=rdt, device=self.dev)
        o_star = torch.empty((T, d), dtype=rdt, device=self.dev)
        u_next = None if last else torch.empty((T, d), dtype=self.dt, device=self.dev)
        fs.fs_combine(self.desc, self.y_perm, self.pos, self.w, o_prev, self.s, o_star, o_k, u_next, wiring)
        torch.cuda.synchronize()
        return o_k, o_star, u_next, idx


def gpu_stack_stepwise(cfg, packed_blocks, x, wiring, DEV="cuda", keep_inputs=False):
    """The FarSkip stack driven from Python through the single-step entry
    points, keeping each block's routing (and, with keep_inputs, its inputs
    u_k and o_{k-1}).  Returns (o_L, o_L*, [topk_idx per block], [(u, o_prev)])."""
    run = GpuBlockRunner(cfg, x.shape[0], DEV)
    u, o_prev = x, x
    routing, inputs = [], []
    o_k = o_star = None
    L = len(packed_blocks)
    for b, pw in enumerate(packed_blocks):
        if keep_inputs:
            inputs.append((u, o_prev))
        o_k, o_star, u_next, idx = run.run(pw, u, o_prev, b == L - 1, wiring)
        routing.append(idx)
        u, o_prev = u_next, o_k
    return o_k, o_star, routing, inputs


def explained_drift(cfg, w_r, bias, u_gpu: np.ndarray, gpu_idx: np.ndarray, ref_idx: np.ndarray,
                    ref_logits: np.ndarray, what: str = ""):
    """Routing of a block whose GPU input differs from the oracle's (a later
    block of a stack, where the bf16 block inputs differ by rounding flips of the
    residual).  A token may route differently only if that input difference can
    close its oracle k-th/(k+1)-th logit gap: with z_o the oracle's logits on its
    own input and z_g the oracle's logits on the GPU's input u_gpu (bf16 rows as
    uint16), a swap of a chosen and an unchosen expert needs
        gap(z_o) < 2 max_j |z_g[j] - z_o[j]| + 1e-4
    (the 1e-4 being the GPU's own fp32 logits against fp64 on identical inputs).
    Every differing token must meet this; returns (count, the largest gap and the
    largest perturbation among them).  ref_logits include the bias."""
    bad = np.any(np.sort(gpu_idx, 1) != np.sort(ref_idx, 1), axis=1)
    n_bad = int(bad.sum())
    if n_bad == 0:
        return 0, 0.0, 0.0
    z_o = ref_logits[bad]
    z_g, _, _ = oracle.router(oracle_cfg(cfg), np.ascontiguousarray(u_gpu[bad]), w_r, bias)
    delta = np.abs(z_g - z_o).max(axis=1)
    gaps = kth_gap(z_o, cfg.k)
    ok = gaps < 2.0 * delta + GAP
    assert ok.all(), "%s: routing differs on tokens the input perturbation does not explain: gaps %s, 2 delta %s" % (
        what, gaps[~ok][:5], 2.0 * delta[~ok][:5])
    return n_bad, float(gaps.max()), float(delta.max())


def gpu_attn_layer(run, pw, wiring, a_in, u, o_prev, last, u_plain=None):
    """One layer of the attention-wiring stack (FS_WIRE_ATTN_FARSKIP / _PLAIN)
    through the single-step entry points, as fs_farskip_stack runs it: the
    stand-in attention A_k on the attention input a_in, then the MoE block on
    the MoE input u (farskip) or on u = bf16(h_k), h_k = o_prev + A_k(a_in)
    (plain; that fp32 add and its bf16 rounding are formed here with torch --
    the same single IEEE roundings as the library's kernel, which the caller
    checks against fs_farskip_stack bit for bit); u_plain, when given, replaces
    the plain layer's bf16(h_k) as the MoE input (a per-layer check on the
    oracle's own MoE input).  Returns (o_k, o_k*, topk_idx numpy, the MoE input
    u, next attention input, next MoE input)."""
    fs, cfg, T, d, dt = run.fs, run.cfg, run.T, run.cfg.d, run.dt
    att = torch.empty((T, d), dtype=torch.float32, device=run.dev)
    fs.fs_attn_standin(run.desc, a_in, pw["w_att"], att, run.ws)
    base, extra = o_prev, att
    if wiring == "attn_plain":
        base = o_prev.float() + att
        u = base.to(dt) if u_plain is None else u_plain
        extra = None
    fs.fs_router_topk(run.desc, u, pw["w_r"], pw["bias"], run.idx, run.w, None, run.ws)
    idx = run.idx.cpu().numpy().copy()
    fs.fs_dispatch(run.desc, run.idx, u, run.counts, run.offsets, run.pos, run.perm, run.x_perm, run.ws)
    fs.fs_grouped_swiglu(run.desc, run.x_perm, run.offsets, pw["w13"], pw["w3"], run.y_perm, run.ws)
    if run.s is not None:
        fs.fs_shared_expert(run.desc, u, pw["w13_shared"], pw["w3_shared"], run.s, run.ws)
    rdt = dt if last else torch.float32
    o_k = torch.empty((T, d), dtype=rdt, device=run.dev)
    o_star = torch.empty((T, d), dtype=rdt, device=run.dev)
    a_next = None if last else torch.empty((T, d), dtype=dt, device=run.dev)
    u_next = None if last or wiring == "attn_plain" else torch.empty((T, d), dtype=dt, device=run.dev)
    if wiring == "attn_farskip":
        # next attention input bf16(o_k*) = bf16(o_k - R_k), next MoE input bf16(o_k)
        fs.fs_combine(run.desc, run.y_perm, run.pos, run.w, base, run.s, o_star, o_k, a_next, "partial",
                      extra=extra, u_full=u_next)
    else:
        fs.fs_combine(run.desc, run.y_perm, run.pos, run.w, base, run.s, o_star, o_k, None, "partial",
                      u_full=a_next)
    torch.cuda.synchronize()
    return o_k, o_star, idx, u, a_next, u_next


def gpu_attn_stepwise(cfg, packed_blocks, x, wiring, DEV="cuda"):
    """The attention-wiring stack layer by layer (gpu_attn_layer).  Returns
    (o_L, o_L*, [topk_idx per layer], [MoE input u_k per layer])."""
    run = GpuBlockRunner(cfg, x.shape[0], DEV)
    a_in, u, o_prev = x, x, x
    routing, inputs = [], []
    o_k = o_star = None
    L = len(packed_blocks)
    for b, pw in enumerate(packed_blocks):
        o_k, o_star, idx, u_used, a_in, u = gpu_attn_layer(run, pw, wiring, a_in, u, o_prev, b == L - 1)
        routing.append(idx)
        inputs.append(u_used)
        o_prev = o_k
    return o_k, o_star, routing, inputs
