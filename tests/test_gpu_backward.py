"""GPU parity of the MoE stack's backward (fs_farskip_stack_train +
fs_farskip_stack_backward) against the oracle's backward, on the same seeded
inputs and output gradients.

The backward's stored operands are bf16 on both sides at the same points (dy,
dg/da, the per-slot dx, dS, dz) and every sum is fp32 (GPU) / fp64 (oracle),
so the two sides differ by accumulation order and by bf16 rounding flips of
stored values, compounded through the L blocks.  Bounds: relative Frobenius
<= L x 5e-3 (the end-to-end forward bound) for the input gradient and for every weight gradient, computed
over the tokens whose routing agrees in every block (near-ties are counted
and explained as in the forward: block 1 routes identical inputs, and a later
block may route a token differently only where the bf16 difference of its
input explains it); a weight gradient sums over all tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_expert_gb300 import configs, fs, synth
from parity import explained_drift, gpu_stack_stepwise, oracle_cfg, oracle_weights, record, to64, topk_mismatch

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL = 5e-3
KEYS = ("dW_R", "dW1", "dW2", "dW3", "dW1s", "dW2s", "dW3s")


def routing_agrees(cfg, blocks, routing, inputs, fwd, rows):
    """Tokens (of `rows`) routed the same in every block by the GPU stack (routing,
    inputs: per block over all T tokens) and the oracle forward on those rows:
    block 1 under the strict near-tie rule, later blocks with every difference
    explained by the input difference (explained_drift)."""
    rows_t = torch.as_tensor(rows, device=DEV)
    same = np.ones(len(rows), bool)
    for b in range(cfg.L):
        bias = blocks[b]["bias"]
        bnp = None if bias is None else synth.to_numpy(bias)
        if b == 0:
            z = fwd["logits"][0] - (0 if bnp is None else bnp.astype(np.float64)[None, :])
            bad = topk_mismatch(routing[0][rows], fwd["topk_idx"][0], z, cfg.k, bnp)
        else:
            explained_drift(cfg, synth.to_numpy(blocks[b]["w_r"]), bnp, synth.to_numpy(inputs[b][0][rows_t]),
                            routing[b][rows], fwd["topk_idx"][b], fwd["logits"][b], "block %d" % (b + 1))
            bad = np.any(np.sort(routing[b][rows], 1) != np.sort(fwd["topk_idx"][b], 1), axis=1)
        same &= ~bad
    return same


def _run(cfg, wiring, seed=5, mutate=None):
    prob = synth.make_problem(cfg, DEV)
    if mutate is not None:
        mutate(prob)
    x = prob["x"]
    tr = fs.FarSkipTrainer(cfg, prob["blocks"], wiring=wiring)
    o, o_star = tr.forward(x)
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    ref_o, ref_os, routing, inputs = gpu_stack_stepwise(cfg, tr.blocks, x, wiring, keep_inputs=True)
    assert torch.equal(o, ref_o) and torch.equal(o_star, ref_os), "training forward != inference forward"
    g = torch.Generator(device=DEV).manual_seed(seed)
    dO = torch.randn((cfg.T, cfg.d), generator=g, device=DEV)
    dOs = torch.randn((cfg.T, cfg.d), generator=g, device=DEV)
    dx, grads = tr.backward(dO, dOs)
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    ref = oracle.stack_backward(oracle_cfg(cfg), oracle_weights(prob["blocks"]), wiring, synth.to_numpy(x),
                                to64(dO), to64(dOs))
    fwd = oracle.stack(oracle_cfg(cfg), oracle_weights(prob["blocks"]), wiring, synth.to_numpy(x))
    same = routing_agrees(cfg, prob["blocks"], routing, inputs, fwd, np.arange(cfg.T))
    bound = REL * cfg.L
    got = to64(dx)[same]
    want = ref["dx"][same]
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    stats = {"dx": rel}
    assert rel <= bound, "dx: relative Frobenius %.3e > %.1e" % (rel, bound)
    for b in range(cfg.L):
        for key in KEYS:
            if key not in grads[b]:
                continue
            gw = to64(grads[b][key])
            rw = ref[key][b]
            r = np.linalg.norm(gw - rw) / max(np.linalg.norm(rw), 1e-30)
            stats["%s[%d]" % (key, b)] = r
            assert r <= bound, "block %d %s: relative Frobenius %.3e > %.1e" % (b + 1, key, r, bound)
    record("backward", workload=cfg.name, wiring=wiring, L=cfg.L, excluded=int((~same).sum()), **stats)
    print("backward parity", cfg.name, wiring, {k: "%.2e" % v for k, v in stats.items()})
    return stats


@pytest.mark.parametrize("gate", ["sigmoid_norm", "softmax", "softmax_renorm", "sigmoid"])
def test_block_backward_gates(fs, gate):
    cfg = configs.LayerConfig("bw", T=300, d=256, E=8, k=2, c=128, n_shared=1, c_shared=128, L=1, gate=gate,
                              dtype="bf16")
    _run(cfg, "partial")


@pytest.mark.parametrize("wiring", ["partial", "outdated", "disabled"])
def test_stack_backward_wirings(fs, wiring):
    L = 3
    cfg = configs.LayerConfig("bws", T=333, d=256, E=8, k=2, c=192, n_shared=2, c_shared=128, L=L,
                              gate="softmax_renorm", dtype="bf16")
    _run(cfg, wiring)


def test_backward_multi_tile_ragged(fs):
    """Several M/N tiles, ragged expert segments (the last 64-row K block of each
    expert's weight-gradient contraction partly filled), 16 experts, top-4."""
    cfg = configs.LayerConfig("bwm", T=1000, d=384, E=16, k=4, c=256, n_shared=1, c_shared=256, L=2,
                              gate="sigmoid_norm", dtype="bf16")
    _run(cfg, "partial")


def test_backward_skewed_routing_and_small_E(fs):
    """Zipf-skewed router bias (experts with few or no rows; empty segments
    give zero gradients), E = 16 < 64 (padded router operands), top-1, no shared."""
    cfg = configs.LayerConfig("bwz", T=520, d=192, E=16, k=1, c=128, n_shared=0, c_shared=0, L=2,
                              gate="sigmoid", dtype="bf16", zipf_s=1.2)
    _run(cfg, "outdated")


@pytest.mark.parametrize("T", [1, 15, 16, 64, 65, 130])
def test_backward_exact_segment_lengths(fs, T):
    """A router bias that sends every token to experts 0 and 1 (top-2 of 8), so
    both experts' row segments are exactly T long and the other six are empty.
    The weight-gradient contractions then see a lone row, a block ending one row
    short of a 16-row MMA step, whole steps, one whole 64-row block, one row into
    a second block, and two rows after two full blocks; the shared expert's and
    the router's contractions run over the same T rows."""
    cfg = configs.LayerConfig("bwt", T=T, d=256, E=8, k=2, c=128, n_shared=1, c_shared=128, L=2,
                              gate="softmax_renorm", dtype="bf16")

    def force(prob):
        for w in prob["blocks"]:
            b = torch.zeros(cfg.E, device=DEV)
            b[0], b[1] = 30.0, 29.0
            w["bias"] = b

    _run(cfg, "partial", mutate=force)


def _saved_offsets_at(cfg):
    """Byte offset of block 1's expert offsets inside the training state: u, logits,
    routing indices and weights come first, each region 256-byte aligned."""
    up = lambda n: (n + 255) // 256 * 256
    T, rows = cfg.T, cfg.T * cfg.k
    return up(T * cfg.d * 2) + up(T * cfg.E * 4) + up(rows * 4) + up(rows * 4)


def test_backward_corrupt_offsets_sets_error(fs):
    """Expert offsets in the training state made inconsistent on the host before
    the backward: the plans and the weight-gradient GEMM record DEV_ERR_OFFSETS
    (code 2) and treat every expert as empty (routed weight gradients all zero);
    the next forward rewrites the offsets and the backward is correct again."""
    cfg = configs.LayerConfig("bwo", T=300, d=256, E=8, k=2, c=128, n_shared=1, c_shared=128, L=1,
                              gate="sigmoid_norm", dtype="bf16")
    prob = synth.make_problem(cfg, DEV)
    tr = fs.FarSkipTrainer(cfg, prob["blocks"])
    tr.forward(prob["x"])
    torch.cuda.synchronize()
    at = _saved_offsets_at(cfg)
    offs = tr.saved[at:at + 4 * (cfg.E + 1)].view(torch.int32)
    want = offs.clone()
    assert int(want[0]) == 0 and int(want[-1]) == cfg.T * cfg.k and bool((want[1:] >= want[:-1]).all())
    offs[1] = want[2] + 1                 # offsets[1] > offsets[2]
    g = torch.Generator(device=DEV).manual_seed(2)
    dO = torch.randn((cfg.T, cfg.d), generator=g, device=DEV)
    _, grads = tr.backward(dO)
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (5, 2)
    for key in ("dW1", "dW2", "dW3"):
        assert not grads[0][key].any(), key
    _run(cfg, "partial")                  # a fresh trainer: the error word is clear and parity holds


# ------------------------------------------------------ full-size workloads

# sampled tokens per workload: the oracle's backward costs about three forwards per
# token, so the sample is sized to keep the GPU suite within its time budget
# (Qwen3, the cheapest, at 1,024 tokens with every weight gradient compared)
SAMPLE_BWD = {"v2lite": 512, "qwen3": 1024, "scout": 256, "v3": 512}


@pytest.mark.slow
@pytest.mark.parametrize("name,grads", [("v2lite", False), ("qwen3", True), ("scout", False), ("v3", False)])
def test_full_size_backward_sampled(fs, name, grads):
    """The full-size training step (one forward call keeping state, one backward
    call) with output gradients nonzero only on a seeded sample of tokens.  Token
    rows are independent through the stack, so dx of the sampled rows -- and,
    where the oracle's weight-gradient arrays fit in host memory, every weight
    gradient -- equal the oracle's on the sample alone, and dx of every other
    token is exactly zero."""
    cfg = configs.CONFIGS[name]
    prob = synth.make_problem(cfg, DEV)
    x = prob["x"]
    tr = fs.FarSkipTrainer(cfg, prob["blocks"])
    tr.forward(x)
    g = np.random.default_rng(1)
    rows = np.sort(g.choice(cfg.T, size=SAMPLE_BWD[name], replace=False))
    rows_t = torch.as_tensor(rows, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(9)
    dO = torch.zeros((cfg.T, cfg.d), device=DEV)
    dOs = torch.zeros((cfg.T, cfg.d), device=DEV)
    dO[rows_t] = torch.randn((len(rows), cfg.d), generator=gen, device=DEV)
    dOs[rows_t] = torch.randn((len(rows), cfg.d), generator=gen, device=DEV)
    dx, gr = tr.backward(dO, dOs)
    torch.cuda.synchronize()
    assert fs.fs_get_error() == (0, 0)
    others = torch.ones(cfg.T, dtype=torch.bool, device=DEV)
    others[rows_t] = False
    assert not dx[others].any(), "nonzero input gradient outside the sampled tokens"
    xs = x[rows_t]
    _, _, routing, inputs = gpu_stack_stepwise(cfg, tr.blocks, x, cfg.wiring, keep_inputs=True)
    ocfg, ow = oracle_cfg(cfg), oracle_weights(prob["blocks"])
    fwd = oracle.stack(ocfg, ow, cfg.wiring, synth.to_numpy(xs))
    same = routing_agrees(cfg, prob["blocks"], routing, inputs, fwd, rows)
    ref = oracle.stack_backward(ocfg, ow, cfg.wiring, synth.to_numpy(xs), to64(dO[rows_t]), to64(dOs[rows_t]),
                                want_grads=grads and same.all())
    bound = REL * cfg.L
    got, want = to64(dx[rows_t])[same], ref["dx"][same]
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel <= bound, "dx: relative Frobenius %.3e > %.1e" % (rel, bound)
    stats = {"dx": rel}
    if grads and same.all():
        for b in range(cfg.L):
            for key in KEYS:
                if key not in gr[b]:
                    continue
                rw = ref[key][b]
                r = np.linalg.norm(to64(gr[b][key]) - rw) / max(np.linalg.norm(rw), 1e-30)
                stats["%s[%d]" % (key, b)] = r
                assert r <= bound, "block %d %s: relative Frobenius %.3e > %.1e" % (b + 1, key, r, bound)
    record("backward_full_size", workload=name, tokens=len(rows), excluded=int((~same).sum()), **stats)
    print("full-size backward parity", name, {k: "%.2e" % v for k, v in stats.items()})
