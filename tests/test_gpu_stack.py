"""GPU parity of the whole FarSkip stack (fs_farskip_stack through the C ABI)
against the CPU oracle: small multi-tile shapes for every wiring and gate, the
fp32 workload in full, and the full-size bf16 workloads on sampled tokens
(token rows are independent through the whole stack, so the oracle can follow
any subset of tokens through all L blocks)."""
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_expert_gb300 import configs, fs, synth
from parity import (compare, gpu_stack_stepwise, oracle_cfg, oracle_weights, routing_mismatch_all_blocks,
                    to64, topk_mismatch)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_gpu(cfg, prob, wiring):
    stack = fs.FarSkipStack(cfg, prob["blocks"], wiring=wiring)
    o, o_star = stack.forward(prob["x"])
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    assert st == 0, "device error word %d" % code
    return stack, o, o_star


def _gpu_routing(cfg, stack, u):
    """Top-k indices the GPU picks for input u with block 0's router."""
    T = u.shape[0]
    desc = fs.make_desc(cfg, T)
    ws = fs.alloc_workspace(desc, 0)
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, cfg.k), dtype=torch.float32, device=DEV)
    fs.fs_router_topk(desc, u, stack.blocks[0]["w_r"], stack.blocks[0]["bias"], idx, w, None, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy()


def _check_stack(cfg, prob, wiring):
    """fs_farskip_stack vs the oracle on every token; the same stack driven
    step by step through the single-step entry points must give identical
    bits and supplies each block's routing for the mismatch rule."""
    stack, o, o_star = _run_gpu(cfg, prob, wiring)
    so, so_star, routing = gpu_stack_stepwise(cfg, stack.blocks, prob["x"], wiring)
    assert torch.equal(so, o) and torch.equal(so_star, o_star), "stack driver != single-step calls"
    ref = oracle.stack(oracle_cfg(cfg), oracle_weights(prob["blocks"]), wiring, synth.to_numpy(prob["x"]))
    bad, stats = routing_mismatch_all_blocks(cfg, routing, ref, prob["blocks"])
    keep = ~bad
    compare(to64(o)[keep], ref["o"][keep], cfg.dtype, "o_L")
    compare(to64(o_star)[keep], ref["o_star"][keep], cfg.dtype, "o_L*")
    return ref


@pytest.mark.parametrize("wiring", ["partial", "outdated", "disabled"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_stack_wirings(fs, wiring, dtype):
    cfg = configs.LayerConfig("s", T=333, d=256, E=8, k=2, c=192, n_shared=1, c_shared=128, L=3,
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
SAMPLE = int(os.environ.get("FS_PARITY_SAMPLE", "128"))


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(fs, name):
    """Full-size workload, in the launch configuration the benchmark times
    (one fs_farskip_stack call over all T tokens); the oracle follows a seeded
    sample of tokens through all L blocks, and block-1 routing of every token
    is checked against the oracle's router."""
    cfg = configs.CONFIGS[name]
    prob = synth.make_problem(cfg, DEV)
    stack, o, o_star = _run_gpu(cfg, prob, cfg.wiring)
    g = np.random.default_rng(0)
    rows = np.sort(g.choice(cfg.T, size=min(SAMPLE, cfg.T), replace=False))
    x_s = prob["x"][torch.as_tensor(rows, device=DEV)]
    ref = oracle.stack(oracle_cfg(cfg), oracle_weights(prob["blocks"]), cfg.wiring, synth.to_numpy(x_s))
    _, _, routing = gpu_stack_stepwise(cfg, stack.blocks, x_s, cfg.wiring)
    bad, stats = routing_mismatch_all_blocks(cfg, routing, ref, prob["blocks"])
    keep = ~bad
    rows_t = torch.as_tensor(rows, device=DEV)
    compare(to64(o[rows_t])[keep], ref["o"][keep], cfg.dtype, name + " o_L")
    compare(to64(o_star[rows_t])[keep], ref["o_star"][keep], cfg.dtype, name + " o_L*")
