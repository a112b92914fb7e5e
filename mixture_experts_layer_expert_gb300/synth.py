"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds none of the layer's arithmetic: it only draws random tensors.
Recipe (stated once here and in the design notes):
  * x ~ N(0, 1); every weight ~ N(0, 1/fan_in) with fan_in = d for W_R, W1, W2
    and fan_in = c for W3 (c_shared for the shared W3).
  * Drawn in fp32 from a torch.Generator seeded ``seed * 1000 + tensor_id`` (one
    generator per tensor, so a tensor does not depend on the others' sizes),
    then rounded to bf16 (RNE) for the bf16 workloads.
  * Router bias: zero, or for a Zipf-skewed load b_j = -s * ln(1 + pi(j)) with
    pi a seeded permutation of the experts, so exp(b_j) is proportional to the
    Zipf(s) weight of expert j's rank.
Weights are returned in the page's layout: W1 (up) and W2 (gate) [E, c, d],
W3 (down) [E, d, c]; shared experts [n_shared, c_shared, d] / [n_shared, d, c_shared].
"""
from __future__ import annotations

import math

import torch

from .configs import LayerConfig

X_ID = 0


def _ids(block: int) -> dict:
    base = 1 + 16 * block
    return {"w_r": base, "w1": base + 1, "w2": base + 2, "w3": base + 3,
            "w1s": base + 4, "w2s": base + 5, "w3s": base + 6, "bias": base + 7}


def _randn(shape, seed: int, device, scale: float, dtype: torch.dtype) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    return t.to(dtype)


def storage_dtype(cfg: LayerConfig) -> torch.dtype:
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def make_x(cfg: LayerConfig, device="cpu", T: int | None = None) -> torch.Tensor:
    T = cfg.T if T is None else T
    return _randn((T, cfg.d), cfg.seed * 1000 + X_ID, device, 1.0, storage_dtype(cfg))


def zipf_bias(E: int, s: float, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(E, generator=g)
    return torch.tensor([-s * math.log(1.0 + float(perm[j])) for j in range(E)], dtype=torch.float32)


def make_block_weights(cfg: LayerConfig, block: int, device="cpu") -> dict:
    """Weights of block `block` (0-based) in the page's layout."""
    ids = _ids(block)
    s0 = cfg.seed * 1000
    dt = storage_dtype(cfg)
    d, E, c = cfg.d, cfg.E, cfg.c
    w = {
        "w_r": _randn((E, d), s0 + ids["w_r"], device, 1.0 / math.sqrt(d), dt),
        "w1": _randn((E, c, d), s0 + ids["w1"], device, 1.0 / math.sqrt(d), dt),
        "w2": _randn((E, c, d), s0 + ids["w2"], device, 1.0 / math.sqrt(d), dt),
        "w3": _randn((E, d, c), s0 + ids["w3"], device, 1.0 / math.sqrt(c), dt),
        "bias": None,
        "w1s": None, "w2s": None, "w3s": None,
    }
    if cfg.zipf_s:
        w["bias"] = zipf_bias(E, cfg.zipf_s, s0 + ids["bias"]).to(device)
    if cfg.n_shared:
        ns, cs = cfg.n_shared, cfg.c_shared
        w["w1s"] = _randn((ns, cs, d), s0 + ids["w1s"], device, 1.0 / math.sqrt(d), dt)
        w["w2s"] = _randn((ns, cs, d), s0 + ids["w2s"], device, 1.0 / math.sqrt(d), dt)
        w["w3s"] = _randn((ns, d, cs), s0 + ids["w3s"], device, 1.0 / math.sqrt(cs), dt)
    return w


def add_attention_standin(blocks: list, cfg: LayerConfig, device="cpu") -> list:
    """Stand-in attention weights W_att [d, d] ~ N(0, 1/d) per block (attention wirings)."""
    dt = storage_dtype(cfg)
    for b, w in enumerate(blocks):
        w["w_att"] = _randn((cfg.d, cfg.d), cfg.seed * 1000 + _ids(b)["bias"] + 8, device, 1.0 / math.sqrt(cfg.d), dt)
    return blocks


def make_problem(cfg: LayerConfig, device="cpu", T: int | None = None) -> dict:
    return {"x": make_x(cfg, device, T),
            "blocks": [make_block_weights(cfg, b, device) for b in range(cfg.L)]}


def to_numpy(t: torch.Tensor | None):
    """Host copy for the oracle: bf16 as its raw uint16 bit pattern."""
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
