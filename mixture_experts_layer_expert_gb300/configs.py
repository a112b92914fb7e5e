"""Workload registry: the MoE layer shapes the FarSkip-Collective pages evaluate.

The shapes are those of the models named in "FarSkip-Collective: Unhobbling
Blocking Communication in Mixture of Experts Models" (papercache.org summary),
§A4 (experimental setup: DeepSeek-V2-Lite, Qwen3-30B MoE, Llama-4 Scout,
DeepSeek-V3) at the batch x context sizes of its inference experiments
(32 x 2048 = 65,536 prefill tokens; a 1,024-token decode batch).
Inputs are synthetic and seeded (see ``synth.py``); no dataset is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int               # tokens
    d: int               # model dim
    E: int               # routed experts
    k: int               # top-k
    c: int               # routed expert intermediate width
    n_shared: int        # shared experts (0 = none)
    c_shared: int        # shared expert width
    L: int               # FarSkip blocks
    gate: str            # softmax | softmax_renorm | sigmoid | sigmoid_norm
    dtype: str           # "bf16" (bf16 storage, fp32 accumulate), "f32", "fp8"
                         # (bf16 storage, FP8 E4M3 expert GEMM operands with row scales)
                         # or "mxfp8" (the same with one scale per 32-element block)
    zipf_s: float | None = None   # router-bias skew (Zipf exponent) or None
    wiring: str = "partial"
    seed: int = 0

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)

    # algorithmic work per block (router + routed + shared GEMM FLOPs)
    def flops_per_block(self) -> float:
        T, d = self.T, self.d
        return (2.0 * T * d * self.E + 6.0 * T * self.k * d * self.c
                + 6.0 * T * self.n_shared * d * self.c_shared)

    def gemm_flops_per_block(self) -> float:
        """FLOPs of the grouped/dense SwiGLU GEMMs (routed + shared)."""
        T, d = self.T, self.d
        return 6.0 * T * self.k * d * self.c + 6.0 * T * self.n_shared * d * self.c_shared

    def alg_bytes_per_block(self) -> float:
        """Algorithmic HBM bytes of one block: read u and o_prev, write o* and o,
        read every expert's, the shared experts' and the router's weights once."""
        es = 4 if self.dtype == "f32" else 2
        # FP8 expert weights: one byte per element (MX: plus one scale byte per 32)
        wes = 1.0 if self.dtype == "fp8" else (1.0 + 1.0 / 32 if self.dtype == "mxfp8" else es)
        T, d = self.T, self.d
        act = 4.0 * T * d * es
        w = (3.0 * self.E * d * self.c + 3.0 * self.n_shared * d * self.c_shared) * wes + self.E * d * es
        return act + w


CONFIGS = {
    "tiny_f32": LayerConfig("tiny_f32", T=256, d=128, E=8, k=2, c=256, n_shared=1, c_shared=256,
                            L=2, gate="softmax_renorm", dtype="f32"),
    "v2lite": LayerConfig("v2lite", T=8192, d=2048, E=64, k=6, c=1408, n_shared=2, c_shared=1408,
                          L=4, gate="softmax", dtype="bf16"),
    "qwen3": LayerConfig("qwen3", T=16384, d=2048, E=128, k=8, c=768, n_shared=0, c_shared=0,
                         L=1, gate="softmax_renorm", dtype="bf16", zipf_s=1.2),
    "scout": LayerConfig("scout", T=32768, d=5120, E=16, k=1, c=8192, n_shared=1, c_shared=8192,
                         L=2, gate="sigmoid", dtype="bf16"),
    "v3": LayerConfig("v3", T=65536, d=7168, E=256, k=8, c=2048, n_shared=1, c_shared=2048,
                      L=1, gate="sigmoid_norm", dtype="bf16"),
    "v3_decode": LayerConfig("v3_decode", T=1024, d=7168, E=256, k=8, c=2048, n_shared=1,
                             c_shared=2048, L=1, gate="sigmoid_norm", dtype="bf16"),
    # DeepSeek-V3's per-expert GEMM shapes (d = 7168, c = 2048, 2048 rows per expert)
    # with 32 of its 256 experts: about 5 GB on the device, small enough for
    # multi-pass profiler captures of the headline kernels
    "v3_e32": LayerConfig("v3_e32", T=8192, d=7168, E=32, k=8, c=2048, n_shared=1, c_shared=2048,
                          L=1, gate="sigmoid_norm", dtype="bf16"),
}
# The FP8 expert path on the same shapes (the pages' inference precision).
for _name in ("v2lite", "qwen3", "scout", "v3", "v3_decode", "v3_e32"):
    CONFIGS[_name + "_fp8"] = CONFIGS[_name].with_(name=_name + "_fp8", dtype="fp8")
    # block-scaled FP8 (MX: one UE8M0 scale per 32 elements along the contraction)
    CONFIGS[_name + "_mxfp8"] = CONFIGS[_name].with_(name=_name + "_mxfp8", dtype="mxfp8")


def describe(cfg: LayerConfig) -> str:
    sh = "%dx%d shared" % (cfg.n_shared, cfg.c_shared) if cfg.n_shared else "no shared"
    return ("%s: T=%d d=%d E=%d top-%d %s c=%d %s L=%d %s%s" % (
        cfg.name, cfg.T, cfg.d, cfg.E, cfg.k, cfg.gate, cfg.c, sh, cfg.L, cfg.dtype,
        " zipf(%.1f) bias" % cfg.zipf_s if cfg.zipf_s else ""))
