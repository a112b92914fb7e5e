"""CPU oracle for the FarSkip-Collective MoE layer stack -- TEST INFRASTRUCTURE.

A ctypes wrapper around ``oracle.c`` (plain C, fp64 accumulation).  Only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
arm may import this package.  It imports nothing from the CUDA library and the
library imports nothing from it.

Every function takes numpy arrays.  bf16 tensors are passed as ``uint16`` arrays
(the raw bit patterns) together with ``dtype="bf16"``.

Source of the formulas: "FarSkip-Collective: Unhobbling Blocking Communication
in Mixture of Experts Models" (papercache.org summary), §2.1 (MLP and MoE
equations, Dispatch/Combine) and §3 (FarSkip equation, eq. 8a/8b).  The readings
taken where the page is silent are stated in ``oracle.c``.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, hand-derived golden values, brute force, reductions to a dense
MLP, invariants).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
EXACT, STORE_BF16, STORE_F32 = 0, 1, 2
GATES = {"softmax": 0, "softmax_renorm": 1, "sigmoid": 2, "sigmoid_norm": 3}
WIRINGS = {"partial": 0, "outdated": 1, "disabled": 2, "attn_farskip": 3, "attn_plain": 4}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (OpenMP over tokens).  Returns its path."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or any(
            os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
        if force or stale:
            tmp = _LIB + ".%d.tmp" % os.getpid()
            subprocess.check_call(["gcc", "-O2", "-fopenmp", "-std=c11", "-shared", "-fPIC",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("d", "E", "k", "c", "n_shared", "c_shared", "gate", "in_dtype", "storage", "fp8")]


class _W(ctypes.Structure):
    _fields_ = [("w_r", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("w1", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w3", ctypes.c_void_p),
                ("w1s", ctypes.c_void_p), ("w2s", ctypes.c_void_p), ("w3s", ctypes.c_void_p),
                ("w_att", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_round.restype = ctypes.c_double
        L.oracle_round.argtypes = [ctypes.c_double, ctypes.c_int]
        _lib = L
    return _lib


def _dt(a: np.ndarray, dtype: str | None = None) -> int:
    if dtype == "bf16" or a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float64:
        return F64
    raise TypeError("unsupported oracle input dtype %s" % a.dtype)


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def round_storage(x: float, storage: int) -> float:
    return float(lib().oracle_round(float(x), int(storage)))


FP8_MODES = {False: 0, True: 1, "row": 1, "mx": 2, 0: 0, 1: 1, 2: 2}


def make_cfg(d, E, k, c, n_shared=0, c_shared=0, gate="softmax_renorm", in_dtype=F32,
             storage=EXACT, fp8=False) -> _Cfg:
    """fp8=True / "row": expert GEMM operands in FP8 E4M3 with one power-of-two
    scale per row along the contraction (tokens, hidden rows, weight output
    channels); fp8="mx": one such scale per block of 32 consecutive elements
    along the contraction."""
    g = GATES[gate] if isinstance(gate, str) else int(gate)
    return _Cfg(d, E, k, c, n_shared, c_shared, g, in_dtype, storage, FP8_MODES[fp8])


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed (rc=%d)" % (what, rc))


def e4m3(x: np.ndarray):
    """Nearest FP8 E4M3 values (ties to even, saturating at +-448) and their codes."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    codes = np.zeros(x.shape, np.uint8)
    _check(lib().oracle_e4m3_array(ctypes.c_int64(x.size), _p(x), _p(out), _p(codes)), "e4m3")
    return out, codes


def quant_rows(x: np.ndarray, dtype: str | None = None):
    """Per-row FP8 quantisation of x [rows, cols]: codes [rows, cols] uint8, the row
    exponents e [rows] (scale 2^e) and the dequantised values e4m3(x 2^-e) 2^e."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    codes = np.zeros((rows, cols), np.uint8)
    exps = np.zeros(rows, np.int32)
    deq = np.zeros((rows, cols), np.float64)
    _check(lib().oracle_quant_rows(ctypes.c_int(rows), ctypes.c_int(cols), _p(x), ctypes.c_int(_dt(x, dtype)),
                                   _p(codes), _p(exps), _p(deq)), "quant_rows")
    return codes, exps, deq


def quant_blocks(x: np.ndarray, blk: int, dtype: str | None = None):
    """FP8 quantisation of x [rows, cols] in blocks of blk consecutive elements per
    row (blk = cols: per row): codes [rows, cols] uint8, the block exponents e
    [rows, cols / blk] (scale 2^e) and the dequantised values."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    codes = np.zeros((rows, cols), np.uint8)
    exps = np.zeros((rows, cols // blk), np.int32)
    deq = np.zeros((rows, cols), np.float64)
    _check(lib().oracle_quant_blocks(ctypes.c_int(rows), ctypes.c_int(cols), ctypes.c_int(blk), _p(x),
                                     ctypes.c_int(_dt(x, dtype)), _p(codes), _p(exps), _p(deq)), "quant_blocks")
    return codes, exps, deq


def router(cfg: _Cfg, u: np.ndarray, w_r: np.ndarray, bias: np.ndarray | None = None):
    """Logits z = u W_R^T + b (fp64), top-k indices and gate weights."""
    u = np.ascontiguousarray(u)
    n = u.shape[0]
    logits = np.zeros((n, cfg.E), np.float64)
    idx = np.zeros((n, cfg.k), np.int32)
    w = np.zeros((n, cfg.k), np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _check(lib().oracle_router(ctypes.byref(cfg), ctypes.c_int(n), _p(u), ctypes.c_int(_dt(u)),
                               _p(np.ascontiguousarray(w_r)), _p(b),
                               _p(logits), _p(idx), _p(w)), "router")
    return logits, idx, w


def expert_rows(cfg: _Cfg, a: np.ndarray, expert: np.ndarray, w1, w2, w3):
    """Per row r: h = SiLU(a W2[e]^T) * (a W1[e]^T) and y = h W3[e]^T (rounded per storage).
    With cfg.fp8 the FP8 form: a, the weight rows and h quantised per row (h is
    returned before its quantisation)."""
    a = np.ascontiguousarray(a)
    n = a.shape[0]
    h = np.zeros((n, cfg.c), np.float64)
    y = np.zeros((n, cfg.d), np.float64)
    ex = np.ascontiguousarray(expert, dtype=np.int32)
    _check(lib().oracle_expert_rows(ctypes.byref(cfg), ctypes.c_int(n), _p(a), ctypes.c_int(_dt(a)),
                                    _p(ex), _p(np.ascontiguousarray(w1)), _p(np.ascontiguousarray(w2)),
                                    _p(np.ascontiguousarray(w3)), _p(h), _p(y)), "expert_rows")
    return h, y


class Weights:
    """One block's weights in the page's layout (numpy; bf16 as uint16)."""

    def __init__(self, w_r, w1, w2, w3, bias=None, w1s=None, w2s=None, w3s=None, w_att=None):
        c = np.ascontiguousarray
        self.w_r, self.w1, self.w2, self.w3 = c(w_r), c(w1), c(w2), c(w3)
        self.bias = None if bias is None else c(bias, dtype=np.float32)
        self.w1s = None if w1s is None else c(w1s)
        self.w2s = None if w2s is None else c(w2s)
        self.w3s = None if w3s is None else c(w3s)
        self.w_att = None if w_att is None else c(w_att)

    def struct(self) -> _W:
        return _W(_p(self.w_r), _p(self.bias), _p(self.w1), _p(self.w2), _p(self.w3),
                  _p(self.w1s), _p(self.w2s), _p(self.w3s), _p(self.w_att))


def stack(cfg: _Cfg, weights: list, wiring: str, x: np.ndarray, want_rs: bool = False,
          want_logits: bool = True, want_inputs: bool = False):
    """Run L = len(weights) FarSkip blocks on the rows of x.

    Returns a dict with o (= o_L), o_star (= o_L*), topk_idx [L,n,k], topk_w [L,n,k],
    logits [L,n,E], with want_rs R and S [L,n,d], and with want_inputs the
    block inputs U (u_k, the MoE input) and P (o_{k-1}), the attention inputs
    A (attention wirings), and block outputs O (o_k), OS (o_k*) [L,n,d]."""
    x = np.ascontiguousarray(x)
    L = len(weights)
    n = x.shape[0]
    arr = (_W * L)(*[w.struct() for w in weights])
    out = {
        "o": np.zeros((n, cfg.d), np.float64),
        "o_star": np.zeros((n, cfg.d), np.float64),
        "topk_idx": np.zeros((L, n, cfg.k), np.int32),
        "topk_w": np.zeros((L, n, cfg.k), np.float64),
        "logits": np.zeros((L, n, cfg.E), np.float64) if want_logits else None,
        "R": np.zeros((L, n, cfg.d), np.float64) if want_rs else None,
        "S": np.zeros((L, n, cfg.d), np.float64) if want_rs else None,
        "U": np.zeros((L, n, cfg.d), np.float64) if want_inputs else None,
        "P": np.zeros((L, n, cfg.d), np.float64) if want_inputs else None,
        "O": np.zeros((L, n, cfg.d), np.float64) if want_inputs else None,
        "OS": np.zeros((L, n, cfg.d), np.float64) if want_inputs else None,
        "A": np.zeros((L, n, cfg.d), np.float64) if want_inputs else None,
    }
    _check(lib().oracle_stack(ctypes.byref(cfg), arr, ctypes.c_int(L), ctypes.c_int(WIRINGS[wiring]),
                              ctypes.c_int(n), _p(x), ctypes.c_int(_dt(x)),
                              _p(out["o"]), _p(out["o_star"]), _p(out["topk_idx"]), _p(out["topk_w"]),
                              _p(out["logits"]), _p(out["R"]), _p(out["S"]), _p(out["U"]), _p(out["P"]),
                              _p(out["O"]), _p(out["OS"]), _p(out["A"])),
           "stack")
    return out


def attn_standin(cfg: _Cfg, a: np.ndarray, w_att: np.ndarray):
    """Stand-in attention A(a) = a W_att^T (fp64)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    _check(lib().oracle_attn_standin(ctypes.byref(cfg), ctypes.c_int(a.shape[0]), _p(a),
                                     _p(np.ascontiguousarray(w_att)), _p(out)), "attn_standin")
    return out


def dispatch(T: int, k: int, E: int, topk_idx: np.ndarray):
    """Counting-sort Dispatch: counts[E], offsets[E+1], pos[T*k], perm_src[T*k]."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    pos = np.zeros(T * k, np.int32)
    perm = np.zeros(T * k, np.int32)
    _check(lib().oracle_dispatch(ctypes.c_int(T), ctypes.c_int(k), ctypes.c_int(E), _p(idx),
                                 _p(counts), _p(offsets), _p(pos), _p(perm)), "dispatch")
    return counts, offsets, pos, perm


def combine(T, k, d, y_perm, pos, topk_w, o_prev, shared_out=None, storage=EXACT):
    """o* = o_prev + S and o = o_prev + S + sum_s w_s y_perm[pos] (fp64, rounded per storage)."""
    y_perm = np.ascontiguousarray(y_perm)
    o_prev = np.ascontiguousarray(o_prev)
    dt = _dt(y_perm)
    assert _dt(o_prev) == dt and (shared_out is None or _dt(shared_out) == dt)
    o_star = np.zeros((T, d), np.float64)
    o = np.zeros((T, d), np.float64)
    _check(lib().oracle_combine(ctypes.c_int(T), ctypes.c_int(k), ctypes.c_int(d), ctypes.c_int(dt),
                                ctypes.c_int(storage), _p(y_perm),
                                _p(np.ascontiguousarray(pos, dtype=np.int32)),
                                _p(np.ascontiguousarray(topk_w, dtype=np.float32)), _p(o_prev),
                                _p(None if shared_out is None else np.ascontiguousarray(shared_out)),
                                _p(o_star), _p(o)), "combine")
    return o_star, o


def _grad_arrays(cfg: _Cfg, L: int | None):
    pre = () if L is None else (L,)
    E, d, c, ns, cs = cfg.E, cfg.d, cfg.c, cfg.n_shared, cfg.c_shared
    g = {"dW_R": np.zeros(pre + (E, d)), "dW1": np.zeros(pre + (E, c, d)), "dW2": np.zeros(pre + (E, c, d)),
         "dW3": np.zeros(pre + (E, d, c))}
    if ns:
        g.update(dW1s=np.zeros(pre + (ns, cs, d)), dW2s=np.zeros(pre + (ns, cs, d)), dW3s=np.zeros(pre + (ns, d, cs)))
    else:
        g.update(dW1s=None, dW2s=None, dW3s=None)
    return g


def block_backward(cfg: _Cfg, weights: Weights, u: np.ndarray, dO: np.ndarray, dOs: np.ndarray | None = None):
    """Backward of one block at its input rows u (fp64 values): du, do_prev, the
    gate-weight gradients dw [n, k] and the weight gradients dW_R, dW1, dW2, dW3
    (+ shared dW1s, dW2s, dW3s)."""
    u = np.ascontiguousarray(u, dtype=np.float64)
    n = u.shape[0]
    out = {"du": np.zeros((n, cfg.d)), "do_prev": np.zeros((n, cfg.d)), "dw": np.zeros((n, cfg.k))}
    out.update(_grad_arrays(cfg, None))
    dO = np.ascontiguousarray(dO, dtype=np.float64)
    dOs = None if dOs is None else np.ascontiguousarray(dOs, dtype=np.float64)
    _check(lib().oracle_block_backward(ctypes.byref(cfg), ctypes.byref(weights.struct()), ctypes.c_int(n), _p(u),
                                       _p(dO), _p(dOs), _p(out["du"]), _p(out["do_prev"]), _p(out["dw"]),
                                       _p(out["dW_R"]), _p(out["dW1"]), _p(out["dW2"]), _p(out["dW3"]),
                                       _p(out["dW1s"]), _p(out["dW2s"]), _p(out["dW3s"])), "block_backward")
    return out


def stack_backward(cfg: _Cfg, weights: list, wiring: str, x: np.ndarray, dOL: np.ndarray,
                   dOLs: np.ndarray | None = None, want_grads: bool = True):
    """Backward of stack() for the MoE wirings: dx and (want_grads) the per-block
    weight gradients [L, ...]."""
    x = np.ascontiguousarray(x)
    L = len(weights)
    n = x.shape[0]
    arr = (_W * L)(*[w.struct() for w in weights])
    out = {"dx": np.zeros((n, cfg.d))}
    if want_grads:
        out.update(_grad_arrays(cfg, L))
    else:
        out.update({k: None for k in ("dW_R", "dW1", "dW2", "dW3", "dW1s", "dW2s", "dW3s")})
    dOL = np.ascontiguousarray(dOL, dtype=np.float64)
    dOLs = None if dOLs is None else np.ascontiguousarray(dOLs, dtype=np.float64)
    _check(lib().oracle_stack_backward(ctypes.byref(cfg), arr, ctypes.c_int(L), ctypes.c_int(WIRINGS[wiring]),
                                       ctypes.c_int(n), _p(x), ctypes.c_int(_dt(x)), _p(dOL), _p(dOLs),
                                       _p(out["dx"]), _p(out["dW_R"]), _p(out["dW1"]), _p(out["dW2"]),
                                       _p(out["dW3"]), _p(out["dW1s"]), _p(out["dW2s"]), _p(out["dW3s"])),
           "stack_backward")
    return out
