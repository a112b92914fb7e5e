"""Thin Python binding of libfs (the C ABI in include/fs.h).

Argument marshalling only: every function passes tensor data pointers, sizes
and the current CUDA stream to the library entry point of the same name.  The
library is loaded from the in-tree build (``_build/libfs.so``); if it is
missing, ``lib()`` raises -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .configs import LayerConfig

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfs.so")
_lib = None

FS_BF16, FS_F32, FS_FP8, FS_MXFP8 = 0, 1, 2, 3
DTYPES = {"bf16": FS_BF16, "f32": FS_F32, "fp8": FS_FP8, "mxfp8": FS_MXFP8}
GATES = {"softmax": 0, "softmax_renorm": 1, "sigmoid": 2, "sigmoid_norm": 3}
WIRINGS = {"partial": 0, "outdated": 1, "disabled": 2, "attn_farskip": 3, "attn_plain": 4}
STATUS = {0: "FS_OK", 1: "FS_ERR_INVALID_ARG", 2: "FS_ERR_UNSUPPORTED", 3: "FS_ERR_WORKSPACE",
          4: "FS_ERR_CUDA", 5: "FS_ERR_DEVICE_STATE"}


class FsError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        super().__init__("%s failed: %s%s" % (what, STATUS.get(status, status), (" (%s)" % detail) if detail else ""))


class LayerDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "d", "E", "k", "c", "n_shared", "c_shared", "dtype", "gate")]


class BlockWeights(ctypes.Structure):
    _fields_ = [("w_r", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("w13", ctypes.c_void_p),
                ("w3", ctypes.c_void_p), ("w13_shared", ctypes.c_void_p), ("w3_shared", ctypes.c_void_p),
                ("w_att", ctypes.c_void_p)]


class BlockWeightsT(ctypes.Structure):
    _fields_ = [("w13t", ctypes.c_void_p), ("w3t", ctypes.c_void_p), ("w13t_shared", ctypes.c_void_p),
                ("w3t_shared", ctypes.c_void_p), ("w_rt", ctypes.c_void_p)]


class BlockGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dw_r", "dw1", "dw2", "dw3", "dw1_shared", "dw2_shared", "dw3_shared")]


_VP, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_SIGS = {
    "fs_workspace_bytes": (_SZ, [ctypes.POINTER(LayerDesc), ctypes.c_int]),
    "fs_pack_w13": (_I32, [_I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP]),
    "fs_pack_w3_shared": (_I32, [_I32, _I32, _I32, _I32, _VP, _VP, _VP]),
    "fs_pack_w3": (_I32, [_I32, _I32, _I32, _I32, _VP, _VP, _VP]),
    "fs_packed_bytes": (_SZ, [_I32, _I32, _I32, _I32]),
    "fs_router_topk": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "fs_dispatch": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "fs_dispatch_noalloc": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "fs_grouped_swiglu": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "fs_grouped_swiglu_gather": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "fs_shared_expert": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "fs_combine": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP, _VP, _I32, _VP, _I32,
                          _VP, _VP]),
    "fs_attn_standin": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _SZ, _VP]),
    "fs_shared_expert_combine": (_I32, [ctypes.POINTER(LayerDesc), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _VP,
                                        _I32, _VP, _I32, _VP, _SZ, _VP]),
    "fs_farskip_stack": (_I32, [ctypes.POINTER(LayerDesc), _I32, _I32, ctypes.POINTER(BlockWeights), _VP, _VP,
                                _VP, _VP, _SZ, _VP]),
    "fs_farskip_stack_overlap": (_I32, [ctypes.POINTER(LayerDesc), _I32, _I32, ctypes.POINTER(BlockWeights), _VP,
                                        _VP, _VP, _VP, _SZ, _VP, _VP]),
    "fs_workspace_bytes_overlap": (_SZ, [ctypes.POINTER(LayerDesc), ctypes.c_int]),
    "fs_workspace_bytes_attn": (_SZ, [ctypes.POINTER(LayerDesc), ctypes.c_int]),
    "fs_fp8_rows_bytes": (_SZ, [ctypes.c_int64, _I32]),
    "fs_pack_w13t": (_I32, [_I32, _I32, _I32, _VP, _VP, _VP, _VP]),
    "fs_pack_w3t": (_I32, [_I32, _I32, _I32, _VP, _VP, _VP]),
    "fs_pack_w3t_shared": (_I32, [_I32, _I32, _I32, _VP, _VP, _VP]),
    "fs_pack_wrt": (_I32, [_I32, _I32, _VP, _VP, _VP]),
    "fs_train_saved_bytes": (_SZ, [ctypes.POINTER(LayerDesc), ctypes.c_int]),
    "fs_workspace_bytes_backward": (_SZ, [ctypes.POINTER(LayerDesc), ctypes.c_int]),
    "fs_farskip_stack_train": (_I32, [ctypes.POINTER(LayerDesc), _I32, _I32, ctypes.POINTER(BlockWeights), _VP, _VP,
                                      _VP, _VP, _SZ, _VP, _SZ, _VP]),
    "fs_farskip_stack_backward": (_I32, [ctypes.POINTER(LayerDesc), _I32, _I32, ctypes.POINTER(BlockWeights),
                                         ctypes.POINTER(BlockWeightsT), _VP, _SZ, _VP, _VP, _VP,
                                         ctypes.POINTER(BlockGrads), _VP, _SZ, _VP]),
    "fs_quantize_rows_fp8": (_I32, [ctypes.c_int64, _I32, _VP, _VP, _VP]),
    "fs_mx_rows_bytes": (_SZ, [ctypes.c_int64, _I32]),
    "fs_quantize_rows_mx": (_I32, [ctypes.c_int64, _I32, _VP, _VP, _VP]),
    "fs_dispatch_rows": (ctypes.c_int64, [ctypes.POINTER(LayerDesc)]),
    "fs_get_error": (_I32, [ctypes.POINTER(ctypes.c_int32)]),
    "fs_launch_count": (ctypes.c_uint64, []),
    "fs_selftest_wait_timeout": (_I32, [_I32, _VP]),
    "fs_last_cuda_error": (ctypes.c_char_p, []),
    "fs_status_string": (ctypes.c_char_p, [_I32]),
}


def lib():
    """Load libfs.so (built in-tree).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfs.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        detail = ""
        if status in (3, 4):
            detail = (lib().fs_last_cuda_error() or b"").decode()
        raise FsError(status, what, detail)


def _p(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def make_desc(cfg: LayerConfig, T: int | None = None) -> LayerDesc:
    return LayerDesc(cfg.T if T is None else T, cfg.d, cfg.E, cfg.k, cfg.c, cfg.n_shared, cfg.c_shared,
                     DTYPES[cfg.dtype], GATES[cfg.gate])


# ----------------------------------------------------------------- entry points

def fs_workspace_bytes(desc: LayerDesc, L: int = 0) -> int:
    return int(lib().fs_workspace_bytes(ctypes.byref(desc), L))


def fs_pack_w13(G, c, d, dtype, w1, w2, w13, stream=None):
    _check(lib().fs_pack_w13(G, c, d, dtype, _p(w1), _p(w2), _p(w13), _stream(stream)), "fs_pack_w13")


def fs_packed_bytes(G, N, K, dtype) -> int:
    return int(lib().fs_packed_bytes(G, N, K, dtype))


def fs_pack_w3(G, d, c, dtype, w3, w3p, stream=None):
    _check(lib().fs_pack_w3(G, d, c, dtype, _p(w3), _p(w3p), _stream(stream)), "fs_pack_w3")


def fs_pack_w3_shared(n_shared, c_shared, d, dtype, w3s, w3cat, stream=None):
    _check(lib().fs_pack_w3_shared(n_shared, c_shared, d, dtype, _p(w3s), _p(w3cat), _stream(stream)),
           "fs_pack_w3_shared")


def fs_fp8_rows_bytes(rows: int, cols: int) -> int:
    return int(lib().fs_fp8_rows_bytes(rows, cols))


def fs_quantize_rows_fp8(rows, cols, x, q, stream=None):
    _check(lib().fs_quantize_rows_fp8(rows, cols, _p(x), _p(q), _stream(stream)), "fs_quantize_rows_fp8")


def fs_mx_rows_bytes(rows: int, cols: int) -> int:
    return int(lib().fs_mx_rows_bytes(rows, cols))


def fs_quantize_rows_mx(rows, cols, x, q, stream=None):
    _check(lib().fs_quantize_rows_mx(rows, cols, _p(x), _p(q), _stream(stream)), "fs_quantize_rows_mx")


def fs_dispatch_rows(desc) -> int:
    return int(lib().fs_dispatch_rows(ctypes.byref(desc)))


def mx_rows_empty(rows: int, cols: int, device="cuda") -> torch.Tensor:
    """A byte buffer for an MX matrix [rows, cols] (codes, then block-scale chunks)."""
    return torch.empty(fs_mx_rows_bytes(rows, cols), dtype=torch.uint8, device=device)


def mx_rows_split(buf: torch.Tensor, rows: int, cols: int):
    """Views (codes [rows128, cols] uint8, scale bytes [rows128 / 128, cols / 128, 512]) of an MX matrix."""
    r128 = (rows + 127) // 128 * 128
    off = (r128 * cols + 255) // 256 * 256
    return (buf[:r128 * cols].view(r128, cols),
            buf[off:off + r128 // 128 * cols // 128 * 512].view(r128 // 128, cols // 128, 512))


def fp8_rows_empty(rows: int, cols: int, device="cuda") -> torch.Tensor:
    """A byte buffer for an FP8 row-scaled matrix [rows, cols] (codes, then scales)."""
    return torch.empty(fs_fp8_rows_bytes(rows, cols), dtype=torch.uint8, device=device)


def fp8_rows_split(buf: torch.Tensor, rows: int, cols: int):
    """Views (codes [rows, cols] uint8, scales [rows] fp32) of an FP8 row-scaled matrix."""
    off = (rows * cols + 255) // 256 * 256
    return buf[:rows * cols].view(rows, cols), buf[off:off + 4 * rows].view(torch.float32)


def fs_router_topk(desc, u, w_r, bias, topk_idx, topk_w, logits, ws, stream=None):
    _check(lib().fs_router_topk(ctypes.byref(desc), _p(u), _p(w_r), _p(bias), _p(topk_idx), _p(topk_w),
                                _p(logits), _p(ws), _nbytes(ws), _stream(stream)), "fs_router_topk")


def fs_dispatch(desc, topk_idx, u, counts, offsets, pos, perm_src, x_perm, ws, stream=None):
    _check(lib().fs_dispatch(ctypes.byref(desc), _p(topk_idx), _p(u), _p(counts), _p(offsets), _p(pos),
                             _p(perm_src), _p(x_perm), _p(ws), _nbytes(ws), _stream(stream)), "fs_dispatch")


def fs_dispatch_noalloc(desc, topk_idx, u, counts, offsets, pos, perm_src, x_perm, stream=None):
    """fs_dispatch with the library's fixed static scratch instead of a workspace
    (for callers that cannot provide device scratch memory)."""
    _check(lib().fs_dispatch_noalloc(ctypes.byref(desc), _p(topk_idx), _p(u), _p(counts), _p(offsets), _p(pos),
                                     _p(perm_src), _p(x_perm), _stream(stream)), "fs_dispatch_noalloc")


def fs_grouped_swiglu(desc, x_perm, offsets, w13, w3, y_perm, ws, stream=None):
    _check(lib().fs_grouped_swiglu(ctypes.byref(desc), _p(x_perm), _p(offsets), _p(w13), _p(w3), _p(y_perm),
                                   _p(ws), _nbytes(ws), _stream(stream)), "fs_grouped_swiglu")


def fs_grouped_swiglu_gather(desc, u, perm_src, offsets, w13, w3, y_perm, ws, stream=None):
    _check(lib().fs_grouped_swiglu_gather(ctypes.byref(desc), _p(u), _p(perm_src), _p(offsets), _p(w13), _p(w3),
                                          _p(y_perm), _p(ws), _nbytes(ws), _stream(stream)),
           "fs_grouped_swiglu_gather")


def fs_shared_expert(desc, u, w13_shared, w3_shared, s_out, ws, stream=None):
    _check(lib().fs_shared_expert(ctypes.byref(desc), _p(u), _p(w13_shared), _p(w3_shared), _p(s_out), _p(ws),
                                  _nbytes(ws), _stream(stream)), "fs_shared_expert")


def _dtype_code(t):
    return FS_BF16 if t.dtype == torch.bfloat16 else FS_F32


def fs_combine(desc, y_perm, pos, topk_w, o_prev, shared_out, o_partial, o_full, u_next=None, wiring="partial",
               extra=None, u_full=None, stream=None):
    """Residual dtypes (bf16 or fp32) are taken from the o_prev and o_full tensors."""
    if o_partial is not None:
        assert o_partial.dtype == o_full.dtype
    w = WIRINGS[wiring] if isinstance(wiring, str) else int(wiring)
    _check(lib().fs_combine(ctypes.byref(desc), _p(y_perm), _p(pos), _p(topk_w), _p(o_prev), _dtype_code(o_prev),
                            _p(shared_out), _p(extra), _p(o_partial), _p(o_full), _dtype_code(o_full), _p(u_next), w,
                            _p(u_full), _stream(stream)), "fs_combine")


def fs_shared_expert_combine(desc, u, w13_shared, w3_shared, y_perm, pos, topk_w, o_prev, o_partial, o_full,
                             u_next=None, wiring="partial", ws=None, stream=None):
    """fs_shared_expert + fs_combine in one pass; residual dtypes from o_prev and o_full."""
    if o_partial is not None:
        assert o_partial.dtype == o_full.dtype
    w = WIRINGS[wiring] if isinstance(wiring, str) else int(wiring)
    _check(lib().fs_shared_expert_combine(ctypes.byref(desc), _p(u), _p(w13_shared), _p(w3_shared), _p(y_perm),
                                          _p(pos), _p(topk_w), _p(o_prev), _dtype_code(o_prev), _p(o_partial),
                                          _p(o_full), _dtype_code(o_full), _p(u_next), w, _p(ws), _nbytes(ws),
                                          _stream(stream)), "fs_shared_expert_combine")


def fs_attn_standin(desc, a, w_att, out, ws, stream=None):
    _check(lib().fs_attn_standin(ctypes.byref(desc), _p(a), _p(w_att), _p(out), _p(ws), _nbytes(ws),
                                 _stream(stream)), "fs_attn_standin")


def block_struct(packed: dict) -> BlockWeights:
    return BlockWeights(_p(packed["w_r"]), _p(packed.get("bias")), _p(packed["w13"]), _p(packed["w3"]),
                        _p(packed.get("w13_shared")), _p(packed.get("w3_shared")), _p(packed.get("w_att")))


def fs_farskip_stack(desc, L, wiring, blocks, x, o_full, o_partial, ws, stream=None):
    """`blocks`: list of L packed-weight dicts (see pack_block)."""
    arr = (BlockWeights * L)(*[block_struct(b) for b in blocks])
    w = WIRINGS[wiring] if isinstance(wiring, str) else int(wiring)
    _check(lib().fs_farskip_stack(ctypes.byref(desc), L, w, arr, _p(x), _p(o_full), _p(o_partial), _p(ws),
                                  _nbytes(ws), _stream(stream)), "fs_farskip_stack")


def fs_workspace_bytes_overlap(desc: LayerDesc, L: int) -> int:
    return int(lib().fs_workspace_bytes_overlap(ctypes.byref(desc), L))


def fs_farskip_stack_overlap(desc, L, wiring, blocks, x, o_full, o_partial, ws, stream=None, stream2=None):
    """Two-stream stack: `stream2` (a torch.cuda.Stream) runs router/dispatch/shared."""
    arr = (BlockWeights * L)(*[block_struct(b) for b in blocks])
    w = WIRINGS[wiring] if isinstance(wiring, str) else int(wiring)
    _check(lib().fs_farskip_stack_overlap(ctypes.byref(desc), L, w, arr, _p(x), _p(o_full), _p(o_partial), _p(ws),
                                          _nbytes(ws), _stream(stream), _stream(stream2)),
           "fs_farskip_stack_overlap")


def fs_get_error():
    code = ctypes.c_int32(0)
    st = lib().fs_get_error(ctypes.byref(code))
    return int(st), int(code.value)


def fs_selftest_wait_timeout(limit_us: int, stream=None):
    _check(lib().fs_selftest_wait_timeout(limit_us, _stream(stream)), "fs_selftest_wait_timeout")


def fs_launch_count() -> int:
    return int(lib().fs_launch_count())


# -------------------------------------------------------------- conveniences

def fs_workspace_bytes_attn(desc: LayerDesc, L: int) -> int:
    return int(lib().fs_workspace_bytes_attn(ctypes.byref(desc), L))


def alloc_workspace(desc: LayerDesc, L: int, device="cuda", attn: bool = False) -> torch.Tensor:
    n = fs_workspace_bytes_attn(desc, L) if attn else fs_workspace_bytes(desc, L)
    if n == 0:
        raise FsError(1, "fs_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _packed(G, N, K, dt, like):
    n = fs_packed_bytes(G, N, K, dt)
    if n == 0:
        raise FsError(1, "fs_packed_bytes")
    if dt in (FS_FP8, FS_MXFP8):
        return torch.empty(n, dtype=torch.uint8, device=like.device)
    return torch.empty(n // like.element_size(), dtype=like.dtype, device=like.device)


def pack_block(cfg: LayerConfig, w: dict, stream=None) -> dict:
    """Repack one block's page-layout weights (on the GPU) into the library layout
    (FP8: quantised from the bf16 weights)."""
    dt = DTYPES[cfg.dtype]
    E, c, d = cfg.E, cfg.c, cfg.d
    out = {"w_r": w["w_r"].contiguous(), "bias": None if w.get("bias") is None else w["bias"].contiguous().float()}
    out["w13"] = _packed(E, 2 * c, d, dt, w["w1"])
    fs_pack_w13(E, c, d, dt, w["w1"].contiguous(), w["w2"].contiguous(), out["w13"], stream)
    out["w3"] = _packed(E, d, c, dt, w["w3"])
    fs_pack_w3(E, d, c, dt, w["w3"].contiguous(), out["w3"], stream)
    if w.get("w_att") is not None:
        out["w_att"] = w["w_att"].contiguous()
    if cfg.n_shared:
        cw = cfg.n_shared * cfg.c_shared
        out["w13_shared"] = _packed(1, 2 * cw, d, dt, w["w1s"])
        fs_pack_w13(1, cw, d, dt, w["w1s"].contiguous(), w["w2s"].contiguous(), out["w13_shared"], stream)
        out["w3_shared"] = _packed(1, d, cw, dt, w["w3s"])
        fs_pack_w3_shared(cfg.n_shared, cfg.c_shared, d, dt, w["w3s"].contiguous(), out["w3_shared"], stream)
    return out


class FarSkipStack:
    """L FarSkip MoE blocks on one GPU: packed weights + workspace, one
    fs_farskip_stack call per forward."""

    def __init__(self, cfg: LayerConfig, raw_blocks: list, wiring: str | None = None, T: int | None = None,
                 device="cuda"):
        self.cfg = cfg
        self.T = cfg.T if T is None else T
        self.wiring = wiring or cfg.wiring
        self.desc = make_desc(cfg, self.T)
        self.blocks = [pack_block(cfg, b) for b in raw_blocks]
        self.ws = alloc_workspace(self.desc, len(self.blocks), device, attn=self.wiring.startswith("attn"))
        dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
        self.o_full = torch.empty((self.T, cfg.d), dtype=dt, device=device)
        self.o_partial = torch.empty((self.T, cfg.d), dtype=dt, device=device)

    def forward(self, x: torch.Tensor, stream=None):
        fs_farskip_stack(self.desc, len(self.blocks), self.wiring, self.blocks, x, self.o_full, self.o_partial,
                         self.ws, stream)
        return self.o_full, self.o_partial

    def capture(self, x: torch.Tensor, overlap: bool = False):
        """Record one forward (the library's launches for all L blocks, reading x and
        writing o_full, o_partial) into a CUDA graph; replay() re-runs it.  Warm the
        stack up (one eager forward) first so that one-time setup happens outside
        the capture."""
        self.graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.o_full.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                if overlap:
                    self.forward_overlap(x, stream=s)
                else:
                    self.forward(x, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        return self.graph

    def replay(self):
        """Re-run the captured forward (same x buffer, same outputs)."""
        self.graph.replay()
        return self.o_full, self.o_partial

    def forward_overlap(self, x: torch.Tensor, stream=None):
        """Two-stream FarSkip schedule (partial/outdated wiring)."""
        if not hasattr(self, "ws_overlap"):
            n = fs_workspace_bytes_overlap(self.desc, len(self.blocks))
            self.ws_overlap = torch.empty(n, dtype=torch.uint8, device=self.o_full.device)
            self.stream2 = torch.cuda.Stream(device=self.o_full.device)
        fs_farskip_stack_overlap(self.desc, len(self.blocks), self.wiring, self.blocks, x, self.o_full,
                                 self.o_partial, self.ws_overlap, stream, self.stream2)
        return self.o_full, self.o_partial


# ------------------------------------------------------------------ training

def fs_train_saved_bytes(desc: LayerDesc, L: int) -> int:
    return int(lib().fs_train_saved_bytes(ctypes.byref(desc), L))


def fs_workspace_bytes_backward(desc: LayerDesc, L: int) -> int:
    return int(lib().fs_workspace_bytes_backward(ctypes.byref(desc), L))


def fs_pack_w13t(G, c, d, w1, w2, out, stream=None):
    _check(lib().fs_pack_w13t(G, c, d, _p(w1), _p(w2), _p(out), _stream(stream)), "fs_pack_w13t")


def fs_pack_w3t(G, d, c, w3, out, stream=None):
    _check(lib().fs_pack_w3t(G, d, c, _p(w3), _p(out), _stream(stream)), "fs_pack_w3t")


def fs_pack_w3t_shared(n_shared, c_shared, d, w3s, out, stream=None):
    _check(lib().fs_pack_w3t_shared(n_shared, c_shared, d, _p(w3s), _p(out), _stream(stream)), "fs_pack_w3t_shared")


def fs_pack_wrt(E, d, w_r, out, stream=None):
    _check(lib().fs_pack_wrt(E, d, _p(w_r), _p(out), _stream(stream)), "fs_pack_wrt")


def pack_block_t(cfg: LayerConfig, w: dict, stream=None) -> dict:
    """Transposed packs of one block's bf16 weights for the input-gradient GEMMs."""
    E, c, d = cfg.E, cfg.c, cfg.d
    epad = (E + 63) // 64 * 64
    out = {"w13t": _packed(E, d, 2 * c, FS_BF16, w["w1"]), "w3t": _packed(E, c, d, FS_BF16, w["w3"]),
           "w_rt": _packed(1, d, epad, FS_BF16, w["w_r"])}
    fs_pack_w13t(E, c, d, w["w1"].contiguous(), w["w2"].contiguous(), out["w13t"], stream)
    fs_pack_w3t(E, d, c, w["w3"].contiguous(), out["w3t"], stream)
    fs_pack_wrt(E, d, w["w_r"].contiguous(), out["w_rt"], stream)
    if cfg.n_shared:
        cw = cfg.n_shared * cfg.c_shared
        out["w13t_shared"] = _packed(1, d, 2 * cw, FS_BF16, w["w1s"])
        out["w3t_shared"] = _packed(1, cw, d, FS_BF16, w["w3s"])
        fs_pack_w13t(1, cw, d, w["w1s"].contiguous(), w["w2s"].contiguous(), out["w13t_shared"], stream)
        fs_pack_w3t_shared(cfg.n_shared, cfg.c_shared, d, w["w3s"].contiguous(), out["w3t_shared"], stream)
    return out


def _block_t_struct(p: dict) -> BlockWeightsT:
    return BlockWeightsT(_p(p["w13t"]), _p(p["w3t"]), _p(p.get("w13t_shared")), _p(p.get("w3t_shared")),
                         _p(p["w_rt"]))


def _grads_struct(g: dict) -> BlockGrads:
    return BlockGrads(*[_p(g.get(k)) for k in ("dW_R", "dW1", "dW2", "dW3", "dW1s", "dW2s", "dW3s")])


class FarSkipTrainer:
    """Forward (keeping what the backward reads) and backward of an L-block
    FarSkip MoE stack on one GPU (bf16, MoE wirings): two library calls."""

    def __init__(self, cfg: LayerConfig, raw_blocks: list, wiring: str | None = None, T: int | None = None,
                 device="cuda"):
        self.cfg = cfg
        self.T = cfg.T if T is None else T
        self.wiring = wiring or cfg.wiring
        self.desc = make_desc(cfg, self.T)
        L = len(raw_blocks)
        self.L = L
        self.blocks = [pack_block(cfg, b) for b in raw_blocks]
        self.blocks_t = [pack_block_t(cfg, b) for b in raw_blocks]
        self.saved = torch.empty(fs_train_saved_bytes(self.desc, L), dtype=torch.uint8, device=device)
        self.ws = alloc_workspace(self.desc, L, device)
        self.ws_b = torch.empty(fs_workspace_bytes_backward(self.desc, L), dtype=torch.uint8, device=device)
        E, c, d, ns, cs = cfg.E, cfg.c, cfg.d, cfg.n_shared, cfg.c_shared
        f32 = dict(dtype=torch.float32, device=device)
        self.grads = []
        for _ in range(L):
            g = {"dW_R": torch.empty((E, d), **f32), "dW1": torch.empty((E, c, d), **f32),
                 "dW2": torch.empty((E, c, d), **f32), "dW3": torch.empty((E, d, c), **f32)}
            if ns:
                g.update(dW1s=torch.empty((ns, cs, d), **f32), dW2s=torch.empty((ns, cs, d), **f32),
                         dW3s=torch.empty((ns, d, cs), **f32))
            self.grads.append(g)
        self.o_full = torch.empty((self.T, d), dtype=torch.bfloat16, device=device)
        self.o_partial = torch.empty((self.T, d), dtype=torch.bfloat16, device=device)
        self.dx = torch.empty((self.T, d), **f32)

    def forward(self, x: torch.Tensor, stream=None):
        arr = (BlockWeights * self.L)(*[block_struct(b) for b in self.blocks])
        _check(lib().fs_farskip_stack_train(ctypes.byref(self.desc), self.L, WIRINGS[self.wiring], arr, _p(x),
                                            _p(self.o_full), _p(self.o_partial), _p(self.saved), _nbytes(self.saved),
                                            _p(self.ws), _nbytes(self.ws), _stream(stream)), "fs_farskip_stack_train")
        return self.o_full, self.o_partial

    def backward(self, d_o: torch.Tensor, d_os: torch.Tensor | None = None, stream=None,
                 dx: torch.Tensor | None = None):
        """Gradients for the last forward: dx (into `dx` when given, else self.dx)
        and the weight gradients (self.grads)."""
        out = self.dx if dx is None else dx
        arr = (BlockWeights * self.L)(*[block_struct(b) for b in self.blocks])
        arr_t = (BlockWeightsT * self.L)(*[_block_t_struct(b) for b in self.blocks_t])
        gr = (BlockGrads * self.L)(*[_grads_struct(g) for g in self.grads])
        _check(lib().fs_farskip_stack_backward(ctypes.byref(self.desc), self.L, WIRINGS[self.wiring], arr, arr_t,
                                               _p(self.saved), _nbytes(self.saved), _p(d_o), _p(d_os), _p(out),
                                               gr, _p(self.ws_b), _nbytes(self.ws_b), _stream(stream)),
               "fs_farskip_stack_backward")
        return out, self.grads
