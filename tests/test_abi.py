"""The C ABI without a GPU: the library loads, exports every function that
include/fs.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_expert_gb300 import build, configs, fs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fs.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return fs.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fs_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fs_router_topk", "fs_dispatch", "fs_grouped_swiglu", "fs_combine", "fs_farskip_stack",
              "fs_shared_expert", "fs_workspace_bytes", "fs_get_error", "fs_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), "libfs.so does not export %s" % n


def test_binding_covers_the_header():
    for n in declared_functions():
        assert n in fs._SIGS, "fs.py has no binding for %s" % n


def test_status_strings(L):
    for code, name in fs.STATUS.items():
        assert L.fs_status_string(code).decode() == name


def desc(**kw):
    cfg = configs.CONFIGS["v3"]
    d = fs.make_desc(cfg)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_mx_sizes(L):
    d = desc(dtype=3)                                     # FS_MXFP8, V3 shapes
    assert fs.fs_dispatch_rows(d) == (65536 * 8 + 127 * 256 + 127) // 128 * 128
    assert fs.fs_dispatch_rows(desc()) == 65536 * 8
    assert fs.fs_mx_rows_bytes(300, 256) == 384 * 256 + 3 * 2 * 512          # rows rounded up to 128
    assert fs.fs_mx_rows_bytes(300, 200) == 0                                # cols % 128
    assert fs.fs_packed_bytes(2, 384, 256, 3) == 2 * 512 * 256 + 2 * 2 * 2 * 1024
    assert fs.fs_packed_bytes(2, 320, 256, 3) == 0                           # N % 128
    big = desc(dtype=3, T=(2 ** 31 - 1024 - 127 * 256 - 64) // 8, k=8)
    assert fs.fs_workspace_bytes(big, 0) == 0                                # padded rows beyond int32
    assert L.fs_quantize_rows_mx(10, 200, _vp(FAKE), _vp(FAKE), None) == 2
    assert L.fs_quantize_rows_mx(0, 256, _vp(FAKE), _vp(FAKE), None) == 1


def test_workspace_bytes(L):
    assert fs.fs_workspace_bytes(desc(), 0) > 0
    assert fs.fs_workspace_bytes(desc(), 1) > fs.fs_workspace_bytes(desc(), 0)
    assert fs.fs_workspace_bytes(desc(), 4) > fs.fs_workspace_bytes(desc(), 1)
    # invalid descriptors -> 0
    for bad in (dict(T=0), dict(k=300), dict(d=100), dict(c=100), dict(E=1024), dict(dtype=7), dict(gate=9),
                dict(k=17, E=64)):
        assert fs.fs_workspace_bytes(desc(**bad), 1) == 0, bad
    # the V3 stack: X_perm and Y_perm dominate (2 x 7.5 GB)
    v3 = fs.fs_workspace_bytes(desc(), 1)
    assert 15.0e9 < v3 < 25.0e9


FAKE = 0x10000          # 16-byte aligned, never dereferenced: every call below fails validation first
MIS = 0x10001


def _vp(x):
    return ctypes.c_void_p(x)


def test_router_rejects_bad_args(L):
    d = desc()
    ws_ok = fs.fs_workspace_bytes(d, 0)
    f = L.fs_router_topk
    args = [ctypes.byref(d), _vp(FAKE), _vp(FAKE), None, _vp(FAKE), _vp(FAKE), None, _vp(FAKE * 256), ws_ok, None]
    a = list(args); a[1] = None
    assert f(*a) == 1                                     # null u
    a = list(args); a[1] = _vp(MIS)
    assert f(*a) == 2                                     # misaligned u
    a = list(args); a[8] = ws_ok - 1
    assert f(*a) == 3                                     # workspace too small
    a = list(args); a[7] = _vp(FAKE * 256 + 16)
    assert f(*a) == 3                                     # workspace misaligned
    bad = desc(k=9, E=8)
    a = list(args); a[0] = ctypes.byref(bad)
    assert f(*a) == 1                                     # k > E
    bad = desc(d=7100)
    a = list(args); a[0] = ctypes.byref(bad)
    assert f(*a) == 2                                     # d not a multiple of 64


def test_other_entry_points_reject_bad_args(L):
    d = desc()
    assert L.fs_dispatch(ctypes.byref(d), None, _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE),
                         _vp(FAKE * 256), 1 << 40, None) == 1
    assert L.fs_grouped_swiglu(ctypes.byref(d), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE),
                               _vp(FAKE * 256), 16, None) == 3
    # fs_combine(desc, y, pos, w, o_prev, prev_dtype, S, extra, o_partial, o_full, out_dtype, u_next, wiring, u_full, st)
    assert L.fs_combine(ctypes.byref(d), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), 0, None, None, None, None, 0,
                        None, 0, None, None) == 1                           # null o_full
    assert L.fs_combine(ctypes.byref(d), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), 0, _vp(MIS), None, None,
                        _vp(FAKE), 0, None, 0, None, None) == 2             # misaligned S
    assert L.fs_combine(ctypes.byref(d), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), 3, None, None, None,
                        _vp(FAKE), 0, None, 0, None, None) == 1             # bad residual dtype
    assert L.fs_combine(ctypes.byref(d), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), 0, None, None, None,
                        _vp(FAKE), 0, _vp(FAKE), 9, None, None) == 1        # bad wiring for u_next
    assert L.fs_combine(ctypes.byref(d), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), 0, None, _vp(MIS), None,
                        _vp(FAKE), 0, None, 0, None, None) == 2             # misaligned extra
    # fs_shared_expert_combine(desc, u, w13s, w3s, y, pos, w, o_prev, prev_dtype, o_partial, o_full, out_dtype,
    #                          u_next, wiring, ws, ws_bytes, st)
    sc = lambda dd, *a: L.fs_shared_expert_combine(ctypes.byref(dd), *a)
    V = _vp(FAKE)
    assert sc(d, V, V, V, V, V, V, V, 0, None, None, 0, None, 0, _vp(FAKE * 256), 1 << 40, None) == 1   # null o_full
    assert sc(d, V, V, V, V, V, V, V, 2, None, V, 0, None, 0, _vp(FAKE * 256), 1 << 40, None) == 1      # bad dtype
    assert sc(d, V, V, V, V, V, V, V, 0, None, V, 0, V, 7, _vp(FAKE * 256), 1 << 40, None) == 1         # bad wiring
    assert sc(d, V, V, V, V, V, V, V, 0, _vp(MIS), V, 0, None, 0, _vp(FAKE * 256), 1 << 40, None) == 2  # misaligned
    assert sc(desc(n_shared=0), V, V, V, V, V, V, V, 0, None, V, 0, None, 0, _vp(FAKE * 256), 1 << 40,
              None) == 1                                                                            # no shared expert
    assert sc(desc(dtype=1), V, V, V, V, V, V, V, 0, None, V, 0, None, 0, _vp(FAKE * 256), 1 << 40,
              None) == 2                                                                            # fp32: unfused only
    assert sc(d, V, V, V, V, V, V, V, 0, None, V, 0, None, 0, _vp(FAKE * 256), 16, None) == 3           # small ws
    assert L.fs_attn_standin(ctypes.byref(d), None, _vp(FAKE), _vp(FAKE), _vp(FAKE * 256), 1 << 40, None) == 1
    blocks1 = (fs.BlockWeights * 1)(fs.BlockWeights(FAKE, None, FAKE, FAKE, FAKE, FAKE, None))
    assert L.fs_farskip_stack(ctypes.byref(d), 1, 3, blocks1, _vp(FAKE), _vp(FAKE), None, _vp(FAKE * 256),
                              1 << 40, None) == 1              # attention wiring without w_att
    nd = desc(n_shared=0)
    assert L.fs_shared_expert(ctypes.byref(nd), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE), _vp(FAKE * 256),
                              1 << 40, None) == 1
    assert L.fs_pack_w13(0, 64, 64, 0, _vp(FAKE), _vp(FAKE), _vp(FAKE), None) == 1
    assert L.fs_pack_w13(1, 65, 64, 0, _vp(FAKE), _vp(FAKE), _vp(FAKE), None) == 2
    assert L.fs_pack_w3_shared(1, 64, 64, 9, _vp(FAKE), _vp(FAKE), None) == 1
    blocks = (fs.BlockWeights * 1)()
    assert L.fs_farskip_stack(ctypes.byref(d), 1, 0, blocks, _vp(FAKE), _vp(FAKE), None, _vp(FAKE * 256),
                              1 << 40, None) == 1              # null block weights
    assert L.fs_farskip_stack(ctypes.byref(d), 0, 0, blocks, _vp(FAKE), _vp(FAKE), None, _vp(FAKE * 256),
                              1 << 40, None) == 1              # L = 0
    assert L.fs_farskip_stack(ctypes.byref(d), 1, 5, blocks, _vp(FAKE), _vp(FAKE), None, _vp(FAKE * 256),
                              1 << 40, None) == 1              # bad wiring


def test_fp8_argument_checks(L):
    """FS_FP8 needs d, c, c_shared multiples of 128; rejected before any launch."""
    ok = desc(dtype=2)
    assert fs.fs_workspace_bytes(ok, 1) > 0
    # FP8 x_perm (1 byte per element) is smaller than the bf16 one
    assert fs.fs_workspace_bytes(ok, 1) < fs.fs_workspace_bytes(desc(), 1)
    for bad in (dict(d=7168 + 64), dict(c=2048 + 64), dict(c_shared=2048 + 64)):
        assert fs.fs_workspace_bytes(desc(dtype=2, **bad), 1) == 0, bad
    assert fs.fs_packed_bytes(256, 4096, 7168, 2) == 256 * 4096 * 7168 + 256 * 4096 * 4
    assert fs.fs_packed_bytes(1, 384, 256, 2) == 512 * 256 + 384 * 4      # rows padded to 256
    assert fs.fs_packed_bytes(1, 256, 192, 2) == 0                        # K % 128
    assert fs.fs_fp8_rows_bytes(3, 128) == 512 + 12
    assert fs.fs_fp8_rows_bytes(0, 128) == 0
    assert L.fs_pack_w13(1, 192, 256, 2, _vp(FAKE), _vp(FAKE), _vp(FAKE), None) == 2
    assert L.fs_pack_w3(1, 256, 192, 2, _vp(FAKE), _vp(FAKE), None) == 2
    assert L.fs_pack_w3_shared(2, 192, 256, 2, _vp(FAKE), _vp(FAKE), None) == 2
    assert L.fs_quantize_rows_fp8(10, 100, _vp(FAKE), _vp(FAKE), None) == 2
    assert L.fs_quantize_rows_fp8(0, 128, _vp(FAKE), _vp(FAKE), None) == 1
    assert L.fs_quantize_rows_fp8(10, 128, _vp(MIS), _vp(FAKE), None) == 2
    assert L.fs_pack_w13(1, 128, 128, 9, _vp(FAKE), _vp(FAKE), _vp(FAKE), None) == 1      # unknown dtype
    assert fs.fs_launch_count() == 0


def test_training_argument_checks(L):
    """The training entry points: bf16 and the MoE wirings only; bad arguments
    are rejected before any launch."""
    d = desc()
    assert fs.fs_train_saved_bytes(d, 1) > 0
    assert fs.fs_train_saved_bytes(d, 2) == 2 * fs.fs_train_saved_bytes(d, 1)
    assert fs.fs_workspace_bytes_backward(d, 1) > 0
    assert fs.fs_train_saved_bytes(desc(dtype=2), 1) == 0          # FP8: no backward
    assert fs.fs_train_saved_bytes(desc(dtype=1), 1) == 0          # fp32: no backward
    assert fs.fs_workspace_bytes_backward(d, 0) == 0
    blocks = (fs.BlockWeights * 1)(fs.BlockWeights(FAKE, None, FAKE, FAKE, FAKE, FAKE, None))
    args = [ctypes.byref(d), 1, 0, blocks, _vp(FAKE), _vp(FAKE), None, _vp(FAKE * 256), 1 << 40, _vp(FAKE * 256),
            1 << 40, None]
    a = list(args); a[2] = 3
    assert L.fs_farskip_stack_train(*a) == 1                         # attention wiring
    a = list(args); a[1] = 0
    assert L.fs_farskip_stack_train(*a) == 1                         # L = 0
    f32 = desc(dtype=1)
    a = list(args); a[0] = ctypes.byref(f32)
    assert L.fs_farskip_stack_train(*a) == 2                         # fp32
    a = list(args); a[8] = 16
    assert L.fs_farskip_stack_train(*a) == 3                         # saved buffer too small
    bt = (fs.BlockWeightsT * 1)(fs.BlockWeightsT(FAKE, FAKE, FAKE, FAKE, FAKE))
    gr = (fs.BlockGrads * 1)(fs.BlockGrads(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE))
    bargs = [ctypes.byref(d), 1, 0, blocks, bt, _vp(FAKE * 256), 1 << 40, _vp(FAKE), None, _vp(FAKE), gr,
             _vp(FAKE * 256), 1 << 40, None]
    a = list(bargs); a[10] = None
    assert L.fs_farskip_stack_backward(*a) == 1                      # no gradient array
    a = list(bargs); a[8] = _vp(MIS)
    assert L.fs_farskip_stack_backward(*a) == 2                      # misaligned d_os
    a = list(bargs); a[12] = 16
    assert L.fs_farskip_stack_backward(*a) == 3                      # workspace too small
    assert L.fs_pack_w13t(0, 64, 64, _vp(FAKE), _vp(FAKE), _vp(FAKE), None) == 1
    assert L.fs_pack_w3t(1, 64, 65, _vp(FAKE), _vp(FAKE), None) == 2
    assert L.fs_pack_wrt(16, 100, _vp(FAKE), _vp(FAKE), None) == 2
    assert fs.fs_launch_count() == 0


def test_no_launch_on_rejected_calls(L):
    assert fs.fs_launch_count() == 0
