"""ctypes binding of liblrm.so: argument marshalling only.

Every function has the name and argument order of its C entry point in
include/lrm.h; tensors are passed as device pointers (torch tensors are
accepted and their data_ptr() is used), ``stream`` defaults to torch's
current CUDA stream. A status other than LRM_OK raises LrmError. The library
is required: importing this module without a built liblrm.so raises.
"""

from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblrm.so")

LRM_OK, LRM_ERR_INVALID_ARG, LRM_ERR_UNSUPPORTED, LRM_ERR_WORKSPACE, LRM_ERR_CUDA = range(5)
LRM_F32, LRM_BF16 = 0, 1
LRM_DEVERR_EXPERT_ID, LRM_DEVERR_QUOTA, LRM_DEVERR_INDEX, LRM_DEVERR_TIMEOUT = 1, 2, 4, 8
LRM_DEVERR_QUEUE = 16

# Every symbol include/lrm.h declares.
EXPORTS = (
    "lrm_workspace_bytes", "lrm_clear_device_error", "lrm_get_device_error",
    "lrm_status_string", "lrm_dispatch_permute", "lrm_permute_rows",
    "lrm_quota_from_rate", "lrm_score", "lrm_select_quota", "lrm_compact",
    "lrm_expert_bwd_grouped", "lrm_expert_fc2_dgrad", "lrm_expert_fc2_wgrad",
    "lrm_expert_fc1_wgrad", "lrm_expert_fc1_dgrad", "lrm_scatter_dx",
    "lrm_dispatch_permute_noalloc", "lrm_selftest_wait_timeout", "lrm_score_variant",
    "lrm_gather_tokens", "lrm_expert_fc1_fwd", "lrm_expert_fc2_fwd", "lrm_combine",
    "lrm_expert_fwd_grouped", "lrm_expert_fc1_recompute", "lrm_expert_bwd_gathered",
    "lrm_select_rate",
)
LRM_BWD_FC2_DGRAD, LRM_BWD_FC2_WGRAD, LRM_BWD_FC1_WGRAD = 1, 2, 4
LRM_BWD_FC1_DGRAD, LRM_BWD_SCATTER_DX, LRM_BWD_ALL = 8, 16, 31
LRM_METRIC_LRM, LRM_METRIC_GRAD_SQ, LRM_METRIC_GRAD_ABS, LRM_METRIC_RANDOM = range(4)
LRM_NOALLOC_MAX_CHUNK_ENTRIES = 65536


class LrmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status_string(status)}")


class lrm_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("D", ctypes.c_int32), ("H", ctypes.c_int32),
                ("E", ctypes.c_int32), ("K", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"liblrm.so not built at {_LIB_PATH}; run "
            "`python -m demand_side_expert_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    sp = ctypes.POINTER(lrm_shape)
    sig = {
        "lrm_workspace_bytes": (sz, [sp]),
        "lrm_clear_device_error": (i32, [vp, sz, vp]),
        "lrm_get_device_error": (i32, [vp, sz, ctypes.POINTER(i32), vp]),
        "lrm_status_string": (ctypes.c_char_p, [i32]),
        "lrm_dispatch_permute": (i32, [sp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_permute_rows": (i32, [vp, i32, vp, vp, i64, vp]),
        "lrm_quota_from_rate": (i32, [vp, i32, i32, i32, i32, vp, vp]),
        "lrm_score": (i32, [sp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_select_quota": (i32, [sp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_compact": (i32, [sp] + [vp] * 15 + [vp, sz, vp]),
        "lrm_expert_bwd_grouped": (i32, [sp] + [vp] * 16 + [vp, sz, vp]),
        "lrm_expert_fc2_dgrad": (i32, [sp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_expert_fc2_wgrad": (i32, [sp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_expert_fc1_wgrad": (i32, [sp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_expert_fc1_dgrad": (i32, [sp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_scatter_dx": (i32, [sp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_dispatch_permute_noalloc": (i32, [sp, vp, vp, vp, vp, vp, vp, vp]),
        "lrm_selftest_wait_timeout": (i32, [vp, sz, vp]),
        "lrm_score_variant": (i32, [sp, i32, ctypes.c_uint64, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_gather_tokens": (i32, [sp, vp, vp, vp, vp, sz, vp]),
        "lrm_expert_fc1_fwd": (i32, [sp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_expert_fc2_fwd": (i32, [sp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_combine": (i32, [sp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_expert_fwd_grouped": (i32, [sp] + [vp] * 13 + [vp, sz, vp]),
        "lrm_expert_fc1_recompute": (i32, [sp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "lrm_expert_bwd_gathered": (i32, [sp, i32] + [vp] * 18 + [vp, sz, vp]),
        "lrm_select_rate": (i32, [sp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def library_path() -> str:
    return _LIB_PATH


def _p(x):
    """Device pointer of a tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != LRM_OK:
        raise LrmError(fn, status)


def make_shape(T: int, D: int, H: int, E: int, K: int, dtype: int) -> lrm_shape:
    return lrm_shape(T, D, H, E, K, dtype)


def status_string(status: int) -> str:
    return _lib.lrm_status_string(status).decode()


def lrm_status_string(status: int) -> str:
    return status_string(status)


def lrm_workspace_bytes(shape: lrm_shape) -> int:
    return int(_lib.lrm_workspace_bytes(ctypes.byref(shape)))


def lrm_clear_device_error(ws, ws_bytes: int, stream=None):
    _check("lrm_clear_device_error", _lib.lrm_clear_device_error(_p(ws), ws_bytes, _s(stream)))


def lrm_get_device_error(ws, ws_bytes: int, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("lrm_get_device_error",
           _lib.lrm_get_device_error(_p(ws), ws_bytes, ctypes.byref(out), _s(stream)))
    return int(out.value)


def lrm_dispatch_permute(shape, topk_idx, perm, inv, counts, off, ws, ws_bytes, stream=None):
    _check("lrm_dispatch_permute", _lib.lrm_dispatch_permute(
        ctypes.byref(shape), _p(topk_idx), _p(perm), _p(inv), _p(counts), _p(off),
        _p(ws), ws_bytes, _s(stream)))


def lrm_permute_rows(perm, n_rows: int, src, dst, row_bytes: int, stream=None):
    _check("lrm_permute_rows", _lib.lrm_permute_rows(
        _p(perm), n_rows, _p(src), _p(dst), row_bytes, _s(stream)))


def lrm_quota_from_rate(counts, E: int, num: int, den: int, cap: int, quota, stream=None):
    _check("lrm_quota_from_rate", _lib.lrm_quota_from_rate(
        _p(counts), E, num, den, cap, _p(quota), _s(stream)))


def lrm_score(shape, g, phi, alpha, inv, score, ws, ws_bytes, stream=None):
    _check("lrm_score", _lib.lrm_score(
        ctypes.byref(shape), _p(g), _p(phi), _p(alpha), _p(inv), _p(score),
        _p(ws), ws_bytes, _s(stream)))


def lrm_select_quota(shape, score, off, quota, keep, sel_off, sel_pos, ws, ws_bytes,
                     stream=None):
    _check("lrm_select_quota", _lib.lrm_select_quota(
        ctypes.byref(shape), _p(score), _p(off), _p(quota), _p(keep), _p(sel_off),
        _p(sel_pos), _p(ws), ws_bytes, _s(stream)))


def lrm_compact(shape, perm, keep, sel_off, sel_pos, alpha, x, g, ab, phi, dy_c, x_c, ab_c,
                phi_c, tok_c, row_of_pos, ws, ws_bytes, stream=None):
    _check("lrm_compact", _lib.lrm_compact(
        ctypes.byref(shape), _p(perm), _p(keep), _p(sel_off), _p(sel_pos), _p(alpha), _p(x),
        _p(g), _p(ab), _p(phi), _p(dy_c), _p(x_c), _p(ab_c), _p(phi_c), _p(tok_c),
        _p(row_of_pos), _p(ws), ws_bytes, _s(stream)))


def lrm_expert_bwd_grouped(shape, sel_off, w_gate, w_up, w_down, dy_c, x_c, ab_c, phi_c, inv,
                           row_of_pos, dab_c, dx_c, dw_gate, dw_up, dw_down, dx, ws, ws_bytes,
                           stream=None):
    _check("lrm_expert_bwd_grouped", _lib.lrm_expert_bwd_grouped(
        ctypes.byref(shape), _p(sel_off), _p(w_gate), _p(w_up), _p(w_down), _p(dy_c), _p(x_c),
        _p(ab_c), _p(phi_c), _p(inv), _p(row_of_pos), _p(dab_c), _p(dx_c), _p(dw_gate),
        _p(dw_up), _p(dw_down), _p(dx), _p(ws), ws_bytes, _s(stream)))


def lrm_expert_fc2_dgrad(shape, sel_off, w_down, dy_c, ab_c, dab_c, ws, ws_bytes, stream=None):
    _check("lrm_expert_fc2_dgrad", _lib.lrm_expert_fc2_dgrad(
        ctypes.byref(shape), _p(sel_off), _p(w_down), _p(dy_c), _p(ab_c), _p(dab_c), _p(ws),
        ws_bytes, _s(stream)))


def lrm_expert_fc2_wgrad(shape, sel_off, phi_c, dy_c, dw_down, ws, ws_bytes, stream=None):
    _check("lrm_expert_fc2_wgrad", _lib.lrm_expert_fc2_wgrad(
        ctypes.byref(shape), _p(sel_off), _p(phi_c), _p(dy_c), _p(dw_down), _p(ws), ws_bytes,
        _s(stream)))


def lrm_expert_fc1_wgrad(shape, sel_off, x_c, dab_c, dw_gate, dw_up, ws, ws_bytes, stream=None):
    _check("lrm_expert_fc1_wgrad", _lib.lrm_expert_fc1_wgrad(
        ctypes.byref(shape), _p(sel_off), _p(x_c), _p(dab_c), _p(dw_gate), _p(dw_up), _p(ws),
        ws_bytes, _s(stream)))


def lrm_expert_fc1_dgrad(shape, sel_off, w_gate, w_up, dab_c, dx_c, ws, ws_bytes, stream=None):
    _check("lrm_expert_fc1_dgrad", _lib.lrm_expert_fc1_dgrad(
        ctypes.byref(shape), _p(sel_off), _p(w_gate), _p(w_up), _p(dab_c), _p(dx_c), _p(ws),
        ws_bytes, _s(stream)))


def lrm_scatter_dx(shape, dx_c, inv, row_of_pos, dx, ws, ws_bytes, stream=None):
    _check("lrm_scatter_dx", _lib.lrm_scatter_dx(
        ctypes.byref(shape), _p(dx_c), _p(inv), _p(row_of_pos), _p(dx), _p(ws), ws_bytes,
        _s(stream)))


def lrm_dispatch_permute_noalloc(shape, topk_idx, perm, inv, counts, off, dev_err=None,
                                 stream=None):
    """Dispatch permutation that allocates nothing (scratch built into the library).

    For callers that may not allocate device memory; see include/lrm.h for
    the size limit and the rule that overlapping calls race.
    """
    _check("lrm_dispatch_permute_noalloc", _lib.lrm_dispatch_permute_noalloc(
        ctypes.byref(shape), _p(topk_idx), _p(perm), _p(inv), _p(counts), _p(off),
        _p(dev_err), _s(stream)))


def lrm_selftest_wait_timeout(ws, ws_bytes, stream=None):
    _check("lrm_selftest_wait_timeout",
           _lib.lrm_selftest_wait_timeout(_p(ws), ws_bytes, _s(stream)))


def lrm_score_variant(shape, metric, seed, g, phi, alpha, inv, score, ws, ws_bytes, stream=None):
    _check("lrm_score_variant", _lib.lrm_score_variant(
        ctypes.byref(shape), metric, seed, _p(g), _p(phi), _p(alpha), _p(inv), _p(score),
        _p(ws), ws_bytes, _s(stream)))


def lrm_gather_tokens(shape, perm, x, x_disp, ws, ws_bytes, stream=None):
    _check("lrm_gather_tokens", _lib.lrm_gather_tokens(
        ctypes.byref(shape), _p(perm), _p(x), _p(x_disp), _p(ws), ws_bytes, _s(stream)))


def lrm_expert_fc1_fwd(shape, off, x_disp, w_gate, w_up, ab, phi, ws, ws_bytes, stream=None):
    _check("lrm_expert_fc1_fwd", _lib.lrm_expert_fc1_fwd(
        ctypes.byref(shape), _p(off), _p(x_disp), _p(w_gate), _p(w_up), _p(ab), _p(phi),
        _p(ws), ws_bytes, _s(stream)))


def lrm_expert_fc2_fwd(shape, off, phi, w_down, y, ws, ws_bytes, stream=None):
    _check("lrm_expert_fc2_fwd", _lib.lrm_expert_fc2_fwd(
        ctypes.byref(shape), _p(off), _p(phi), _p(w_down), _p(y), _p(ws), ws_bytes,
        _s(stream)))


def lrm_combine(shape, y, alpha, inv, out, ws, ws_bytes, stream=None):
    _check("lrm_combine", _lib.lrm_combine(
        ctypes.byref(shape), _p(y), _p(alpha), _p(inv), _p(out), _p(ws), ws_bytes,
        _s(stream)))


def lrm_expert_fwd_grouped(shape, perm, inv, off, alpha, x, w_gate, w_up, w_down, x_disp, ab,
                           phi, y, out, ws, ws_bytes, stream=None):
    _check("lrm_expert_fwd_grouped", _lib.lrm_expert_fwd_grouped(
        ctypes.byref(shape), _p(perm), _p(inv), _p(off), _p(alpha), _p(x), _p(w_gate),
        _p(w_up), _p(w_down), _p(x_disp), _p(ab), _p(phi), _p(y), _p(out), _p(ws), ws_bytes,
        _s(stream)))


def lrm_expert_fc1_recompute(shape, sel_off, x_c, w_gate, w_up, ab_c, ws, ws_bytes,
                             stream=None):
    _check("lrm_expert_fc1_recompute", _lib.lrm_expert_fc1_recompute(
        ctypes.byref(shape), _p(sel_off), _p(x_c), _p(w_gate), _p(w_up), _p(ab_c), _p(ws),
        ws_bytes, _s(stream)))


def lrm_expert_bwd_gathered(shape, parts, sel_off, sel_pos, tok_c, w_gate, w_up, w_down, dy_c,
                            x, ab, phi, inv, row_of_pos, dab_c, dx_c, dw_gate, dw_up, dw_down,
                            dx, ws, ws_bytes, stream=None):
    _check("lrm_expert_bwd_gathered", _lib.lrm_expert_bwd_gathered(
        ctypes.byref(shape), parts, _p(sel_off), _p(sel_pos), _p(tok_c), _p(w_gate), _p(w_up),
        _p(w_down), _p(dy_c), _p(x), _p(ab), _p(phi), _p(inv), _p(row_of_pos), _p(dab_c),
        _p(dx_c), _p(dw_gate), _p(dw_up), _p(dw_down), _p(dx), _p(ws), ws_bytes, _s(stream)))


def lrm_select_rate(shape, score, off, num, den, cap, quota, keep, sel_off, sel_pos, ws, ws_bytes,
                    stream=None):
    _check("lrm_select_rate", _lib.lrm_select_rate(
        ctypes.byref(shape), _p(score), _p(off), num, den, cap, _p(quota), _p(keep), _p(sel_off),
        _p(sel_pos), _p(ws), ws_bytes, _s(stream)))
