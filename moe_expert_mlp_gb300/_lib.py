"""ctypes binding of libmoe (include/moe.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, turns torch tensors into device pointers and the current
torch stream into a cudaStream_t, and raises on a non-zero status.  All
computation happens in the library's CUDA kernels.  There is no fallback:
if libmoe.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_DTYPE_BF16 = 1
MOE_DTYPE_MXFP8 = 2
MOE_DTYPE_NVFP4 = 3
MOE_DTYPE_FP32 = 4
MOE_MX_SCALES_ROWMAJOR = 0
MOE_MX_SCALES_MMA = 1
ACTS = {"swiglu": 0, "geglu": 1, "srelu": 2, "sreglu": 3}

EXPORTS = (
    "moe_fc1_padded_width", "moe_workspace_size", "moe_repack_fc1", "moe_unpack_fc1",
    "moe_route_permute", "moe_group_offsets", "moe_mlp_fwd", "moe_unpermute_combine",
    "moe_unpermute_combine_bwd", "moe_mlp_bwd", "moe_permute_bwd", "moe_route_bwd",
    "moe_read_device_status", "moe_status_string", "moe_fc1_glu_fwd", "moe_fc2_fwd",
    "moe_fc2_dgrad_dglu", "moe_fc2_wgrad", "moe_fc1_dgrad", "moe_fc1_wgrad", "moe_bias_grads",
    "moe_route_permute_noalloc", "moe_quantize_mx", "moe_selftest_wait_timeout",
    "moe_fc1_glu_fwd_unfused", "moe_fc2_dgrad_dglu_unfused", "moe_fc1_recompute_h",
    "moe_mx_scale_bytes", "moe_quantize_mx_bf16", "moe_quantize_act_mx",
    "moe_quantize_weights_mx", "moe_mlp_fwd_mx", "moe_mlp_bwd_mx", "moe_fc1_glu_fwd_mx",
    "moe_fc2_fwd_mx", "moe_fc2_dgrad_dglu_mx", "moe_fc2_wgrad_mx", "moe_fc1_dgrad_mx",
    "moe_fc1_wgrad_mx", "moe_route_permute_fused", "moe_nvfp4_scale_bytes", "moe_amax_nvfp4",
    "moe_quantize_nvfp4_bf16", "moe_quantize_act_nvfp4", "moe_quantize_weights_nvfp4",
    "moe_fc1_glu_fwd_nv", "moe_fc2_fwd_nv", "moe_fc2_dgrad_dglu_nv", "moe_fc2_wgrad_nv",
    "moe_fc1_dgrad_nv", "moe_fc1_wgrad_nv", "moe_mlp_fwd_nv", "moe_mlp_bwd_nv",
    "moe_fc1_recompute_h_mx", "moe_fc1_recompute_h_nv", "moe_fc1_glu_fwd_mx_unfused",
    "moe_fc2_dgrad_dglu_mx_unfused", "moe_fc2_dgrad_dglu_recompute",
    "moe_fc2_dgrad_dglu_recompute_mx", "moe_route_permute_mx", "moe_unpermute_combine_bwd_mx",
    "moe_transpose_weights_tf32", "moe_transpose_rows_f32", "moe_fc1_glu_fwd_tf32",
    "moe_fc2_fwd_tf32", "moe_fc2_dgrad_dglu_tf32", "moe_fc2_wgrad_tf32", "moe_fc1_dgrad_tf32",
    "moe_fc1_wgrad_tf32", "moe_selftest_grid_wait_timeout",
)


class MoeError(RuntimeError):
    pass


class moe_mlp_desc_t(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
        ("d", ctypes.c_int32), ("F", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("act", ctypes.c_int32), ("alpha", ctypes.c_float), ("limit", ctypes.c_float),
        ("linear_offset", ctypes.c_float), ("out_scale", ctypes.c_float),
        ("has_b1", ctypes.c_int32), ("has_b2", ctypes.c_int32), ("align", ctypes.c_int32),
        ("sm_margin", ctypes.c_int32), ("capacity", ctypes.c_int32),
        ("recompute_h", ctypes.c_int32),
    ]


class moe_mx_out_t(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("qt", ctypes.c_void_p),
                ("scale_t", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("layout", ctypes.c_int32)]


class moe_mx_weights_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w1", "w1_s", "w1t", "w1t_s", "w2", "w2_s", "w2t", "w2t_s")]


class moe_nv_weights_t(ctypes.Structure):
    _fields_ = [("q", moe_mx_weights_t), ("amax", ctypes.c_void_p)]


def _nvw(w):
    """dict of the eight NVFP4 weight tensors + "amax" (float[4]) ->
    moe_nv_weights_t pointer."""
    q = moe_mx_weights_t(*[_p(w[k]).value for k in
                           ("w1", "w1_s", "w1t", "w1t_s", "w2", "w2_s", "w2t", "w2t_s")])
    return ctypes.byref(moe_nv_weights_t(q, _p(w["amax"]).value))


def _mx(mx):
    """dict of optional tensors {q, scale, qt, scale_t, amax} (+ "layout":
    "mma" for the MMA scale layout) -> struct pointer."""
    if mx is None:
        return None
    st = moe_mx_out_t(*[(_p(mx[k]).value if mx.get(k) is not None else None)
                        for k in ("q", "scale", "qt", "scale_t", "amax")],
                      MOE_MX_SCALES_MMA if mx.get("layout") == "mma" else MOE_MX_SCALES_ROWMAJOR)
    return ctypes.byref(st)


def _mxw(w):
    """dict of the eight MXFP8 weight tensors -> moe_mx_weights_t pointer."""
    st = moe_mx_weights_t(*[_p(w[k]).value for k in
                            ("w1", "w1_s", "w1t", "w1t_s", "w2", "w2_s", "w2t", "w2t_s")])
    return ctypes.byref(st)


def make_desc(T, E, k, d, F, act="swiglu", alpha=1.0, limit=math.inf, linear_offset=0.0,
              out_scale=1.0, has_b1=False, has_b2=False, sm_margin=0, capacity=None,
              recompute_h=False, dtype="bf16"):
    if capacity is None:
        capacity = T * k + E * 127
        capacity = (capacity + 127) // 128 * 128
    dt = {"bf16": MOE_DTYPE_BF16, "mxfp8": MOE_DTYPE_MXFP8, "nvfp4": MOE_DTYPE_NVFP4,
          "fp32": MOE_DTYPE_FP32}[dtype]
    return moe_mlp_desc_t(T, E, k, d, F, dt, ACTS[act], alpha, limit, linear_offset,
                          out_scale, int(has_b1), int(has_b2), 128, sm_margin, capacity,
                          int(recompute_h))


_lib = None


def lib():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoeError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        D = ctypes.POINTER(moe_mlp_desc_t)
        sig = {
            "moe_fc1_padded_width": (ctypes.c_int32, [ctypes.c_int32]),
            "moe_workspace_size": (ctypes.c_int, [D, ctypes.POINTER(ctypes.c_size_t)]),
            "moe_repack_fc1": (ctypes.c_int, [D, P, P, P, P, P]),
            "moe_unpack_fc1": (ctypes.c_int, [D, P, P, ctypes.c_int32, P]),
            "moe_route_permute": (ctypes.c_int, [D] + [P] * 13 + [ctypes.c_size_t, P]),
            "moe_group_offsets": (ctypes.c_int, [D, P, P, P, P, P]),
            "moe_mlp_fwd": (ctypes.c_int, [D] + [P] * 13 + [ctypes.c_size_t, P]),
            "moe_unpermute_combine": (ctypes.c_int, [D, P, P, P, P, P]),
            "moe_unpermute_combine_bwd": (ctypes.c_int, [D] + [P] * 8 + [P]),
            "moe_mlp_bwd": (ctypes.c_int, [D] + [P] * 17 + [ctypes.c_size_t, P]),
            "moe_permute_bwd": (ctypes.c_int, [D, P, P, P, P]),
            "moe_route_bwd": (ctypes.c_int, [D, P, P, P, P, P]),
            "moe_read_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), ctypes.c_int32]),
            "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "moe_fc1_glu_fwd": (ctypes.c_int, [D] + [P] * 9),
            "moe_fc2_fwd": (ctypes.c_int, [D] + [P] * 8),
            "moe_fc2_dgrad_dglu": (ctypes.c_int, [D] + [P] * 8),
            "moe_fc2_wgrad": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_dgrad": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_wgrad": (ctypes.c_int, [D] + [P] * 6),
            "moe_bias_grads": (ctypes.c_int, [D] + [P] * 7),
            "moe_route_permute_noalloc": (ctypes.c_int, [D] + [P] * 12 + [P]),
            "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, P]),
            "moe_selftest_grid_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, P]),
            "moe_fc1_glu_fwd_unfused": (ctypes.c_int, [D] + [P] * 8),
            "moe_fc1_recompute_h": (ctypes.c_int, [D] + [P] * 7),
            "moe_fc2_dgrad_dglu_unfused": (ctypes.c_int, [D] + [P] * 8),
            "moe_quantize_mx": (ctypes.c_int, [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               P, P, P]),
            "moe_mx_scale_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
            "moe_quantize_mx_bf16": (ctypes.c_int, [P, ctypes.c_int64, ctypes.c_int64,
                                                    ctypes.c_int64, P, P]),
            "moe_quantize_act_mx": (ctypes.c_int, [D, P, ctypes.c_int32, P, P, P]),
            "moe_quantize_weights_mx": (ctypes.c_int, [D, P, P, P, P]),
            "moe_mlp_fwd_mx": (ctypes.c_int, [D] + [P] * 11),
            "moe_mlp_bwd_mx": (ctypes.c_int, [D] + [P] * 16),
            "moe_fc1_glu_fwd_mx": (ctypes.c_int, [D] + [P] * 9),
            "moe_route_permute_fused": (ctypes.c_int, [D] + [P] * 14 + [ctypes.c_size_t, P]),
            "moe_fc2_fwd_mx": (ctypes.c_int, [D] + [P] * 7),
            "moe_fc2_dgrad_dglu_mx": (ctypes.c_int, [D] + [P] * 8),
            "moe_fc2_wgrad_mx": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_dgrad_mx": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_wgrad_mx": (ctypes.c_int, [D] + [P] * 6),
            "moe_nvfp4_scale_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
            "moe_amax_nvfp4": (ctypes.c_int, [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                              P, P, P]),
            "moe_quantize_nvfp4_bf16": (ctypes.c_int, [P, ctypes.c_int64, ctypes.c_int64,
                                                       ctypes.c_int64, P, ctypes.c_int32, P]),
            "moe_quantize_act_nvfp4": (ctypes.c_int, [D, P, ctypes.c_int32, P, P,
                                                      ctypes.c_int32, P]),
            "moe_quantize_weights_nvfp4": (ctypes.c_int, [D, P, P, P, P]),
            "moe_fc1_glu_fwd_nv": (ctypes.c_int, [D] + [P] * 9),
            "moe_fc2_fwd_nv": (ctypes.c_int, [D] + [P] * 7),
            "moe_fc2_dgrad_dglu_nv": (ctypes.c_int, [D] + [P] * 8),
            "moe_fc2_wgrad_nv": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_dgrad_nv": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_wgrad_nv": (ctypes.c_int, [D] + [P] * 6),
            "moe_mlp_fwd_nv": (ctypes.c_int, [D] + [P] * 12),
            "moe_fc1_recompute_h_mx": (ctypes.c_int, [D] + [P] * 7),
            "moe_fc1_glu_fwd_mx_unfused": (ctypes.c_int, [D] + [P] * 9),
            "moe_fc2_dgrad_dglu_recompute": (ctypes.c_int, [D] + [P] * 10),
            "moe_route_permute_mx": (ctypes.c_int, [D] + [P] * 14 + [ctypes.c_size_t, P]),
            "moe_unpermute_combine_bwd_mx": (ctypes.c_int, [D] + [P] * 9 + [P]),
            "moe_fc2_dgrad_dglu_recompute_mx": (ctypes.c_int, [D] + [P] * 9),
            "moe_fc2_dgrad_dglu_mx_unfused": (ctypes.c_int, [D] + [P] * 9),
            "moe_fc1_recompute_h_nv": (ctypes.c_int, [D] + [P] * 7),
            "moe_mlp_bwd_nv": (ctypes.c_int, [D] + [P] * 16),
            "moe_transpose_weights_tf32": (ctypes.c_int, [D] + [P] * 5),
            "moe_transpose_rows_f32": (ctypes.c_int, [D, P, ctypes.c_int32, P, P, P]),
            "moe_fc1_glu_fwd_tf32": (ctypes.c_int, [D] + [P] * 9),
            "moe_fc2_fwd_tf32": (ctypes.c_int, [D] + [P] * 7),
            "moe_fc2_dgrad_dglu_tf32": (ctypes.c_int, [D] + [P] * 8),
            "moe_fc2_wgrad_tf32": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_dgrad_tf32": (ctypes.c_int, [D] + [P] * 6),
            "moe_fc1_wgrad_tf32": (ctypes.c_int, [D] + [P] * 6),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(st):
    if st != 0:
        msg = lib().moe_status_string(st).decode()
        raise MoeError(f"libmoe status {st}: {msg}")


def moe_fc1_padded_width(F):
    return int(lib().moe_fc1_padded_width(F))


def moe_workspace_size(desc):
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def moe_repack_fc1(desc, w1, b1, w1p, b1p, stream=None):
    _check(lib().moe_repack_fc1(ctypes.byref(desc), _p(w1), _p(b1), _p(w1p), _p(b1p), _stream(stream)))


def moe_unpack_fc1(desc, w1p, w1, rows_width, stream=None):
    _check(lib().moe_unpack_fc1(ctypes.byref(desc), _p(w1p), _p(w1), rows_width, _stream(stream)))


def moe_route_permute(desc, logits, bias, x, topk_idx, topk_w, counts, offsets, padded_offsets,
                      tile_prefix, row_src, row_of, x_perm, ws, stream=None):
    _check(lib().moe_route_permute(
        ctypes.byref(desc), _p(logits), _p(bias), _p(x), _p(topk_idx), _p(topk_w), _p(counts),
        _p(offsets), _p(padded_offsets), _p(tile_prefix), _p(row_src), _p(row_of), _p(x_perm),
        _p(ws), ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream)))


def moe_route_permute_fused(desc, x, w_router, bias, logits, topk_idx, topk_w, counts, offsets,
                            padded_offsets, tile_prefix, row_src, row_of, x_perm, ws,
                            stream=None):
    _check(lib().moe_route_permute_fused(
        ctypes.byref(desc), _p(x), _p(w_router), _p(bias), _p(logits), _p(topk_idx), _p(topk_w),
        _p(counts), _p(offsets), _p(padded_offsets), _p(tile_prefix), _p(row_src), _p(row_of),
        _p(x_perm), _p(ws), ws.numel() * ws.element_size() if ws is not None else 0,
        _stream(stream)))


def moe_group_offsets(desc, counts, offsets, padded_offsets, tile_prefix, stream=None):
    _check(lib().moe_group_offsets(ctypes.byref(desc), _p(counts), _p(offsets), _p(padded_offsets),
                                   _p(tile_prefix), _stream(stream)))


def moe_mlp_fwd(desc, x_perm, counts, padded_offsets, w1p, b1p, w2, b2, h, a, y, ws=None,
                stream=None, a_mx=None, y_mx=None):
    _check(lib().moe_mlp_fwd(
        ctypes.byref(desc), _p(x_perm), _p(counts), _p(padded_offsets), _p(w1p), _p(b1p), _p(w2),
        _p(b2), _p(h), _p(a), _p(y), _mx(a_mx), _mx(y_mx), _p(ws),
        ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream)))


def moe_unpermute_combine(desc, y, row_of, topk_w, out, stream=None):
    _check(lib().moe_unpermute_combine(ctypes.byref(desc), _p(y), _p(row_of), _p(topk_w), _p(out),
                                       _stream(stream)))


def moe_unpermute_combine_bwd(desc, dout, y, row_of, topk_w, row_src, padded_offsets, dy, dw,
                              stream=None):
    _check(lib().moe_unpermute_combine_bwd(
        ctypes.byref(desc), _p(dout), _p(y), _p(row_of), _p(topk_w), _p(row_src),
        _p(padded_offsets), _p(dy), _p(dw), _stream(stream)))


def moe_mlp_bwd(desc, dy, x_perm, h, a, counts, padded_offsets, w1p, w2, dh, dx_perm, dw1p, db1p,
                dw2, db2, ws=None, stream=None, dh_mx=None, b1p=None):
    _check(lib().moe_mlp_bwd(
        ctypes.byref(desc), _p(dy), _p(x_perm), _p(h), _p(a), _p(counts), _p(padded_offsets),
        _p(w1p), _p(b1p), _p(w2), _p(dh), _p(dx_perm), _p(dw1p), _p(db1p), _p(dw2), _p(db2),
        _mx(dh_mx), _p(ws), ws.numel() * ws.element_size() if ws is not None else 0,
        _stream(stream)))


def moe_permute_bwd(desc, dx_perm, row_of, dx, stream=None):
    _check(lib().moe_permute_bwd(ctypes.byref(desc), _p(dx_perm), _p(row_of), _p(dx), _stream(stream)))


def moe_route_bwd(desc, dw, topk_w, topk_idx, dlogits, stream=None):
    _check(lib().moe_route_bwd(ctypes.byref(desc), _p(dw), _p(topk_w), _p(topk_idx), _p(dlogits),
                               _stream(stream)))


def moe_read_device_status(clear=True):
    v = ctypes.c_int32(0)
    _check(lib().moe_read_device_status(ctypes.byref(v), int(clear)))
    return int(v.value)


def moe_fc1_glu_fwd(desc, x_perm, counts, padded_offsets, w1p, b1p, h, a, stream=None, mx=None):
    _check(lib().moe_fc1_glu_fwd(ctypes.byref(desc), _p(x_perm), _p(counts), _p(padded_offsets),
                                 _p(w1p), _p(b1p), _p(h), _p(a), _mx(mx), _stream(stream)))


def moe_fc2_fwd(desc, a, counts, padded_offsets, w2, b2, y, stream=None, mx=None):
    _check(lib().moe_fc2_fwd(ctypes.byref(desc), _p(a), _p(counts), _p(padded_offsets), _p(w2),
                             _p(b2), _p(y), _mx(mx), _stream(stream)))


def moe_fc2_dgrad_dglu(desc, dy, h, counts, padded_offsets, w2, dh, stream=None, mx=None):
    _check(lib().moe_fc2_dgrad_dglu(ctypes.byref(desc), _p(dy), _p(h), _p(counts),
                                    _p(padded_offsets), _p(w2), _p(dh), _mx(mx), _stream(stream)))


def moe_fc2_wgrad(desc, dy, a, counts, padded_offsets, dw2, stream=None):
    _check(lib().moe_fc2_wgrad(ctypes.byref(desc), _p(dy), _p(a), _p(counts), _p(padded_offsets),
                               _p(dw2), _stream(stream)))


def moe_fc1_dgrad(desc, dh, counts, padded_offsets, w1p, dx_perm, stream=None):
    _check(lib().moe_fc1_dgrad(ctypes.byref(desc), _p(dh), _p(counts), _p(padded_offsets), _p(w1p),
                               _p(dx_perm), _stream(stream)))


def moe_fc1_wgrad(desc, dh, x_perm, counts, padded_offsets, dw1p, stream=None):
    _check(lib().moe_fc1_wgrad(ctypes.byref(desc), _p(dh), _p(x_perm), _p(counts),
                               _p(padded_offsets), _p(dw1p), _stream(stream)))


def moe_bias_grads(desc, dy, dh, counts, padded_offsets, db1p, db2, stream=None):
    _check(lib().moe_bias_grads(ctypes.byref(desc), _p(dy), _p(dh), _p(counts),
                                _p(padded_offsets), _p(db1p), _p(db2), _stream(stream)))


def moe_selftest_wait_timeout(limit_us, stream=None):
    _check(lib().moe_selftest_wait_timeout(int(limit_us), _stream(stream)))


def moe_selftest_grid_wait_timeout(limit_us, stream=None):
    _check(lib().moe_selftest_grid_wait_timeout(int(limit_us), _stream(stream)))


def moe_quantize_mx(x, colwise, q, scales, stream=None):
    """MXFP8-quantize fp32 x [rows, cols] rowwise (colwise=False) or
    columnwise into the transposed q (colwise=True)."""
    rows, cols = x.shape
    _check(lib().moe_quantize_mx(_p(x), rows, cols, int(bool(colwise)), _p(q), _p(scales),
                                 _stream(stream)))


def moe_route_permute_noalloc(desc, logits, bias, x, topk_idx, topk_w, counts, offsets,
                              padded_offsets, tile_prefix, row_src, row_of, x_perm, stream=None):
    """moe_route_permute without a caller-provided workspace (see include/moe.h)."""
    _check(lib().moe_route_permute_noalloc(
        ctypes.byref(desc), _p(logits), _p(bias), _p(x), _p(topk_idx), _p(topk_w), _p(counts),
        _p(offsets), _p(padded_offsets), _p(tile_prefix), _p(row_src), _p(row_of), _p(x_perm),
        _stream(stream)))


def moe_fc1_glu_fwd_unfused(desc, x_perm, counts, padded_offsets, w1p, b1p, h, a, stream=None):
    _check(lib().moe_fc1_glu_fwd_unfused(ctypes.byref(desc), _p(x_perm), _p(counts),
                                         _p(padded_offsets), _p(w1p), _p(b1p), _p(h), _p(a),
                                         _stream(stream)))


def moe_fc2_dgrad_dglu_unfused(desc, dy, h, counts, padded_offsets, w2, da, dh, stream=None):
    _check(lib().moe_fc2_dgrad_dglu_unfused(ctypes.byref(desc), _p(dy), _p(h), _p(counts),
                                            _p(padded_offsets), _p(w2), _p(da), _p(dh),
                                            _stream(stream)))


def moe_fc1_recompute_h(desc, x_perm, counts, padded_offsets, w1p, b1p, h, stream=None):
    _check(lib().moe_fc1_recompute_h(ctypes.byref(desc), _p(x_perm), _p(counts),
                                     _p(padded_offsets), _p(w1p), _p(b1p), _p(h), _stream(stream)))


# ------------------------------------------------------------------ MXFP8
def moe_mx_scale_bytes(rows, cols):
    return int(lib().moe_mx_scale_bytes(rows, cols))


def moe_quantize_mx_bf16(inp, batch, rows, cols, out, stream=None):
    _check(lib().moe_quantize_mx_bf16(_p(inp), batch, rows, cols, _mx(out), _stream(stream)))


def moe_quantize_act_mx(desc, inp, width, padded_offsets, out, stream=None):
    _check(lib().moe_quantize_act_mx(ctypes.byref(desc), _p(inp), width, _p(padded_offsets),
                                     _mx(out), _stream(stream)))


def moe_quantize_weights_mx(desc, w1p, w2, out, stream=None):
    _check(lib().moe_quantize_weights_mx(ctypes.byref(desc), _p(w1p), _p(w2), _mxw(out),
                                         _stream(stream)))


def moe_mlp_fwd_mx(desc, x_mx, counts, padded_offsets, w_mx, b1p, b2, h, a, a_mx, y,
                   stream=None):
    _check(lib().moe_mlp_fwd_mx(ctypes.byref(desc), _mx(x_mx), _p(counts), _p(padded_offsets),
                                _mxw(w_mx), _p(b1p), _p(b2), _p(h), _p(a), _mx(a_mx), _p(y),
                                _stream(stream)))


def moe_mlp_bwd_mx(desc, dy, dy_mx, x_mx, h, a_mx, counts, padded_offsets, w_mx, dh, dh_mx,
                   dx_perm, dw1p, db1p, dw2, db2, stream=None):
    _check(lib().moe_mlp_bwd_mx(ctypes.byref(desc), _p(dy), _mx(dy_mx), _mx(x_mx), _p(h),
                                _mx(a_mx), _p(counts), _p(padded_offsets), _mxw(w_mx), _p(dh),
                                _mx(dh_mx), _p(dx_perm), _p(dw1p), _p(db1p), _p(dw2), _p(db2),
                                _stream(stream)))


def moe_fc1_glu_fwd_mx(desc, x_mx, counts, padded_offsets, w_mx, b1p, h, a, a_mx, stream=None):
    _check(lib().moe_fc1_glu_fwd_mx(ctypes.byref(desc), _mx(x_mx), _p(counts),
                                    _p(padded_offsets), _mxw(w_mx), _p(b1p), _p(h), _p(a),
                                    _mx(a_mx), _stream(stream)))


def moe_fc2_fwd_mx(desc, a_mx, counts, padded_offsets, w_mx, b2, y, stream=None):
    _check(lib().moe_fc2_fwd_mx(ctypes.byref(desc), _mx(a_mx), _p(counts), _p(padded_offsets),
                                _mxw(w_mx), _p(b2), _p(y), _stream(stream)))


def moe_fc2_dgrad_dglu_mx(desc, dy_mx, h, counts, padded_offsets, w_mx, dh, dh_mx,
                          stream=None):
    _check(lib().moe_fc2_dgrad_dglu_mx(ctypes.byref(desc), _mx(dy_mx), _p(h), _p(counts),
                                       _p(padded_offsets), _mxw(w_mx), _p(dh), _mx(dh_mx),
                                       _stream(stream)))


def moe_fc2_wgrad_mx(desc, dy_mx, a_mx, counts, padded_offsets, dw2, stream=None):
    _check(lib().moe_fc2_wgrad_mx(ctypes.byref(desc), _mx(dy_mx), _mx(a_mx), _p(counts),
                                  _p(padded_offsets), _p(dw2), _stream(stream)))


def moe_fc1_dgrad_mx(desc, dh_mx, counts, padded_offsets, w_mx, dx_perm, stream=None):
    _check(lib().moe_fc1_dgrad_mx(ctypes.byref(desc), _mx(dh_mx), _p(counts),
                                  _p(padded_offsets), _mxw(w_mx), _p(dx_perm), _stream(stream)))


def moe_fc1_wgrad_mx(desc, dh_mx, x_mx, counts, padded_offsets, dw1p, stream=None):
    _check(lib().moe_fc1_wgrad_mx(ctypes.byref(desc), _mx(dh_mx), _mx(x_mx), _p(counts),
                                  _p(padded_offsets), _p(dw1p), _stream(stream)))


# ------------------------------------------------------------------ NVFP4
def moe_nvfp4_scale_bytes(rows, cols):
    return int(lib().moe_nvfp4_scale_bytes(rows, cols))


def moe_amax_nvfp4(inp, batch, rows, cols, amax, row_limit=None, stream=None):
    _check(lib().moe_amax_nvfp4(_p(inp), batch, rows, cols, _p(row_limit), _p(amax),
                                _stream(stream)))


def moe_quantize_nvfp4_bf16(inp, batch, rows, cols, out, rotate_t=False, stream=None):
    _check(lib().moe_quantize_nvfp4_bf16(_p(inp), batch, rows, cols, _mx(out),
                                         int(bool(rotate_t)), _stream(stream)))


def moe_quantize_act_nvfp4(desc, inp, width, padded_offsets, out, compute_amax, stream=None):
    _check(lib().moe_quantize_act_nvfp4(ctypes.byref(desc), _p(inp), width, _p(padded_offsets),
                                        _mx(out), int(bool(compute_amax)), _stream(stream)))


def moe_quantize_weights_nvfp4(desc, w1p, w2, out, stream=None):
    _check(lib().moe_quantize_weights_nvfp4(ctypes.byref(desc), _p(w1p), _p(w2), _nvw(out),
                                            _stream(stream)))


def moe_fc1_glu_fwd_nv(desc, x_nv, counts, padded_offsets, w_nv, b1p, h, a, a_amax, stream=None):
    _check(lib().moe_fc1_glu_fwd_nv(ctypes.byref(desc), _mx(x_nv), _p(counts),
                                    _p(padded_offsets), _nvw(w_nv), _p(b1p), _p(h), _p(a),
                                    _p(a_amax), _stream(stream)))


def moe_fc2_fwd_nv(desc, a_nv, counts, padded_offsets, w_nv, b2, y, stream=None):
    _check(lib().moe_fc2_fwd_nv(ctypes.byref(desc), _mx(a_nv), _p(counts), _p(padded_offsets),
                                _nvw(w_nv), _p(b2), _p(y), _stream(stream)))


def moe_fc2_dgrad_dglu_nv(desc, dy_nv, h, counts, padded_offsets, w_nv, dh, dh_amax,
                          stream=None):
    _check(lib().moe_fc2_dgrad_dglu_nv(ctypes.byref(desc), _mx(dy_nv), _p(h), _p(counts),
                                       _p(padded_offsets), _nvw(w_nv), _p(dh), _p(dh_amax),
                                       _stream(stream)))


def moe_fc2_wgrad_nv(desc, dy_nv, a_nv, counts, padded_offsets, dw2, stream=None):
    _check(lib().moe_fc2_wgrad_nv(ctypes.byref(desc), _mx(dy_nv), _mx(a_nv), _p(counts),
                                  _p(padded_offsets), _p(dw2), _stream(stream)))


def moe_fc1_dgrad_nv(desc, dh_nv, counts, padded_offsets, w_nv, dx_perm, stream=None):
    _check(lib().moe_fc1_dgrad_nv(ctypes.byref(desc), _mx(dh_nv), _p(counts),
                                  _p(padded_offsets), _nvw(w_nv), _p(dx_perm), _stream(stream)))


def moe_fc1_wgrad_nv(desc, dh_nv, x_nv, counts, padded_offsets, dw1p, stream=None):
    _check(lib().moe_fc1_wgrad_nv(ctypes.byref(desc), _mx(dh_nv), _mx(x_nv), _p(counts),
                                  _p(padded_offsets), _p(dw1p), _stream(stream)))


def moe_mlp_fwd_nv(desc, x_perm, x_nv, counts, padded_offsets, w_nv, b1p, b2, h, a, a_nv, y,
                   stream=None):
    _check(lib().moe_mlp_fwd_nv(ctypes.byref(desc), _p(x_perm), _mx(x_nv), _p(counts),
                                _p(padded_offsets), _nvw(w_nv), _p(b1p), _p(b2), _p(h), _p(a),
                                _mx(a_nv), _p(y), _stream(stream)))


def moe_mlp_bwd_nv(desc, dy, dy_nv, x_nv, h, a_nv, counts, padded_offsets, w_nv, dh, dh_nv,
                   dx_perm, dw1p, db1p, dw2, db2, stream=None):
    _check(lib().moe_mlp_bwd_nv(ctypes.byref(desc), _p(dy), _mx(dy_nv), _mx(x_nv), _p(h),
                                _mx(a_nv), _p(counts), _p(padded_offsets), _nvw(w_nv), _p(dh),
                                _mx(dh_nv), _p(dx_perm), _p(dw1p), _p(db1p), _p(dw2), _p(db2),
                                _stream(stream)))


def moe_fc1_recompute_h_mx(desc, x_mx, counts, padded_offsets, w_mx, b1p, h, stream=None):
    _check(lib().moe_fc1_recompute_h_mx(ctypes.byref(desc), _mx(x_mx), _p(counts),
                                        _p(padded_offsets), _mxw(w_mx), _p(b1p), _p(h),
                                        _stream(stream)))


def moe_route_permute_mx(desc, logits, bias, x, topk_idx, topk_w, counts, offsets,
                         padded_offsets, tile_prefix, row_src, row_of, x_perm, x_mx, ws,
                         stream=None):
    """moe_route_permute that also writes x_perm's rowwise MXFP8 copy."""
    _check(lib().moe_route_permute_mx(
        ctypes.byref(desc), _p(logits), _p(bias), _p(x), _p(topk_idx), _p(topk_w), _p(counts),
        _p(offsets), _p(padded_offsets), _p(tile_prefix), _p(row_src), _p(row_of), _p(x_perm),
        _mx(x_mx), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_unpermute_combine_bwd_mx(desc, dout, y, row_of, topk_w, row_src, padded_offsets, dy,
                                 dy_mx, dw, stream=None):
    """moe_unpermute_combine_bwd that also writes dy's rowwise MXFP8 copy."""
    _check(lib().moe_unpermute_combine_bwd_mx(
        ctypes.byref(desc), _p(dout), _p(y), _p(row_of), _p(topk_w), _p(row_src),
        _p(padded_offsets), _p(dy), _mx(dy_mx), _p(dw), _stream(stream)))


def moe_fc2_dgrad_dglu_recompute(desc, x_perm, dy, counts, padded_offsets, w1p, b1p, w2, dh,
                                 stream=None, mx=None):
    """FC2 dgrad + dGLU with H recomputed inside the kernel (see include/moe.h)."""
    _check(lib().moe_fc2_dgrad_dglu_recompute(ctypes.byref(desc), _p(x_perm), _p(dy), _p(counts),
                                              _p(padded_offsets), _p(w1p), _p(b1p), _p(w2),
                                              _p(dh), _mx(mx), _stream(stream)))


def moe_fc2_dgrad_dglu_recompute_mx(desc, x_mx, dy_mx, counts, padded_offsets, w_mx, b1p, dh,
                                    dh_mx, stream=None):
    """The same on the MXFP8 operands (see include/moe.h)."""
    _check(lib().moe_fc2_dgrad_dglu_recompute_mx(ctypes.byref(desc), _mx(x_mx), _mx(dy_mx),
                                                 _p(counts), _p(padded_offsets), _mxw(w_mx),
                                                 _p(b1p), _p(dh), _mx(dh_mx), _stream(stream)))


def moe_fc1_glu_fwd_mx_unfused(desc, x_mx, counts, padded_offsets, w_mx, b1p, h, a, a_mx,
                               stream=None):
    """FC1 plain GEMM, GLU pass, MXFP8 quantize pass (see include/moe.h)."""
    _check(lib().moe_fc1_glu_fwd_mx_unfused(ctypes.byref(desc), _mx(x_mx), _p(counts),
                                            _p(padded_offsets), _mxw(w_mx), _p(b1p), _p(h), _p(a),
                                            _mx(a_mx), _stream(stream)))


def moe_fc2_dgrad_dglu_mx_unfused(desc, dy_mx, h, counts, padded_offsets, w_mx, da, dh, dh_mx,
                                  stream=None):
    """FC2 dgrad plain GEMM, dGLU pass, MXFP8 quantize pass (see include/moe.h)."""
    _check(lib().moe_fc2_dgrad_dglu_mx_unfused(ctypes.byref(desc), _mx(dy_mx), _p(h), _p(counts),
                                               _p(padded_offsets), _mxw(w_mx), _p(da), _p(dh),
                                               _mx(dh_mx), _stream(stream)))


def moe_fc1_recompute_h_nv(desc, x_nv, counts, padded_offsets, w_nv, b1p, h, stream=None):
    _check(lib().moe_fc1_recompute_h_nv(ctypes.byref(desc), _mx(x_nv), _p(counts),
                                        _p(padded_offsets), _nvw(w_nv), _p(b1p), _p(h),
                                        _stream(stream)))


# ------------------------------------------------------- fp32 / TF32 path
def moe_transpose_weights_tf32(desc, w1p, w2, w1t, w2t, stream=None):
    _check(lib().moe_transpose_weights_tf32(ctypes.byref(desc), _p(w1p), _p(w2), _p(w1t),
                                            _p(w2t), _stream(stream)))


def moe_transpose_rows_f32(desc, x, width, padded_offsets, out, stream=None):
    _check(lib().moe_transpose_rows_f32(ctypes.byref(desc), _p(x), width, _p(padded_offsets),
                                        _p(out), _stream(stream)))


def moe_fc1_glu_fwd_tf32(desc, x_perm, counts, padded_offsets, w1p, b1p, h, a, a_t=None,
                         stream=None):
    _check(lib().moe_fc1_glu_fwd_tf32(ctypes.byref(desc), _p(x_perm), _p(counts),
                                      _p(padded_offsets), _p(w1p), _p(b1p), _p(h), _p(a),
                                      _p(a_t), _stream(stream)))


def moe_fc2_fwd_tf32(desc, a, counts, padded_offsets, w2, b2, y, stream=None):
    _check(lib().moe_fc2_fwd_tf32(ctypes.byref(desc), _p(a), _p(counts), _p(padded_offsets),
                                  _p(w2), _p(b2), _p(y), _stream(stream)))


def moe_fc2_dgrad_dglu_tf32(desc, dy, h, counts, padded_offsets, w2t, dh, dh_t=None,
                            stream=None):
    _check(lib().moe_fc2_dgrad_dglu_tf32(ctypes.byref(desc), _p(dy), _p(h), _p(counts),
                                         _p(padded_offsets), _p(w2t), _p(dh), _p(dh_t),
                                         _stream(stream)))


def moe_fc2_wgrad_tf32(desc, dy_t, a_t, counts, padded_offsets, dw2, stream=None):
    _check(lib().moe_fc2_wgrad_tf32(ctypes.byref(desc), _p(dy_t), _p(a_t), _p(counts),
                                    _p(padded_offsets), _p(dw2), _stream(stream)))


def moe_fc1_dgrad_tf32(desc, dh, counts, padded_offsets, w1t, dx_perm, stream=None):
    _check(lib().moe_fc1_dgrad_tf32(ctypes.byref(desc), _p(dh), _p(counts), _p(padded_offsets),
                                    _p(w1t), _p(dx_perm), _stream(stream)))


def moe_fc1_wgrad_tf32(desc, dh_t, x_t, counts, padded_offsets, dw1p, stream=None):
    _check(lib().moe_fc1_wgrad_tf32(ctypes.byref(desc), _p(dh_t), _p(x_t), _p(counts),
                                    _p(padded_offsets), _p(dw1p), _stream(stream)))
