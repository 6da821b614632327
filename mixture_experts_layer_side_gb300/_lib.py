"""ctypes binding of libmok.so (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors for device buffers, and passes their data pointers, sizes and the
current CUDA stream through the C ABI declared in ``include/mok.h``.  No step
of the layer runs in Python; if the library is missing the import fails.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmok.so")

MOK_BF16 = 0
MOK_MXFP8 = 1
MOK_DEBUG_SKIP_RING_SIGNAL = 1
MOK_DEBUG_SERIAL_RING = 2
MOK_DEBUG_FUSED_WGRAD_GATHER = 4
MOK_DEBUG_SINGLE_CTA_WGRAD = 8
MOK_DEBUG_SINGLE_CTA_ROWS = 16
MOK_DEBUG_SINGLE_CTA_RING = 32
MOK_DEBUG_GATHER_X_RING = 64
MOK_DEBUG_NO_OVERLAP = 128

STATUS = {0: "MOK_OK", 1: "MOK_ERR_INVALID_ARG", 2: "MOK_ERR_UNSUPPORTED", 3: "MOK_ERR_WORKSPACE_TOO_SMALL",
          4: "MOK_ERR_CUDA", 5: "MOK_ERR_BAD_INDEX", 6: "MOK_ERR_TIMEOUT"}

# every entry point include/mok.h declares
EXPORTS = ["mok_workspace_size", "mok_ctx_size", "mok_workspace_layout", "mok_build_schedule", "mok_forward",
           "mok_forward_fused",
           "mok_backward", "mok_mxfp8_quantize", "mok_gather_rows", "mok_gemm_bf16", "mok_check",
           "mok_device_sm_count", "mok_status_string", "mok_version", "mok_trace_enable", "mok_trace_read",
           "mok_launch_count", "mok_build_schedule_noalloc", "mok_gemm_mxfp8", "mok_router_workspace_size",
           "mok_router_forward", "mok_router_backward", "mok_schedule_workspace_size", "mok_ep_first_expert",
           "mok_ep_plan", "mok_ep_pack_rows", "mok_ep_combine_rows", "mok_ep_unsort_scores"]

PHASES = ["schedule", "fwd_gemm", "fwd_combine", "bwd_da", "bwd_ds", "bwd_dx", "bwd_dx_combine", "bwd_wg13",
          "bwd_wg2", "quant", "bwd_sort", "router_fwd", "router_bwd", "bwd_replay", "fwd_fused", "fwd_sort"]


class MokError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class MokShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32)]


class MokConfig(ctypes.Structure):
    _fields_ = [("minibatch_rows", ctypes.c_int32), ("ring_slots", ctypes.c_int32),
                ("capacity_mult", ctypes.c_float), ("comm_sms", ctypes.c_int32), ("debug_flags", ctypes.c_int32),
                ("replay", ctypes.c_int32), ("overlap_sms", ctypes.c_int32)]


class MokMx(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class MokLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("header", "counts", "offsets", "padded_offsets", "perm", "inv_perm",
                                               "pad_perm", "pad_inv", "tile_expert")] + \
               [("pad_capacity", ctypes.c_int64), ("tile_capacity", ctypes.c_int64)]


class MokScheduleBuffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("header", "counts", "offsets", "padded_offsets", "perm",
                                               "inv_perm", "pad_perm", "pad_inv", "tile_expert")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run mixture_experts_layer_side_gb300.build.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    S = ctypes.POINTER(MokShape)
    C = ctypes.POINTER(MokConfig)
    i32, sz = ctypes.c_int32, ctypes.c_size_t
    sig = {
        "mok_workspace_size": (sz, [S, C, i32]),
        "mok_ctx_size": (sz, [S, C, i32]),
        "mok_workspace_layout": (i32, [S, C, i32, ctypes.POINTER(MokLayout)]),
        "mok_build_schedule": (i32, [S, C, P, sz, P, P]),
        "mok_forward": (i32, [S, C, i32, P, sz, P, P, P, P, P, P, P, P]),
        "mok_forward_fused": (i32, [S, C, i32, P, sz, P, P, P, P, P, P, P, P, P]),
        "mok_backward": (i32, [S, C, i32, P, sz, P, P, P, P, P, P, P, P, P, P, P, P, P]),
        "mok_mxfp8_quantize": (i32, [P, i32, i32, i32, i32, P, P, P]),
        "mok_gather_rows": (i32, [S, C, P, sz, P, P, P]),
        "mok_gemm_bf16": (i32, [i32, i32, i32, P, i32, P, i32, P, P, P]),
        "mok_check": (i32, [P, P]),
        "mok_device_sm_count": (i32, []),
        "mok_status_string": (ctypes.c_char_p, [i32]),
        "mok_version": (ctypes.c_char_p, []),
        "mok_trace_enable": (i32, [i32]),
        "mok_trace_read": (i32, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int32)]),
        "mok_launch_count": (ctypes.c_int64, []),
        "mok_build_schedule_noalloc": (i32, [S, P, ctypes.POINTER(MokScheduleBuffers), P]),
        "mok_gemm_mxfp8": (i32, [i32, i32, i32, P, P, i32, P, P, i32, P, P, sz, P]),
        "mok_router_workspace_size": (sz, [S]),
        "mok_router_forward": (i32, [S, P, sz, P, P, P, P, P, P, P]),
        "mok_router_backward": (i32, [S, P, sz, P, P, P, P, P, P, P, P]),
        "mok_schedule_workspace_size": (sz, [S, C]),
        "mok_ep_first_expert": (i32, [i32, i32, i32]),
        "mok_ep_plan": (i32, [i32, i32, i32, P, P, P, P, P, ctypes.c_int64, P]),
        "mok_ep_pack_rows": (i32, [S, C, P, sz, P, P, P, P, P]),
        "mok_ep_combine_rows": (i32, [S, C, P, sz, P, P, P, P]),
        "mok_ep_unsort_scores": (i32, [S, C, P, sz, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, MokMx):
        return ctypes.cast(ctypes.pointer(t), ctypes.c_void_p)
    if isinstance(t, ctypes.Array):  # consecutive mok_mx descriptors
        return ctypes.cast(t, ctypes.c_void_p)
    return ctypes.c_void_p(t.data_ptr())


def _ok(status, where):
    if status != 0:
        raise MokError(status, where)


def shape_of(T, H, I, E, k):
    return MokShape(T, H, I, E, k)


def config(minibatch_rows=0, ring_slots=0, capacity_mult=0.0, comm_sms=0, debug_flags=0, replay=0, overlap_sms=0):
    return MokConfig(minibatch_rows, ring_slots, capacity_mult, comm_sms, debug_flags, replay, overlap_sms)


def mx(q, scale):
    """MXFP8 tensor descriptor (codes, scales) for mok_forward / mok_backward."""
    return MokMx(q.data_ptr(), scale.data_ptr())


def mok_version():
    return LIB.mok_version().decode()


def mok_status_string(status):
    return LIB.mok_status_string(status).decode()


def mok_device_sm_count():
    return LIB.mok_device_sm_count()


def mok_workspace_size(shape, cfg, prec=MOK_BF16):
    return LIB.mok_workspace_size(ctypes.byref(shape), ctypes.byref(cfg), prec)


def mok_ctx_size(shape, cfg, prec=MOK_BF16):
    return LIB.mok_ctx_size(ctypes.byref(shape), ctypes.byref(cfg), prec)


def mok_workspace_layout(shape, cfg, prec=MOK_BF16):
    out = MokLayout()
    _ok(LIB.mok_workspace_layout(ctypes.byref(shape), ctypes.byref(cfg), prec, ctypes.byref(out)),
        "mok_workspace_layout")
    return {name: getattr(out, name) for name, _ in MokLayout._fields_}


def mok_build_schedule(shape, cfg, ws, topk_idx, stream=None):
    _ok(LIB.mok_build_schedule(ctypes.byref(shape), ctypes.byref(cfg), _ptr(ws), ws.numel() * ws.element_size(),
                               _ptr(topk_idx), _stream(stream)), "mok_build_schedule")


def mok_forward(shape, cfg, prec, ws, x, scores, W1, W3, W2, out, ctx, stream=None):
    _ok(LIB.mok_forward(ctypes.byref(shape), ctypes.byref(cfg), prec, _ptr(ws), ws.numel() * ws.element_size(),
                        _ptr(x), _ptr(scores), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(out), _ptr(ctx),
                        _stream(stream)), "mok_forward")


def mok_forward_fused(shape, cfg, prec, ws, idx, x, scores, W1, W3, W2, out, ctx, stream=None):
    _ok(LIB.mok_forward_fused(ctypes.byref(shape), ctypes.byref(cfg), prec, _ptr(ws), ws.numel() * ws.element_size(),
                              _ptr(idx), _ptr(x), _ptr(scores), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(out),
                              _ptr(ctx), _stream(stream)), "mok_forward_fused")


def mok_backward(shape, cfg, prec, ws, ctx, x, scores, W1, W3, W2, dout, dX, dW1, dW3, dW2, dscores, stream=None):
    _ok(LIB.mok_backward(ctypes.byref(shape), ctypes.byref(cfg), prec, _ptr(ws), ws.numel() * ws.element_size(),
                         _ptr(ctx), _ptr(x), _ptr(scores), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dout), _ptr(dX),
                         _ptr(dW1), _ptr(dW3), _ptr(dW2), _ptr(dscores), _stream(stream)), "mok_backward")


def mok_mxfp8_quantize(src, block_axis, q, scale, stream=None):
    b, r, c = (src.shape if src.dim() == 3 else (1,) + tuple(src.shape))
    _ok(LIB.mok_mxfp8_quantize(_ptr(src), b, r, c, block_axis, _ptr(q), _ptr(scale), _stream(stream)),
        "mok_mxfp8_quantize")


def mok_router_workspace_size(shape):
    return LIB.mok_router_workspace_size(ctypes.byref(shape))


def mok_router_forward(shape, rws, x, Wr, bias, topk_idx, scores, logits=None, stream=None):
    _ok(LIB.mok_router_forward(ctypes.byref(shape), _ptr(rws), rws.numel() * rws.element_size(), _ptr(x), _ptr(Wr),
                               _ptr(bias), _ptr(topk_idx), _ptr(scores), _ptr(logits), _stream(stream)),
        "mok_router_forward")


def mok_router_backward(shape, rws, x, Wr, topk_idx, scores, dscores, dWr, dx_router, stream=None):
    _ok(LIB.mok_router_backward(ctypes.byref(shape), _ptr(rws), rws.numel() * rws.element_size(), _ptr(x), _ptr(Wr),
                                _ptr(topk_idx), _ptr(scores), _ptr(dscores), _ptr(dWr), _ptr(dx_router),
                                _stream(stream)), "mok_router_backward")


def mok_gather_rows(shape, cfg, ws, x, xg, stream=None):
    _ok(LIB.mok_gather_rows(ctypes.byref(shape), ctypes.byref(cfg), _ptr(ws), ws.numel() * ws.element_size(),
                            _ptr(x), _ptr(xg), _stream(stream)), "mok_gather_rows")


def mok_gemm_bf16(A, a_mn_major, B, b_mn_major, C, scratch, stream=None):
    M, N = C.shape
    K = A.shape[0] if a_mn_major else A.shape[1]
    _ok(LIB.mok_gemm_bf16(M, N, K, _ptr(A), int(a_mn_major), _ptr(B), int(b_mn_major), _ptr(C), _ptr(scratch),
                          _stream(stream)), "mok_gemm_bf16")


def mok_gemm_mxfp8(Aq, Asf, a_mn_major, Bq, Bsf, b_mn_major, C, scratch, stream=None):
    M, N = C.shape
    K = Aq.shape[0] if a_mn_major else Aq.shape[1]
    _ok(LIB.mok_gemm_mxfp8(M, N, K, _ptr(Aq), _ptr(Asf), int(a_mn_major), _ptr(Bq), _ptr(Bsf), int(b_mn_major),
                           _ptr(C), _ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream)),
        "mok_gemm_mxfp8")


def mok_trace_enable(on=True):
    _ok(LIB.mok_trace_enable(1 if on else 0), "mok_trace_enable")


def mok_trace_read():
    """{phase: (summed ms, runs)} since the last read (synchronises)."""
    ms = (ctypes.c_float * len(PHASES))()
    cnt = (ctypes.c_int32 * len(PHASES))()
    _ok(LIB.mok_trace_read(ms, cnt), "mok_trace_read")
    return {name: (ms[i], cnt[i]) for i, name in enumerate(PHASES)}


def mok_launch_count():
    return LIB.mok_launch_count()


def mok_build_schedule_noalloc(shape, topk_idx, buffers, stream=None):
    """``buffers``: dict of int32 device tensors named as MokScheduleBuffers."""
    b = MokScheduleBuffers(*[buffers[n].data_ptr() for n, _ in MokScheduleBuffers._fields_])
    _ok(LIB.mok_build_schedule_noalloc(ctypes.byref(shape), _ptr(topk_idx), ctypes.byref(b), _stream(stream)),
        "mok_build_schedule_noalloc")


def mok_check(ws, stream=None):
    """Synchronise and return the device status recorded in the workspace (int)."""
    return LIB.mok_check(_ptr(ws), _stream(stream))


# ---------------------------------------------------------------- expert parallelism
def mok_schedule_workspace_size(shape, cfg):
    return LIB.mok_schedule_workspace_size(ctypes.byref(shape), ctypes.byref(cfg))


def mok_ep_first_expert(E, G, g):
    return LIB.mok_ep_first_expert(E, G, g)


def mok_ep_plan(E, G, rank, local_counts, recv_counts, recv_capacity=None):
    """Host-only exchange plan.  ``local_counts``: int32 [E]; ``recv_counts``:
    int32 [G, E_rank] (array-likes on the host).  Returns (send_rows list,
    recv_rows list, recv_expert int32 numpy array or None, n_recv)."""
    import numpy as np
    lc = np.ascontiguousarray(np.asarray(local_counts, dtype=np.int32))
    rc = np.ascontiguousarray(np.asarray(recv_counts, dtype=np.int32))
    send = np.zeros(G, dtype=np.int64)
    recv = np.zeros(G, dtype=np.int64)
    n = ctypes.c_int64(0)
    if recv_capacity is None:
        recv_capacity = int(rc.sum())
    experts = np.zeros(max(int(recv_capacity), 1), dtype=np.int32)
    _ok(LIB.mok_ep_plan(E, G, rank, lc.ctypes.data, rc.ctypes.data, send.ctypes.data, recv.ctypes.data,
                        experts.ctypes.data, int(recv_capacity), ctypes.byref(n)), "mok_ep_plan")
    return send.tolist(), recv.tolist(), experts[:n.value], n.value


def mok_ep_pack_rows(shape, cfg, ws, x, scores, rows, row_scores=None, stream=None):
    _ok(LIB.mok_ep_pack_rows(ctypes.byref(shape), ctypes.byref(cfg), _ptr(ws), ws.numel() * ws.element_size(),
                             _ptr(x), _ptr(scores), _ptr(rows), _ptr(row_scores), _stream(stream)),
        "mok_ep_pack_rows")


def mok_ep_combine_rows(shape, cfg, ws, rows, scores, out, stream=None):
    _ok(LIB.mok_ep_combine_rows(ctypes.byref(shape), ctypes.byref(cfg), _ptr(ws), ws.numel() * ws.element_size(),
                                _ptr(rows), _ptr(scores), _ptr(out), _stream(stream)), "mok_ep_combine_rows")


def mok_ep_unsort_scores(shape, cfg, ws, row_vals, out, stream=None):
    _ok(LIB.mok_ep_unsort_scores(ctypes.byref(shape), ctypes.byref(cfg), _ptr(ws), ws.numel() * ws.element_size(),
                                 _ptr(row_vals), _ptr(out), _stream(stream)), "mok_ep_unsort_scores")
