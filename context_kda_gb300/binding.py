"""ctypes binding of libkda (argument marshalling only).

Each function has the name of the C entry point it calls (declared in
include/kda.h); tensors are passed by ``data_ptr()``, the stream is the current
torch CUDA stream unless one is given.  Every step of the computation runs in
libkda's CUDA kernels; there is no Python or CPU fallback, and importing this
module fails if libkda.so has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
KDA_ERR_RANGE = -6
HEAD_DIM_K = HEAD_DIM_V = 128
CHUNK = 64


class KDAError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkda.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_last_cuda_error.restype = ctypes.c_int
    lib.kda_device_status.argtypes = []
    lib.kda_device_status.restype = ctypes.c_int
    lib.kda_selftest_wait_expiry.argtypes = [P]
    lib.kda_selftest_wait_expiry.restype = ctypes.c_int
    lib.kda_selftest_state_abort.argtypes = [P, P, I32, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, SZ, P]
    lib.kda_selftest_state_abort.restype = ctypes.c_int
    lib.kda_plan_segments.argtypes = [P, I32, I32, P, I32, P, ctypes.POINTER(SZ)]
    lib.kda_plan_check.argtypes = [P]
    lib.kda_plan_segments_refined.argtypes = [P, I32, I32, P, I32, I32, I32, P, ctypes.POINTER(SZ)]
    lib.kda_workspace_layout.argtypes = [P, I32, ctypes.POINTER(SZ)]
    lib.kda_workspace_bytes.argtypes = [P, I32]
    lib.kda_workspace_bytes.restype = SZ
    lib.kda_segment_forward.argtypes = [P, P, I32, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, SZ, P]
    lib.kda_compose_summaries.argtypes = [P, P, I32, P, P, P, P, P]
    lib.kda_compose_summaries_blocked.argtypes = [P, P, I32, P, P, P, P, P, SZ, P]
    lib.kda_scan_workspace_bytes.argtypes = [P, I32]
    lib.kda_scan_workspace_bytes.restype = SZ
    lib.kda_apply_boundary.argtypes = [P, P, I32, P, P, SZ, P, P, P]
    lib.kda_forward_segmented.argtypes = [P, P, I32, P, P, P, P, P, P, ctypes.c_float, P, P, P, SZ, P]
    lib.kda_forward_segmented_noalloc.argtypes = [P, P, I32, P, P, P, P, P, P, ctypes.c_float, P, P, P]
    lib.kda_forward_two_pass.argtypes = [P, P, I32, P, P, P, P, P, P, ctypes.c_float, P, P, P, SZ, P]
    lib.kda_backward_segmented.argtypes = [P, P, I32, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, P, P, P,
                                           P, SZ, P]
    lib.kda_backward_workspace_bytes.argtypes = [P, I32]
    lib.kda_backward_workspace_bytes.restype = SZ
    for name in ("kda_plan_segments", "kda_plan_check", "kda_plan_segments_refined", "kda_workspace_layout", "kda_segment_forward", "kda_compose_summaries",
                 "kda_compose_summaries_blocked", "kda_apply_boundary", "kda_forward_segmented", "kda_forward_segmented_noalloc", "kda_backward_segmented",
                 "kda_forward_two_pass"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


_lib = _load()


def _check(fn: str, rc: int):
    if rc != KDA_OK:
        msg = _lib.kda_status_string(rc).decode()
        if rc == KDA_ERR_CUDA:
            msg += f" (cudaError {_lib.kda_last_cuda_error()})"
        raise KDAError(fn, rc, msg)


def kda_device_status() -> int:
    """Synchronises the current device and returns (and clears) the kernels' device-side status:
    KDA_OK, or the first error a kernel recorded: KDA_ERR_TIMEOUT (a bounded wait expired),
    KDA_ERR_RANGE (a chunk's summed decay out of range) or KDA_ERR_INVALID_ARG (a device plan
    that is not the host plan's copy)."""
    return int(_lib.kda_device_status())


def kda_selftest_state_abort(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, A, B, final_state, ws, stream=None):
    """The state pass with the second chunk's package copies withheld (see include/kda.h): its waits run
    out, it returns cleanly, and kda_device_status() then reports KDA_ERR_TIMEOUT."""
    p = _words(plan)
    _check("kda_selftest_state_abort",
           _lib.kda_selftest_state_abort(_hp(p), _dp(plan_dev), int(H), _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta),
                                         _dp(h0), float(scale), _dp(o), _dp(A), _dp(B), _dp(final_state), _dp(ws),
                                         _nbytes(ws), _stream(stream)))


def kda_selftest_wait_expiry(stream=None):
    """Enqueues a kernel whose bounded wait expires (about two seconds); kda_device_status() then
    reports KDA_ERR_TIMEOUT."""
    _check("kda_selftest_wait_expiry", _lib.kda_selftest_wait_expiry(_stream(stream)))


def _words(plan) -> np.ndarray:
    return np.ascontiguousarray(plan, dtype=np.int32)


def _hp(plan):
    return plan.ctypes.data_as(ctypes.c_void_p)


def _dp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)


def kda_status_string(status: int) -> str:
    return _lib.kda_status_string(int(status)).decode()


def kda_plan_segments(cu_seqlens, num_segments: int, seg_bounds=None, chunk: int = CHUNK) -> np.ndarray:
    """Host plan words (int32) for packed sequences ``cu_seqlens`` cut into ``num_segments``."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    sb = None if seg_bounds is None else np.ascontiguousarray(seg_bounds, dtype=np.int32)
    sbp = None if sb is None else sb.ctypes.data_as(ctypes.c_void_p)
    n = ctypes.c_size_t(0)
    args = (cu.ctypes.data_as(ctypes.c_void_p), cu.shape[0] - 1, int(num_segments), sbp, int(chunk))
    _check("kda_plan_segments", _lib.kda_plan_segments(*args, None, ctypes.byref(n)))
    out = np.zeros(n.value, dtype=np.int32)
    _check("kda_plan_segments", _lib.kda_plan_segments(*args, out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n)))
    return out


def kda_plan_segments_refined(cu_seqlens, num_segments: int, heads: int, num_sms: int, seg_bounds=None,
                              chunk: int = CHUNK) -> np.ndarray:
    """A plan whose segments refine ``num_segments`` into chunk-aligned sub-segments (see include/kda.h)."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    sb = None if seg_bounds is None else np.ascontiguousarray(seg_bounds, dtype=np.int32)
    sbp = None if sb is None else sb.ctypes.data_as(ctypes.c_void_p)
    n = ctypes.c_size_t(0)
    args = (cu.ctypes.data_as(ctypes.c_void_p), cu.shape[0] - 1, int(num_segments), sbp, int(chunk), int(heads),
            int(num_sms))
    _check("kda_plan_segments_refined", _lib.kda_plan_segments_refined(*args, None, ctypes.byref(n)))
    out = np.zeros(n.value, dtype=np.int32)
    _check("kda_plan_segments_refined",
           _lib.kda_plan_segments_refined(*args, out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n)))
    return out


def kda_plan_check(plan) -> int:
    """Whole-plan validation (see include/kda.h): KDA_OK or KDA_ERR_INVALID_ARG."""
    return int(_lib.kda_plan_check(_hp(_words(plan))))


def kda_workspace_layout(plan, H: int):
    """Byte offsets (qhat, fin, packages, A, B, S_in, total) of the device workspace."""
    p = _words(plan)
    off = (ctypes.c_size_t * 7)()
    _check("kda_workspace_layout", _lib.kda_workspace_layout(_hp(p), int(H), off))
    return tuple(int(x) for x in off)


def kda_workspace_bytes(plan, H: int) -> int:
    p = _words(plan)
    return int(_lib.kda_workspace_bytes(_hp(p), int(H)))


def upload_plan(plan, device="cuda"):
    """Device copy of the plan words (the caller keeps it alive while calls use it)."""
    import torch
    return torch.from_numpy(_words(plan).copy()).to(device)


def kda_segment_forward(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, A, B, final_state, ws, stream=None):
    p = _words(plan)
    rc = _lib.kda_segment_forward(_hp(p), _dp(plan_dev), int(H), _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta),
                                  _dp(h0), float(scale), _dp(o), _dp(A), _dp(B), _dp(final_state), _dp(ws),
                                  _nbytes(ws), _stream(stream))
    _check("kda_segment_forward", rc)


def kda_compose_summaries(plan, plan_dev, H, A, B, h0, S_in, stream=None):
    p = _words(plan)
    rc = _lib.kda_compose_summaries(_hp(p), _dp(plan_dev), int(H), _dp(A), _dp(B), _dp(h0), _dp(S_in),
                                    _stream(stream))
    _check("kda_compose_summaries", rc)


def kda_scan_workspace_bytes(plan, H: int) -> int:
    return int(_lib.kda_scan_workspace_bytes(_hp(_words(plan)), int(H)))


def kda_compose_summaries_blocked(plan, plan_dev, H, A, B, h0, S_in, ws, stream=None):
    """S_in by the two-level (log-depth across groups) scan; ws holds kda_scan_workspace_bytes."""
    p = _words(plan)
    rc = _lib.kda_compose_summaries_blocked(_hp(p), _dp(plan_dev), int(H), _dp(A), _dp(B), _dp(h0), _dp(S_in),
                                            _dp(ws), _nbytes(ws), _stream(stream))
    _check("kda_compose_summaries_blocked", rc)


def kda_apply_boundary(plan, plan_dev, H, S_in, ws, o, final_state, stream=None):
    p = _words(plan)
    rc = _lib.kda_apply_boundary(_hp(p), _dp(plan_dev), int(H), _dp(S_in), _dp(ws), _nbytes(ws), _dp(o),
                                 _dp(final_state), _stream(stream))
    _check("kda_apply_boundary", rc)


def kda_forward_segmented(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, final_state, ws, stream=None):
    p = _words(plan)
    rc = _lib.kda_forward_segmented(_hp(p), _dp(plan_dev), int(H), _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta),
                                    _dp(h0), float(scale), _dp(o), _dp(final_state), _dp(ws), _nbytes(ws),
                                    _stream(stream))
    _check("kda_forward_segmented", rc)


def kda_forward_two_pass(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, final_state, ws, stream=None):
    """The segmented forward from preceding summaries (see include/kda.h): the same arguments and
    results as kda_forward_segmented, with the state pass run twice and no fix-up."""
    p = _words(plan)
    rc = _lib.kda_forward_two_pass(_hp(p), _dp(plan_dev), int(H), _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta),
                                   _dp(h0), float(scale), _dp(o), _dp(final_state), _dp(ws), _nbytes(ws),
                                   _stream(stream))
    _check("kda_forward_two_pass", rc)


def kda_backward_workspace_bytes(plan, H: int) -> int:
    return int(_lib.kda_backward_workspace_bytes(_hp(_words(plan)), int(H)))


def kda_backward_segmented(plan, plan_dev, H, q, k, v, g, beta, h0, scale, dout, dfinal, dq, dk, dv, dg, dbeta,
                           dh0, ws, stream=None):
    """Gradients of the segmented forward (see include/kda.h); dfinal and dh0 may be None."""
    p = _words(plan)
    rc = _lib.kda_backward_segmented(_hp(p), _dp(plan_dev), int(H), _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta),
                                     _dp(h0), float(scale), _dp(dout), _dp(dfinal), _dp(dq), _dp(dk), _dp(dv),
                                     _dp(dg), _dp(dbeta), _dp(dh0), _dp(ws), _nbytes(ws), _stream(stream))
    _check("kda_backward_segmented", rc)


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def kda_forward_segmented_noalloc(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, final_state, stream=None):
    """kda_forward_segmented with the library's fixed 32 MiB device workspace instead of a
    caller buffer, for callers that cannot allocate device memory (see include/kda.h)."""
    p = _words(plan)
    rc = _lib.kda_forward_segmented_noalloc(_hp(p), _dp(plan_dev), int(H), _dp(q), _dp(k), _dp(v), _dp(g),
                                            _dp(beta), _dp(h0), float(scale), _dp(o), _dp(final_state),
                                            _stream(stream))
    _check("kda_forward_segmented_noalloc", rc)
