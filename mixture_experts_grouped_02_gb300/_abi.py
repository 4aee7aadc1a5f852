"""ctypes binding of libmoe_gb300.so (declared in include/moe.h).

Argument marshalling only: each function here has the name of the C entry
point it calls, takes torch tensors where the C function takes device
pointers, passes ``tensor.data_ptr()`` and the current CUDA stream, and turns
a non-zero status into :class:`MoEError`.  Every step of the computation runs
in the library's CUDA kernels; there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_BAD_ID = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_BOUNDS = 7

MOE_F32, MOE_BF16, MOE_E4M3, MOE_E2M1_MX = 0, 1, 2, 3

(MOE_WS_STATUS, MOE_WS_COUNTS, MOE_WS_OFFSETS, MOE_WS_PADDED_OFFSETS, MOE_WS_SORTED_IDS,
 MOE_WS_INV_PERM, MOE_WS_BLOCK_INFO, MOE_WS_NUM_BLOCKS, MOE_WS_XQ, MOE_WS_X_SCALE, MOE_WS_H,
 MOE_WS_Y, MOE_WS_ALIGN, MOE_WS_NUM) = range(14)

# every symbol include/moe.h declares
EXPORTS = ("moe_status_string", "moe_abi_version", "moe_resolve_block_m", "moe_align_capacity",
           "moe_gemm2_default_splits", "moe_workspace_size", "moe_workspace_offsets", "moe_align",
           "moe_quantize_x_fp8", "moe_gemm1_silu", "moe_gemm2_weighted", "moe_combine",
           "moe_forward", "moe_forward_noalloc", "moe_get_device_status", "moe_mx_packed_bytes",
           "moe_pack_mx_weights", "moe_quantize_gather_x_fp8", "moe_device_info",
           "moe_gather_rows", "moe_align_local", "moe_route_align", "moe_align_scratch_bytes",
           "moe_combine_finish", "moe_forward_noalloc_status", "moe_test_gemm_wait_timeout",
           "moe_gemm1_silu_gather")

MOE_STATIC_SCRATCH_BYTES = 64 << 20
MOE_ACT_SILU, MOE_ACT_SWIGLU_CLAMP = 0, 1


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Problem(ctypes.Structure):
    """moe_problem_t."""
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("E", ctypes.c_int), ("K", ctypes.c_int), ("act", ctypes.c_int),
                ("weight", ctypes.c_int), ("block_m", ctypes.c_int), ("h_scale", ctypes.c_float),
                ("expert_base", ctypes.c_int), ("local_experts", ctypes.c_int),
                ("activation", ctypes.c_int), ("swiglu_alpha", ctypes.c_float),
                ("swiglu_limit", ctypes.c_float), ("gate_up_interleaved", ctypes.c_int),
                ("w13_bias", ctypes.c_void_p), ("w2_bias", ctypes.c_void_p),
                ("fused_combine", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """Load libmoe_gb300.so (building it first if it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"{_build.LIB} is missing; build it with "
                                   "`python -m mixture_experts_grouped_02_gb300.build`")
            L = ctypes.CDLL(_build.LIB)
            _declare(L)
            _lib = L
    return _lib


def checked_lib():
    """libmoe_gb300_checked.so (built if absent or stale): the same entry
    points with every kernel index range-checked (MOE_ERR_BOUNDS), loaded
    beside the product library; call its functions directly."""
    with _lock:
        if not _build.up_to_date(checked=True):
            _build.build(checked=True)
        L = ctypes.CDLL(_build.LIB_CHECKED)
        _declare(L)
        return L


def _declare(L):
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    PP = ctypes.POINTER(Problem)
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [i32]
    L.moe_abi_version.restype = i32
    L.moe_abi_version.argtypes = []
    L.moe_resolve_block_m.restype = i32
    L.moe_resolve_block_m.argtypes = [PP]
    L.moe_align_capacity.restype = sz
    L.moe_align_capacity.argtypes = [i32, i32, i32, i32]
    L.moe_gemm2_default_splits.restype = i32
    L.moe_gemm2_default_splits.argtypes = [PP]
    L.moe_workspace_size.restype = sz
    L.moe_workspace_size.argtypes = [PP]
    L.moe_workspace_offsets.restype = i32
    L.moe_workspace_offsets.argtypes = [PP, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.moe_align.restype = i32
    L.moe_align.argtypes = [vp, i32, i32, i32, i32] + [vp] * 8 + [vp]
    L.moe_route_align.restype = i32
    L.moe_route_align.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32] + [vp] * 9 + [vp, vp]
    L.moe_align_local.restype = i32
    L.moe_align_local.argtypes = [vp, i32, i32, i32, i32, i32, i32] + [vp] * 7 + [vp, sz] + [vp, vp]
    L.moe_align_scratch_bytes.restype = sz
    L.moe_align_scratch_bytes.argtypes = [i32, i32, i32]
    L.moe_quantize_x_fp8.restype = i32
    L.moe_quantize_x_fp8.argtypes = [vp, i32, i32, i32, vp, vp, vp]
    L.moe_gather_rows.restype = i32
    L.moe_gather_rows.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    L.moe_quantize_gather_x_fp8.restype = i32
    L.moe_quantize_gather_x_fp8.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    L.moe_combine_finish.restype = i32
    L.moe_combine_finish.argtypes = [vp, i32, i32, i32, vp, vp, vp]
    L.moe_gemm1_silu.restype = i32
    L.moe_gemm1_silu.argtypes = [PP] + [vp] * 10
    L.moe_gemm1_silu_gather.restype = i32
    L.moe_gemm1_silu_gather.argtypes = [PP] + [vp] * 8
    L.moe_gemm2_weighted.restype = i32
    L.moe_gemm2_weighted.argtypes = [PP, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp]
    L.moe_combine.restype = i32
    L.moe_combine.argtypes = [vp, i32, sz, vp, i32, i32, i32, i32, vp, vp, vp]
    L.moe_forward.restype = i32
    L.moe_forward.argtypes = [PP] + [vp] * 9 + [sz, vp]
    L.moe_forward_noalloc.restype = i32
    L.moe_forward_noalloc.argtypes = [PP] + [vp] * 9
    L.moe_test_gemm_wait_timeout.restype = i32
    L.moe_test_gemm_wait_timeout.argtypes = [PP, i32] + [vp] * 9 + [i32, ctypes.c_ulonglong,
                                                                  vp, vp]
    L.moe_forward_noalloc_status.restype = i32
    L.moe_forward_noalloc_status.argtypes = [vp]
    L.moe_get_device_status.restype = i32
    L.moe_get_device_status.argtypes = [vp, vp]
    L.moe_device_info.restype = i32
    L.moe_device_info.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.moe_mx_packed_bytes.restype = sz
    L.moe_mx_packed_bytes.argtypes = [i32, i32, i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.moe_pack_mx_weights.restype = i32
    L.moe_pack_mx_weights.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]


def status_string(status: int) -> str:
    try:
        return lib().moe_status_string(int(status)).decode()
    except Exception:  # the library itself failed to load
        return f"status {status}"


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc, where):
    if rc != MOE_OK:
        raise MoEError(rc, where)


# ------------------------------------------------------------------ queries

def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_resolve_block_m(p: Problem) -> int:
    return lib().moe_resolve_block_m(ctypes.byref(p))


def moe_align_capacity(T, K, E, block_m) -> int:
    return int(lib().moe_align_capacity(T, K, E, block_m))


def moe_gemm2_default_splits(p: Problem) -> int:
    return lib().moe_gemm2_default_splits(ctypes.byref(p))


def moe_workspace_size(p: Problem) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(p)))


def moe_workspace_offsets(p: Problem):
    off = (ctypes.c_size_t * MOE_WS_NUM)()
    size = (ctypes.c_size_t * MOE_WS_NUM)()
    _check(lib().moe_workspace_offsets(ctypes.byref(p), off, size), "moe_workspace_offsets")
    return list(off), list(size)


# ------------------------------------------------------------------ stages

def moe_align(topk_ids, T, K, E, block_m, counts, offsets, padded_offsets, sorted_ids, inv_perm,
              block_info, num_blocks, dev_status=None, stream=None):
    _check(lib().moe_align(_p(topk_ids), T, K, E, block_m, _p(counts), _p(offsets),
                           _p(padded_offsets), _p(sorted_ids), _p(inv_perm), _p(block_info),
                           _p(num_blocks), _p(dev_status), _stream(stream)), "moe_align")


def moe_align_local(topk_ids, T, K, E, expert_base, local_experts, block_m, counts, offsets,
                    padded_offsets, sorted_ids, inv_perm, block_info, num_blocks, dev_status=None,
                    stream=None, scratch=None):
    nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _check(lib().moe_align_local(_p(topk_ids), T, K, E, expert_base, local_experts, block_m,
                                 _p(counts), _p(offsets), _p(padded_offsets), _p(sorted_ids),
                                 _p(inv_perm), _p(block_info), _p(num_blocks), _p(scratch),
                                 nbytes, _p(dev_status), _stream(stream)), "moe_align_local")


def moe_align_scratch_bytes(T, K, local_experts):
    return int(lib().moe_align_scratch_bytes(T, K, local_experts))


def moe_route_align(logits, logit_dtype, T, E, K, expert_base, local_experts, block_m, topk_ids,
                    topk_weights, counts, offsets, padded_offsets, sorted_ids, inv_perm,
                    block_info, num_blocks, dev_status=None, stream=None):
    _check(lib().moe_route_align(_p(logits), logit_dtype, T, E, K, expert_base, local_experts,
                                 block_m, _p(topk_ids), _p(topk_weights), _p(counts), _p(offsets),
                                 _p(padded_offsets), _p(sorted_ids), _p(inv_perm),
                                 _p(block_info), _p(num_blocks), _p(dev_status),
                                 _stream(stream)), "moe_route_align")


def moe_quantize_x_fp8(x, x_dtype, T, H, xq, row_scale, stream=None):
    _check(lib().moe_quantize_x_fp8(_p(x), x_dtype, T, H, _p(xq), _p(row_scale),
                                    _stream(stream)), "moe_quantize_x_fp8")


def moe_gather_rows(x, dtype, T, H, K, inv_perm, x_sorted, dev_status=None, stream=None,
                    acc_zero=None):
    _check(lib().moe_gather_rows(_p(x), dtype, T, H, K, _p(inv_perm), _p(x_sorted),
                                 _p(acc_zero), _p(dev_status), _stream(stream)),
           "moe_gather_rows")


def moe_quantize_gather_x_fp8(x, x_dtype, T, H, K, inv_perm, xq_sorted, row_scale,
                              dev_status=None, stream=None, acc_zero=None):
    _check(lib().moe_quantize_gather_x_fp8(_p(x), x_dtype, T, H, K, _p(inv_perm), _p(xq_sorted),
                                           _p(row_scale), _p(acc_zero), _p(dev_status),
                                           _stream(stream)),
           "moe_quantize_gather_x_fp8")


def moe_combine_finish(acc, T, H, out_dtype, out, dev_status=None, stream=None):
    _check(lib().moe_combine_finish(_p(acc), T, H, out_dtype, _p(out), _p(dev_status),
                                    _stream(stream)), "moe_combine_finish")


def moe_gemm1_silu(p: Problem, x, x_row_scale, w13, w13_scale, sorted_ids, block_info,
                   num_blocks, h, dev_status=None, stream=None):
    _check(lib().moe_gemm1_silu(ctypes.byref(p), _p(x), _p(x_row_scale), _p(w13), _p(w13_scale),
                                _p(sorted_ids), _p(block_info), _p(num_blocks), _p(h),
                                _p(dev_status), _stream(stream)), "moe_gemm1_silu")


def moe_gemm1_silu_gather(p: Problem, x, w13, sorted_ids, block_info, num_blocks, h,
                          dev_status=None, stream=None):
    _check(lib().moe_gemm1_silu_gather(ctypes.byref(p), _p(x), _p(w13), _p(sorted_ids),
                                       _p(block_info), _p(num_blocks), _p(h), _p(dev_status),
                                       _stream(stream)), "moe_gemm1_silu_gather")


def moe_gemm2_weighted(p: Problem, h, w2, w2_scale, topk_weights, sorted_ids, block_info,
                       num_blocks, y, k_splits, dev_status=None, stream=None):
    _check(lib().moe_gemm2_weighted(ctypes.byref(p), _p(h), _p(w2), _p(w2_scale),
                                    _p(topk_weights), _p(sorted_ids), _p(block_info),
                                    _p(num_blocks), _p(y), int(k_splits), _p(dev_status),
                                    _stream(stream)), "moe_gemm2_weighted")


def moe_combine(y, k_splits, cap, inv_perm, T, K, H, out_dtype, out, dev_status=None,
                stream=None):
    _check(lib().moe_combine(_p(y), int(k_splits), int(cap), _p(inv_perm), T, K, H, out_dtype,
                             _p(out), _p(dev_status), _stream(stream)), "moe_combine")


def moe_forward(p: Problem, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, out,
                workspace, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_forward(ctypes.byref(p), _p(x), _p(topk_ids), _p(topk_weights), _p(w13),
                             _p(w13_scale), _p(w2), _p(w2_scale), _p(out), _p(workspace),
                             int(workspace_bytes), _stream(stream)), "moe_forward")


def moe_forward_noalloc(p: Problem, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale,
                        out, stream=None):
    """moe_forward with the intermediates in the library's static scratch
    array (MOE_STATIC_SCRATCH_BYTES per GPU) instead of a workspace: for
    callers that cannot allocate device memory where they run the layer."""
    _check(lib().moe_forward_noalloc(ctypes.byref(p), _p(x), _p(topk_ids), _p(topk_weights),
                                     _p(w13), _p(w13_scale), _p(w2), _p(w2_scale), _p(out),
                                     _stream(stream)), "moe_forward_noalloc")


def moe_test_gemm_wait_timeout(p: Problem, gemm, a_rows, x_row_scale, w, w_scale, topk_weights,
                               sorted_ids, block_info, num_blocks, out, k_splits, wait_limit_ns,
                               dev_status, stream=None):
    """The GEMM `gemm` (1: gate/up, 2: down) launched with starved pipelines
    and a short wait limit: the kernels' failure path, for tests."""
    _check(lib().moe_test_gemm_wait_timeout(ctypes.byref(p), int(gemm), _p(a_rows),
                                            _p(x_row_scale), _p(w), _p(w_scale),
                                            _p(topk_weights), _p(sorted_ids), _p(block_info),
                                            _p(num_blocks), _p(out), int(k_splits),
                                            int(wait_limit_ns), _p(dev_status),
                                            _stream(stream)), "moe_test_gemm_wait_timeout")


def moe_forward_noalloc_status(stream=None) -> int:
    """The device status word of the last moe_forward_noalloc on the current
    device (synchronises the stream): 0, or the kernels' error code."""
    rc = lib().moe_forward_noalloc_status(_stream(stream))
    if rc == MOE_ERR_CUDA:
        raise MoEError(rc, "moe_forward_noalloc_status")
    return rc


def moe_mx_packed_bytes(E, R, K, sections):
    vb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    total = lib().moe_mx_packed_bytes(E, R, K, sections, ctypes.byref(vb), ctypes.byref(sb))
    if total == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_mx_packed_bytes")
    return vb.value, sb.value


def moe_pack_mx_weights(w, w_scale, E, R, K, sections, interleaved, w_packed, scale_packed,
                        stream=None):
    _check(lib().moe_pack_mx_weights(_p(w), _p(w_scale), E, R, K, sections, interleaved,
                                     _p(w_packed),
                                     _p(scale_packed), _stream(stream)), "moe_pack_mx_weights")


def moe_device_info():
    """(SM count, CTA pairs of the gate/up pair kernel the device holds)."""
    sms, pairs = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().moe_device_info(ctypes.byref(sms), ctypes.byref(pairs)), "moe_device_info")
    return sms.value, pairs.value


def moe_get_device_status(dev_status, stream=None) -> int:
    return lib().moe_get_device_status(_p(dev_status), _stream(stream))
