"""CPU oracle for the MoE expert-FFN forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.  The arithmetic lives in ``moe_oracle.c`` (plain C,
fp64); this module compiles it with gcc when needed and marshals numpy arrays
into it.  Every function cites, in ``moe_oracle.c``, the passage it follows.

Storage conventions of the numpy arguments:
  * bf16 tensors are passed as ``np.uint16`` bit patterns,
  * fp32 tensors as ``np.float32``,
  * mxfp4 weights as ``np.uint8`` packed e2m1 pairs (low nibble = lower K
    index) plus ``np.uint8`` e8m0 scales, one per 32 K elements.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")

F32, BF16, MXFP4 = 0, 1, 3
EXACT, EMULATE = 0, 1

_lock = threading.Lock()
_lib = None


class Problem(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int),
        ("H", ctypes.c_int),
        ("I", ctypes.c_int),
        ("E", ctypes.c_int),
        ("K", ctypes.c_int),
        ("x_dtype", ctypes.c_int),
        ("w_dtype", ctypes.c_int),
        ("quantize_x", ctypes.c_int),
        ("h_e4m3", ctypes.c_int),
        ("h_scale", ctypes.c_double),
        ("expert_base", ctypes.c_int),
        ("local_experts", ctypes.c_int),
        ("activation", ctypes.c_int),
        ("swiglu_alpha", ctypes.c_double),
        ("swiglu_limit", ctypes.c_double),
        ("gate_up_interleaved", ctypes.c_int),
        ("w13_bias", ctypes.c_void_p),
        ("w2_bias", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, OpenMP, no fast-math,
    no FMA contraction so x86 and Arm hosts round alike)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


def _declare(L):
    P = ctypes.POINTER
    vp, i32p, f32p, f64p, u8p = (ctypes.c_void_p, P(ctypes.c_int32), P(ctypes.c_float),
                                 P(ctypes.c_double), P(ctypes.c_uint8))
    ci = ctypes.c_int
    L.orc_align.restype = ci
    L.orc_align.argtypes = [i32p, ci, ci, ci, ci, i32p, i32p, i32p, i32p, i32p, i32p, i32p]
    L.orc_align_local.restype = ci
    L.orc_align_local.argtypes = [i32p, ci, ci, ci, ci, ci, ci, i32p, i32p, i32p, i32p, i32p, i32p,
                                  i32p]
    L.orc_route.restype = ci
    L.orc_route.argtypes = [vp, ci, ci, ci, ci, i32p, f64p]
    L.orc_align_capacity.restype = ctypes.c_long
    L.orc_align_capacity.argtypes = [ci, ci, ci, ci]
    L.orc_moe_forward.restype = ci
    L.orc_moe_forward.argtypes = [P(Problem), ci, vp, i32p, f32p, vp, u8p, vp, u8p, i32p, ci, f64p]
    L.orc_moe_forward_by_expert.restype = ci
    L.orc_moe_forward_by_expert.argtypes = [P(Problem), ci, vp, i32p, f32p, vp, u8p, vp, u8p, f64p]
    L.orc_gemm1_silu_rows.restype = None
    L.orc_gemm1_silu_rows.argtypes = [P(Problem), ci, vp, vp, u8p, i32p, i32p, i32p, ci, f64p]
    L.orc_gemm2_weighted_rows.restype = None
    L.orc_gemm2_weighted_rows.argtypes = [P(Problem), vp, ci, vp, u8p, f32p, i32p, i32p, i32p, ci,
                                          f64p]
    L.orc_combine.restype = None
    L.orc_combine.argtypes = [f32p, i32p, ci, ci, ci, f64p]
    L.orc_quantize_x_fp8.restype = None
    L.orc_quantize_x_fp8.argtypes = [vp, ci, ci, ci, u8p, f32p]
    L.orc_e4m3_to_double.restype = ctypes.c_double
    L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    L.orc_e2m1_to_double.restype = ctypes.c_double
    L.orc_e2m1_to_double.argtypes = [ctypes.c_uint8]
    L.orc_e8m0_to_double.restype = ctypes.c_double
    L.orc_e8m0_to_double.argtypes = [ctypes.c_uint8]
    L.orc_float_to_e4m3.restype = ctypes.c_uint8
    L.orc_float_to_e4m3.argtypes = [ctypes.c_float]


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _vptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _storage(a):
    """Keep the raw storage dtype (uint16 bf16 bits / float32 / uint8)."""
    return None if a is None else np.ascontiguousarray(a)


def _dtype_code(a):
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint8:
        return MXFP4
    raise TypeError(f"unsupported storage dtype {a.dtype}")


ACT_SILU, ACT_SWIGLU_CLAMP = 0, 1


def make_problem(T, H, I, E, K, x, w13, quantize_x=False, h_e4m3=False, h_scale=1.0,
                 expert_base=0, local_experts=0, activation=ACT_SILU, swiglu_alpha=1.0,
                 swiglu_limit=float("inf"), gate_up_interleaved=False, w13_bias=None,
                 w2_bias=None):
    """local_experts > 0: an expert-parallel shard holding experts
    [expert_base, expert_base + local_experts); the weights passed with it
    hold those experts only.  activation ACT_SWIGLU_CLAMP: the clamped
    SwiGLU with swiglu_alpha / swiglu_limit; gate_up_interleaved: w13 rows
    2j (gate) and 2j+1 (up); w13_bias (experts, 2I) in w13's row order and
    w2_bias (experts, H), fp32, optional."""
    b13 = _c(w13_bias, np.float32)
    b2 = _c(w2_bias, np.float32)
    P = Problem(T, H, I, E, K, _dtype_code(x), _dtype_code(w13), int(quantize_x), int(h_e4m3),
                float(h_scale), int(expert_base), int(local_experts), int(activation),
                float(swiglu_alpha), float(swiglu_limit), int(gate_up_interleaved),
                None if b13 is None else b13.ctypes.data, None if b2 is None else b2.ctypes.data)
    P._keep = (b13, b2)  # the arrays the pointers refer to live as long as P
    return P


def route(logits, K):
    """Top-K experts (descending logit, ties to the lower id) and their
    softmax weights renormalised over the K chosen, for (T, E) logits stored
    as fp32 or bf16 bits."""
    logits = _storage(logits)
    T, E = logits.shape
    ids = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float64)
    rc = lib().orc_route(_vptr(logits), _dtype_code(logits), T, E, K, _ptr(ids, ctypes.c_int32),
                         _ptr(w, ctypes.c_double))
    if rc != 0:
        raise ValueError("K outside [1, E]")
    return ids, w


def align_capacity(T, K, E, bm):
    return int(lib().orc_align_capacity(T, K, E, bm))


def align(ids, E, bm, expert_base=0, local_experts=0):
    """Align (T, K) top-k ids into per-expert, bm-padded sorted lists (of the
    shard's experts when local_experts > 0)."""
    ids = _c(ids, np.int32)
    T, K = ids.shape
    L = local_experts if local_experts > 0 else E
    cap = align_capacity(T, K, L, bm)
    out = dict(
        counts=np.zeros(L, np.int32),
        offsets=np.zeros(L + 1, np.int32),
        padded_offsets=np.zeros(L + 1, np.int32),
        sorted_ids=np.zeros(cap, np.int32),
        inv_perm=np.zeros(T * K, np.int32),
        block_info=np.zeros((cap // bm, 4), np.int32),
        num_blocks=np.zeros(1, np.int32),
    )
    rc = lib().orc_align_local(_ptr(ids, ctypes.c_int32), T, K, E, expert_base, L, bm,
                         *[_ptr(out[k], ctypes.c_int32) for k in
                           ("counts", "offsets", "padded_offsets", "sorted_ids", "inv_perm",
                            "block_info", "num_blocks")])
    if rc != 0:
        raise ValueError("expert id outside [0, E)")
    out["num_blocks"] = int(out["num_blocks"][0])
    return out


def forward(prob, x, ids, topk_w, w13, w2, w13_scale=None, w2_scale=None, mode=EXACT,
            tokens=None):
    """out[t, :] (fp64) for the tokens listed (all when tokens is None)."""
    x, w13, w2 = _storage(x), _storage(w13), _storage(w2)
    ids, topk_w = _c(ids, np.int32), _c(topk_w, np.float32)
    w13_scale, w2_scale = _c(w13_scale, np.uint8), _c(w2_scale, np.uint8)
    toks = None if tokens is None else _c(tokens, np.int32)
    n = prob.T if toks is None else len(toks)
    out = np.zeros((n, prob.H), np.float64)
    rc = lib().orc_moe_forward(ctypes.byref(prob), mode, _vptr(x), _ptr(ids, ctypes.c_int32),
                               _ptr(topk_w, ctypes.c_float), _vptr(w13),
                               _ptr(w13_scale, ctypes.c_uint8), _vptr(w2),
                               _ptr(w2_scale, ctypes.c_uint8), _ptr(toks, ctypes.c_int32),
                               0 if toks is None else len(toks), _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("expert id outside [0, E)")
    return out


def forward_by_expert(prob, x, ids, topk_w, w13, w2, w13_scale=None, w2_scale=None, mode=EXACT):
    x, w13, w2 = _storage(x), _storage(w13), _storage(w2)
    ids, topk_w = _c(ids, np.int32), _c(topk_w, np.float32)
    w13_scale, w2_scale = _c(w13_scale, np.uint8), _c(w2_scale, np.uint8)
    out = np.zeros((prob.T, prob.H), np.float64)
    rc = lib().orc_moe_forward_by_expert(ctypes.byref(prob), mode, _vptr(x),
                                         _ptr(ids, ctypes.c_int32), _ptr(topk_w, ctypes.c_float),
                                         _vptr(w13), _ptr(w13_scale, ctypes.c_uint8), _vptr(w2),
                                         _ptr(w2_scale, ctypes.c_uint8),
                                         _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("expert id outside [0, E)")
    return out


def gemm1_silu_rows(prob, x, w13, sorted_ids, expert_of_row, rows, w13_scale=None, mode=EXACT):
    """h[r, :] for the sorted slots `rows` (fp64; sentinel slots stay zero)."""
    x, w13 = _storage(x), _storage(w13)
    sorted_ids, eor, rows = _c(sorted_ids, np.int32), _c(expert_of_row, np.int32), _c(rows,
                                                                                       np.int32)
    h = np.zeros((len(rows), prob.I), np.float64)
    lib().orc_gemm1_silu_rows(ctypes.byref(prob), mode, _vptr(x), _vptr(w13),
                              _ptr(_c(w13_scale, np.uint8), ctypes.c_uint8),
                              _ptr(sorted_ids, ctypes.c_int32), _ptr(eor, ctypes.c_int32),
                              _ptr(rows, ctypes.c_int32), len(rows), _ptr(h, ctypes.c_double))
    return h


def gemm2_weighted_rows(prob, h, w2, topk_w, sorted_ids, expert_of_row, rows, w2_scale=None,
                        h_is_e4m3=False):
    """y[r, :] = w_i * W2[e] h[rows[r]] (fp64) for the sorted slots `rows`."""
    h, w2 = _storage(h), _storage(w2)
    hcode = 2 if h_is_e4m3 else _dtype_code(h)
    topk_w = _c(topk_w, np.float32)
    sorted_ids, eor, rows = _c(sorted_ids, np.int32), _c(expert_of_row, np.int32), _c(rows,
                                                                                       np.int32)
    y = np.zeros((len(rows), prob.H), np.float64)
    lib().orc_gemm2_weighted_rows(ctypes.byref(prob), _vptr(h), hcode, _vptr(w2),
                                  _ptr(_c(w2_scale, np.uint8), ctypes.c_uint8),
                                  _ptr(topk_w, ctypes.c_float), _ptr(sorted_ids, ctypes.c_int32),
                                  _ptr(eor, ctypes.c_int32), _ptr(rows, ctypes.c_int32),
                                  len(rows), _ptr(y, ctypes.c_double))
    return y


def combine(y_sorted, inv_perm, T, K, H):
    y_sorted, inv_perm = _c(y_sorted, np.float32), _c(inv_perm, np.int32)
    out = np.zeros((T, H), np.float64)
    lib().orc_combine(_ptr(y_sorted, ctypes.c_float), _ptr(inv_perm, ctypes.c_int32), T, K, H,
                      _ptr(out, ctypes.c_double))
    return out


def quantize_x_fp8(x):
    """Per-row e4m3 codes and fp32 row scales of x (bf16 bits or fp32)."""
    x = _storage(x)
    T, H = x.shape
    xq = np.zeros((T, H), np.uint8)
    s = np.zeros(T, np.float32)
    lib().orc_quantize_x_fp8(_vptr(x), _dtype_code(x), T, H, _ptr(xq, ctypes.c_uint8),
                             _ptr(s, ctypes.c_float))
    return xq, s


def e4m3_to_float(codes):
    L = lib()
    return np.array([L.orc_e4m3_to_double(int(c)) for c in np.ravel(codes)]).reshape(
        np.shape(codes))


def float_to_e4m3(vals):
    L = lib()
    return np.array([L.orc_float_to_e4m3(float(v)) for v in np.ravel(vals)],
                    np.uint8).reshape(np.shape(vals))


def e2m1_to_float(nibbles):
    L = lib()
    return np.array([L.orc_e2m1_to_double(int(c)) for c in np.ravel(nibbles)]).reshape(
        np.shape(nibbles))


def e8m0_to_float(codes):
    L = lib()
    return np.array([L.orc_e8m0_to_double(int(c)) for c in np.ravel(codes)]).reshape(
        np.shape(codes))


def build_variant(source_text: str, out_dir: str, name: str) -> str:
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle and check that a pin catches it)."""
    src = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, "lib" + name + ".so")
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    src, "-o", so, "-lm"], check=True)
    return so


def source() -> str:
    with open(_SRC) as f:
        return f.read()


class using_library:
    """Context manager: route this module's functions to another build."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        with _lock:
            self.prev = _lib
            L = ctypes.CDLL(self.path)
            _declare(L)
            _lib = L
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.prev
        return False
