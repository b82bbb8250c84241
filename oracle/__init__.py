"""ctypes front end of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it; the product path never does.

Arrays cross this boundary as numpy arrays: 16-bit element types as their raw
``uint16`` codes, fp32 as ``float32``.  The DAG is a list of
``(op, a, b, slot)`` tuples whose ``op`` is one of ``accum, load, scalar,
broadcast, mul, add, relu, store, sub, div, min, max, col_broadcast, sigmoid,
tanh, gelu, silu, hardswish, leaky_relu`` (the node kinds of the epilogue DAG in
"CUTLASS Operator API: Custom epilogue fusions for GEMMs", section "How the
epilogue fusion API works").
"""
import ctypes
import os

import numpy as np

from . import build as _build

_TYPES = {"f16": 0, "bf16": 1, "f32": 2}
_OPS = {"accum": 0, "load": 1, "scalar": 2, "broadcast": 3, "mul": 4, "add": 5,
        "relu": 6, "store": 7, "sub": 8, "div": 9, "min": 10, "max": 11, "col_broadcast": 12,
        "sigmoid": 13, "tanh": 14, "gelu": 15, "silu": 16, "hardswish": 17, "leaky_relu": 18}


class _Node(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("a", ctypes.c_int32), ("b", ctypes.c_int32),
                ("slot", ctypes.c_int32)]


_lib = None


def lib(path=None):
    """Load (building first if needed) and return the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _bind(L):
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    L.orc_f16_to_f64.restype = ctypes.c_double
    L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_f64.restype = ctypes.c_double
    L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.orc_f64_to_f16.restype = ctypes.c_uint16
    L.orc_f64_to_f16.argtypes = [ctypes.c_double]
    L.orc_f64_to_bf16.restype = ctypes.c_uint16
    L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
    for name in ("orc_f16_to_f64_array", "orc_bf16_to_f64_array", "orc_f64_to_f16_array",
                 "orc_f64_to_bf16_array"):
        getattr(L, name).restype = None
        getattr(L, name).argtypes = [P, P, i64]
    L.orc_gemm_epilogue.restype = ctypes.c_int
    L.orc_gemm_epilogue.argtypes = [i64, i64, i64, i64, i32, P, P, i32, P, P, i32, P, i32, P,
                                    i32, P, P, P, i64, P, i32]
    L.orc_gemm_accum.restype = ctypes.c_int
    L.orc_gemm_accum.argtypes = [i64, i64, i64, i64, i32, P, P, P, i64, P, i32]
    return L


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _codes(a, dtype):
    a = np.ascontiguousarray(a)
    if dtype == "f32":
        if a.dtype != np.float32:
            raise TypeError("f32 operand must be a float32 array")
        return a
    if a.dtype == np.float16 and dtype == "f16":
        return a.view(np.uint16)
    if a.dtype not in (np.uint16, np.int16):
        raise TypeError("16-bit operand must be given as raw uint16 codes")
    return a.view(np.uint16)


# ---------------------------------------------------------------- codecs --

def f16_to_f64(codes, L=None):
    c = np.ascontiguousarray(codes, dtype=np.uint16)
    out = np.empty(c.shape, np.float64)
    (L or lib()).orc_f16_to_f64_array(_ptr(c), _ptr(out), c.size)
    return out


def bf16_to_f64(codes, L=None):
    c = np.ascontiguousarray(codes, dtype=np.uint16)
    out = np.empty(c.shape, np.float64)
    (L or lib()).orc_bf16_to_f64_array(_ptr(c), _ptr(out), c.size)
    return out


def f64_to_f16(x, L=None):
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    (L or lib()).orc_f64_to_f16_array(_ptr(v), _ptr(out), v.size)
    return out


def f64_to_bf16(x, L=None):
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    (L or lib()).orc_f64_to_bf16_array(_ptr(v), _ptr(out), v.size)
    return out


def decode(codes, dtype, L=None):
    """Element codes (or float32 values) of ``dtype`` -> float64."""
    if dtype == "f16":
        return f16_to_f64(codes, L)
    if dtype == "bf16":
        return bf16_to_f64(codes, L)
    return np.asarray(codes, dtype=np.float32).astype(np.float64)


# ------------------------------------------------------------ GEMM + DAG --

def gemm_epilogue(L, M, N, K, ab_dtype, A, B, aux, aux_dtypes, scalars, dag, out_dtypes,
                  rows=None, threads=0, want_pre=False, lib_handle=None):
    """Evaluate the GEMM and the epilogue DAG on the CPU in fp64.

    Returns ``(outs, pre)``: ``outs[o]`` has shape ``(n_rows, N)`` (codes for
    16-bit outputs, float32 for f32), ``pre[o]`` the fp64 value each store
    rounded (or None unless ``want_pre``).  ``rows`` lists flattened rows
    ``l*M + i``; None means every row in order.
    """
    h = lib_handle or lib()
    A = _codes(A, ab_dtype)
    B = _codes(B, ab_dtype)
    if A.size != L * M * K or B.size != L * K * N:
        raise ValueError("A or B size does not match L, M, N, K")
    aux_arrays = [_codes(a, t) for a, t in zip(aux, aux_dtypes)]
    n_aux = len(aux_arrays)
    aux_types = (ctypes.c_int32 * max(n_aux, 1))(*[_TYPES[t] for t in aux_dtypes])
    aux_ptrs = (ctypes.c_void_p * max(n_aux, 1))(*[a.ctypes.data for a in aux_arrays])
    sc = np.ascontiguousarray(np.asarray(scalars, dtype=np.float64).reshape(-1))
    nodes = (_Node * len(dag))(*[_Node(_OPS[op], a, b, s) for (op, a, b, s) in dag])
    if rows is None:
        n_rows, rows_arr, rows_ptr = L * M, None, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows, rows_ptr = rows_arr.size, _ptr(rows_arr)
    outs = [np.zeros((n_rows, N), np.float32 if t == "f32" else np.uint16) for t in out_dtypes]
    pres = [np.zeros((n_rows, N), np.float64) for _ in out_dtypes] if want_pre else []
    out_types = (ctypes.c_int32 * len(out_dtypes))(*[_TYPES[t] for t in out_dtypes])
    out_ptrs = (ctypes.c_void_p * len(outs))(*[o.ctypes.data for o in outs])
    pre_ptrs = (ctypes.c_void_p * len(outs))(*[p.ctypes.data for p in pres]) if want_pre else None
    st = h.orc_gemm_epilogue(L, M, N, K, _TYPES[ab_dtype], _ptr(A), _ptr(B), n_aux, aux_types,
                             aux_ptrs, sc.size, _ptr(sc) if sc.size else None, len(dag), nodes,
                             len(outs), out_types, out_ptrs, pre_ptrs, n_rows, rows_ptr, threads)
    if st != 0:
        raise ValueError("oracle rejected the problem (status %d)" % st)
    return outs, (pres if want_pre else None)


def grouped_gemm_epilogue(problems, ab_dtype, As, Bs, auxs, aux_dtypes, scalars, dag, out_dtypes,
                          threads=0, lib_handle=None):
    """A grouped GEMM by its definition: every problem ``g`` (sizes
    ``problems[g] = (M, N, K)``) is an independent one-batch GEMM with the
    shared epilogue DAG and scalars ("Grouped GEMM", example three of the
    Python interface walkthrough).  ``auxs[g]`` lists problem g's aux
    operands.  Returns one ``outs`` list (as gemm_epilogue) per problem."""
    result = []
    for (M, N, K), A, B, aux in zip(problems, As, Bs, auxs):
        outs, _ = gemm_epilogue(1, M, N, K, ab_dtype, A, B, aux, aux_dtypes, scalars, dag,
                                out_dtypes, threads=threads, lib_handle=lib_handle)
        result.append(outs)
    return result


def gemm_accum(L, M, N, K, ab_dtype, A, B, rows=None, threads=0, lib_handle=None):
    """fp64 accumulator rows ``accum[l,i,:]`` (no epilogue)."""
    h = lib_handle or lib()
    A = _codes(A, ab_dtype)
    B = _codes(B, ab_dtype)
    if rows is None:
        n_rows, rows_arr, rows_ptr = L * M, None, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows, rows_ptr = rows_arr.size, _ptr(rows_arr)
    acc = np.zeros((n_rows, N), np.float64)
    st = h.orc_gemm_accum(L, M, N, K, _TYPES[ab_dtype], _ptr(A), _ptr(B), _ptr(acc), n_rows,
                          rows_ptr, threads)
    if st != 0:
        raise ValueError("oracle rejected the problem (status %d)" % st)
    return acc


def threads_default():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
