"""Thin ctypes binding of libgemm_epi.so (include/gemm_epi.h).

Argument marshalling only: every step of the GEMM and the epilogue runs in the
library's CUDA kernels.  Functions keep the C names; tensors may be given as
torch tensors (their data pointers are passed) or as raw integer addresses.
Importing this module raises if the library has not been built: there is no
fallback.
"""
import ctypes
import os

from . import build as _build

GE_F16, GE_BF16, GE_F32 = 0, 1, 2
(GE_ACCFETCH, GE_LOAD, GE_SCALAR, GE_BROADCAST, GE_MUL, GE_ADD, GE_RELU, GE_STORE, GE_SUB, GE_DIV,
 GE_MIN, GE_MAX, GE_COL_BROADCAST, GE_SIGMOID, GE_TANH, GE_GELU, GE_SILU, GE_HARDSWISH,
 GE_LEAKY_RELU) = range(19)
GE_MAX_NODES, GE_MAX_AUX, GE_MAX_TMA_AUX, GE_MAX_OUT, GE_MAX_SCALARS = 16, 8, 4, 4, 16
GE_DEBUG_SKIP_FIRST_LOAD = 1
GE_DEBUG_FORCE_INTERPRETER = 2
GE_DEBUG_NO_TAIL_SPLIT = 4
GE_ROW_MAJOR, GE_COL_MAJOR = 0, 1

STATUS = ["GE_OK", "GE_ERR_NO_ACCUM", "GE_ERR_NO_D", "GE_ERR_SSA", "GE_ERR_MISSING_ARG",
          "GE_ERR_UNSUPPORTED", "GE_ERR_MISALIGNED", "GE_ERR_ARCH", "GE_ERR_SHAPE",
          "GE_ERR_TIMEOUT", "GE_ERR_CUDA", "GE_ERR_INVALID", "GE_ERR_SMEM", "GE_ERR_WORKSPACE"]
for _i, _n in enumerate(STATUS):
    globals()[_n] = _i

DTYPE = {"f16": GE_F16, "bf16": GE_BF16, "f32": GE_F32}
OP = {"accum": GE_ACCFETCH, "load": GE_LOAD, "scalar": GE_SCALAR, "broadcast": GE_BROADCAST,
      "mul": GE_MUL, "add": GE_ADD, "relu": GE_RELU, "store": GE_STORE, "sub": GE_SUB,
      "div": GE_DIV, "min": GE_MIN, "max": GE_MAX, "col_broadcast": GE_COL_BROADCAST,
      "sigmoid": GE_SIGMOID, "tanh": GE_TANH, "gelu": GE_GELU, "silu": GE_SILU,
      "hardswish": GE_HARDSWISH, "leaky_relu": GE_LEAKY_RELU}

# exported symbols of include/gemm_epi.h
EXPORTS = ["gemm_epi_plan_create", "gemm_epi_plan_create_ex", "gemm_epi_validate", "gemm_epi_run",
           "gemm_epi_unfused_workspace_bytes", "gemm_epi_run_unfused", "gemm_epi_plan_destroy",
           "gemm_epi_plan_info", "gemm_epi_status_string", "gemm_epi_last_error",
           "gemm_epi_run_unfused_noalloc", "gemm_epi_grouped_plan_create", "gemm_epi_grouped_run"]
GE_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
GE_MAX_GROUPS = 4096


class ge_node(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("a", ctypes.c_int32), ("b", ctypes.c_int32),
                ("slot", ctypes.c_int32)]


class ge_dag(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("node", ge_node * GE_MAX_NODES)]


class ge_dtypes(ctypes.Structure):
    _fields_ = [("ab", ctypes.c_int32), ("acc", ctypes.c_int32), ("n_aux", ctypes.c_int32),
                ("n_scalar", ctypes.c_int32), ("n_out", ctypes.c_int32),
                ("aux", ctypes.c_int32 * GE_MAX_AUX), ("out", ctypes.c_int32 * GE_MAX_OUT)]


class ge_options(ctypes.Structure):
    _fields_ = [("cta_group", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("max_ctas", ctypes.c_int32),
                ("raster_group", ctypes.c_int32), ("timeout_ms", ctypes.c_int32),
                ("debug_flags", ctypes.c_uint32), ("cluster_n", ctypes.c_int32),
                ("a_major", ctypes.c_int32), ("b_major", ctypes.c_int32),
                ("cd_major", ctypes.c_int32), ("epi_warps", ctypes.c_int32),
                ("specialize", ctypes.c_int32), ("no_pdl", ctypes.c_int32)]


class ge_problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class ge_plan_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("cta_group", "tile_m", "tile_n", "tile_k", "stages", "epi_chunk", "aux_stages",
                 "grid", "num_tiles", "smem_bytes", "n_instr", "n_regs", "num_sms",
                 "epi_variant", "cluster_n", "epi_warps", "raster_group")]


class GemmEpiError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        name = STATUS[status] if 0 <= status < len(STATUS) else "GE_ERR_UNKNOWN"
        super().__init__("%s%s (%d)" % (where + ": " if where else "", name, status))


def library_path():
    return _build.LIB


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError("libgemm_epi.so is not built (%s); run __graft_entry__.build() or "
                          "python -m dense_gemm_elementwise_gb300.build" % path)
    L = ctypes.CDLL(path)
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    pp = ctypes.POINTER(ctypes.c_void_p)
    L.gemm_epi_plan_create.restype = ctypes.c_int
    L.gemm_epi_plan_create.argtypes = [pp, i64, i64, i64, i64, ctypes.POINTER(ge_dtypes),
                                       ctypes.POINTER(ge_dag)]
    L.gemm_epi_plan_create_ex.restype = ctypes.c_int
    L.gemm_epi_plan_create_ex.argtypes = [pp, i64, i64, i64, i64, ctypes.POINTER(ge_dtypes),
                                          ctypes.POINTER(ge_dag), ctypes.POINTER(ge_options)]
    L.gemm_epi_validate.restype = ctypes.c_int
    L.gemm_epi_validate.argtypes = [ctypes.POINTER(ge_dtypes), ctypes.POINTER(ge_dag)]
    L.gemm_epi_run.restype = ctypes.c_int
    L.gemm_epi_run.argtypes = [P, P, P, pp, ctypes.POINTER(ctypes.c_float), pp, P]
    L.gemm_epi_unfused_workspace_bytes.restype = ctypes.c_size_t
    L.gemm_epi_unfused_workspace_bytes.argtypes = [P]
    L.gemm_epi_run_unfused.restype = ctypes.c_int
    L.gemm_epi_run_unfused.argtypes = [P, P, P, pp, ctypes.POINTER(ctypes.c_float), pp, P,
                                       ctypes.c_size_t, P]
    L.gemm_epi_run_unfused_noalloc.restype = ctypes.c_int
    L.gemm_epi_run_unfused_noalloc.argtypes = [P, P, P, pp, ctypes.POINTER(ctypes.c_float), pp, P]
    L.gemm_epi_grouped_plan_create.restype = ctypes.c_int
    L.gemm_epi_grouped_plan_create.argtypes = [pp, i32, ctypes.POINTER(ge_problem),
                                               ctypes.POINTER(ge_dtypes), ctypes.POINTER(ge_dag),
                                               ctypes.POINTER(ge_options)]
    L.gemm_epi_grouped_run.restype = ctypes.c_int
    L.gemm_epi_grouped_run.argtypes = [P, pp, pp, pp, ctypes.POINTER(ctypes.c_float), pp, P]
    L.gemm_epi_plan_destroy.restype = None
    L.gemm_epi_plan_destroy.argtypes = [P]
    L.gemm_epi_plan_info.restype = ctypes.c_int
    L.gemm_epi_plan_info.argtypes = [P, ctypes.POINTER(ge_plan_info)]
    L.gemm_epi_status_string.restype = ctypes.c_char_p
    L.gemm_epi_status_string.argtypes = [ctypes.c_int]
    L.gemm_epi_last_error.restype = ctypes.c_int
    L.gemm_epi_last_error.argtypes = [P]
    return L


lib = _load()


# ------------------------------------------------------------ marshalling --

def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptr_array(items):
    n = max(len(items), 1)
    arr = (ctypes.c_void_p * n)()
    for i, x in enumerate(items):
        arr[i] = _addr(x)
    return arr


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_dtypes(ab, aux_dtypes, n_scalar, out_dtypes):
    d = ge_dtypes()
    d.ab = DTYPE[ab] if isinstance(ab, str) else ab
    d.acc = GE_F32
    d.n_aux = len(aux_dtypes)
    d.n_scalar = n_scalar
    d.n_out = len(out_dtypes)
    for i, t in enumerate(aux_dtypes):
        d.aux[i] = DTYPE[t] if isinstance(t, str) else t
    for i, t in enumerate(out_dtypes):
        d.out[i] = DTYPE[t] if isinstance(t, str) else t
    return d


def make_dag(nodes):
    """``nodes``: (op, a, b, slot) tuples, op a name or a GE_* code."""
    g = ge_dag()
    g.n = len(nodes)
    for i, (op, a, b, s) in enumerate(nodes):
        g.node[i] = ge_node(OP[op] if isinstance(op, str) else op, a, b, s)
    return g


# ----------------------------------------------------------------- C API --

def gemm_epi_validate(dtypes, dag):
    return lib.gemm_epi_validate(ctypes.byref(dtypes), ctypes.byref(dag))


def gemm_epi_plan_create(L, M, N, K, dtypes, dag, options=None):
    """Returns the plan handle; raises GemmEpiError with the status code."""
    h = ctypes.c_void_p()
    if options is None:
        st = lib.gemm_epi_plan_create(ctypes.byref(h), L, M, N, K, ctypes.byref(dtypes),
                                      ctypes.byref(dag))
    else:
        st = lib.gemm_epi_plan_create_ex(ctypes.byref(h), L, M, N, K, ctypes.byref(dtypes),
                                         ctypes.byref(dag), ctypes.byref(options))
    if st != GE_OK:
        raise GemmEpiError(st, "gemm_epi_plan_create")
    return h


def gemm_epi_plan_destroy(plan):
    lib.gemm_epi_plan_destroy(plan)


def gemm_epi_plan_info(plan):
    info = ge_plan_info()
    st = lib.gemm_epi_plan_info(plan, ctypes.byref(info))
    if st != GE_OK:
        raise GemmEpiError(st, "gemm_epi_plan_info")
    return {n: getattr(info, n) for n, _ in ge_plan_info._fields_}


def _scalars(scalars):
    n = max(len(scalars), 1)
    return (ctypes.c_float * n)(*[float(s) for s in scalars])


def gemm_epi_run(plan, A, B, aux, scalars, outs, stream=None, check=True):
    st = lib.gemm_epi_run(plan, _addr(A), _addr(B), _ptr_array(aux), _scalars(scalars),
                          _ptr_array(outs), _stream(stream))
    if check and st != GE_OK:
        raise GemmEpiError(st, "gemm_epi_run")
    return st


def gemm_epi_unfused_workspace_bytes(plan):
    return lib.gemm_epi_unfused_workspace_bytes(plan)


def gemm_epi_run_unfused(plan, A, B, aux, scalars, outs, workspace, workspace_bytes=None,
                         stream=None, check=True):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib.gemm_epi_run_unfused(plan, _addr(A), _addr(B), _ptr_array(aux), _scalars(scalars),
                                  _ptr_array(outs), _addr(workspace), workspace_bytes,
                                  _stream(stream))
    if check and st != GE_OK:
        raise GemmEpiError(st, "gemm_epi_run_unfused")
    return st


def gemm_epi_run_unfused_noalloc(plan, A, B, aux, scalars, outs, stream=None, check=True):
    """The unfused path on the library's built-in workspace: for callers that
    cannot allocate device memory themselves (see include/gemm_epi.h)."""
    st = lib.gemm_epi_run_unfused_noalloc(plan, _addr(A), _addr(B), _ptr_array(aux),
                                          _scalars(scalars), _ptr_array(outs), _stream(stream))
    if check and st != GE_OK:
        raise GemmEpiError(st, "gemm_epi_run_unfused_noalloc")
    return st


def gemm_epi_grouped_plan_create(problems, dtypes, dag, options=None):
    """``problems``: (M, N, K) triples.  Returns the plan handle; raises
    GemmEpiError with the status code."""
    n = len(problems)
    arr = (ge_problem * max(n, 1))(*[ge_problem(int(m), int(nn), int(k)) for m, nn, k in problems])
    h = ctypes.c_void_p()
    st = lib.gemm_epi_grouped_plan_create(ctypes.byref(h), n, arr, ctypes.byref(dtypes),
                                          ctypes.byref(dag),
                                          ctypes.byref(options) if options is not None else None)
    if st != GE_OK:
        raise GemmEpiError(st, "gemm_epi_grouped_plan_create")
    return h


def gemm_epi_grouped_run(plan, As, Bs, aux, scalars, outs, stream=None, check=True):
    """``As``, ``Bs``: one tensor per problem; ``aux``, ``outs``: one list per
    problem (its aux slots / output slots), flattened problem-major."""
    flat_aux = [x for per in aux for x in per]
    flat_out = [x for per in outs for x in per]
    st = lib.gemm_epi_grouped_run(plan, _ptr_array(As), _ptr_array(Bs),
                                  _ptr_array(flat_aux) if flat_aux else None, _scalars(scalars),
                                  _ptr_array(flat_out), _stream(stream))
    if check and st != GE_OK:
        raise GemmEpiError(st, "gemm_epi_grouped_run")
    return st


def prepare_grouped_run(plan, As, Bs, aux, scalars, outs, stream=None):
    """Marshal the arguments of gemm_epi_grouped_run once; the returned
    callable issues the run with no per-call Python marshalling and returns
    its status."""
    flat_aux = [x for per in aux for x in per]
    flat_out = [x for per in outs for x in per]
    args = (plan, _ptr_array(As), _ptr_array(Bs), _ptr_array(flat_aux) if flat_aux else None,
            _scalars(scalars), _ptr_array(flat_out), _stream(stream))
    fn = lib.gemm_epi_grouped_run
    return lambda: fn(*args)


def prepare_run(plan, A, B, aux, scalars, outs, stream=None):
    """As prepare_grouped_run, for gemm_epi_run."""
    args = (plan, _addr(A), _addr(B), _ptr_array(aux), _scalars(scalars), _ptr_array(outs),
            _stream(stream))
    fn = lib.gemm_epi_run
    return lambda: fn(*args)


def gemm_epi_status_string(status):
    return lib.gemm_epi_status_string(status).decode()


def gemm_epi_last_error(plan=None):
    return lib.gemm_epi_last_error(plan)
