"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every function include/gemm_epi.h declares, DAG validation returns
the documented status codes (the pages' failure cases), and plan creation
reports the missing device instead of falling back to anything."""
import ctypes
import os
import re

import pytest

from dense_gemm_elementwise_gb300 import build as gbuild

gbuild.build()
from dense_gemm_elementwise_gb300 import binding as B  # noqa: E402
from dense_gemm_elementwise_gb300 import workloads as W  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    with open(os.path.join(ROOT, "include", "gemm_epi.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(gemm_epi_\w+)\(", text, re.M)))


def test_header_declares_the_boundary():
    names = header_functions()
    assert set(names) == set(B.EXPORTS), names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.library_path())
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for code, name in enumerate(B.STATUS):
        assert B.gemm_epi_status_string(code) == name
    assert B.gemm_epi_status_string(999) == "GE_ERR_UNKNOWN"


def _dt(w):
    return B.make_dtypes(w.ab, [s[2] for s in w.aux], len(w.scalars), [dt for _, dt in w.outs])


@pytest.mark.parametrize("w", W.WORKLOADS + W.page_examples(), ids=lambda w: w.name)
def test_workload_dags_validate(w):
    assert B.gemm_epi_validate(_dt(w), B.make_dag(w.dag)) == B.GE_OK


def _base():
    w = W.MY_EPILOGUE_128
    return _dt(w), list(w.dag)


def test_missing_accum():
    # "accum must be an input to the epilogue function": D = C * beta
    dt, _ = _base()
    dag = [("load", 0, 0, 0), ("scalar", 0, 0, 1), ("mul", 0, 1, 0), ("store", 2, 0, 0)]
    dt.n_out = 1
    assert B.gemm_epi_validate(dt, B.make_dag(dag)) == B.GE_ERR_NO_ACCUM


def test_missing_D():
    # "Output node D is not found": F is returned, D never stored
    dt, _ = _base()
    dag = [("accum", 0, 0, 0), ("store", 0, 0, 1)]
    assert B.gemm_epi_validate(dt, B.make_dag(dag)) == B.GE_ERR_NO_D


def test_ssa_violations():
    dt, dag = _base()
    # an output stored twice ("Variable 'tmp' cannot be defined twice")
    bad = dag + [("store", 0, 0, 1)]
    assert B.gemm_epi_validate(dt, B.make_dag(bad)) == B.GE_ERR_SSA
    # an operand that refers to itself / a later node
    bad = [("accum", 0, 0, 0), ("mul", 1, 0, 0), ("store", 1, 0, 0)]
    dt.n_out = 1
    assert B.gemm_epi_validate(dt, B.make_dag(bad)) == B.GE_ERR_SSA
    # an operand that is a store (stores produce no value)
    bad = [("accum", 0, 0, 0), ("store", 0, 0, 0), ("relu", 1, 0, 0)]
    assert B.gemm_epi_validate(dt, B.make_dag(bad)) == B.GE_ERR_SSA


def test_missing_arguments():
    # "Argument alpha is not provided": scalar slot beyond n_scalar
    dt, dag = _base()
    dt.n_scalar = 2
    assert B.gemm_epi_validate(dt, B.make_dag(dag)) == B.GE_ERR_MISSING_ARG
    # "Argument D is not provided": store slot beyond n_out
    dt, dag = _base()
    dt.n_out = 1
    assert B.gemm_epi_validate(dt, B.make_dag(dag)) == B.GE_ERR_MISSING_ARG
    # aux slot beyond n_aux
    dt, dag = _base()
    dt.n_aux = 0
    assert B.gemm_epi_validate(dt, B.make_dag(dag)) == B.GE_ERR_MISSING_ARG


def test_unsupported():
    dt, dag = _base()
    bad = [("accum", 0, 0, 0), (42, 0, 0, 0), ("store", 0, 0, 0)]
    assert B.gemm_epi_validate(dt, B.make_dag(bad)) == B.GE_ERR_UNSUPPORTED
    dt2, _ = _base()
    dt2.acc = B.GE_F16  # the accumulator must be fp32
    assert B.gemm_epi_validate(dt2, B.make_dag(dag)) == B.GE_ERR_UNSUPPORTED
    dt3, _ = _base()
    dt3.ab = B.GE_F32  # A/B are fp16 or bf16
    assert B.gemm_epi_validate(dt3, B.make_dag(dag)) == B.GE_ERR_UNSUPPORTED
    # one aux slot used both as a tensor and as a row vector
    dt4, _ = _base()
    bad = [("accum", 0, 0, 0), ("load", 0, 0, 0), ("broadcast", 0, 0, 0), ("add", 0, 1, 0),
           ("add", 3, 2, 0), ("store", 4, 0, 0), ("store", 0, 0, 1)]
    assert B.gemm_epi_validate(dt4, B.make_dag(bad)) == B.GE_ERR_UNSUPPORTED


def test_activation_nodes():
    """Unary activations take one earlier value; leaky ReLU two (value,
    slope); any of them referring to itself or a later node is an SSA error."""
    dt, _ = _base()
    dt.n_out = 1
    for act in W.ACTIVATIONS[:-1]:
        ok = [("accum", 0, 0, 0), ("load", 0, 0, 0), (act, 1, 0, 0), ("add", 0, 2, 0),
              (act, 3, 0, 0), ("store", 4, 0, 0)]
        assert B.gemm_epi_validate(dt, B.make_dag(ok)) == B.GE_OK, act
        bad = [("accum", 0, 0, 0), (act, 2, 0, 0), ("store", 1, 0, 0)]
        assert B.gemm_epi_validate(dt, B.make_dag(bad)) == B.GE_ERR_SSA, act
    ok = [("accum", 0, 0, 0), ("scalar", 0, 0, 0), ("leaky_relu", 0, 1, 0), ("store", 2, 0, 0)]
    assert B.gemm_epi_validate(dt, B.make_dag(ok)) == B.GE_OK
    bad = [("accum", 0, 0, 0), ("leaky_relu", 0, 2, 0), ("scalar", 0, 0, 0), ("store", 1, 0, 0)]
    assert B.gemm_epi_validate(dt, B.make_dag(bad)) == B.GE_ERR_SSA
    # PReLU: the slope is a row vector
    ok = [("accum", 0, 0, 0), ("broadcast", 0, 0, 0), ("leaky_relu", 0, 1, 0), ("store", 2, 0, 0)]
    assert B.gemm_epi_validate(dt, B.make_dag(ok)) == B.GE_OK


def test_program_register_counts():
    """Five values live at once: more than the 4 registers of the compact
    interpreter, within the 8 the program may use (16 nodes cannot keep more
    than 7 values live), so the DAG is accepted."""
    g = W.Dag()
    acc = g.accum()
    sc = g.scalar(0)
    vals = [g.mul(acc, sc)] + [g.mul(g.load(i), sc) for i in range(4)]
    s = vals[0]
    for v in vals[1:]:
        s = g.add(s, v)
    g.store(s, 0)
    dt = B.make_dtypes("f16", ["f16"] * 4, 1, ["f16"])
    assert B.gemm_epi_validate(dt, B.make_dag(g.nodes)) == B.GE_OK
    # the same sum accumulated as it goes needs only two
    g = W.Dag()
    sc = g.scalar(0)
    s = g.mul(g.accum(), sc)
    for i in range(4):
        s = g.add(s, g.mul(g.load(i), sc))
    g.store(s, 0)
    assert B.gemm_epi_validate(dt, B.make_dag(g.nodes)) == B.GE_OK


def test_empty_and_oversized_dags():
    dt, _ = _base()
    assert B.gemm_epi_validate(dt, B.make_dag([])) == B.GE_ERR_UNSUPPORTED
    big = B.ge_dag()
    big.n = B.GE_MAX_NODES + 1
    assert B.gemm_epi_validate(dt, big) == B.GE_ERR_UNSUPPORTED


def test_plan_create_checks_before_device():
    dt, dag = _base()
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_plan_create(1, 0, 128, 128, dt, B.make_dag(dag))
    assert e.value.status == B.GE_ERR_SHAPE
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_plan_create(1, 128, 128, 100, dt, B.make_dag(dag))  # K*2 bytes not 16-aligned
    assert e.value.status == B.GE_ERR_MISALIGNED
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_plan_create(1, 128, 12, 128, dt, B.make_dag(dag))   # N*2 bytes not 16-aligned
    assert e.value.status == B.GE_ERR_MISALIGNED


def test_plan_create_without_gpu_reports_arch():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    dt, dag = _base()
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_plan_create(1, 128, 128, 128, dt, B.make_dag(dag))
    assert e.value.status == B.GE_ERR_ARCH


def _grouped_base():
    w = W.GROUPED_BY_NAME["grouped_gemm_50"]
    return B.make_dtypes(w.ab, [s[2] for s in w.aux], len(w.scalars),
                         [dt for _, dt in w.outs]), B.make_dag(w.dag)


def test_grouped_plan_create_checks_before_device():
    dt, dag = _grouped_base()
    cases = [([], B.GE_ERR_SHAPE),                                   # no problems
             ([(128, 128, 128)] * (B.GE_MAX_GROUPS + 1), B.GE_ERR_SHAPE),
             ([(128, 128, 128), (0, 128, 128)], B.GE_ERR_SHAPE),     # M = 0
             ([(128, 128, 128), (128, 128, -8)], B.GE_ERR_SHAPE),    # K < 0
             ([(128, 128, 128), (128, 128, 100)], B.GE_ERR_MISALIGNED),  # K*2 bytes
             ([(64, 12, 64)], B.GE_ERR_MISALIGNED)]                  # N*2 bytes
    for problems, want in cases:
        with pytest.raises(B.GemmEpiError) as e:
            B.gemm_epi_grouped_plan_create(problems, dt, dag)
        assert e.value.status == want, (problems[:2], e.value.status)
    bad = [("accum", 0, 0, 0), ("relu", 0, 0, 0)]  # D never stored
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_grouped_plan_create([(128, 128, 128)], dt, B.make_dag(bad))
    assert e.value.status == B.GE_ERR_NO_D


def test_grouped_plan_create_without_gpu_reports_arch():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    dt, dag = _grouped_base()
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_grouped_plan_create([(128, 256, 64), (256, 128, 128)], dt, dag)
    assert e.value.status == B.GE_ERR_ARCH


def test_grouped_run_rejects_null_plan():
    assert B.lib.gemm_epi_grouped_run(None, None, None, None, None, None, None) == \
        B.GE_ERR_INVALID


def test_majors_checked_before_device():
    """Storage orders: bad values, the contiguous dimension of each tensor
    (per its major) in whole 16-byte units; no cluster of more than one
    CTA pair (cluster_n 2 was an A-multicast option, since removed)."""
    dt, dag = _base()
    cases = [(dict(a_major=1), (1, 100, 128, 128), B.GE_ERR_MISALIGNED),
             (dict(b_major=1), (1, 128, 128, 100), B.GE_ERR_MISALIGNED),
             (dict(b_major=1), (1, 128, 12, 128), B.GE_ERR_MISALIGNED),   # C, D rows still N
             (dict(cd_major=1), (1, 100, 128, 128), B.GE_ERR_MISALIGNED),
             (dict(cd_major=-1), (1, 128, 128, 128), B.GE_ERR_INVALID),
             (dict(b_major=3), (1, 128, 128, 128), B.GE_ERR_INVALID),
             (dict(cluster_n=2), (1, 128, 128, 128), B.GE_ERR_UNSUPPORTED),
             (dict(cluster_n=-1), (1, 128, 128, 128), B.GE_ERR_UNSUPPORTED)]
    for kw, (L, M, N, K), want in cases:
        with pytest.raises(B.GemmEpiError) as e:
            B.gemm_epi_plan_create(L, M, N, K, dt, B.make_dag(dag), B.ge_options(**kw))
        assert e.value.status == want, (kw, e.value.status)
    gdt, gdag = _grouped_base()
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_grouped_plan_create([(128, 128, 128), (100, 128, 128)], gdt, gdag,
                                       B.ge_options(a_major=1))
    assert e.value.status == B.GE_ERR_MISALIGNED
