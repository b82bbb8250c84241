"""Kernels compiled at plan time for epilogues outside the built-in set
(ge_options.specialize): bit-identical to the interpreter, and to the
oracle where the inputs make every value exact, in batched, grouped and
column-major launches."""
import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu

import _gpu  # noqa: E402
import test_gpu_grouped as G  # noqa: E402
import test_gpu_random_dags as R  # noqa: E402
from _gpu import B, W  # noqa: E402

NOT_BUILT_IN = ["relu_aux_store", "relu_scale_return_acc", "clamp_f16", "aux_normalize_f16",
                "scale_shift_bf16", "act_sigmoid", "act_leaky_relu"]
EXAMPLES = {x.name: x for x in W.page_examples(L=2, M=264, N=392, K=200)}


@pytest.mark.parametrize("name", NOT_BUILT_IN)
@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=lambda v: "cg%d_n%d" % v)
def test_specialized_matches_interpreter(name, variant):
    w = EXAMPLES[name]
    inputs = W.make_inputs(w)
    base = dict(cta_group=variant[0], tile_n=variant[1])
    spec, info = _gpu.run_gpu(w, inputs, options=B.ge_options(**base))
    interp, info2 = _gpu.run_gpu(w, inputs, options=B.ge_options(specialize=-1, **base))
    assert info["epi_variant"] == -3 and info2["epi_variant"] in (-1, -2)
    _gpu.bitwise_equal(spec, interp)
    _gpu.compare(w, spec, _gpu.oracle_rows(w, inputs))


@pytest.mark.parametrize("seed", [1, 5, 11, 17, 23, 31])
def test_specialized_random_dags(seed):
    w = R.random_workload(seed)
    inputs = W.make_inputs(w)
    spec, info = _gpu.run_gpu(w, inputs)
    assert info["epi_variant"] in (-3,) or info["epi_variant"] >= 0
    interp, _ = _gpu.run_gpu(w, inputs, options=B.ge_options(specialize=-1))
    _gpu.bitwise_equal(spec, interp)
    _gpu.compare(w, spec, _gpu.oracle_rows(w, inputs))


def test_specialized_grouped_and_column_major():
    """A grouped launch of a DAG outside the built-in set, and the same DAG
    with every operand column-major."""
    w = G.W.GROUPED_BY_NAME["grouped_bias_relu_ragged"]
    info = G.run_and_check(w)
    assert info["epi_variant"] == -3
    import test_gpu_majors as M
    wb = EXAMPLES["relu_aux_store"]
    inputs = W.make_inputs(wb)
    gpu = M.run_majors(wb, inputs, (1, 1, 1))
    _gpu.compare(wb, gpu, _gpu.oracle_rows(wb, inputs))


def test_plan_time_compilation_is_cached():
    """The second plan of the same program and launch shape reuses the
    compiled kernel (plan creation then takes milliseconds)."""
    import time
    w = dataclasses.replace(EXAMPLES["clamp_f16"], M=520, N=264)
    dt, dag = _gpu.dtypes_of(w), B.make_dag(w.dag)
    opts = B.ge_options(cta_group=1, tile_n=64, stages=3)
    t0 = time.time()
    p1 = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, dt, dag, opts)
    first = time.time() - t0
    t0 = time.time()
    p2 = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, dt, dag, opts)
    second = time.time() - t0
    try:
        assert B.gemm_epi_plan_info(p1)["epi_variant"] == -3
        assert B.gemm_epi_plan_info(p2)["epi_variant"] == -3
        assert second < 0.1, (first, second)
    finally:
        B.gemm_epi_plan_destroy(p1)
        B.gemm_epi_plan_destroy(p2)


def test_specialized_four_warps_at_long_k():
    """A compiled epilogue on 4 warps (the option) at long K: the compiled
    kernel is then the 4-warp instance, still bit-identical to the
    interpreter and exact against the oracle."""
    w = dataclasses.replace(EXAMPLES["relu_aux_store"], L=1, M=256, N=264, K=8192)
    inputs = W.make_inputs(w)
    spec, info = _gpu.run_gpu(w, inputs, options=B.ge_options(epi_warps=4))
    assert info["epi_variant"] == -3 and info["epi_warps"] == 4, info
    interp, info2 = _gpu.run_gpu(w, inputs, options=B.ge_options(specialize=-1))
    assert info2["epi_variant"] in (-1, -2)
    _gpu.bitwise_equal(spec, interp)
    _gpu.compare(w, spec, _gpu.oracle_rows(w, inputs))
