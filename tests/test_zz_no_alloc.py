"""The allocation-free entry point, gemm_epi_run_unfused_noalloc, checked
against the ordinary unfused entry point through the C ABI.

The variant is for callers that cannot allocate device memory (allocator
callbacks, applications that reserve all device memory up front): it runs the
unfused path on a workspace built into the library instead of one the caller
passes.  This file is collected last on purpose, so a run that stops at the
first failure has already run every other test; it also passes on its own in
a fresh process (the first call on the device does the one-time set-up).
"""
import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu

import _gpu  # noqa: E402
from _gpu import B, W  # noqa: E402


def _outputs(w):
    return [torch.empty(w.L, w.M, w.N, dtype=W.TORCH_DTYPE[dt], device="cuda")
            for _, dt in w.outs]


def test_noalloc_matches_unfused_on_two_calls_in_a_row():
    # one plan, two calls with different inputs: the second must not see the
    # first call's workspace contents
    w = dataclasses.replace(W.BIAS_RELU_SQUARE_L8, L=2, M=256, N=520, K=264, sample_rows=None)
    assert B.gemm_epi_unfused_workspace_bytes  # exported
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag))
    try:
        assert B.gemm_epi_unfused_workspace_bytes(plan) <= B.GE_NOALLOC_SCRATCH_BYTES
        ws = torch.empty(B.gemm_epi_unfused_workspace_bytes(plan) // 4, dtype=torch.float32,
                         device="cuda")
        for seed in (11, 12):
            inputs = W.make_inputs(dataclasses.replace(w, seed=seed))
            A, Bm, aux, sc = inputs
            Ad, Bd, auxd = A.cuda(), Bm.cuda(), [a.cuda() for a in aux]
            ref, got = _outputs(w), _outputs(w)
            B.gemm_epi_run_unfused(plan, Ad, Bd, auxd, sc, ref, ws)
            B.gemm_epi_run_unfused_noalloc(plan, Ad, Bd, auxd, sc, got)
            torch.cuda.synchronize()
            assert B.gemm_epi_last_error(plan) == B.GE_OK
            ref_h, got_h = [t.cpu() for t in ref], [t.cpu() for t in got]
            # against the oracle, as every parity test: the tolerance of the
            # N(0,1) workloads, elementwise
            _gpu.compare(w, got_h, _gpu.oracle_rows(w, inputs))
            # against the caller-workspace entry point: the tolerance the
            # parity tests use, and in fact identical bits (same program on
            # the same fp32 accumulator)
            _gpu.compare(w, got_h, [W.to_codes(t).reshape(w.L * w.M, w.N) for t in ref_h])
            _gpu.bitwise_equal(got_h, ref_h)
    finally:
        B.gemm_epi_plan_destroy(plan)


def test_noalloc_call_allocates_no_device_memory():
    """The property the entry point exists for: once the device is set up
    (a first call, which also loads the kernels), a call leaves the device's
    free memory and torch's allocator exactly where they were, and its
    results still match the oracle."""
    w = dataclasses.replace(W.MY_EPILOGUE_128, L=2, M=200, N=264, K=200, sample_rows=None)
    inputs = W.make_inputs(w)
    A, Bm, aux, sc = inputs
    Ad, Bd, auxd = A.cuda(), Bm.cuda(), [a.cuda() for a in aux]
    outs = _outputs(w)
    stream = torch.cuda.Stream()
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag))
    try:
        B.gemm_epi_run_unfused_noalloc(plan, Ad, Bd, auxd, sc, outs, stream=stream)
        torch.cuda.synchronize()
        for o in outs:
            o.zero_()
        torch.cuda.synchronize()
        free_before, _ = torch.cuda.mem_get_info()
        torch_before = torch.cuda.memory_allocated()
        B.gemm_epi_run_unfused_noalloc(plan, Ad, Bd, auxd, sc, outs, stream=stream)
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
        assert free_after == free_before, (free_before, free_after)
        assert torch.cuda.memory_allocated() == torch_before
        assert B.gemm_epi_last_error(plan) == B.GE_OK
    finally:
        B.gemm_epi_plan_destroy(plan)
    _gpu.compare(w, [o.cpu() for o in outs], _gpu.oracle_rows(w, inputs))


def test_noalloc_rejects_problems_beyond_its_workspace():
    w = W.ALPHA_BETA_X_8192  # 8192^3: 256 MiB of fp32 workspace
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag))
    try:
        assert B.gemm_epi_unfused_workspace_bytes(plan) > B.GE_NOALLOC_SCRATCH_BYTES
        dummy = torch.empty(16, dtype=torch.float16, device="cuda")
        st = B.gemm_epi_run_unfused_noalloc(plan, dummy, dummy, [dummy, dummy], [1.0, 1.0, 1.0],
                                            [dummy, dummy], check=False)
        assert st == B.GE_ERR_WORKSPACE
    finally:
        B.gemm_epi_plan_destroy(plan)
