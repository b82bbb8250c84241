"""GPU parity for the other storage orders (a_major, b_major, cd_major of
"Custom Epilogue Example", step "Define tensor arguments"): the logical
problem is the same, only the device copies are transposed; the oracle sees
the logical row-major tensors."""
import dataclasses
import itertools

import pytest
import torch

pytestmark = pytest.mark.gpu

import _gpu  # noqa: E402
from _gpu import B, W  # noqa: E402

DEV = torch.device("cuda", 0)
MAJORS = list(itertools.product([B.GE_ROW_MAJOR, B.GE_COL_MAJOR], repeat=3))


def mid(m):
    return "A%s_B%s_CD%s" % tuple("col" if x else "row" for x in m)


def to_device(t, col):
    """(L, R, C) logical -> device copy, stored (L, C, R) when col."""
    t = t.transpose(-1, -2).contiguous() if col else t
    return t.to(DEV)


def run_majors(w, inputs, majors, unfused=False, **opt):
    a_major, b_major, cd_major = majors
    A, Bm, aux, scalars = inputs
    Ad, Bd = to_device(A, a_major), to_device(Bm, b_major)
    auxd = [to_device(a, cd_major) if a.dim() == 3 else a.to(DEV) for a in aux]
    shape = (w.L, w.N, w.M) if cd_major else (w.L, w.M, w.N)
    outs = [torch.full(shape, float("nan"), dtype=W.TORCH_DTYPE[dt], device=DEV)
            for _, dt in w.outs]
    options = B.ge_options(a_major=a_major, b_major=b_major, cd_major=cd_major, **opt)
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag),
                                  options)
    try:
        if unfused:
            ws = torch.empty(B.gemm_epi_unfused_workspace_bytes(plan) // 4, dtype=torch.float32,
                             device=DEV)
            B.gemm_epi_run_unfused(plan, Ad, Bd, auxd, scalars, outs, ws)
        else:
            B.gemm_epi_run(plan, Ad, Bd, auxd, scalars, outs)
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(plan) == B.GE_OK
    finally:
        B.gemm_epi_plan_destroy(plan)
    return [(o.transpose(-1, -2) if cd_major else o).contiguous().cpu() for o in outs]


BASE = dataclasses.replace(W.MY_EPILOGUE_128, L=2, M=264, N=392, K=200, sample_rows=None)


@pytest.mark.parametrize("majors", MAJORS, ids=mid)
@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=lambda v: "cg%d_n%d" % v)
def test_majors_exact(majors, variant):
    """Integer inputs, the Aux/D epilogue of my_epilogue: bit-exact for every
    combination of majors, on a ragged shape spanning several tiles."""
    w = BASE
    inputs = W.make_inputs(w)
    gpu = run_majors(w, inputs, majors, cta_group=variant[0], tile_n=variant[1])
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


@pytest.mark.parametrize("majors", [(1, 1, 1), (0, 0, 1), (1, 0, 0)], ids=mid)
def test_majors_unfused_and_broadcasts(majors):
    """Row and column bias with an M-major aux tensor, fused and unfused,
    bf16 operands: identical bits and equal to the oracle."""
    ex = {x.name: x for x in W.page_examples(L=2, M=136, N=264, K=72)}
    w = ex["row_col_bias_f16"]
    inputs = W.make_inputs(w)
    fused = run_majors(w, inputs, majors)
    unf = run_majors(w, inputs, majors, unfused=True)
    _gpu.bitwise_equal(fused, unf)
    _gpu.compare(w, fused, _gpu.oracle_rows(w, inputs))
    w5 = dataclasses.replace(W.BIAS_RELU_SQUARE_L8, L=2, M=200, N=264, K=136, dist="randint",
                             sample_rows=None)
    inputs = W.make_inputs(w5)
    fused = run_majors(w5, inputs, majors, cta_group=2, tile_n=256)
    unf = run_majors(w5, inputs, majors, unfused=True, cta_group=2, tile_n=256)
    _gpu.bitwise_equal(fused, unf)
    _gpu.compare(w5, fused, _gpu.oracle_rows(w5, inputs))


def test_majors_normal_inputs_full_tiles():
    """N(0,1) inputs through the alpha-beta-x epilogue, column-major
    everything, several full 256x256 tiles: within the fp32 tolerance."""
    w = dataclasses.replace(W.ALPHA_BETA_X_8192, L=1, M=1024, N=768, K=512, sample_rows=None)
    inputs = W.make_inputs(w)
    gpu = run_majors(w, inputs, (1, 1, 1))
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


def test_majors_alignment_and_option_errors():
    w = BASE
    dt, dag = _gpu.dtypes_of(w), B.make_dag(w.dag)
    cases = [(dict(a_major=1), (1, 100, 128, 128), B.GE_ERR_MISALIGNED),   # M*2 bytes
             (dict(a_major=0), (1, 100, 128, 128), B.GE_OK),
             (dict(b_major=1), (1, 128, 128, 100), B.GE_ERR_MISALIGNED),   # K*2 bytes
             (dict(cd_major=1), (1, 100, 128, 128), B.GE_ERR_MISALIGNED),  # M*2 bytes (C, D)
             (dict(a_major=2), (1, 128, 128, 128), B.GE_ERR_INVALID)]
    for kw, (L, M, N, K), want in cases:
        try:
            plan = B.gemm_epi_plan_create(L, M, N, K, dt, dag, B.ge_options(**kw))
            B.gemm_epi_plan_destroy(plan)
            st = B.GE_OK
        except B.GemmEpiError as e:
            st = e.status
        assert st == want, (kw, st)


def test_grouped_with_majors():
    """A grouped launch with M-major A, K-major B and M-major epilogue
    tensors: each problem bit-exact against the oracle."""
    import test_gpu_grouped as G
    w = W.GROUPED_BY_NAME["grouped_bias_relu_ragged"]
    w = dataclasses.replace(w, problems=[p for p in w.problems if p[0] % 8 == 0])
    inputs = W.make_grouped_inputs(w)
    As, Bs, auxs, scalars = inputs
    Ad = [a.t().contiguous().to(DEV) for a in As]
    Bd = [b.t().contiguous().to(DEV) for b in Bs]
    auxd = [[x.t().contiguous().to(DEV) if x.dim() == 2 else x.to(DEV) for x in per]
            for per in auxs]
    outs = [[torch.full((n, m), float("nan"), dtype=W.TORCH_DTYPE[dt], device=DEV)
             for _, dt in w.outs] for m, n, k in w.problems]
    plan = B.gemm_epi_grouped_plan_create(
        w.problems, G.dtypes_of(w), B.make_dag(w.dag),
        B.ge_options(a_major=1, b_major=1, cd_major=1))
    try:
        B.gemm_epi_grouped_run(plan, Ad, Bd, auxd, scalars, outs)
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(plan) == B.GE_OK
    finally:
        B.gemm_epi_plan_destroy(plan)
    gpu = [[o.t().contiguous().cpu() for o in per] for per in outs]
    G.compare_grouped(w, gpu, G.oracle_grouped(w, inputs))
