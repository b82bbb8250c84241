"""The last-wave split: when the last wave of tiles would leave at least half
of the CTAs (pairs) idle, its tiles run as two half-width tiles each.  Every
output element's sum still runs over K in the same order, so the split and
unsplit schedules (GE_DEBUG_NO_TAIL_SPLIT) must agree bit for bit, and both
with the oracle."""
import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu

import _gpu  # noqa: E402
import test_gpu_majors as MJ  # noqa: E402
from _gpu import B, W  # noqa: E402

NO_SPLIT = B.GE_DEBUG_NO_TAIL_SPLIT
MYEPI = W.MY_EPILOGUE_128   # D = 0.5 * (acc + 2 C), Aux = acc + 2 C: integer inputs, exact
BRS = W.BIAS_RELU_SQUARE_L8   # bf16, D = relu(0.5 acc + C + bias), E = D * D: N(0,1) inputs


def both_schedules(w, unfused=False, **opt):
    """Outputs and plan info with the default (split) schedule and without it."""
    inputs = W.make_inputs(w)
    flags = opt.pop("debug_flags", 0)
    split, info_s = _gpu.run_gpu(w, inputs, options=B.ge_options(debug_flags=flags, **opt),
                                 unfused=unfused)
    plain, info_p = _gpu.run_gpu(w, inputs,
                                 options=B.ge_options(debug_flags=flags | NO_SPLIT, **opt),
                                 unfused=unfused)
    return inputs, split, plain, info_s, info_p


def check(w, unfused=False, expect_split=True, **opt):
    inputs, split, plain, info_s, info_p = both_schedules(w, unfused, **opt)
    if expect_split:
        # r tiles of the last wave became 2r half tiles
        assert info_s["num_tiles"] > info_p["num_tiles"], (info_s, info_p)
    _gpu.bitwise_equal(split, plain)
    _gpu.compare(w, split, _gpu.oracle_rows(w, inputs))
    return info_s, info_p


# (L, M, N, K, cta_group, tile_n): each leaves a last wave at most half full
# (76 CTA pairs or 152 single CTAs)
SHAPES = [
    (1, 2048, 1000, 256, 2, 256),   # 8 x 4 pair tiles, all split; the last n-block ragged
    (1, 2048, 896, 192, 2, 256),    # the last n-block's second half lies past N
    (1, 2560, 4608, 64, 2, 256),    # 180 pair tiles: two full waves, then 28 split
    (2, 1024, 2560, 64, 1, 256),    # 160 single-CTA tiles over two batches: 152, then 8 split
    (1, 640, 904, 320, 1, 128),     # 40 single-CTA 128 x 128 tiles, the last n-block ragged
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "L%d_%dx%dx%d_cg%d_n%d" % s)
def test_split_matches_unsplit_exact(shape):
    L, M, N, K, cg, bn = shape
    w = dataclasses.replace(MYEPI, L=L, M=M, N=N, K=K, sample_rows=None)
    info_s, _ = check(w, cta_group=cg, tile_n=bn)
    assert info_s["cta_group"] == cg and info_s["tile_n"] == bn


def test_split_bf16_broadcast_two_outputs():
    """Row-vector bias read at the half tile's own columns, two outputs."""
    w = dataclasses.replace(BRS, L=2, M=512, N=640, K=128, sample_rows=None)
    check(w, cta_group=2, tile_n=256)


def test_split_four_epilogue_warps_and_interpreter():
    w = dataclasses.replace(MYEPI, L=1, M=2048, N=1000, K=128, sample_rows=None)
    check(w, cta_group=2, tile_n=256, epi_warps=4)
    check(w, cta_group=2, tile_n=256, debug_flags=B.GE_DEBUG_FORCE_INTERPRETER)


def test_split_unfused_path():
    """The unfused path's fp32-accumulator GEMM uses the same schedule."""
    w = dataclasses.replace(MYEPI, L=1, M=2048, N=1000, K=192, sample_rows=None)
    check(w, unfused=True, cta_group=2, tile_n=256)


@pytest.mark.parametrize("majors", [(0, 1, 0), (1, 0, 0), (1, 1, 1)], ids=str)
def test_split_with_majors(majors):
    """K-major B (half tiles load whole boxes), M-major A, M-major epilogue."""
    w = dataclasses.replace(MYEPI, L=1, M=2048, N=1024, K=128, sample_rows=None)
    inputs = W.make_inputs(w)
    split = MJ.run_majors(w, inputs, majors, cta_group=2, tile_n=256)
    plain = MJ.run_majors(w, inputs, majors, cta_group=2, tile_n=256, debug_flags=NO_SPLIT)
    _gpu.bitwise_equal(split, plain)
    _gpu.compare(w, split, _gpu.oracle_rows(w, inputs))


def test_no_split_when_the_last_wave_is_more_than_half_full():
    """60 pair tiles (more than half of the 76 pairs) stay whole."""
    w = dataclasses.replace(MYEPI, L=1, M=2560, N=1536, K=64, sample_rows=None)  # 10 x 6
    _, _, _, info_s, info_p = both_schedules(w, cta_group=2, tile_n=256)
    assert info_s["num_tiles"] == info_p["num_tiles"] == 60


def test_split_runs_in_a_cuda_graph():
    w = dataclasses.replace(MYEPI, L=1, M=2048, N=1000, K=128, sample_rows=None)
    inputs = W.make_inputs(w)
    ref, _ = _gpu.run_gpu(w, inputs, options=B.ge_options(cta_group=2, tile_n=256))
    A, Bm, aux, scalars = inputs
    dev = torch.device("cuda", 0)
    Ad, Bd = A.to(dev), Bm.to(dev)
    auxd = [a.to(dev) for a in aux]
    outs = [torch.empty(w.L, w.M, w.N, dtype=W.TORCH_DTYPE[dt], device=dev) for _, dt in w.outs]
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag),
                                  B.ge_options(cta_group=2, tile_n=256))
    try:
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            B.gemm_epi_run(plan, Ad, Bd, auxd, scalars, outs, stream=s)
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(plan) == B.GE_OK
    finally:
        B.gemm_epi_plan_destroy(plan)
    _gpu.bitwise_equal([o.cpu() for o in outs], ref)
