"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, on the same seeded inputs."""
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import _gpu  # noqa: E402
from _gpu import B, W  # noqa: E402


def small(w, L, M, N, K, **kw):
    return dataclasses.replace(w, L=L, M=M, N=N, K=K, sample_rows=None, **kw)


# --------------------------------------------------- the five workloads --

@pytest.mark.parametrize("w", W.WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(w):
    """The three integer workloads on every element; the two N(0,1) ones
    (the full 8192^3 and L=8 sizes, in the launch configuration the
    benchmark times) on 64 seeded rows per batch, including each batch's
    first and last row."""
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs)
    rows = None if w.sample_rows is None else W.sample_rows(w)
    ref = _gpu.oracle_rows(w, inputs, rows)
    _gpu.compare(w, gpu, ref, rows)


def test_plan_choices_for_headline_sizes():
    w = W.BY_NAME["alpha_beta_x_8192"]
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag))
    try:
        info = B.gemm_epi_plan_info(plan)
    finally:
        B.gemm_epi_plan_destroy(plan)
    assert info["cta_group"] == 2 and info["tile_m"] == 256 and info["tile_n"] == 256
    assert info["stages"] >= 4 and info["grid"] % 2 == 0


# ------------------------------------------------------ page examples --

@pytest.mark.parametrize("w", W.page_examples(L=2, M=256, N=256, K=320), ids=lambda w: w.name)
def test_page_examples(w):
    inputs = W.make_inputs(w)
    gpu, _ = _gpu.run_gpu(w, inputs)
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


# ------------------------------------------------ shapes and variants --

SHAPES = [(1, 1, 8, 8), (1, 8, 8, 8), (1, 129, 136, 72), (3, 200, 264, 200),
          (2, 257, 520, 1000), (1, 300, 24, 64), (1, 64, 1032, 136), (2, 513, 392, 8)]
# (cta_group, tile N)
VARIANTS = [(1, 64), (1, 128), (1, 256), (2, 128), (2, 256)]


def opts(variant, **kw):
    return B.ge_options(cta_group=variant[0], tile_n=variant[1], **kw)


def vid(v):
    return "cg%d_n%d" % v


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("variant", VARIANTS, ids=vid)
def test_ragged_shapes_exact(shape, variant):
    """Integer inputs: every kernel variant must be bit-exact on ragged M, N,
    K (TMA zero-fills loads and clips stores at the edges)."""
    w = small(W.MY_EPILOGUE_128, *shape)
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=opts(variant))
    assert (info["cta_group"], info["tile_n"]) == variant
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


@pytest.mark.parametrize("variant", VARIANTS, ids=vid)
def test_bf16_bias_relu_square_variants(variant):
    w = small(W.BIAS_RELU_SQUARE_L8, 2, 384, 520, 264)
    inputs = W.make_inputs(w)
    gpu, _ = _gpu.run_gpu(w, inputs, options=opts(variant))
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_few_stages(stages):
    """Short rings wrap the stage/phase bookkeeping many times per tile."""
    w = small(W.ALPHA_BETA_X_8192, 1, 512, 1024, 1024)
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=B.ge_options(
        stages=stages, cta_group=2, tile_n=256))
    assert info["stages"] == stages
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


@pytest.mark.parametrize("stages", [6, 7])
def test_more_stages_than_default(stages):
    """A requested stage count above the default takes its room from the aux
    prefetch ring (128 x 64 tiles: 24 KiB a stage), bit-exact."""
    w = small(W.MY_EPILOGUE_128, 2, 520, 776, 1000)
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=B.ge_options(
        stages=stages, cta_group=1, tile_n=64))
    assert info["stages"] == stages and info["aux_stages"] >= 1
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=lambda v: "cg%d_n%d" % v)
def test_many_batches(variant):
    """L = 200 small problems in one batched launch: the batch coordinate of
    every TMA box and the (l, m, n) order of the persistent schedule,
    bit-exact against the oracle."""
    w = small(W.MY_EPILOGUE_128, 200, 136, 264, 72)
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=opts(variant))
    assert info["num_tiles"] >= 200
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


def test_wide_and_tall_extents():
    """One very wide (N = 65,544) and one very tall (M = 65,537) problem:
    column and row coordinates far past any tile count, ragged at the far
    edge, bit-exact against the oracle."""
    for (M, N, K) in ((130, 65544, 40), (65537, 136, 24)):
        w = small(W.MY_EPILOGUE_128, 1, M, N, K)
        inputs = W.make_inputs(w)
        gpu, _ = _gpu.run_gpu(w, inputs)
        _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


def test_small_grid_many_tiles_per_cta():
    """Four CTAs loop over many tiles: both TMEM accumulators, the aux
    prefetch across tile boundaries and the raster order all wrap."""
    w = small(W.ALPHA_BETA_X_8192, 2, 1024, 768, 256)
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=B.ge_options(
        max_ctas=4, raster_group=3, cta_group=2, tile_n=256))
    assert info["grid"] <= 4 and info["cluster_n"] == 1
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=lambda v: "cg%d_n%d" % v)
def test_k_snake_with_ragged_k(variant):
    """A few CTAs loop over many tiles, so half of their tiles walk K
    backwards and start on the partial last k-block (K = 200 and 1000 are
    not multiples of 64): bit-exact against the oracle, and the unfused
    path (same schedule) bit-identical."""
    cg, bn = variant
    for K in (200, 1000):
        w = small(W.MY_EPILOGUE_128, 2, 520, 776, K)
        inputs = W.make_inputs(w)
        opts = B.ge_options(max_ctas=2 * cg, cta_group=cg, tile_n=bn)
        gpu, info = _gpu.run_gpu(w, inputs, options=opts)
        assert info["num_tiles"] >= 4 * info["grid"] // cg
        _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))
        unf, _ = _gpu.run_gpu(w, inputs, options=opts, unfused=True)
        _gpu.bitwise_equal(gpu, unf)


def test_fused_and_unfused_share_the_k_order():
    """N(0,1) inputs, where the order of the sum over K shows in the last
    bits, and many tiles per CTA, half of them walking K backwards: the
    unfused path's GEMM must use the same schedule, bit for bit."""
    w = small(W.ALPHA_BETA_X_8192, 1, 1040, 776, 1000)
    inputs = W.make_inputs(w)
    opts = B.ge_options(max_ctas=4, cta_group=2, tile_n=256)
    fused, info = _gpu.run_gpu(w, inputs, options=opts)
    assert info["num_tiles"] >= 4 * info["grid"] // 2
    unf, _ = _gpu.run_gpu(w, inputs, options=opts, unfused=True)
    _gpu.bitwise_equal(fused, unf)
    _gpu.compare(w, fused, _gpu.oracle_rows(w, inputs))


# ------------------------------------------------------------ unfused --

@pytest.mark.parametrize("w", [W.MY_EPILOGUE_1024, small(W.BIAS_RELU_SQUARE_L8, 2, 256, 392, 520),
                               small(W.ALPHA_BETA_X_8192, 1, 300, 264, 200)], ids=lambda w: w.name)
def test_unfused_matches_fused_bitwise(w):
    """Same compiled program on the same fp32 accumulator: identical bits."""
    inputs = W.make_inputs(w)
    fused, _ = _gpu.run_gpu(w, inputs)
    unfused, _ = _gpu.run_gpu(w, inputs, unfused=True)
    _gpu.bitwise_equal(fused, unfused)
    _gpu.compare(w, unfused, _gpu.oracle_rows(w, inputs))


def test_variants_agree_on_normal_inputs():
    w = small(W.ALPHA_BETA_X_8192, 1, 512, 512, 2048)
    inputs = W.make_inputs(w)
    base, _ = _gpu.run_gpu(w, inputs, options=opts(VARIANTS[4]))
    for v in VARIANTS[:4]:
        other, _ = _gpu.run_gpu(w, inputs, options=opts(v))
        for a, b in zip(base, other):
            assert torch.allclose(a.float(), b.float(), rtol=1e-3, atol=1e-2)


def test_repeated_runs_and_side_stream():
    w = small(W.MY_EPILOGUE_128, 1, 384, 256, 512)
    inputs = W.make_inputs(w)
    s = torch.cuda.Stream()
    gpu, _ = _gpu.run_gpu(w, inputs, stream=s, repeat=3)
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


# ------------------------------------------------------ error behaviour --

def test_run_argument_errors():
    w = small(W.MY_EPILOGUE_128, 1, 128, 128, 128)
    A, Bm, aux, sc = [x for x in W.make_inputs(w)]
    dev = torch.device("cuda")
    Ad, Bd, Cd = A.cuda(), Bm.cuda(), aux[0].cuda()
    D = torch.empty(1, 128, 128, dtype=torch.float16, device=dev)
    X = torch.empty(1, 128, 128, dtype=torch.float16, device=dev)
    plan = B.gemm_epi_plan_create(1, 128, 128, 128, _gpu.dtypes_of(w), B.make_dag(w.dag))
    try:
        assert B.gemm_epi_run(plan, Ad, Bd, [Cd], sc, [D, None], check=False) == \
            B.GE_ERR_MISSING_ARG
        assert B.gemm_epi_run(plan, Ad, Bd, [None], sc, [D, X], check=False) == \
            B.GE_ERR_MISSING_ARG
        mis = Ad.data_ptr() + 2
        assert B.gemm_epi_run(plan, mis, Bd, [Cd], sc, [D, X], check=False) == \
            B.GE_ERR_MISALIGNED
        ws = torch.empty(16, dtype=torch.float32, device=dev)
        assert B.gemm_epi_run_unfused(plan, Ad, Bd, [Cd], sc, [D, X], ws, check=False) == \
            B.GE_ERR_WORKSPACE
        # nothing was launched by the rejected calls; a good call still works
        assert B.gemm_epi_run(plan, Ad, Bd, [Cd], sc, [D, X]) == B.GE_OK
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(plan) == B.GE_OK
    finally:
        B.gemm_epi_plan_destroy(plan)


def test_device_wait_timeout_is_reported():
    """A k-block that is never loaded: the MMA warp's bounded wait runs out,
    the kernel records GE_ERR_TIMEOUT, drains and exits; the context stays
    usable and the next run is correct."""
    w = small(W.MY_EPILOGUE_128, 1, 256, 256, 256)
    inputs = W.make_inputs(w)
    opt = B.ge_options(timeout_ms=50, debug_flags=B.GE_DEBUG_SKIP_FIRST_LOAD,
                       max_ctas=2, cta_group=2, tile_n=256)
    A, Bm, aux, sc = inputs
    dev = torch.device("cuda")
    outs = [torch.empty(1, 256, 256, dtype=torch.float16, device=dev) for _ in range(2)]
    plan = B.gemm_epi_plan_create(1, 256, 256, 256, _gpu.dtypes_of(w), B.make_dag(w.dag), opt)
    try:
        assert B.gemm_epi_run(plan, A.cuda(), Bm.cuda(), [aux[0].cuda()], sc, outs) == B.GE_OK
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(plan) == B.GE_ERR_TIMEOUT
        assert B.gemm_epi_last_error(plan) == B.GE_OK  # read-and-clear
    finally:
        B.gemm_epi_plan_destroy(plan)
    gpu, _ = _gpu.run_gpu(w, inputs)
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


# ------------------------------------------ catalog vs interpreter --

def test_headline_workloads_use_builtin_epilogues():
    for w in W.WORKLOADS:
        plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag))
        try:
            info = B.gemm_epi_plan_info(plan)
        finally:
            B.gemm_epi_plan_destroy(plan)
        assert info["epi_variant"] >= 0, w.name


CATALOG_CASES = [small(W.MY_EPILOGUE_128, 2, 300, 392, 200), small(W.RELU_2400X3232X4096, 1, 264, 520, 136),
                 small(W.ALPHA_BETA_X_8192, 1, 384, 264, 520), small(W.BIAS_RELU_SQUARE_L8, 3, 200, 264, 200)] + \
    [small(w, 2, 136, 264, 72) for w in W.page_examples()]


@pytest.mark.parametrize("w", CATALOG_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("variant", [(1, 64), (2, 256)], ids=vid)
def test_builtin_and_interpreter_agree_bitwise(w, variant):
    """The straight-line kernels and the interpreter evaluate the same
    compiled program in the same order: identical bits, fused and unfused."""
    inputs = W.make_inputs(w)
    base = dict(cta_group=variant[0], tile_n=variant[1])
    fast, info = _gpu.run_gpu(w, inputs, options=B.ge_options(**base))
    slow, info2 = _gpu.run_gpu(w, inputs, options=B.ge_options(
        debug_flags=B.GE_DEBUG_FORCE_INTERPRETER, **base))
    assert info2["epi_variant"] == -1
    _gpu.bitwise_equal(fast, slow)
    slow_unfused, _ = _gpu.run_gpu(w, inputs, unfused=True, options=B.ge_options(
        debug_flags=B.GE_DEBUG_FORCE_INTERPRETER, **base))
    _gpu.bitwise_equal(fast, slow_unfused)
    _gpu.compare(w, fast, _gpu.oracle_rows(w, inputs))


# ------------------------------------------------- wider node set --

def _reverse_ops_workload():
    """Exercises the two-address compiler's reversed forms: C - alpha*accum
    and C / (beta*X) reuse the register of their second operand."""
    g = W.Dag()
    acc = g.accum()
    t = g.mul(acc, g.scalar(0))
    c = g.load(0)
    u = g.sub(c, t)
    v = g.mul(g.load(1), g.scalar(1))
    w_ = g.div(c, v)
    g.store(g.minimum(u, w_), 0)
    g.store(u, 1)
    return W.Workload(name="reverse_ops", L=2, M=264, N=392, K=200, ab="f16",
                      aux=[("C", "tensor", "f16"), ("X", "tensor", "f16", "pow2")],
                      scalars=[("alpha", 1.0), ("beta", 2.0)],
                      outs=[("D", "f16"), ("U", "f16")], dag=g.nodes, dist="randint", seed=31,
                      exact=True)


@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=vid)
def test_reversed_sub_div_and_min(variant):
    w = _reverse_ops_workload()
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=opts(variant))
    assert info["epi_variant"] < 0  # not a built-in epilogue
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))
    unf, _ = _gpu.run_gpu(w, inputs, unfused=True, options=opts(variant))
    _gpu.bitwise_equal(gpu, unf)


def test_row_col_bias_uses_catalog():
    w = [x for x in W.page_examples(L=2, M=300, N=264, K=136) if x.name == "row_col_bias_f16"][0]
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs)
    assert info["epi_variant"] >= 0
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


# ------------------------------------------------------- activations --

ACT_CASES = [x for x in W.page_examples(L=2, M=264, N=392, K=200)
             if x.name.startswith("act_") or x.name.startswith("complex_")]


def _ulp(v, dt):
    """Spacing of the output type at magnitude v."""
    p, emin = {"f16": (11, -14), "bf16": (8, -126), "f32": (24, -126)}[dt]
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (e - (p - 1))


@pytest.mark.parametrize("w", ACT_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=vid)
def test_activations_within_one_ulp(w, variant):
    """The fp32 activations (CUDA math library) against the fp64 oracle.
    The activation's argument differs between the two sides by at most the
    fp32 summation bound K * 2^-24 * sum_k |a_ik b_kj| (times the scalar
    applied to accum) plus a few fp32 roundings of its own size, and the
    math library adds a few fp32 ulps; with every activation's slope at most
    1.5, each output then lies within one unit in the last place of its type,
    plus 1.5 times that bound, plus 32 fp32 ulps of the oracle's, and nearly
    all are identical."""
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=opts(variant))
    ref = _gpu.oracle_rows(w, inputs)
    A, Bm = inputs[0].double().numpy(), inputs[1].double().numpy()
    S = np.einsum("lik,lkj->lij", np.abs(A), np.abs(Bm)).reshape(w.L * w.M, w.N)
    u = 2.0 ** -24
    arg_err = abs(w.scalars[0][1]) * w.K * u * S
    for (name, dt), g, r in zip(w.outs, gpu, ref):
        gv = _gpu.decode(W.to_codes(g).reshape(w.L * w.M, w.N), dt)
        rv = _gpu.decode(r, dt)
        assert not np.isnan(gv).any()
        lim = (_ulp(np.maximum(np.abs(gv), np.abs(rv)), dt) + 1.5 * arg_err +
               32 * u * (1 + np.abs(rv)))
        err = np.abs(gv - rv)
        assert (err <= lim).all(), (name, float((err - lim).max()), gv[err > lim][:4],
                                    rv[err > lim][:4])
        assert (gv == rv).mean() > 0.97, (name, float((gv == rv).mean()))


def test_activation_special_inputs():
    """Large-magnitude and zero arguments: sigmoid saturates to 0 and 1,
    tanh to -1 and 1, gelu and silu to 0 and x, hardswish to 0 and x,
    without NaN (K = 8, accum = 64 * a row of A)."""
    import torch
    for act in W.ACTIVATIONS:
        w = [x for x in W.page_examples(L=1, M=128, N=64, K=8) if x.name == "act_" + act][0]
        w = dataclasses.replace(w, outs=[("D", "f32")])
        A = torch.zeros(1, 128, 8, dtype=torch.float16)
        A[0, :, 0] = torch.linspace(-60, 60, 128).to(torch.float16)
        Bm = torch.zeros(1, 8, 64, dtype=torch.float16)
        Bm[0, 0, :] = 64.0
        C = torch.zeros(1, 128, 64, dtype=torch.float16)
        inputs = (A, Bm, [C], [0.25] + ([0.1] if act == "leaky_relu" else []))
        gpu, _ = _gpu.run_gpu(w, inputs)
        ref = _gpu.oracle_rows(w, inputs)
        gv = _gpu.decode(W.to_codes(gpu[0]).reshape(128, 64), "f32")
        rv = _gpu.decode(ref[0], "f32")
        assert not np.isnan(gv).any(), act
        assert np.allclose(gv, rv, rtol=4e-6, atol=1e-30), (act, np.abs(gv - rv).max())


def _leaky_workloads():
    """Leaky ReLU with the slope in a register that dies while the value
    lives on (the reversed form), and PReLU with a per-column slope vector;
    integer inputs and half-integer slopes keep both bit-exact."""
    g = W.Dag()
    t = g.mul(g.accum(), g.scalar(0))
    s = g.mul(g.load(0), g.scalar(1))
    g.store(g.leaky_relu(t, s), 0)
    g.store(t, 1)
    rev = W.Workload(name="leaky_reversed", L=2, M=264, N=392, K=200, ab="f16",
                     aux=[("C", "tensor", "f16")], scalars=[("alpha", 1.0), ("half", 0.5)],
                     outs=[("D", "f16"), ("T", "f16")], dag=g.nodes, dist="randint", seed=32,
                     exact=True)
    g = W.Dag()
    g.store(g.leaky_relu(g.accum(), g.broadcast(0)), 0)
    prelu = W.Workload(name="prelu_row_slope", L=2, M=200, N=264, K=136, ab="bf16",
                       aux=[("slope", "row", "f32")], scalars=[], outs=[("D", "bf16")],
                       dag=g.nodes, dist="randint", seed=33, exact=True)
    return [rev, prelu]


@pytest.mark.parametrize("w", _leaky_workloads(), ids=lambda w: w.name)
@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=vid)
def test_leaky_relu_forms(w, variant):
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=opts(variant))
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))
    unf, _ = _gpu.run_gpu(w, inputs, unfused=True, options=opts(variant))
    _gpu.bitwise_equal(gpu, unf)


# ------------------------------------------------ eight epilogue warps --

@pytest.mark.parametrize("w", CATALOG_CASES[:4] + [small(W.BIAS_RELU_SQUARE_L8, 2, 264, 520, 136)] +
                         [x for x in CATALOG_CASES if x.name in ("complex_gelu_tanh",
                                                                  "row_col_bias_f16")],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("variant", [(1, 64), (1, 256), (2, 128), (2, 256)], ids=vid)
def test_eight_epilogue_warps_bitwise(w, variant):
    """Two warps per accumulator lane quarter, each taking every other
    32-column step: the same bits as four warps, and the oracle's values."""
    inputs = W.make_inputs(w)
    base = dict(cta_group=variant[0], tile_n=variant[1])
    four, i4 = _gpu.run_gpu(w, inputs, options=B.ge_options(epi_warps=4, **base))
    eight, i8 = _gpu.run_gpu(w, inputs, options=B.ge_options(epi_warps=8, **base))
    assert i8["epi_variant"] >= 0
    _gpu.bitwise_equal(four, eight)
    _gpu.compare(w, eight, _gpu.oracle_rows(w, inputs))


def test_eight_epilogue_warps_rules():
    w = small(W.MY_EPILOGUE_128, 1, 256, 256, 256)
    dt, dag = _gpu.dtypes_of(w), B.make_dag(w.dag)
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_plan_create(1, 256, 256, 256, dt, dag, B.ge_options(epi_warps=6))
    assert e.value.status == B.GE_ERR_INVALID


@pytest.mark.parametrize("w", [small(W.BIAS_RELU_SQUARE_L8, 2, 264, 520, 136)] +
                         [x for x in CATALOG_CASES if x.name in ("act_sigmoid", "clamp_f16",
                                                                  "aux_normalize_f16")],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("variant", [(1, 128), (2, 256)], ids=vid)
def test_interpreter_eight_warps_bitwise(w, variant):
    """The interpreter on 8 warps: the same bits as on 4 and as the
    built-in kernels."""
    inputs = W.make_inputs(w)
    base = dict(cta_group=variant[0], tile_n=variant[1],
                debug_flags=B.GE_DEBUG_FORCE_INTERPRETER)
    four, i4 = _gpu.run_gpu(w, inputs, options=B.ge_options(epi_warps=4, **base))
    eight, i8 = _gpu.run_gpu(w, inputs, options=B.ge_options(epi_warps=8, **base))
    assert i4["epi_variant"] == -1 and i8["epi_warps"] == 8
    _gpu.bitwise_equal(four, eight)
    _gpu.compare(w, eight, _gpu.oracle_rows(w, inputs))


def test_eight_epilogue_warps_timeout_is_reported():
    w = small(W.MY_EPILOGUE_128, 1, 256, 256, 256)
    inputs = W.make_inputs(w)
    A, Bm, aux, sc = inputs
    opt = B.ge_options(timeout_ms=50, debug_flags=B.GE_DEBUG_SKIP_FIRST_LOAD, max_ctas=2,
                       cta_group=2, tile_n=256, epi_warps=8)
    outs = [torch.empty(1, 256, 256, dtype=torch.float16, device="cuda") for _ in range(2)]
    plan = B.gemm_epi_plan_create(1, 256, 256, 256, _gpu.dtypes_of(w), B.make_dag(w.dag), opt)
    try:
        assert B.gemm_epi_run(plan, A.cuda(), Bm.cuda(), [aux[0].cuda()], sc, outs) == B.GE_OK
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(plan) == B.GE_ERR_TIMEOUT
    finally:
        B.gemm_epi_plan_destroy(plan)
    gpu, _ = _gpu.run_gpu(w, inputs, options=B.ge_options(epi_warps=8))
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))


def test_program_with_more_than_four_registers():
    """Five values live at once: the interpreter variant with 8 program
    registers (plan epi_variant -2, 4 epilogue warps), fused and unfused,
    bit-exact on integer inputs."""
    g = W.Dag()
    acc = g.accum()
    sc = g.scalar(0)
    vals = [g.mul(acc, sc)] + [g.mul(g.load(i), sc) for i in range(4)]
    s = vals[0]
    for v in vals[1:]:
        s = g.add(s, v)
    g.store(s, 0)
    w = W.Workload(name="five_live", L=2, M=200, N=264, K=136, ab="f16",
                   aux=[("C%d" % i, "tensor", "f16") for i in range(4)], scalars=[("s", 2.0)],
                   outs=[("D", "f16")], dag=g.nodes, dist="randint", seed=37, exact=True)
    inputs = W.make_inputs(w)
    gpu, info = _gpu.run_gpu(w, inputs, options=B.ge_options(specialize=-1))
    assert info["epi_variant"] == -2 and info["epi_warps"] == 4 and info["n_regs"] == 5
    _gpu.compare(w, gpu, _gpu.oracle_rows(w, inputs))
    unf, _ = _gpu.run_gpu(w, inputs, unfused=True)
    _gpu.bitwise_equal(gpu, unf)
    with pytest.raises(B.GemmEpiError) as e:
        B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag),
                               B.ge_options(epi_warps=8, specialize=-1))
    assert e.value.status == B.GE_ERR_UNSUPPORTED
    # compiled for this program: all 8 registers in straight-line code, 8 warps
    spec, info = _gpu.run_gpu(w, inputs)
    assert info["epi_variant"] == -3 and info["epi_warps"] == 8
    _gpu.bitwise_equal(gpu, spec)


def test_run_captured_in_cuda_graph():
    """gemm_epi_run only launches once its tensor maps are encoded (first
    run), so it can be captured into a CUDA graph and replayed; replays give
    the plain run's bits, including after the inputs change in place."""
    w = small(W.BIAS_RELU_SQUARE_L8, 2, 264, 520, 136)
    inputs = W.make_inputs(w)
    A, Bm, aux, sc = inputs
    dev = torch.device("cuda")
    Ad, Bd, auxd = A.to(dev), Bm.to(dev), [a.to(dev) for a in aux]
    outs = [torch.empty(w.L, w.M, w.N, dtype=W.TORCH_DTYPE[dt], device=dev) for _, dt in w.outs]
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag))
    s = torch.cuda.Stream()
    try:
        B.gemm_epi_run(plan, Ad, Bd, auxd, sc, outs, stream=s)
        torch.cuda.synchronize()
        plain = [o.clone() for o in outs]
        call = B.prepare_run(plan, Ad, Bd, auxd, sc, outs, stream=s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            assert call() == B.GE_OK
        for o in outs:
            o.zero_()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        _gpu.bitwise_equal([o.cpu() for o in outs], [p.cpu() for p in plain])
        # new values in the same buffers: the replay reads them
        Ad.neg_()
        graph.replay()
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(plan) == B.GE_OK
        neg = (W.make_inputs(w)[0].neg(), Bm, aux, sc)
        _gpu.compare(w, [o.cpu() for o in outs], _gpu.oracle_rows(w, neg))
    finally:
        B.gemm_epi_plan_destroy(plan)


def test_epilogue_warps_default_and_option():
    """Compiled epilogues and the 4-register interpreter take 8 warps at any
    K; the option overrides."""
    def warps(w, **opt):
        plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, _gpu.dtypes_of(w), B.make_dag(w.dag),
                                      B.ge_options(**opt) if opt else None)
        try:
            return B.gemm_epi_plan_info(plan)["epi_warps"]
        finally:
            B.gemm_epi_plan_destroy(plan)
    ab, brs = W.ALPHA_BETA_X_8192, W.BIAS_RELU_SQUARE_L8
    assert warps(ab) == 8                                     # K = 8192: 128 k-blocks a tile
    assert warps(dataclasses.replace(ab, K=1024)) == 8        # 16 k-blocks a tile
    assert warps(brs) == 8                                    # K = 2048, three epilogue tensors
    assert warps(ab, epi_warps=4) == 4
    assert warps(ab, debug_flags=B.GE_DEBUG_FORCE_INTERPRETER) == 8


@pytest.mark.parametrize("no_pdl", [0, 1])
def test_back_to_back_runs_read_and_write_each_others_buffers(no_pdl):
    """Batched runs are launched with programmatic stream serialization: a
    run's set-up may overlap the previous kernel's tail, but its reads of
    inputs and writes of outputs wait for that kernel.  Run 1 (Aux/D of
    my_epilogue, a few CTAs) writes D1; run 2 reads D1 as its A (read after
    write) and stores its fp32 product over the memory run 1 read its A
    from (write after read).  Twenty pairs in a row on one stream, then
    both results against the oracle, with the overlap and without it."""
    w1 = small(W.MY_EPILOGUE_128, 1, 256, 256, 136)
    A1, B1, aux1, sc1 = W.make_inputs(w1)
    w2 = [x for x in W.page_examples(L=1, M=256, N=136, K=256) if x.name == "identity_f32_out"][0]
    _, B2, _, _ = W.make_inputs(w2)
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    nbytes = max(A1.numel() * 2, w2.M * w2.N * 4)
    X = torch.empty(nbytes // 2, dtype=torch.int16, device=dev)
    A1d = X[:A1.numel()].view(torch.float16).view(A1.shape)
    out2 = X.view(torch.float32)[:w2.M * w2.N].view(1, w2.M, w2.N)
    B1d, C1d, B2d = B1.to(dev), aux1[0].to(dev), B2.to(dev)
    D1 = torch.empty(1, 256, 256, dtype=torch.float16, device=dev)
    Aux1 = torch.empty_like(D1)
    opt = B.ge_options(no_pdl=no_pdl)
    p1 = B.gemm_epi_plan_create(1, 256, 256, 136, _gpu.dtypes_of(w1), B.make_dag(w1.dag), opt)
    p2 = B.gemm_epi_plan_create(1, 256, 136, 256, _gpu.dtypes_of(w2), B.make_dag(w2.dag), opt)
    try:
        for _ in range(20):
            with torch.cuda.stream(s):
                A1d.copy_(A1.to(dev))  # run 2 of the previous pair overwrote it
            B.gemm_epi_run(p1, A1d, B1d, [C1d], sc1, [D1, Aux1], stream=s)
            B.gemm_epi_run(p2, D1, B2d, [], [], [out2], stream=s)
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(None) == B.GE_OK
        d1, aux1_out, o2 = D1.cpu(), Aux1.cpu(), out2.cpu().clone()
    finally:
        B.gemm_epi_plan_destroy(p1)
        B.gemm_epi_plan_destroy(p2)
    _gpu.compare(w1, [d1, aux1_out], _gpu.oracle_rows(w1, (A1, B1, aux1, sc1)))
    _gpu.compare(w2, [o2], _gpu.oracle_rows(w2, (d1, B2, [], [])))
