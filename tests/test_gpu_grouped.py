"""GPU parity of the grouped GEMM (one launch over problems of different
sizes) against the oracle, problem by problem, through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import _gpu  # noqa: E402
import oracle  # noqa: E402
from _gpu import B, W  # noqa: E402

DEV = torch.device("cuda", 0)


def dtypes_of(w):
    return B.make_dtypes(w.ab, [s[2] for s in w.aux], len(w.scalars), [dt for _, dt in w.outs])


class Grouped:
    """Device buffers (outputs inside sentinel guard bands) and a plan for a
    grouped workload."""

    def __init__(self, w, inputs, options=None):
        self.w = w
        As, Bs, auxs, self.scalars = inputs
        self.As = [a.to(DEV) for a in As]
        self.Bs = [b.to(DEV) for b in Bs]
        self.auxs = [[x.to(DEV) for x in per] for per in auxs]
        self.bufs, self.outs = [], []
        for m, n, k in w.problems:
            wg = W.Workload(name="g", L=1, M=m, N=n, K=k, ab=w.ab, aux=w.aux, scalars=w.scalars,
                            outs=w.outs, dag=w.dag, dist=w.dist, seed=0, exact=w.exact)
            per_b, per_o = [], []
            for _, dt in w.outs:
                buf, view = _gpu.alloc_out(wg, dt, DEV)
                per_b.append(buf)
                per_o.append(view)
            self.bufs.append(per_b)
            self.outs.append(per_o)
        self.plan = B.gemm_epi_grouped_plan_create(w.problems, dtypes_of(w), B.make_dag(w.dag),
                                                   options)
        self.info = B.gemm_epi_plan_info(self.plan)

    def run(self, stream=None, outs=None):
        B.gemm_epi_grouped_run(self.plan, self.As, self.Bs, self.auxs, self.scalars,
                               outs or self.outs, stream=stream)

    def finish(self):
        torch.cuda.synchronize()
        st = B.gemm_epi_last_error(self.plan)
        assert st == B.GE_OK, B.gemm_epi_status_string(st)
        for per_b in self.bufs:
            for buf, (_, dt) in zip(per_b, self.w.outs):
                _gpu.check_guards(buf, dt)
        return [[o.cpu() for o in per] for per in self.outs]

    def close(self):
        B.gemm_epi_plan_destroy(self.plan)


def oracle_grouped(w, inputs):
    As, Bs, auxs, scalars = inputs
    return oracle.grouped_gemm_epilogue(
        w.problems, w.ab, [W.to_codes(a) for a in As], [W.to_codes(b) for b in Bs],
        [[W.to_codes(x) for x in per] for per in auxs], [s[2] for s in w.aux], scalars, w.dag,
        [dt for _, dt in w.outs], threads=oracle.threads_default())


def compare_grouped(w, gpu, ref):
    for g, (m, n, k) in enumerate(w.problems):
        wg = W.Workload(name="%s[%d]" % (w.name, g), L=1, M=m, N=n, K=k, ab=w.ab, aux=w.aux,
                        scalars=w.scalars, outs=w.outs, dag=w.dag, dist=w.dist, seed=0,
                        exact=w.exact)
        _gpu.compare(wg, gpu[g], ref[g])


def run_and_check(w, options=None):
    inputs = W.make_grouped_inputs(w)
    G = Grouped(w, inputs, options)
    try:
        G.run()
        gpu = G.finish()
    finally:
        G.close()
    compare_grouped(w, gpu, oracle_grouped(w, inputs))
    return G.info


@pytest.mark.parametrize("w", W.grouped_workloads(), ids=lambda w: w.name)
def test_grouped_parity(w):
    """The grouped-GEMM notebook's 50 problems and a custom epilogue over
    ragged problems: bit-exact (integer inputs) against the oracle."""
    info = run_and_check(w)
    assert info["num_tiles"] > 0 and info["grid"] > 0


VARIANTS = [(1, 64), (1, 128), (1, 256), (2, 128), (2, 256)]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "cg%d_n%d" % v)
def test_grouped_tile_variants(variant):
    w = W.GROUPED_BY_NAME["grouped_bias_relu_ragged"]
    info = run_and_check(w, B.ge_options(cta_group=variant[0], tile_n=variant[1]))
    assert (info["cta_group"], info["tile_n"]) == variant


def test_grouped_interpreter_matches_builtin():
    w = W.GROUPED_BY_NAME["grouped_gemm_50"]
    w = dataclasses.replace(w, problems=w.problems[:12], scalars=[("alpha", 1.0), ("beta", 2.0)])
    inputs = W.make_grouped_inputs(w)
    fast = Grouped(w, inputs)
    slow = Grouped(w, inputs, B.ge_options(debug_flags=B.GE_DEBUG_FORCE_INTERPRETER))
    try:
        assert fast.info["epi_variant"] >= 0 and slow.info["epi_variant"] == -1
        fast.run()
        slow.run()
        a, b = fast.finish(), slow.finish()
    finally:
        fast.close()
        slow.close()
    for pa, pb in zip(a, b):
        _gpu.bitwise_equal(pa, pb)
    compare_grouped(w, a, oracle_grouped(w, inputs))


def test_grouped_normal_inputs_and_activation():
    """N(0,1) bf16 inputs through GELU: within the fp32 tolerance."""
    g = W.Dag()
    g.store(g.gelu(g.add(g.mul(g.accum(), g.scalar(0)), g.load(0))), 0)
    w = W.GroupedWorkload(name="grouped_gelu", problems=[(256, 512, 1024), (100, 136, 520),
                                                         (1024, 256, 64), (8, 8, 2048)],
                          ab="bf16", aux=[("C", "tensor", "bf16")], scalars=[("alpha", 0.125)],
                          outs=[("D", "bf16")], dag=g.nodes, dist="normal", seed=41, exact=False)
    run_and_check(w)


def test_grouped_table_reuse_and_rotation():
    """Same pointers: the table is reused; new output buffers on every run
    rotate through the four tables (the fifth run waits for the first) and
    every run's outputs are complete and identical."""
    w = W.GROUPED_BY_NAME["grouped_bias_relu_ragged"]
    inputs = W.make_grouped_inputs(w)
    G = Grouped(w, inputs)
    try:
        for _ in range(3):
            G.run()
        first = G.finish()
        extra = []
        for r in range(6):
            outs = [[torch.full_like(o, float("nan")) for o in per] for per in G.outs]
            G.run(outs=outs)
            extra.append(outs)
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(G.plan) == B.GE_OK
    finally:
        G.close()
    for outs in extra:
        for pa, pb in zip(first, outs):
            _gpu.bitwise_equal(pa, [o.cpu() for o in pb])
    compare_grouped(w, first, oracle_grouped(w, inputs))


def test_grouped_across_streams():
    """A table built on one stream and reused on another: the second run is
    ordered after the first and both are correct."""
    w = W.GROUPED_BY_NAME["grouped_gemm_50"]
    w = dataclasses.replace(w, problems=w.problems[:20])
    inputs = W.make_grouped_inputs(w)
    G = Grouped(w, inputs)
    s1, s2 = torch.cuda.Stream(device=DEV), torch.cuda.Stream(device=DEV)
    try:
        G.run(stream=s1)
        G.run(stream=s2)
        gpu = G.finish()
    finally:
        G.close()
    compare_grouped(w, gpu, oracle_grouped(w, inputs))


def test_grouped_argument_errors():
    w = W.GROUPED_BY_NAME["grouped_gemm_50"]
    w = dataclasses.replace(w, problems=w.problems[:3])
    inputs = W.make_grouped_inputs(w)
    G = Grouped(w, inputs)
    try:
        st = B.gemm_epi_grouped_run(G.plan, G.As[:2] + [None], G.Bs, G.auxs, G.scalars, G.outs,
                                    check=False)
        assert st == B.GE_ERR_MISSING_ARG
        bad = [[G.outs[0][0].view(-1)[1:]]] + G.outs[1:]
        st = B.gemm_epi_grouped_run(G.plan, G.As, G.Bs, G.auxs, G.scalars, bad, check=False)
        assert st == B.GE_ERR_MISALIGNED
        # a grouped plan is not a batched plan and vice versa
        assert B.gemm_epi_run(G.plan, G.As[0], G.Bs[0], G.auxs[0], G.scalars, G.outs[0],
                              check=False) == B.GE_ERR_INVALID
        assert B.gemm_epi_unfused_workspace_bytes(G.plan) == 0
    finally:
        G.close()
    wb = W.MY_EPILOGUE_128
    plan = B.gemm_epi_plan_create(wb.L, wb.M, wb.N, wb.K, _gpu.dtypes_of(wb), B.make_dag(wb.dag))
    try:
        st = B.gemm_epi_grouped_run(plan, G.As, G.Bs, G.auxs, G.scalars, G.outs, check=False)
        assert st == B.GE_ERR_INVALID
    finally:
        B.gemm_epi_plan_destroy(plan)


def test_grouped_device_wait_timeout_is_reported():
    """The skip-first-load test hook in a grouped launch: the bounded wait
    expires, the status reads GE_ERR_TIMEOUT, and the next run is correct."""
    w = W.GROUPED_BY_NAME["grouped_bias_relu_ragged"]
    inputs = W.make_grouped_inputs(w)
    G = Grouped(w, inputs, B.ge_options(debug_flags=B.GE_DEBUG_SKIP_FIRST_LOAD, timeout_ms=50))
    try:
        G.run()
        torch.cuda.synchronize()
        assert B.gemm_epi_last_error(G.plan) == B.GE_ERR_TIMEOUT
    finally:
        G.close()
    run_and_check(w)


def test_grouped_eight_epilogue_warps():
    """A built-in epilogue (alpha*accum + beta*C) with two warps per lane
    quarter over problems of every size."""
    w = W.GROUPED_BY_NAME["grouped_gemm_50"]
    w = dataclasses.replace(w, scalars=[("alpha", 1.0), ("beta", 2.0)])
    for cg, bn in [(1, 128), (2, 256), (1, 64)]:
        info = run_and_check(w, B.ge_options(epi_warps=8, cta_group=cg, tile_n=bn))
        assert (info["cta_group"], info["tile_n"]) == (cg, bn) and info["epi_variant"] >= 0


def test_grouped_reused_table_waits_for_the_previous_kernel():
    """A run that reuses its problem table may overlap the previous kernel on
    the stream (programmatic dependent launch) but must read its inputs only
    after that kernel: each run follows an in-place negation of every A
    (stream-ordered), five times; the result matches the oracle on the
    final inputs."""
    w = W.GROUPED_BY_NAME["grouped_bias_relu_ragged"]
    inputs = W.make_grouped_inputs(w)
    G = Grouped(w, inputs)
    s = torch.cuda.Stream(device=DEV)
    try:
        G.run(stream=s)  # builds the table
        for _ in range(5):
            with torch.cuda.stream(s):
                for a in G.As:
                    a.neg_()
            G.run(stream=s)
        gpu = G.finish()
    finally:
        G.close()
    As, Bs, auxs, sc = inputs
    compare_grouped(w, gpu, oracle_grouped(w, ([a.neg() for a in As], Bs, auxs, sc)))
