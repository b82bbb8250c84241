"""Helpers for the GPU parity tests: run a workload through the C ABI and
compare with the oracle on the same seeded inputs."""
import numpy as np
import torch

import _pins
import oracle
from dense_gemm_elementwise_gb300 import build as gbuild

gbuild.build()
from dense_gemm_elementwise_gb300 import binding as B  # noqa: E402
from dense_gemm_elementwise_gb300 import workloads as W  # noqa: E402

GUARD = 128  # guard elements before and after every output (sentinel-filled)
SENTINEL16 = 0x7E5A  # a NaN pattern no store produces from finite inputs
SENTINEL32 = 0x7FC05A5A


def dtypes_of(w):
    return B.make_dtypes(w.ab, [s[2] for s in w.aux], len(w.scalars),
                         [dt for _, dt in w.outs])


def alloc_out(w, dt, dev):
    n = w.L * w.M * w.N
    if dt == "f32":
        buf = torch.full((n + 2 * GUARD,), SENTINEL32, dtype=torch.int32, device=dev)
        view = buf[GUARD:GUARD + n].view(torch.float32)
    else:
        buf = torch.full((n + 2 * GUARD,), SENTINEL16, dtype=torch.int16, device=dev)
        view = buf[GUARD:GUARD + n].view(W.TORCH_DTYPE[dt])
    return buf, view.view(w.L, w.M, w.N)


def check_guards(buf, dt):
    b = buf.cpu()
    head, tail = b[:GUARD], b[-GUARD:]
    want = SENTINEL32 if dt == "f32" else SENTINEL16
    assert bool((head == want).all()) and bool((tail == want).all()), "write outside the output"


def run_gpu(w, inputs, options=None, unfused=False, stream=None, repeat=1):
    """Run the workload on cuda:0 through the C ABI; returns host outputs."""
    A, Bm, aux, scalars = inputs
    dev = torch.device("cuda", 0)
    Ad, Bd = A.to(dev), Bm.to(dev)
    auxd = [a.to(dev) for a in aux]
    bufs, outs = [], []
    for _, dt in w.outs:
        buf, view = alloc_out(w, dt, dev)
        bufs.append(buf)
        outs.append(view)
    plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, dtypes_of(w), B.make_dag(w.dag), options)
    try:
        info = B.gemm_epi_plan_info(plan)
        ws = None
        if unfused:
            nbytes = B.gemm_epi_unfused_workspace_bytes(plan)
            ws = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
        for _ in range(repeat):
            if unfused:
                B.gemm_epi_run_unfused(plan, Ad, Bd, auxd, scalars, outs, ws, stream=stream)
            else:
                B.gemm_epi_run(plan, Ad, Bd, auxd, scalars, outs, stream=stream)
        torch.cuda.synchronize()
        st = B.gemm_epi_last_error(plan)
        assert st == B.GE_OK, B.gemm_epi_status_string(st)
    finally:
        B.gemm_epi_plan_destroy(plan)
    for buf, (_, dt) in zip(bufs, w.outs):
        check_guards(buf, dt)
    return [o.cpu() for o in outs], info


def oracle_rows(w, inputs, rows=None):
    A, Bm, aux, scalars = inputs
    outs, _ = oracle.gemm_epilogue(w.L, w.M, w.N, w.K, w.ab, W.to_codes(A), W.to_codes(Bm),
                                   [W.to_codes(a) for a in aux], [s[2] for s in w.aux],
                                   scalars, w.dag, [dt for _, dt in w.outs], rows=rows,
                                   threads=oracle.threads_default())
    return outs


def decode(codes, dt):
    if dt == "f32":
        return np.asarray(codes, dtype=np.float32).astype(np.float64)
    return _pins.np_decode(codes, dt)


def compare(w, gpu_outs, ref_outs, rows=None, exact=None):
    """Bit-exact (as values: -0 == +0) for integer-valued workloads, else
    |gpu - ref| <= ATOL + RTOL*|ref| with ref rounded to the output type."""
    exact = w.exact if exact is None else exact
    for (name, dt), g, r in zip(w.outs, gpu_outs, ref_outs):
        gc = W.to_codes(g).reshape(w.L * w.M, w.N)
        if rows is not None:
            gc = gc[rows]
        gv, rv = decode(gc, dt), decode(r, dt)
        assert not np.isnan(gv).any(), "%s: NaN in GPU output" % name
        if exact:
            bad = gv != rv
            if bad.any():
                idx = np.argwhere(bad)[:5]
                raise AssertionError("%s: %d of %d elements differ, e.g. %s gpu=%s ref=%s" % (
                    name, bad.sum(), bad.size, idx.tolist(), gv[bad][:5], rv[bad][:5]))
        else:
            err = np.abs(gv - rv)
            lim = W.ATOL + W.RTOL * np.abs(rv)
            bad = err > lim
            if bad.any():
                idx = np.argwhere(bad)[:5]
                raise AssertionError("%s: %d of %d elements out of tolerance, worst %g, e.g. %s "
                                     "gpu=%s ref=%s" % (name, bad.sum(), bad.size,
                                                        float((err - lim).max()), idx.tolist(),
                                                        gv[bad][:5], rv[bad][:5]))


def bitwise_equal(xs, ys):
    for x, y in zip(xs, ys):
        a, b = W.to_codes(x), W.to_codes(y)
        if a.dtype == np.uint16:
            a, b = _pins.zero_norm(a), _pins.zero_norm(b)
            assert np.array_equal(a, b)
        else:
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
