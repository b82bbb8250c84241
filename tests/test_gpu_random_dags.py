"""Random epilogue DAGs through the whole path: the DAG compiler (register
allocation, reversed two-address forms, leaf reads), the built-in or
interpreted executor and the unfused kernel, against the oracle.

Inputs are small integers, scalars are small dyadic numbers and divisors
powers of two; the generator tracks a bound on every value's magnitude and
on its fractional bits and only builds nodes whose result needs at most 24
significant bits, so every fp32 intermediate is exact and results must match
the oracle bit for bit in every output type."""
import math
import random

import pytest

pytestmark = pytest.mark.gpu

import _gpu  # noqa: E402
from _gpu import B, W  # noqa: E402

SCALARS = [0.5, 2.0, -1.0, 3.0, 0.25]
SCALAR_BOUND, SCALAR_FRAC = 3.0, 2


def random_workload(seed):
    """A valid single-assignment DAG of at most 16 nodes over accum (K = 32,
    |accum| <= 128), a Load tensor C, a power-of-two divisor tensor Q, a row
    and a column vector, up to three scalars; 1-3 stores of random types."""
    rng = random.Random(seed)
    g = W.Dag()
    info = {}  # node -> (magnitude bound, fractional bits)

    def add(node, bound, frac):
        info[node] = (bound, frac)
        return node

    def fits(bound, frac):
        return math.log2(max(bound, 1.0)) + frac <= 23

    vals = [add(g.accum(), 128.0, 0)]
    n_scalar = rng.randint(1, 3)
    aux = [("C", "tensor", "f16"), ("Q", "tensor", "f16", "pow2"), ("r", "row", "f32"),
           ("c", "col", "f16")]
    divisor = None
    n_out = rng.randint(1, 3)
    budget = 16 - n_out
    while len(g.nodes) < budget:
        r = rng.random()
        if r < 0.3:
            k = rng.randrange(4)
            if k == 0:
                v = add(g.load(0), 2.0, 0)
            elif k == 1:
                v = divisor = add(g.load(1), 4.0, 0)
            elif k == 2:
                v = add(g.broadcast(2), 2.0, 0)
            else:
                v = add(g.col_broadcast(3), 2.0, 0)
            vals.append(v)
        elif r < 0.4:
            vals.append(add(g.scalar(rng.randrange(n_scalar)), SCALAR_BOUND, SCALAR_FRAC))
        elif r < 0.55:
            a = rng.choice(vals)
            ba, fa = info[a]
            if rng.random() < 0.5 or len(g.nodes) + 2 > budget or not fits(ba * 3, fa + 2):
                vals.append(add(g.relu(a), ba, fa))
            else:
                s = add(g.scalar(0), SCALAR_BOUND, SCALAR_FRAC)
                vals.append(add(g.leaky_relu(a, s), ba * SCALAR_BOUND, fa + SCALAR_FRAC))
        else:
            op = rng.choice(["add", "sub", "mul", "min", "max", "div"])
            a, b = rng.choice(vals), rng.choice(vals)
            (ba, fa), (bb, fb) = info[a], info[b]
            if op == "div":
                if divisor is None or not fits(ba, fa + 2):
                    continue
                vals.append(add(g.div(a, divisor), ba, fa + 2))
            elif op == "mul":
                if not fits(ba * bb, fa + fb):
                    continue
                vals.append(add(g.mul(a, b), ba * bb, fa + fb))
            elif op in ("add", "sub"):
                if not fits(ba + bb, max(fa, fb)):
                    continue
                vals.append(add(getattr(g, op)(a, b), ba + bb, max(fa, fb)))
            else:
                fn = g.minimum if op == "min" else g.maximum
                vals.append(add(fn(a, b), max(ba, bb), max(fa, fb)))
    outs = []
    picks = rng.sample(vals[1:], min(n_out, len(vals) - 1)) if len(vals) > 1 else [vals[0]]
    for o, v in enumerate(picks):
        g.store(v, o)
        outs.append(("O%d" % o, rng.choice(["f32", "f16", "bf16"])))
    scal = [("s%d" % i, rng.choice(SCALARS)) for i in range(n_scalar)]
    return W.Workload(name="random_%d" % seed, L=2, M=136, N=264, K=32, ab="f16", aux=aux,
                      scalars=scal, outs=outs, dag=g.nodes, dist="randint", seed=seed,
                      exact=True)


SEEDS = list(range(48))


@pytest.mark.parametrize("seed", SEEDS)
def test_random_dag(seed):
    w = random_workload(seed)
    dt, dag = _gpu.dtypes_of(w), B.make_dag(w.dag)
    st = B.gemm_epi_validate(dt, dag)
    if st == B.GE_ERR_UNSUPPORTED:
        pytest.skip("more live values than the program's registers")
    assert st == B.GE_OK, B.gemm_epi_status_string(st)
    inputs = W.make_inputs(w)
    ref = _gpu.oracle_rows(w, inputs)
    fused, info = _gpu.run_gpu(w, inputs)
    _gpu.compare(w, fused, ref)
    unfused, _ = _gpu.run_gpu(w, inputs, unfused=True)
    _gpu.bitwise_equal(fused, unfused)
    four, _ = _gpu.run_gpu(w, inputs, options=B.ge_options(epi_warps=4, cta_group=1, tile_n=64))
    _gpu.bitwise_equal(fused, four)
