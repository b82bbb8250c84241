"""Pins for the CPU oracle: checks that fix what the oracle must compute
without calling the oracle to produce the expected values.

Every pin takes the loaded oracle library (so a deliberately mutated build can
be run through the same pins) and raises AssertionError on a mismatch.

Sources of truth used here:
  * the IEEE 754 binary16 layout as implemented by numpy's float16, and the
    bfloat16 layout as the upper half of numpy's float32;
  * exact integer arithmetic (numpy int64) for integer-valued inputs, the
    closed form the legacy basic-GEMM notebook asserts with
    assert_array_equal (D = alpha*(A@B) + beta*C);
  * exact rational arithmetic (fractions.Fraction) plus a table search for the
    nearest representable value, on tiny random problems;
  * hand-worked examples stored under tests/golden/;
  * special cases: A = 0, B = identity.
"""
import json
import os
from fractions import Fraction

import numpy as np

import oracle
from dense_gemm_elementwise_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ references --

def np_decode(codes, fmt):
    """Codes -> float64 through numpy's own IEEE types (independent of the oracle)."""
    c = np.asarray(codes, dtype=np.uint16)
    if fmt == "f16":
        return c.view(np.float16).astype(np.float64)
    if fmt == "bf16":
        with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen quietly
            return (c.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(fmt)


def np_encode_exact(values, fmt):
    """Codes of values that are exactly representable in ``fmt``."""
    v = np.asarray(values, dtype=np.float64)
    if fmt == "f16":
        c = v.astype(np.float16)
        assert np.array_equal(c.astype(np.float64), v), "value not representable in f16"
        return c.view(np.uint16)
    f = v.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), v)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not representable in bf16"
    return (bits >> 16).astype(np.uint16)


_TABLES = {}


def _table(fmt):
    """Sorted non-negative finite values of a 16-bit format and their codes."""
    if fmt not in _TABLES:
        top = 0x7C00 if fmt == "f16" else 0x7F80  # first inf code
        codes = np.arange(0, top, dtype=np.uint16)
        vals = np_decode(codes, fmt)
        assert np.all(np.diff(vals) > 0)
        _TABLES[fmt] = (vals, codes, top)
    return _TABLES[fmt]


def nearest_even_code(x, fmt):
    """Nearest ``fmt`` code to the exact value x (Fraction or exact float),
    ties to the even code, overflow to inf; found by table search with exact
    rational comparisons."""
    x = Fraction(x)
    vals, codes, inf_code = _table(fmt)
    sign = 0x8000 if x < 0 else 0
    ax = abs(x)
    top = Fraction(float(vals[-1]))
    half_ulp_top = (top - Fraction(float(vals[-2]))) / 2
    if ax >= top + half_ulp_top:
        return sign | inf_code
    k = int(np.searchsorted(vals, float(ax)))
    best = None
    for idx in (k - 1, k, k + 1):
        if 0 <= idx < len(vals):
            d = abs(Fraction(float(vals[idx])) - ax)
            if best is None or d < best[0] or (d == best[0] and int(codes[idx]) % 2 == 0):
                best = (d, int(codes[idx]))
    return sign | best[1]


def nearest_even_f32(x):
    """Nearest float32 to the exact value x, ties to even (exact comparisons)."""
    x = Fraction(x)
    g = np.float32(float(x))
    cands = {g, np.nextafter(g, np.float32(np.inf)), np.nextafter(g, np.float32(-np.inf))}
    best = None
    for c in sorted(cands):
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - x)
        even = int(np.array(c, dtype=np.float32).view(np.uint32)) % 2 == 0
        if best is None or d < best[0] or (d == best[0] and even):
            best = (d, c)
    return np.float32(best[1])


def _mpf(x):
    import mpmath
    return mpmath.mpf(x.numerator) / x.denominator


def _frac(m):
    """mpmath number -> exact Fraction of its binary value."""
    import mpmath
    sign, man, exp, _ = mpmath.mpf(m)._mpf_
    return (-1) ** sign * Fraction(int(man)) * (Fraction(2) ** int(exp))


def activation_exact(op, x):
    """The activation at 60 significant digits (mpmath), as a Fraction: the
    definitions, evaluated far beyond fp64 so the result rounds like the
    true value."""
    import mpmath
    with mpmath.workdps(60):
        m = _mpf(Fraction(x))
        if op == "sigmoid":
            r = 1 / (1 + mpmath.exp(-m))
        elif op == "tanh":
            r = mpmath.tanh(m)
        elif op == "gelu":
            r = m * (1 + mpmath.erf(m / mpmath.sqrt(2))) / 2
        elif op == "silu":
            r = m / (1 + mpmath.exp(-m))
        else:  # hardswish
            r = m * min(max(m + 3, 0), 6) / 6
        return _frac(r)


def eval_dag_exact(dag, acc, aux_vals, scalars, n_out):
    """Evaluate a DAG on exact rationals for one element.  ``aux_vals[s]`` is
    the (already selected) exact value of aux slot s at this element."""
    v = [None] * len(dag)
    outs = [None] * n_out
    for n, (op, a, b, s) in enumerate(dag):
        if op == "accum":
            v[n] = acc
        elif op in ("load", "broadcast", "col_broadcast"):
            v[n] = aux_vals[s]
        elif op == "scalar":
            v[n] = Fraction(scalars[s])
        elif op == "mul":
            v[n] = v[a] * v[b]
        elif op == "add":
            v[n] = v[a] + v[b]
        elif op == "sub":
            v[n] = v[a] - v[b]
        elif op == "div":
            v[n] = v[a] / v[b]
        elif op == "min":
            v[n] = min(v[a], v[b])
        elif op == "max":
            v[n] = max(v[a], v[b])
        elif op == "relu":
            v[n] = v[a] if v[a] > 0 else Fraction(0)
        elif op == "leaky_relu":
            v[n] = v[a] if v[a] > 0 else v[b] * v[a]
        elif op in ("sigmoid", "tanh", "gelu", "silu", "hardswish"):
            v[n] = activation_exact(op, v[a])
        elif op == "store":
            outs[s] = v[a]
    return outs


def zero_norm(codes):
    """Map -0 codes to +0 (results are compared as values, -0 == +0)."""
    c = np.array(codes, dtype=np.uint16, copy=True)
    c[c == 0x8000] = 0
    return c


def run_oracle(L_, w, A, B, aux, scalars, rows=None, threads=0, want_pre=False):
    return oracle.gemm_epilogue(w.L, w.M, w.N, w.K, w.ab, W.to_codes(A), W.to_codes(B),
                                [W.to_codes(a) for a in aux], [s[2] for s in w.aux],
                                scalars, w.dag, [dt for _, dt in w.outs], rows=rows,
                                threads=threads, want_pre=want_pre, lib_handle=L_)


def small(w, L, M, N, K, seed=None, dist=None):
    import dataclasses
    return dataclasses.replace(w, L=L, M=M, N=N, K=K, seed=w.seed if seed is None else seed,
                               dist=dist or w.dist, sample_rows=None)


# ------------------------------------------------------------------ pins --

def pin_decode_exhaustive(L_):
    codes = np.arange(65536, dtype=np.uint16)
    for fmt, fn in (("f16", oracle.f16_to_f64), ("bf16", oracle.bf16_to_f64)):
        got = fn(codes, L_)
        ref = np_decode(codes, fmt)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan), fmt + ": NaN codes differ"
        assert np.array_equal(got[~nan], ref[~nan]), fmt + ": decoded values differ"
        assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), fmt + ": sign"


def pin_encode_roundtrip(L_):
    codes = np.arange(65536, dtype=np.uint16)
    for fmt, enc in (("f16", oracle.f64_to_f16), ("bf16", oracle.f64_to_bf16)):
        vals = np_decode(codes, fmt)
        ok = ~np.isnan(vals)
        got = enc(vals[ok], L_)
        assert np.array_equal(got, codes[ok]), fmt + ": encode(decode(c)) != c"
        nan_codes = enc(np.array([np.nan]), L_)
        assert np.isnan(np_decode(nan_codes, fmt)).all(), fmt + ": NaN must stay NaN"


def pin_encode_midpoints(L_):
    """Halfway points between neighbours go to the even code; a hair above or
    below goes to the nearer neighbour; the halfway point above the largest
    finite value goes to inf."""
    for fmt, enc in (("f16", oracle.f64_to_f16), ("bf16", oracle.f64_to_bf16)):
        vals, codes, inf_code = _table(fmt)
        lo, hi = vals[:-1], vals[1:]
        mid = (lo + hi) / 2  # exact: neighbours differ by a power of two in a binade
        assert np.all((mid > lo) & (mid < hi))
        even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
        for sgn in (1.0, -1.0):
            sbit = np.uint16(0x8000) if sgn < 0 else np.uint16(0)
            got = enc(sgn * mid, L_)
            assert np.array_equal(got, even | sbit), fmt + ": ties must go to even"
            # a hair further from zero goes to the larger magnitude, a hair
            # closer to zero to the smaller, whatever the sign
            up = enc(sgn * np.nextafter(mid, np.inf), L_)
            dn = enc(sgn * np.nextafter(mid, -np.inf), L_)
            assert np.array_equal(up, codes[1:] | sbit), fmt + ": above midpoint"
            assert np.array_equal(dn, codes[:-1] | sbit), fmt + ": below midpoint"
        top, prev = vals[-1], vals[-2]
        edge = top + (top - prev) / 2
        assert int(enc(np.array([edge]), L_)[0]) == inf_code, fmt + ": overflow midpoint"
        assert int(enc(np.array([np.nextafter(edge, 0)]), L_)[0]) == int(codes[-1])
        assert int(enc(np.array([-edge]), L_)[0]) == (inf_code | 0x8000)


def pin_encode_random_vs_table(L_):
    """Random doubles over the whole exponent range against the exact table
    search (and, for f16, numpy's own double -> half conversion)."""
    rs = np.random.RandomState(11)
    x = rs.standard_normal(4000) * np.exp2(rs.uniform(-30, 18, 4000))
    got16 = oracle.f64_to_f16(x, L_)
    with np.errstate(over="ignore"):
        np16 = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(zero_norm(got16), zero_norm(np16))
    sub = x[:600]
    ref16 = np.array([nearest_even_code(float(v), "f16") for v in sub], dtype=np.uint16)
    assert np.array_equal(zero_norm(got16[:600]), zero_norm(ref16))
    y = rs.standard_normal(600) * np.exp2(rs.uniform(-140, 130, 600))
    gotb = oracle.f64_to_bf16(y, L_)
    refb = np.array([nearest_even_code(float(v), "bf16") for v in y], dtype=np.uint16)
    assert np.array_equal(zero_norm(gotb), zero_norm(refb))


def _golden_cases():
    dags = {
        "my_epilogue_2x2x2.json": (W.dag_my_epilogue(), [("C", "tensor", "f16")],
                                   [("D", "f16"), ("Aux", "f16")]),
        "relu_linear_2x2x2.json": (W.dag_relu_linear(), [("C", "tensor", "f16")], [("D", "f16")]),
        "alpha_beta_x_2x2x2.json": (W.dag_alpha_beta_x(),
                                    [("C", "tensor", "f16"), ("X", "tensor", "f16")],
                                    [("D", "f16"), ("Y", "f16")]),
        "bias_relu_square_2x2x2x2.json": (W.dag_bias_relu_square(),
                                          [("C", "tensor", "bf16"), ("bias", "row", "f32")],
                                          [("D", "bf16"), ("E", "bf16")]),
        "row_col_bias_2x2x2.json": (W.dag_row_col_bias(),
                                    [("row_bias", "row", "f16"), ("col_bias", "col", "f16")],
                                    [("D", "f16")]),
    }
    for fname, (dag, aux_spec, outs) in dags.items():
        with open(os.path.join(GOLDEN, fname)) as f:
            yield fname, json.load(f), dag, aux_spec, outs


def pin_golden(L_):
    for fname, g, dag, aux_spec, outs in _golden_cases():
        L, M, N, K, ab = g["L"], g["M"], g["N"], g["K"], g["ab"]
        A = np_encode_exact(np.array(g["A"], dtype=np.float64).reshape(L, M, K), ab)
        B = np_encode_exact(np.array(g["B"], dtype=np.float64).reshape(L, K, N), ab)
        aux, aux_dt = [], []
        for name, kind, dt in aux_spec:
            a = np.array(g["aux"][name], dtype=np.float64)
            aux.append(a.astype(np.float32) if dt == "f32" else np_encode_exact(a, dt))
            aux_dt.append(dt)
        res, _ = oracle.gemm_epilogue(L, M, N, K, ab, A, B, aux, aux_dt, g["scalars"], dag,
                                      [dt for _, dt in outs], lib_handle=L_)
        for (name, dt), got in zip(outs, res):
            want = np.array(g["expected"][name], dtype=np.float64).reshape(L * M, N)
            val = got.astype(np.float64) if dt == "f32" else np_decode(got, dt)
            assert np.array_equal(val, want), "%s: %s = %s, hand-worked %s" % (
                fname, name, val.tolist(), want.tolist())
            if "expected_codes" in g and name in g["expected_codes"]:
                wc = np.array(g["expected_codes"][name], dtype=np.uint16).reshape(L * M, N)
                assert np.array_equal(got, wc), fname + ": codes"


def _int_inputs(w):
    A, B, aux, scalars = W.make_inputs(w)
    Ai = A.float().numpy().astype(np.int64)
    Bi = B.float().numpy().astype(np.int64)
    auxi = [a.float().numpy().astype(np.int64) for a in aux]
    return (A, B, aux, scalars), Ai, Bi, auxi


def pin_integer_closed_form(L_):
    """Integer inputs: the exact integer result, as the basic-GEMM notebook
    asserts (assert_array_equal(D, alpha*(A@B) + beta*C))."""
    w = small(W.MY_EPILOGUE_128, L=2, M=24, N=40, K=56)
    (A, B, aux, sc), Ai, Bi, (Ci,) = _int_inputs(w)
    acc = np.einsum("lik,lkj->lij", Ai, Bi)  # exact int64
    aux_ref = 1 * acc + 2 * Ci
    (D, Aux), _ = run_oracle(L_, w, A, B, aux, sc)
    assert np.array_equal(np_decode(Aux, "f16"), aux_ref.reshape(-1, w.N).astype(np.float64))
    assert np.array_equal(np_decode(D, "f16"), 0.5 * aux_ref.reshape(-1, w.N))
    # ceil(uniform(-4, 4)) inputs and the fused ReLU: D = max(A@B + 2*C, 0)
    w3 = small(W.RELU_2400X3232X4096, L=2, M=20, N=24, K=72)
    (A, B, aux, sc), Ai, Bi, (Ci,) = _int_inputs(w3)
    ref = np.maximum(np.einsum("lik,lkj->lij", Ai, Bi) + 2 * Ci, 0).reshape(-1, w3.N)
    (D,), _ = run_oracle(L_, w3, A, B, aux, sc)
    assert np.array_equal(np_decode(D, "f16"), ref.astype(np.float64))


def pin_gemm_accum_closed_form(L_):
    """The accumulator alone, before any epilogue ("CUTLASS Operator API:
    Custom epilogue fusions for GEMMs": accum is the GEMM result the
    epilogue receives), on integer inputs: the exact int64 product, per
    batch, for every row and for an unordered row subset spread over the
    batches, fp16 and bf16 operands, one thread and several."""
    for w in (small(W.MY_EPILOGUE_128, L=3, M=20, N=24, K=72),
              small(W.BIAS_RELU_SQUARE_L8, L=2, M=12, N=40, K=56, dist="randint")):
        (A, B, _, _), Ai, Bi, _ = _int_inputs(w)
        want = np.einsum("lik,lkj->lij", Ai, Bi).reshape(w.L * w.M, w.N).astype(np.float64)
        full = oracle.gemm_accum(w.L, w.M, w.N, w.K, w.ab, W.to_codes(A), W.to_codes(B),
                                 threads=1, lib_handle=L_)
        assert np.array_equal(full, want), w.name
        rows = np.array([w.L * w.M - 1, 0, w.M + 3, 7, w.M, 2 * w.M - 1], dtype=np.int64)
        part = oracle.gemm_accum(w.L, w.M, w.N, w.K, w.ab, W.to_codes(A), W.to_codes(B),
                                 rows=rows, threads=3, lib_handle=L_)
        assert np.array_equal(part, want[rows]), w.name


def pin_new_ops_closed_form(L_):
    """Integer inputs through subtraction, division by powers of two, min,
    max and row + column broadcasts: the exact results, computed in numpy."""
    ex = {x.name: x for x in W.page_examples()}
    w = small(ex["row_col_bias_f16"], L=2, M=12, N=24, K=40)
    (A, B, aux, sc), Ai, Bi, (rb, cb) = _int_inputs(w)
    acc = np.einsum("lik,lkj->lij", Ai, Bi)
    ref = (acc + rb[None, None, :] + cb[None, :, None]).reshape(-1, w.N)
    (D,), _ = run_oracle(L_, w, A, B, aux, sc)
    assert np.array_equal(np_decode(D, "f16"), ref.astype(np.float64))
    w = small(ex["clamp_f16"], L=2, M=10, N=16, K=24)
    (A, B, aux, sc), Ai, Bi, (Ci,) = _int_inputs(w)
    acc = np.einsum("lik,lkj->lij", Ai, Bi)
    ref = np.minimum(np.maximum(acc - Ci, -3.0), 5.5).reshape(-1, w.N)
    (D,), _ = run_oracle(L_, w, A, B, aux, sc)
    assert np.array_equal(np_decode(D, "f16"), ref)
    w = small(ex["aux_normalize_f16"], L=1, M=8, N=16, K=24)
    A, B, aux, sc = W.make_inputs(w)
    acc = np.einsum("lik,lkj->lij", A.double().numpy(), B.double().numpy())
    ref = (acc / aux[0].double().numpy()).reshape(-1, w.N)
    assert set(np.unique(np.abs(aux[0].double().numpy()))) <= {1.0, 2.0, 4.0}
    (D,), _ = run_oracle(L_, w, A, B, aux, sc)
    assert np.array_equal(np_decode(D, "f16"), ref)
    w = small(ex["scale_shift_bf16"], L=1, M=8, N=16, K=24)
    A, B, aux, sc = W.make_inputs(w)
    acc = np.einsum("lik,lkj->lij", A.double().numpy(), B.double().numpy()).reshape(-1, w.N)
    (D, T), _ = run_oracle(L_, w, A, B, aux, sc)
    assert np.array_equal(D.astype(np.float64), (acc * 2 - 1) / 4)
    assert np.array_equal(np_decode(T, "bf16"), acc * 2)


def _act_values(L_, act, xs, slope=0.25):
    """act(x) through the oracle for fp16-representable xs: K = 1 and B = 1,
    so accum = x exactly; D = act(accum) stored as fp32."""
    import torch
    g = W.Dag()
    a = g.accum()
    g.store(g.leaky_relu(a, g.scalar(0)) if act == "leaky_relu" else getattr(g, act)(a), 0)
    w = W.Workload(name="act_" + act, L=1, M=len(xs), N=1, K=1, ab="f16", aux=[],
                   scalars=[("slope", slope)], outs=[("D", "f32")], dag=g.nodes,
                   dist="normal", seed=0, exact=False)
    A = torch.tensor(xs, dtype=torch.float64).to(torch.float16).reshape(1, -1, 1)
    assert np.array_equal(A.double().numpy().ravel(), np.asarray(xs, dtype=np.float64))
    B = torch.ones(1, 1, 1, dtype=torch.float16)
    (D,), _ = run_oracle(L_, w, A, B, [], [slope])
    return D.ravel().astype(np.float64)


def pin_activation_identities(L_):
    """The activations against textbook values and identities that tie them to
    one another: sigmoid(0) = 1/2 and sigmoid(x) + sigmoid(-x) = 1;
    tanh(x) = 2 sigmoid(2x) - 1 and tanh odd; x Phi(x) with Phi from the
    standard normal table (Phi(1) = 0.8413447460685429, upper tail at 8 =
    6.220960574271785e-16) and gelu(x) - gelu(-x) = x; silu(x) = x sigmoid(x);
    hardswish's three pieces at hand-worked points; leaky ReLU's two sides."""
    u = 2.0 ** -23  # fp32 unit roundoff x 2: results are fp64 rounded once to fp32
    xs = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 8.0, 0.125, 0.75]
    xn = [-x for x in xs]
    sig_p, sig_n = _act_values(L_, "sigmoid", xs), _act_values(L_, "sigmoid", xn)
    assert sig_p[0] == 0.5
    assert np.all(np.abs(sig_p + sig_n - 1.0) <= 2 * u)
    assert np.all(np.diff(_act_values(L_, "sigmoid", sorted(xn + xs[1:]))) >= 0)
    sig_2x = _act_values(L_, "sigmoid", [2 * x for x in xs])
    th_p, th_n = _act_values(L_, "tanh", xs), _act_values(L_, "tanh", xn)
    assert th_p[0] == 0.0 and np.array_equal(th_p, -th_n)
    assert np.all(np.abs(th_p - (2 * sig_2x - 1)) <= 4 * u)
    ge_p, ge_n = _act_values(L_, "gelu", xs), _act_values(L_, "gelu", xn)
    assert ge_p[0] == 0.0
    assert np.all(np.abs((ge_p - ge_n) - np.array(xs)) <= 2 * u * np.maximum(1.0, np.array(xs)))
    assert abs(ge_p[2] - 0.8413447460685429) <= u
    assert abs(ge_n[2] + (1 - 0.8413447460685429)) <= u
    assert ge_p[8] == 8.0
    tail = -8.0 * 6.220960574271785e-16
    assert abs(ge_n[8] - tail) <= 2 * u * abs(tail)
    si_p, si_n = _act_values(L_, "silu", xs), _act_values(L_, "silu", xn)
    assert np.all(np.abs(si_p - np.array(xs) * sig_p) <= 2 * u * np.maximum(1.0, np.array(xs)))
    assert np.all(np.abs(si_n - np.array(xn) * sig_n) <= 2 * u)
    hx = [-8.0, -3.0, -2.0, -1.5, 0.0, 1.0, 1.5, 3.0, 4.0, 8.0]
    hs = _act_values(L_, "hardswish", hx)
    want = [0.0, 0.0, -1 / 3, -0.375, 0.0, 2 / 3, 1.125, 3.0, 4.0, 8.0]
    assert np.array_equal(hs, np.array(want, dtype=np.float32).astype(np.float64))
    lx = [-4.0, -1.5, -0.125, 0.0, 0.125, 1.5, 4.0]
    assert np.array_equal(_act_values(L_, "leaky_relu", lx, slope=0.25),
                          [-1.0, -0.375, -0.03125, 0.0, 0.125, 1.5, 4.0])


def pin_grouped_closed_form(L_):
    """A grouped GEMM is its problems computed independently: integer inputs,
    each problem's D equals its own exact alpha*A_g@B_g + beta*C_g (numpy
    float64 matmul of small integers, exact), the row bias and ReLU of the
    ragged workload likewise, and reversing the problem order reverses the
    outputs."""
    import dataclasses
    w = dataclasses.replace(W.GROUPED_BY_NAME["grouped_gemm_50"],
                            problems=[(8, 16, 24), (24, 8, 40), (16, 32, 8)],
                            scalars=[("alpha", 1.0), ("beta", 2.0)])
    As, Bs, auxs, sc = W.make_grouped_inputs(w)
    assert set(np.unique(As[0].double().numpy())) <= set(range(-3, 3))

    def run(ws, As_, Bs_, auxs_):
        return oracle.grouped_gemm_epilogue(
            ws.problems, ws.ab, [W.to_codes(a) for a in As_], [W.to_codes(b) for b in Bs_],
            [[W.to_codes(x) for x in per] for per in auxs_], [s[2] for s in ws.aux], sc, ws.dag,
            [dt for _, dt in ws.outs], lib_handle=L_)

    res = run(w, As, Bs, auxs)
    for g in range(len(w.problems)):
        ref = As[g].double().numpy() @ Bs[g].double().numpy() + 2 * auxs[g][0].double().numpy()
        assert np.array_equal(np_decode(res[g][0], "f16"), ref), g
    wr = dataclasses.replace(w, problems=w.problems[::-1])
    rev = run(wr, As[::-1], Bs[::-1], auxs[::-1])
    for g in range(len(w.problems)):
        assert np.array_equal(rev[g][0], res[-1 - g][0])
    w = dataclasses.replace(W.GROUPED_BY_NAME["grouped_bias_relu_ragged"],
                            problems=[(5, 8, 9), (3, 16, 2), (9, 8, 17)])
    As, Bs, auxs, sc = W.make_grouped_inputs(w)
    res = oracle.grouped_gemm_epilogue(
        w.problems, w.ab, [W.to_codes(a) for a in As], [W.to_codes(b) for b in Bs],
        [[W.to_codes(x) for x in per] for per in auxs], [s[2] for s in w.aux], sc, w.dag,
        [dt for _, dt in w.outs], lib_handle=L_)
    for g in range(len(w.problems)):
        t = (0.5 * (As[g].double().numpy() @ Bs[g].double().numpy()) +
             auxs[g][0].double().numpy() + auxs[g][1].double().numpy()[None, :])
        assert np.array_equal(np_decode(res[g][0], "bf16"), np.maximum(t, 0.0)), g
        assert np.array_equal(res[g][1].astype(np.float64), t), g


def pin_broadcast_closed_form(L_):
    """Row-broadcast bias indexed by column j, same vector for every row and
    batch: integer inputs, D = relu(0.5*A@B + C + bias), E = D*D rounded."""
    w = small(W.BIAS_RELU_SQUARE_L8, L=3, M=6, N=16, K=8, dist="randint")
    (A, B, aux, sc), Ai, Bi, (Ci, biasi) = _int_inputs(w)
    acc = np.einsum("lik,lkj->lij", Ai, Bi)
    d = np.maximum(0.5 * acc + Ci + biasi[None, None, :], 0.0).reshape(-1, w.N)
    (D, E), _ = run_oracle(L_, w, A, B, aux, sc)
    assert np.array_equal(np_decode(D, "bf16"), d)
    e_ref = np.array([nearest_even_code(v * v, "bf16") for v in d.ravel()], dtype=np.uint16)
    assert np.array_equal(zero_norm(E.ravel()), zero_norm(e_ref))


def _exact_case(L_, w, rs):
    """Fraction brute force for one workload at a tiny size with non-integer
    inputs (N(0,1) rounded to the operand type)."""
    import torch
    g = torch.Generator().manual_seed(int(rs.randint(1 << 30)))
    L, M, N, K = w.L, w.M, w.N, w.K
    A = torch.randn(L, M, K, generator=g).to(W.TORCH_DTYPE[w.ab])
    B = torch.randn(L, K, N, generator=g).to(W.TORCH_DTYPE[w.ab])
    aux = []
    for spec in w.aux:
        shp = {"tensor": (L, M, N), "row": (N,), "col": (M,)}[spec[1]]
        aux.append(torch.randn(shp, generator=g).to(W.TORCH_DTYPE[spec[2]]))
    scalars = [float(np.float32(v)) for v in rs.uniform(-3, 3, len(w.scalars))]
    outs, _ = run_oracle(L_, w, A, B, aux, scalars)
    Af = [[[Fraction(float(x)) for x in r] for r in m] for m in A.double().tolist()]
    Bf = [[[Fraction(float(x)) for x in r] for r in m] for m in B.double().tolist()]
    auxf = [a.double().numpy() for a in aux]
    for l in range(L):
        for i in range(M):
            for j in range(N):
                acc = sum(Af[l][i][k] * Bf[l][k][j] for k in range(K))
                av = []
                for spec, a in zip(w.aux, auxf):
                    sel = {"tensor": lambda: a[l, i, j], "row": lambda: a[j],
                           "col": lambda: a[i]}[spec[1]]()
                    av.append(Fraction(float(sel)))
                want = eval_dag_exact(w.dag, acc, av, scalars, len(w.outs))
                for o, (_, dt) in enumerate(w.outs):
                    got = outs[o][l * M + i, j]
                    if dt == "f32":
                        ref = nearest_even_f32(want[o])
                        assert got == ref or (got == 0 and ref == 0), (w.name, l, i, j)
                    else:
                        ref = nearest_even_code(want[o], dt)
                        assert zero_norm([got])[0] == zero_norm([ref])[0], (
                            w.name, l, i, j, hex(int(got)), hex(ref), float(want[o]))


def pin_fraction_brute_force(L_):
    rs = np.random.RandomState(5)
    cases = list(W.WORKLOADS[1:]) + W.page_examples()
    for w in cases:
        _exact_case(L_, small(w, L=2, M=3, N=5, K=7), rs)


def pin_special_cases(L_):
    # A = 0: accum = 0, so Aux = beta*C and D = extra_scalar*beta*C
    w = small(W.MY_EPILOGUE_128, L=1, M=8, N=16, K=24)
    A, B, aux, sc = W.make_inputs(w)
    A = A * 0
    (D, Aux), _ = run_oracle(L_, w, A, B, aux, sc)
    C = aux[0].double().numpy().reshape(-1, w.N)
    assert np.array_equal(np_decode(Aux, "f16"), 2 * C)
    assert np.array_equal(np_decode(D, "f16"), C)
    # B = identity (K = N): accum = A exactly; Y is A's codes and D rounds
    # 2A + C + 3X (exact in fp64 for fp16 operands) once
    import torch
    w4 = small(W.ALPHA_BETA_X_8192, L=2, M=8, N=16, K=16)
    A, B, aux, sc = W.make_inputs(w4)
    B = torch.eye(16, dtype=torch.float16).expand(2, 16, 16).contiguous()
    (D, Y), _ = run_oracle(L_, w4, A, B, aux, sc)
    assert np.array_equal(zero_norm(Y), zero_norm(W.to_codes(A).reshape(-1, 16)))
    a, c, x = (t.double().numpy().reshape(-1, 16) for t in (A, aux[0], aux[1]))
    ref = (2 * a + c + 3 * x).astype(np.float16).view(np.uint16)
    assert np.array_equal(zero_norm(D), zero_norm(ref))


def pin_relu_positive_zero(L_):
    """ReLU of a non-positive value is +0 ("where(d > 0, d, 0)"), including
    ReLU of -0: with negative scalars, a zero row of A and a zero row of C
    make alpha*accum + beta*C = (-0) + (-0) = -0 there."""
    w = small(W.RELU_2400X3232X4096, L=1, M=16, N=16, K=16)
    A, B, aux, sc = W.make_inputs(w)
    A[0, 0, :] = 0
    aux[0][0, 0, :] = 0
    sc = [-1.0, -2.0]
    (D,), _ = run_oracle(L_, w, A, B, aux, sc)
    (F,), _ = run_oracle(L_, small(w, 1, 16, 16, 16), A, B, aux, [1.0, 2.0])
    vals = np_decode(D, "f16")
    assert np.all(vals >= 0)
    assert (vals == 0).sum() > 100
    assert np.all(D[vals == 0] == 0), "relu must give +0 (code 0x0000)"
    assert np.all(D[0] == 0)
    # with the signs flipped every element that was cut to zero is positive
    flip = np_decode(F, "f16")
    assert np.all((vals > 0) | (flip >= 0))


def pin_rows_and_threads(L_):
    """A row subset equals the same rows of the full result; thread count
    does not change any bit."""
    w = small(W.ALPHA_BETA_X_8192, L=2, M=12, N=24, K=40)
    A, B, aux, sc = W.make_inputs(w)
    full, _ = run_oracle(L_, w, A, B, aux, sc, threads=1)
    rows = np.array([0, 5, 11, 12, 23], dtype=np.int64)
    part, _ = run_oracle(L_, w, A, B, aux, sc, rows=rows, threads=3)
    for f, p in zip(full, part):
        assert np.array_equal(f[rows], p)
    many, _ = run_oracle(L_, w, A, B, aux, sc, threads=7)
    for f, m in zip(full, many):
        assert np.array_equal(f, m)


ALL_PINS = [pin_decode_exhaustive, pin_encode_roundtrip, pin_encode_midpoints,
            pin_encode_random_vs_table, pin_golden, pin_integer_closed_form,
            pin_gemm_accum_closed_form,
            pin_broadcast_closed_form, pin_new_ops_closed_form, pin_activation_identities,
            pin_grouped_closed_form,
            pin_fraction_brute_force,
            pin_special_cases,
            pin_relu_positive_zero, pin_rows_and_threads]


def run_all(lib_path):
    """Run every pin against the library at ``lib_path``; used on mutated
    builds of the oracle.  Exit status 1 when some pin fails."""
    L_ = oracle.lib(lib_path)
    failed = []
    for p in ALL_PINS:
        try:
            p(L_)
        except Exception as e:  # any failure counts as caught
            failed.append("%s: %s" % (p.__name__, str(e)[:120]))
    return failed
