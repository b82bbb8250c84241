"""Workload table and seeded synthetic input generators.

This module holds data only: problem shapes, element types, the epilogue of
each workload written as a DAG (plain tuples), scalar values, and the seeded
generators that draw the operands on the host.  It contains none of the
GEMM or epilogue arithmetic; both the CUDA path (through the C-ABI binding)
and the CPU oracle consume what it produces.

DAG tuples are ``(op, a, b, slot)`` with ``op`` one of ``accum, load, scalar,
broadcast, col_broadcast, mul, add, sub, div, min, max, relu, sigmoid, tanh,
gelu, silu, hardswish, leaky_relu, store``;
``a``/``b`` index earlier nodes; ``slot`` selects the aux tensor (load, row or
column broadcast), the scalar (scalar) or the output (store).  Output slot 0
is D.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np
import torch

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
ESIZE = {"f16": 2, "bf16": 2, "f32": 4}


class Dag:
    """Tiny builder for epilogue DAGs in single assignment order."""

    def __init__(self):
        self.nodes: List[Tuple[str, int, int, int]] = []

    def _add(self, op, a=0, b=0, slot=0):
        self.nodes.append((op, a, b, slot))
        return len(self.nodes) - 1

    def accum(self):
        return self._add("accum")

    def load(self, slot):
        return self._add("load", slot=slot)

    def broadcast(self, slot):
        return self._add("broadcast", slot=slot)

    def col_broadcast(self, slot):
        return self._add("col_broadcast", slot=slot)

    def sub(self, a, b):
        return self._add("sub", a, b)

    def div(self, a, b):
        return self._add("div", a, b)

    def minimum(self, a, b):
        return self._add("min", a, b)

    def maximum(self, a, b):
        return self._add("max", a, b)

    def sigmoid(self, a):
        return self._add("sigmoid", a)

    def tanh(self, a):
        return self._add("tanh", a)

    def gelu(self, a):
        return self._add("gelu", a)

    def silu(self, a):
        return self._add("silu", a)

    def hardswish(self, a):
        return self._add("hardswish", a)

    def leaky_relu(self, a, slope):
        return self._add("leaky_relu", a, slope)

    def scalar(self, slot):
        return self._add("scalar", slot=slot)

    def mul(self, a, b):
        return self._add("mul", a, b)

    def add(self, a, b):
        return self._add("add", a, b)

    def relu(self, a):
        return self._add("relu", a)

    def store(self, a, slot):
        return self._add("store", a, 0, slot)


@dataclass
class Workload:
    name: str
    L: int
    M: int
    N: int
    K: int
    ab: str                                   # element type of A and B
    aux: List[tuple]                          # (name, "tensor" (L,M,N) | "row" (N,) |
                                              #  "col" (M,), dtype[, "pow2"])
    scalars: List[Tuple[str, float]]          # (name, value)
    outs: List[Tuple[str, str]]               # (name, dtype); outs[0] is D
    dag: List[Tuple[str, int, int, int]]
    dist: str                                 # "randint", "ceil_uniform", "normal"
    seed: int
    exact: bool                               # integer-valued: results must be bit-exact
    sample_rows: Optional[int] = None         # oracle rows per batch at full size (None: all)
    cite: str = ""
    notes: str = field(default="")

    def flops(self) -> float:
        return 2.0 * self.L * self.M * self.N * self.K

    def alg_bytes(self) -> int:
        """Read A, B and each aux once; write each output once."""
        L, M, N, K = self.L, self.M, self.N, self.K
        b = (L * M * K + L * K * N) * ESIZE[self.ab]
        for spec in self.aux:
            kind, dt = spec[1], spec[2]
            b += {"tensor": L * M * N, "row": N, "col": M}[kind] * ESIZE[dt]
        for _, dt in self.outs:
            b += L * M * N * ESIZE[dt]
        return b


# ---------------------------------------------------------------- DAGs ----

def dag_my_epilogue():
    """Aux = alpha*accum + beta*C ; D = extra_scalar*Aux ; returns D, Aux.
    ("CUTLASS Operator API: Custom epilogue fusions for GEMMs", cell [2])."""
    g = Dag()
    acc = g.accum()
    alpha = g.scalar(0)
    t0 = g.mul(alpha, acc)
    c = g.load(0)
    beta = g.scalar(1)
    t1 = g.mul(beta, c)
    aux = g.add(t0, t1)
    s = g.scalar(2)
    d = g.mul(s, aux)
    g.store(d, 0)
    g.store(aux, 1)
    return g.nodes


def dag_relu_linear():
    """D = relu(alpha*accum + beta*C) ("Custom Epilogue Example",
    "Activation Functions"; the legacy epilogue notebook's fused ReLU)."""
    g = Dag()
    acc = g.accum()
    t0 = g.mul(acc, g.scalar(0))
    t1 = g.mul(g.load(0), g.scalar(1))
    d = g.relu(g.add(t0, t1))
    g.store(d, 0)
    return g.nodes


def dag_alpha_beta_x():
    """Y = accum ; D = accum*alpha + C*beta + X*x_factor ("Custom Epilogue
    Example", "Basic Example: Alpha-Beta Scaling").  Outputs: D (slot 0), Y."""
    g = Dag()
    acc = g.accum()
    t0 = g.mul(acc, g.scalar(0))
    t1 = g.mul(g.load(0), g.scalar(1))
    t2 = g.add(t0, t1)
    t3 = g.mul(g.load(1), g.scalar(2))
    d = g.add(t2, t3)
    g.store(d, 0)
    g.store(acc, 1)
    return g.nodes


def dag_bias_relu_square():
    """D = relu(alpha*accum + beta*C + bias) ; E = D*D (row-broadcast bias,
    "Row and column broadcasts"; squared second output, "Multiple Outputs")."""
    g = Dag()
    acc = g.accum()
    t0 = g.mul(g.scalar(0), acc)
    t1 = g.mul(g.scalar(1), g.load(0))
    t2 = g.add(t0, t1)
    t3 = g.add(t2, g.broadcast(1))
    d = g.relu(t3)
    e = g.mul(d, d)
    g.store(d, 0)
    g.store(e, 1)
    return g.nodes


def dag_relu_aux_store():
    """F = accum*alpha + C*2.0 ; D = relu(F) ; returns D, F (cell [6]); the
    constant 2.0 is passed as scalar slot 1."""
    g = Dag()
    acc = g.accum()
    f = g.add(g.mul(acc, g.scalar(0)), g.mul(g.load(0), g.scalar(1)))
    d = g.relu(f)
    g.store(d, 0)
    g.store(f, 1)
    return g.nodes


def dag_relu_scale_return_acc():
    """F = relu(accum*alpha + C*beta) ; D = F*scale ; returns D, F, accum
    (cell [7]; accum is stored as fp32)."""
    g = Dag()
    acc = g.accum()
    f = g.relu(g.add(g.mul(acc, g.scalar(0)), g.mul(g.load(0), g.scalar(1))))
    d = g.mul(f, g.scalar(2))
    g.store(d, 0)
    g.store(f, 1)
    g.store(acc, 2)
    return g.nodes


def dag_row_bias():
    """D = accum*alpha + row_bias (cell [9], row part)."""
    g = Dag()
    acc = g.accum()
    d = g.add(g.mul(acc, g.scalar(0)), g.broadcast(0))
    g.store(d, 0)
    return g.nodes


def dag_add_square():
    """d = accum + c ; d_squared = d*d ("Multiple Outputs", first two)."""
    g = Dag()
    d = g.add(g.accum(), g.load(0))
    g.store(d, 0)
    g.store(g.mul(d, d), 1)
    return g.nodes


def dag_identity():
    """D = accum (a plain GEMM stored through the epilogue)."""
    g = Dag()
    g.store(g.accum(), 0)
    return g.nodes


def dag_row_col_bias():
    """D = (accum*alpha) + row_bias + col_bias ("Custom epilogue fusions for
    GEMMs", cell [9]: row bias (N,) and column bias (M, 1) in one epilogue)."""
    g = Dag()
    acc = g.accum()
    t = g.add(g.mul(acc, g.scalar(0)), g.broadcast(0))
    g.store(g.add(t, g.col_broadcast(1)), 0)
    return g.nodes


def dag_aux_normalize():
    """D = accum / aux ("Defining an epilogue via a Python function",
    aux_normalize)."""
    g = Dag()
    g.store(g.div(g.accum(), g.load(0)), 0)
    return g.nodes


def dag_scale_shift():
    """tmp = accum*2.0 ; tmp2 = tmp - 1.0 ; D = tmp2 / 4.0 ; returns D, tmp
    (the computation of the SSA failure example, cell [12], written with a new
    name for the second assignment as single assignment requires)."""
    g = Dag()
    tmp = g.mul(g.accum(), g.scalar(0))
    tmp2 = g.sub(tmp, g.scalar(1))
    g.store(g.div(tmp2, g.scalar(2)), 0)
    g.store(tmp, 1)
    return g.nodes


ACTIVATIONS = ["sigmoid", "tanh", "gelu", "silu", "hardswish", "leaky_relu"]


def dag_activation(act):
    """D = act(alpha*accum + C): one of the activations of the legacy
    interface's registry (gelu, hardswish, leaky_relu, sigmoid, silu, tanh;
    relu and identity have their own workloads).  leaky_relu takes its
    negative slope from scalar slot 1."""
    g = Dag()
    t = g.add(g.mul(g.accum(), g.scalar(0)), g.load(0))
    d = g.leaky_relu(t, g.scalar(1)) if act == "leaky_relu" else getattr(g, act)(t)
    g.store(d, 0)
    return g.nodes


def dag_complex():
    """result = (accum + bias)*scale + c + tanh(x) ; D = gelu(result)
    ("Custom Epilogue Example", section "Complex Expressions"; bias read as a
    row vector)."""
    g = Dag()
    r = g.mul(g.add(g.accum(), g.broadcast(2)), g.scalar(0))
    r = g.add(r, g.load(0))
    r = g.add(r, g.tanh(g.load(1)))
    g.store(g.gelu(r), 0)
    return g.nodes


def dag_clamp():
    """D = min(max(alpha*accum - C, lo), hi): subtraction and binary
    maximum/minimum ("Defining an epilogue via a Python function")."""
    g = Dag()
    t = g.sub(g.mul(g.scalar(0), g.accum()), g.load(0))
    t = g.maximum(t, g.scalar(1))
    g.store(g.minimum(t, g.scalar(2)), 0)
    return g.nodes


# ----------------------------------------------------------- workloads ----

def my_epilogue(L, M, N, K, seed=2025, name=None):
    return Workload(
        name=name or "my_epilogue_%dx%dx%dx%d" % (L, M, N, K), L=L, M=M, N=N, K=K, ab="f16",
        aux=[("C", "tensor", "f16")],
        scalars=[("alpha", 1.0), ("beta", 2.0), ("extra_scalar", 0.5)],
        outs=[("D", "f16"), ("Aux", "f16")], dag=dag_my_epilogue(), dist="randint",
        seed=seed, exact=True,
        cite="CUTLASS Operator API: Custom epilogue fusions for GEMMs, cells [2]-[5]")


# The five workloads of the pages' examples (shapes, types, seeds and epilogues
# as the workload table states them).
WORKLOADS = [
    my_epilogue(1, 128, 128, 128, name="my_epilogue_128"),
    my_epilogue(1, 1024, 1024, 1024, name="my_epilogue_1024"),
    Workload(
        name="relu_2400x3232x4096", L=1, M=2400, N=3232, K=4096, ab="f16",
        aux=[("C", "tensor", "f16")], scalars=[("alpha", 1.0), ("beta", 2.0)],
        outs=[("D", "f16")], dag=dag_relu_linear(), dist="ceil_uniform", seed=1234,
        exact=True,
        cite="CUTLASS Python examples walkthrough: basic GEMM notebook (2400x3232x4096, "
             "beta=2) and epilogue notebook (fused ReLU)"),
    Workload(
        name="alpha_beta_x_8192", L=1, M=8192, N=8192, K=8192, ab="f16",
        aux=[("C", "tensor", "f16"), ("X", "tensor", "f16")],
        scalars=[("alpha", 2.0), ("beta", 1.0), ("x_factor", 3.0)],
        outs=[("D", "f16"), ("Y", "f16")], dag=dag_alpha_beta_x(), dist="normal", seed=2026,
        exact=False, sample_rows=64,
        cite="Custom Epilogue Example: Basic Example: Alpha-Beta Scaling; Running the Example"),
    Workload(
        name="bias_relu_square_8x4096x4096x2048", L=8, M=4096, N=4096, K=2048, ab="bf16",
        aux=[("C", "tensor", "bf16"), ("bias", "row", "f32")],
        scalars=[("alpha", 0.5), ("beta", 1.0)],
        outs=[("D", "bf16"), ("E", "bf16")], dag=dag_bias_relu_square(), dist="normal",
        seed=2027, exact=False, sample_rows=64,
        cite="Custom Epilogue Fusions: Row and column broadcasts; Custom Epilogue Example: "
             "Activation Functions, Multiple Outputs"),
]

MY_EPILOGUE_128, MY_EPILOGUE_1024, RELU_2400X3232X4096, ALPHA_BETA_X_8192, BIAS_RELU_SQUARE_L8 = \
    WORKLOADS

BY_NAME = {w.name: w for w in WORKLOADS}

# Tolerance for the non-integer workloads: |gpu - ref| <= ATOL + RTOL*|ref|,
# ref being the oracle's value rounded to the output type.
ATOL = 1e-2
RTOL = 1e-2


def page_examples(L=1, M=256, N=256, K=256):
    """Further epilogues printed on the pages, at a small size: integer inputs
    where the result is exact, N(0,1) inputs for the activations."""
    return [
        Workload(name="relu_aux_store", L=L, M=M, N=N, K=K, ab="f16",
                 aux=[("C", "tensor", "f16")], scalars=[("alpha", 3.0), ("two", 2.0)],
                 outs=[("D", "f16"), ("F", "f16")], dag=dag_relu_aux_store(), dist="randint",
                 seed=2025, exact=True, cite="Custom epilogue fusions for GEMMs, cell [6]"),
        Workload(name="relu_scale_return_acc", L=L, M=M, N=N, K=K, ab="f16",
                 aux=[("C", "tensor", "f16")],
                 scalars=[("alpha", 1.0), ("beta", 2.0), ("scale", 0.5)],
                 outs=[("D", "f16"), ("F", "f16"), ("accum", "f32")],
                 dag=dag_relu_scale_return_acc(), dist="randint", seed=2025, exact=True,
                 cite="Custom epilogue fusions for GEMMs, cell [7]"),
        Workload(name="string_epilogue_beta_half", L=L, M=M, N=N, K=K, ab="f16",
                 aux=[("C", "tensor", "f16")], scalars=[("alpha", 1.0), ("beta", 0.5)],
                 outs=[("D", "f16"), ("F", "f16")], dag=dag_relu_aux_store(), dist="randint",
                 seed=2025, exact=True, cite="Custom epilogue fusions for GEMMs, cell [8]"),
        Workload(name="row_bias_f16", L=L, M=M, N=N, K=K, ab="f16",
                 aux=[("row_bias", "row", "f16")], scalars=[("alpha", 1.0)],
                 outs=[("D", "f16")], dag=dag_row_bias(), dist="randint", seed=2025,
                 exact=True, cite="Custom epilogue fusions for GEMMs, cell [9] (row part)"),
        Workload(name="add_square_bf16", L=L, M=M, N=N, K=K, ab="bf16",
                 aux=[("c", "tensor", "bf16")], scalars=[],
                 outs=[("d", "bf16"), ("d_squared", "bf16")], dag=dag_add_square(),
                 dist="randint", seed=2025, exact=True,
                 cite="Custom Epilogue Example: Multiple Outputs"),
        Workload(name="identity_f32_out", L=L, M=M, N=N, K=K, ab="f16", aux=[], scalars=[],
                 outs=[("D", "f32")], dag=dag_identity(), dist="ceil_uniform", seed=1234,
                 exact=True, cite="Python examples walkthrough: basic GEMM (f32 accumulate)"),
        Workload(name="row_col_bias_f16", L=L, M=M, N=N, K=K, ab="f16",
                 aux=[("row_bias", "row", "f16"), ("col_bias", "col", "f16")],
                 scalars=[("alpha", 1.0)], outs=[("D", "f16")], dag=dag_row_col_bias(),
                 dist="randint", seed=2025, exact=True,
                 cite="Custom epilogue fusions for GEMMs, cell [9]"),
        Workload(name="aux_normalize_f16", L=L, M=M, N=N, K=K, ab="f16",
                 aux=[("aux", "tensor", "f16", "pow2")], scalars=[], outs=[("D", "f16")],
                 dag=dag_aux_normalize(), dist="randint", seed=2025, exact=True,
                 cite="Defining an epilogue via a Python function: aux_normalize"),
        Workload(name="scale_shift_bf16", L=L, M=M, N=N, K=K, ab="bf16", aux=[],
                 scalars=[("two", 2.0), ("one", 1.0), ("four", 4.0)],
                 outs=[("D", "f32"), ("tmp", "bf16")], dag=dag_scale_shift(), dist="randint",
                 seed=2025, exact=True,
                 cite="Custom epilogue fusions for GEMMs, cell [12] (computation only)"),
        Workload(name="clamp_f16", L=L, M=M, N=N, K=K, ab="f16", aux=[("C", "tensor", "f16")],
                 scalars=[("alpha", 1.0), ("lo", -3.0), ("hi", 5.5)], outs=[("D", "f16")],
                 dag=dag_clamp(), dist="randint", seed=2025, exact=True,
                 cite="Defining an epilogue via a Python function: binary min and max"),
    ] + [
        Workload(name="act_" + act, L=L, M=M, N=N, K=K, ab="f16", aux=[("C", "tensor", "f16")],
                 scalars=[("alpha", 0.25)] + ([("slope", 0.1)] if act == "leaky_relu" else []),
                 outs=[("D", "f16")], dag=dag_activation(act), dist="normal", seed=2028,
                 exact=False,
                 cite="Python examples walkthrough: epilogue notebook, activation registry")
        for act in ACTIVATIONS
    ] + [
        Workload(name="complex_gelu_tanh", L=L, M=M, N=N, K=K, ab="bf16",
                 aux=[("c", "tensor", "bf16"), ("x", "tensor", "bf16"), ("bias", "row", "f32")],
                 scalars=[("scale", 0.125)], outs=[("D", "bf16")], dag=dag_complex(),
                 dist="normal", seed=2029, exact=False,
                 cite="Custom Epilogue Example: Complex Expressions"),
    ]


# ---------------------------------------------------------- generators ----

def _normal(gen, shape, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(TORCH_DTYPE[dtype])


def make_inputs(w: Workload):
    """Seeded host tensors ``(A, B, aux_list, scalars)`` for a workload.

    * ``randint``: integers from {-2,...,2} drawn with torch's CPU generator
      (high end exclusive, as torch.randint(-2, 3, ...) on the page);
    * ``ceil_uniform``: numpy RandomState, ceil(uniform(-4, 4) cast to fp16),
      the basic-GEMM notebook's recipe;
    * ``normal``: N(0, 1) from torch's CPU generator, rounded to the type.
    Operands are drawn in the order A, B, then the aux slots; aux slots marked
    "pow2" (divisors) are then redrawn from +-{1, 2, 4}.
    """
    L, M, N, K = w.L, w.M, w.N, w.K
    shapes = [(L, M, K), (L, K, N)]
    for spec in w.aux:
        shapes.append({"tensor": (L, M, N), "row": (N,), "col": (M,)}[spec[1]])
    dts = [w.ab, w.ab] + [spec[2] for spec in w.aux]
    out = []
    if w.dist == "randint":
        g = torch.Generator().manual_seed(w.seed)
        for shp, dt in zip(shapes, dts):
            out.append(torch.randint(-2, 3, shp, generator=g, dtype=torch.float32)
                       .to(TORCH_DTYPE[dt]))
    elif w.dist == "ceil_uniform":
        rs = np.random.RandomState(w.seed)
        for shp, dt in zip(shapes, dts):
            v = np.ceil(rs.uniform(-4.0, 4.0, size=shp).astype(np.float16))
            out.append(torch.from_numpy(v.astype(np.float32)).to(TORCH_DTYPE[dt]))
    elif w.dist == "normal":
        g = torch.Generator().manual_seed(w.seed)
        for shp, dt in zip(shapes, dts):
            out.append(_normal(g, shp, dt))
    else:
        raise ValueError(w.dist)
    A, B = out[0].contiguous(), out[1].contiguous()
    aux = [t.contiguous() for t in out[2:]]
    # divisor operands ("pow2"): nonzero powers of two, +-{1, 2, 4}, so a
    # division by them is exact in every precision
    g2 = torch.Generator().manual_seed(w.seed + 1)
    for k, spec in enumerate(w.aux):
        if len(spec) > 3 and spec[3] == "pow2":
            mag = torch.pow(2.0, torch.randint(0, 3, aux[k].shape, generator=g2).float())
            sgn = torch.randint(0, 2, aux[k].shape, generator=g2).float() * 2 - 1
            aux[k] = (mag * sgn).to(aux[k].dtype).contiguous()
    scalars = [float(v) for _, v in w.scalars]
    return A, B, aux, scalars


def sample_rows(w: Workload, per_batch: Optional[int] = None, seed: int = 7):
    """Seeded sample of flattened output rows ``l*M + i`` (sorted), ``per_batch``
    rows from every batch; always includes the first and last row of each batch
    so the ragged last M tile is covered."""
    per = per_batch or w.sample_rows
    if per is None or per >= w.M:
        return np.arange(w.L * w.M, dtype=np.int64)
    rs = np.random.RandomState(seed)
    rows = []
    for l in range(w.L):
        pick = set(rs.choice(w.M, size=per - 2, replace=False).tolist())
        pick.update([0, w.M - 1])
        rows.extend(sorted(l * w.M + i for i in pick))
    return np.asarray(rows, dtype=np.int64)


def to_codes(t: torch.Tensor) -> np.ndarray:
    """Host tensor -> numpy array the oracle takes (uint16 codes or float32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


# ---------------------------------------------------------- grouped GEMM ---

@dataclass
class GroupedWorkload:
    """Independent problems of different sizes sharing one epilogue, its types
    and its scalars.  Per problem: A (M,K), B (K,N), Load tensors and
    outputs (M,N), row vectors (N,), column vectors (M,)."""
    name: str
    problems: List[Tuple[int, int, int]]      # (M, N, K)
    ab: str
    aux: List[tuple]                          # as Workload.aux
    scalars: List[Tuple[str, float]]
    outs: List[Tuple[str, str]]
    dag: List[Tuple[str, int, int, int]]
    dist: str                                 # "randint3" or "randint" or "normal"
    seed: int
    exact: bool
    cite: str = ""

    def flops(self) -> float:
        return float(sum(2 * m * n * k for m, n, k in self.problems))

    def alg_bytes(self) -> int:
        b = 0
        for m, n, k in self.problems:
            b += (m * k + k * n) * ESIZE[self.ab]
            for spec in self.aux:
                b += {"tensor": m * n, "row": n, "col": m}[spec[1]] * ESIZE[spec[2]]
            for _, dt in self.outs:
                b += m * n * ESIZE[dt]
        return b

    def problem(self, g: int) -> Workload:
        """Problem g as a one-batch Workload (same epilogue and types)."""
        m, n, k = self.problems[g]
        return Workload(name="%s[%d]" % (self.name, g), L=1, M=m, N=n, K=k, ab=self.ab,
                        aux=self.aux, scalars=self.scalars, outs=self.outs, dag=self.dag,
                        dist=self.dist, seed=self.seed, exact=self.exact, cite=self.cite)


def generate_problem_sizes(count, seed=2023, sizes=(128, 256, 512, 1024)):
    """M, N, K of each problem drawn in that order from ``sizes`` with Python's
    ``random`` seeded once (the grouped-GEMM notebook's generate_problems)."""
    import random
    rng = random.Random(seed)
    return [tuple(rng.choice(sizes) for _ in range(3)) for _ in range(count)]


def grouped_workloads():
    """The grouped-GEMM notebook's batch (50 problems, fp16, values from
    {-3,...,2}, D = A @ B written as alpha*accum + beta*C with alpha 1 and
    beta 0, the interface's defaults) and a custom epilogue over ragged
    problems ("Combine custom epilogues with grouped operations")."""
    g = Dag()
    t = g.add(g.mul(g.accum(), g.scalar(0)), g.mul(g.load(0), g.scalar(1)))
    g.store(t, 0)
    linear = g.nodes
    g = Dag()
    t = g.add(g.add(g.mul(g.accum(), g.scalar(0)), g.load(0)), g.broadcast(1))
    g.store(g.relu(t), 0)
    g.store(t, 1)
    bias_relu = g.nodes
    ragged = [(72, 136, 200), (264, 520, 64), (200, 8, 1000), (1, 256, 128), (520, 392, 136),
              (129, 264, 72), (384, 1032, 520), (8, 8, 8), (300, 24, 64), (1024, 128, 1024),
              (513, 392, 8), (136, 136, 136)]
    return [
        GroupedWorkload(name="grouped_gemm_50", problems=generate_problem_sizes(50), ab="f16",
                        aux=[("C", "tensor", "f16")], scalars=[("alpha", 1.0), ("beta", 0.0)],
                        outs=[("D", "f16")], dag=linear, dist="randint3", seed=2023, exact=True,
                        cite="Python interface walkthrough, example three: Grouped GEMM"),
        GroupedWorkload(name="grouped_bias_relu_ragged", problems=ragged, ab="bf16",
                        aux=[("C", "tensor", "bf16"), ("bias", "row", "f32")],
                        scalars=[("alpha", 0.5)], outs=[("D", "bf16"), ("T", "f32")],
                        dag=bias_relu, dist="randint", seed=2030, exact=True,
                        cite="Custom Epilogue Example, Next Steps: grouped operations"),
    ]


GROUPED_BY_NAME = {w.name: w for w in grouped_workloads()}


def make_grouped_inputs(w: GroupedWorkload):
    """Seeded host tensors ``(As, Bs, auxs, scalars)``: per problem, in problem
    order, A, B, then its aux slots, all from one torch CPU generator.

    * ``randint3``: integers from {-3,...,2} (torch.randint(-3, 3, ...) as in
      the grouped-GEMM notebook's initialize);
    * ``randint``: integers from {-2,...,2};
    * ``normal``: N(0, 1) rounded to the type.
    """
    g = torch.Generator().manual_seed(w.seed)

    def draw(shp, dt):
        if w.dist == "randint3":
            return torch.randint(-3, 3, shp, generator=g, dtype=torch.float32).to(TORCH_DTYPE[dt])
        if w.dist == "randint":
            return torch.randint(-2, 3, shp, generator=g, dtype=torch.float32).to(TORCH_DTYPE[dt])
        if w.dist == "normal":
            return _normal(g, shp, dt)
        raise ValueError(w.dist)

    As, Bs, auxs = [], [], []
    for m, n, k in w.problems:
        As.append(draw((m, k), w.ab).contiguous())
        Bs.append(draw((k, n), w.ab).contiguous())
        auxs.append([draw({"tensor": (m, n), "row": (n,), "col": (m,)}[spec[1]], spec[2])
                     .contiguous() for spec in w.aux])
    scalars = [float(v) for _, v in w.scalars]
    return As, Bs, auxs, scalars
