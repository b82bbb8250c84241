"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (a dropped term, a wrong sign or index, a transposed
or mis-batched operand, a wrong rounding rule).  The mutated copies are built
in a temporary directory and run in a child process; the real oracle is
untouched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = [
    ("dropped_add_term", "case ORC_ADD: v[n] = v[nd->a] + v[nd->b];",
     "case ORC_ADD: v[n] = v[nd->a];"),
    ("add_sign", "case ORC_ADD: v[n] = v[nd->a] + v[nd->b];",
     "case ORC_ADD: v[n] = v[nd->a] - v[nd->b];"),
    ("mul_as_add", "case ORC_MUL: v[n] = v[nd->a] * v[nd->b];",
     "case ORC_MUL: v[n] = v[nd->a] + v[nd->b];"),
    ("relu_abs", "v[nd->a] > 0.0 ? v[nd->a] : 0.0", "v[nd->a] > 0.0 ? v[nd->a] : -v[nd->a]"),
    ("relu_keeps_neg_zero", "v[nd->a] > 0.0 ? v[nd->a] : 0.0",
     "v[nd->a] >= 0.0 ? v[nd->a] : 0.0"),
    ("scalar_slot", "v[n] = jb->scalars[nd->slot];", "v[n] = jb->scalars[0];"),
    ("k_skips_first", "for (int64_t k = 0; k < K; ++k) {\n      const double a = arow[k];",
     "for (int64_t k = 1; k < K; ++k) {\n      const double a = arow[k];"),
    ("B_row_shift", "const double *brow = jb->Bd + k * N;",
     "const double *brow = jb->Bd + ((k + 1) % K) * N;"),
    ("A_ignores_batch", "arow[k] = decode(jb->ab_type, jb->A, (l * M + i) * K + k);",
     "arow[k] = decode(jb->ab_type, jb->A, i * K + k);"),
    ("aux_ignores_batch", "jb->aux[nd->slot], (l * M + i) * N + j);",
     "jb->aux[nd->slot], i * N + j);"),
    ("broadcast_by_row", "case ORC_BCAST: v[n] = decode(jb->aux_type[nd->slot], jb->aux[nd->slot], j);",
     "case ORC_BCAST: v[n] = decode(jb->aux_type[nd->slot], jb->aux[nd->slot], i % N);"),
    ("ties_away", "if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;",
     "if (d >= 0.5) r += 1.0;"),
    ("truncate", "if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;", ""),
    ("f16_exponent_bias", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);"),
    ("bf16_subnormal_scale", "v = ldexp((double)f, -133);", "v = ldexp((double)f, -134);"),
    ("bf16_as_f16_layout", "return round_to_code(x, 7, 8);", "return round_to_code(x, 8, 7);"),
    ("subnormal_threshold", "if (ax < ldexp(1.0, emin)) {", "if (ax < ldexp(1.0, emin - 1)) {"),
    ("f32_store_via_f16", "default: ((float *)base)[idx] = (float)v; break;",
     "default: ((float *)base)[idx] = (float)orc_f16_to_f64(orc_f64_to_f16(v)); break;"),
    ("sub_operands_swapped", "case ORC_SUB: v[n] = v[nd->a] - v[nd->b];",
     "case ORC_SUB: v[n] = v[nd->b] - v[nd->a];"),
    ("div_operands_swapped", "case ORC_DIV: v[n] = v[nd->a] / v[nd->b];",
     "case ORC_DIV: v[n] = v[nd->b] / v[nd->a];"),
    ("min_as_max", "case ORC_MIN: v[n] = v[nd->b] < v[nd->a] ? v[nd->b] : v[nd->a];",
     "case ORC_MIN: v[n] = v[nd->b] > v[nd->a] ? v[nd->b] : v[nd->a];"),
    ("max_returns_first", "case ORC_MAX: v[n] = v[nd->b] > v[nd->a] ? v[nd->b] : v[nd->a];",
     "case ORC_MAX: v[n] = v[nd->a];"),
    ("col_broadcast_by_column",
     "case ORC_COLBCAST: v[n] = decode(jb->aux_type[nd->slot], jb->aux[nd->slot], i);",
     "case ORC_COLBCAST: v[n] = decode(jb->aux_type[nd->slot], jb->aux[nd->slot], j % M);"),
    ("sigmoid_sign", "case ORC_SIGMOID: v[n] = 1.0 / (1.0 + exp(-v[nd->a]));",
     "case ORC_SIGMOID: v[n] = 1.0 / (1.0 + exp(v[nd->a]));"),
    ("tanh_half_argument", "case ORC_TANH: v[n] = tanh(v[nd->a]);",
     "case ORC_TANH: v[n] = 2.0 / (1.0 + exp(-v[nd->a])) - 1.0;"),
    ("gelu_without_sqrt", "erfc(-v[nd->a] / sqrt(2.0))", "erfc(-v[nd->a] / 2.0)"),
    ("gelu_cancels_tail", "0.5 * v[nd->a] * erfc(-v[nd->a] / sqrt(2.0));",
     "0.5 * v[nd->a] * (1.0 + erf(v[nd->a] / sqrt(2.0)));"),
    ("silu_sign", "case ORC_SILU: v[n] = v[nd->a] / (1.0 + exp(-v[nd->a]));",
     "case ORC_SILU: v[n] = v[nd->a] / (1.0 + exp(v[nd->a]));"),
    ("hardswish_clamp_3", "c = c < 0.0 ? 0.0 : (c > 6.0 ? 6.0 : c);",
     "c = c < 0.0 ? 0.0 : (c > 3.0 ? 3.0 : c);"),
    ("accum_drops_last_column", "memcpy(jb->acc_rows + out_row * N, acc, sizeof(double) * (size_t)N);",
     "memcpy(jb->acc_rows + out_row * N, acc, sizeof(double) * (size_t)(N - 1));"),
    ("accum_row_by_job_index", "memcpy(jb->acc_rows + out_row * N, acc,",
     "memcpy(jb->acc_rows + t * N, acc,"),
    ("leaky_side", "case ORC_LEAKY_RELU: v[n] = v[nd->a] > 0.0 ? v[nd->a] : v[nd->b] * v[nd->a];",
     "case ORC_LEAKY_RELU: v[n] = v[nd->a] < 0.0 ? v[nd->a] : v[nd->b] * v[nd->a];"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, "mutation site for %s not found in oracle.c" % name
    mutated = source.replace(old, new, 1)
    (tmp_path / "oracle.c").write_text(mutated)
    with open(os.path.join(ROOT, "oracle", "oracle.h")) as f:
        (tmp_path / "oracle.h").write_text(f.read())
    lib = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", str(tmp_path / "oracle.c"), "-o", lib, "-lm"], check=True)
    code = ("import sys; sys.path[:0] = [%r, %r]; import _pins; f = _pins.run_all(%r); "
            "print('\\n'.join(f)); sys.exit(1 if f else 0)" % (ROOT, os.path.join(ROOT, "tests"), lib))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s passed every pin:\n%s%s" % (name, r.stdout, r.stderr)
