/*
 * oracle.c -- plain fp64 CPU oracle: batched GEMM + elementwise epilogue DAG.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h for what it computes and where the
 * pages define it).  Deliberately simple: a triple loop in i-k-j order with a
 * sequential sum over k, then the DAG evaluated node by node for every
 * element, then one round-to-nearest-even per store.  Rows are split across
 * POSIX threads; nothing else is reordered.
 */
#define _GNU_SOURCE
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* scalar codecs, from the format definitions                               */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent field 0: subnormal, value = fraction * 2^-24;
 * exponent field 31: inf (fraction 0) or NaN. */
double orc_f16_to_f64(uint16_t h) {
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24);
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
  return (h & 0x8000) ? -v : v;
}

/* bfloat16: sign bit, 8 exponent bits (bias 127), 7 fraction bits (the upper
 * half of an IEEE binary32). */
double orc_bf16_to_f64(uint16_t h) {
  int e = (h >> 7) & 0xff;
  int f = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)f, -133); /* f * 2^(1-127-7) */
  else if (e == 255)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
  return (h & 0x8000) ? -v : v;
}

/*
 * Round x to the nearest value of a binary format with `fb` fraction bits and
 * `eb` exponent bits, ties to even, and return its code.  Works in exact
 * double arithmetic: q below is a power of two, so x/q, floor and the
 * comparisons are all exact.
 */
static uint16_t round_to_code(double x, int fb, int eb) {
  const int bias = (1 << (eb - 1)) - 1;
  const int emin = 1 - bias; /* exponent of the smallest normal */
  const int emax = bias;     /* exponent of the largest finite binade */
  const uint32_t sign = signbit(x) ? (1u << (fb + eb)) : 0u;
  const uint32_t inf_code = sign | (((1u << eb) - 1u) << fb);
  if (isnan(x)) return (uint16_t)(inf_code | (1u << (fb - 1)));
  double ax = fabs(x);
  /* largest finite value is (2 - 2^-fb) * 2^emax; the halfway point to the
   * next (unrepresentable) binade value 2^(emax+1) already rounds to even,
   * i.e. to infinity */
  if (ax >= ldexp(2.0 - ldexp(1.0, -(fb + 1)), emax)) return (uint16_t)inf_code;
  int e; /* binade: 2^e <= ax < 2^(e+1); subnormals share the emin spacing */
  if (ax < ldexp(1.0, emin)) {
    e = emin;
  } else {
    (void)frexp(ax, &e);
    e -= 1;
  }
  const double q = ldexp(1.0, e - fb); /* spacing of representable values */
  const double m = ax / q;
  double r = floor(m);
  const double d = m - r;
  if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;
  /* normal: r = 2^fb + fraction, so ((e+bias-1) << fb) + r puts the biased
   * exponent e+bias in the exponent field (r == 2^(fb+1) carries into the
   * next binade); subnormal (e == emin): the exponent term is 0 and r is the
   * fraction, with r == 2^fb becoming the smallest normal. */
  uint32_t code = ((uint32_t)(e + bias - 1) << fb) + (uint32_t)r;
  return (uint16_t)(sign | code);
}

uint16_t orc_f64_to_f16(double x) { return round_to_code(x, 10, 5); }
uint16_t orc_f64_to_bf16(double x) { return round_to_code(x, 7, 8); }

void orc_f16_to_f64_array(const uint16_t *h, double *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f64(h[i]);
}
void orc_bf16_to_f64_array(const uint16_t *h, double *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(h[i]);
}
void orc_f64_to_f16_array(const double *x, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_f16(x[i]);
}
void orc_f64_to_bf16_array(const double *x, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(x[i]);
}

static double decode(int32_t type, const void *base, int64_t idx) {
  switch (type) {
    case ORC_F16: return orc_f16_to_f64(((const uint16_t *)base)[idx]);
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t *)base)[idx]);
    default: return (double)((const float *)base)[idx];
  }
}

static void encode(int32_t type, void *base, int64_t idx, double v) {
  switch (type) {
    case ORC_F16: ((uint16_t *)base)[idx] = orc_f64_to_f16(v); break;
    case ORC_BF16: ((uint16_t *)base)[idx] = orc_f64_to_bf16(v); break;
    default: ((float *)base)[idx] = (float)v; break; /* C conversion: nearest even */
  }
}

/* ------------------------------------------------------------------------ */
/* GEMM + DAG                                                               */
/* ------------------------------------------------------------------------ */

typedef struct {
  int64_t L, M, N, K;
  int32_t ab_type;
  const uint16_t *A;
  const double *Bd; /* B of the batch being processed, decoded: K*N */
  int64_t batch;    /* that batch */
  int32_t n_aux;
  const int32_t *aux_type;
  const void *const *aux;
  const double *scalars;
  int32_t n_nodes;
  const orc_node *nodes;
  const int32_t *out_type;
  void *const *outs;
  double *const *pre;
  int32_t n_out;
  double *acc_rows; /* orc_gemm_accum: destination, else NULL */
  const int64_t *rows;
  const int64_t *pos; /* positions in the caller's row list */
  int64_t count;      /* rows of this batch handled by the job */
  int status;
} job_t;

/* Decode rows [k0, k1) of B for one batch. */
typedef struct {
  const uint16_t *B;
  double *Bd;
  int32_t type;
  int64_t N, k0, k1;
} decode_job_t;

static void *decode_worker(void *p) {
  decode_job_t *d = (decode_job_t *)p;
  for (int64_t k = d->k0; k < d->k1; ++k)
    for (int64_t j = 0; j < d->N; ++j)
      d->Bd[k * d->N + j] = decode(d->type, d->B, k * d->N + j);
  return NULL;
}

static void *row_worker(void *p) {
  job_t *jb = (job_t *)p;
  const int64_t M = jb->M, N = jb->N, K = jb->K;
  double *arow = (double *)malloc(sizeof(double) * (size_t)K);
  double *acc = (double *)malloc(sizeof(double) * (size_t)N);
  if (!arow || !acc) {
    free(arow);
    free(acc);
    jb->status = ORC_NO_MEM;
    return NULL;
  }
  double v[64];
  for (int64_t t = 0; t < jb->count; ++t) {
    const int64_t r = jb->rows[t]; /* r = l*M + i */
    const int64_t i = r % M;
    const int64_t l = r / M;
    const int64_t out_row = jb->pos[t];
    /* accum[l,i,:] = sum_k A[l,i,k] * B[l,k,:], k ascending */
    for (int64_t k = 0; k < K; ++k) arow[k] = decode(jb->ab_type, jb->A, (l * M + i) * K + k);
    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = arow[k];
      const double *brow = jb->Bd + k * N;
      for (int64_t j = 0; j < N; ++j) acc[j] += a * brow[j];
    }
    if (jb->acc_rows) {
      memcpy(jb->acc_rows + out_row * N, acc, sizeof(double) * (size_t)N);
      continue;
    }
    /* the epilogue, element by element, node by node */
    for (int64_t j = 0; j < N; ++j) {
      for (int32_t n = 0; n < jb->n_nodes; ++n) {
        const orc_node *nd = &jb->nodes[n];
        switch (nd->op) {
          case ORC_ACCUM: v[n] = acc[j]; break;
          case ORC_LOAD:
            v[n] = decode(jb->aux_type[nd->slot], jb->aux[nd->slot], (l * M + i) * N + j);
            break;
          case ORC_BCAST: v[n] = decode(jb->aux_type[nd->slot], jb->aux[nd->slot], j); break;
          case ORC_COLBCAST: v[n] = decode(jb->aux_type[nd->slot], jb->aux[nd->slot], i); break;
          case ORC_SCALAR: v[n] = jb->scalars[nd->slot]; break;
          case ORC_MUL: v[n] = v[nd->a] * v[nd->b]; break;
          case ORC_ADD: v[n] = v[nd->a] + v[nd->b]; break;
          case ORC_SUB: v[n] = v[nd->a] - v[nd->b]; break;
          case ORC_DIV: v[n] = v[nd->a] / v[nd->b]; break;
          case ORC_MIN: v[n] = v[nd->b] < v[nd->a] ? v[nd->b] : v[nd->a]; break;
          case ORC_MAX: v[n] = v[nd->b] > v[nd->a] ? v[nd->b] : v[nd->a]; break;
          case ORC_SIGMOID: v[n] = 1.0 / (1.0 + exp(-v[nd->a])); break;
          case ORC_TANH: v[n] = tanh(v[nd->a]); break;
          /* 1 + erf(x/sqrt2) written as erfc(-x/sqrt2): the same number
           * without the cancellation that leaves 0 for x below about -8 */
          case ORC_GELU: v[n] = 0.5 * v[nd->a] * erfc(-v[nd->a] / sqrt(2.0)); break;
          case ORC_SILU: v[n] = v[nd->a] / (1.0 + exp(-v[nd->a])); break;
          case ORC_HARDSWISH: {
            const double x = v[nd->a];
            double c = x + 3.0;
            c = c < 0.0 ? 0.0 : (c > 6.0 ? 6.0 : c);
            v[n] = x * c / 6.0;
          } break;
          case ORC_LEAKY_RELU: v[n] = v[nd->a] > 0.0 ? v[nd->a] : v[nd->b] * v[nd->a]; break;
          case ORC_RELU: v[n] = v[nd->a] > 0.0 ? v[nd->a] : 0.0; break;
          case ORC_STORE:
            encode(jb->out_type[nd->slot], jb->outs[nd->slot], out_row * N + j, v[nd->a]);
            if (jb->pre && jb->pre[nd->slot]) jb->pre[nd->slot][out_row * N + j] = v[nd->a];
            v[n] = 0.0;
            break;
          default: break;
        }
      }
    }
  }
  free(arow);
  free(acc);
  return NULL;
}

static int check_type(int32_t t) { return t == ORC_F16 || t == ORC_BF16 || t == ORC_F32; }

static int validate_dag(int32_t n_nodes, const orc_node *nodes, int32_t n_aux, int32_t n_scalar,
                        int32_t n_out) {
  if (n_nodes <= 0 || n_nodes > 64 || !nodes) return ORC_BAD_DAG;
  for (int32_t n = 0; n < n_nodes; ++n) {
    const orc_node *nd = &nodes[n];
    switch (nd->op) {
      case ORC_ACCUM: break;
      case ORC_LOAD:
      case ORC_BCAST:
      case ORC_COLBCAST:
        if (nd->slot < 0 || nd->slot >= n_aux) return ORC_BAD_DAG;
        break;
      case ORC_SCALAR:
        if (nd->slot < 0 || nd->slot >= n_scalar) return ORC_BAD_DAG;
        break;
      case ORC_MUL:
      case ORC_ADD:
      case ORC_SUB:
      case ORC_DIV:
      case ORC_MIN:
      case ORC_MAX:
      case ORC_LEAKY_RELU:
        if (nd->b < 0 || nd->b >= n || nodes[nd->b].op == ORC_STORE) return ORC_BAD_DAG;
        /* fall through: operand a */
      case ORC_RELU:
      case ORC_SIGMOID:
      case ORC_TANH:
      case ORC_GELU:
      case ORC_SILU:
      case ORC_HARDSWISH:
        if (nd->a < 0 || nd->a >= n || nodes[nd->a].op == ORC_STORE) return ORC_BAD_DAG;
        break;
      case ORC_STORE:
        if (nd->a < 0 || nd->a >= n || nodes[nd->a].op == ORC_STORE) return ORC_BAD_DAG;
        if (nd->slot < 0 || nd->slot >= n_out) return ORC_BAD_DAG;
        break;
      default: return ORC_BAD_DAG;
    }
  }
  return ORC_OK;
}

static int default_threads(int32_t n_threads) {
  if (n_threads > 0) return n_threads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* Shared driver: batch by batch, decode B once, then split the rows of that
 * batch over the threads. */
static int run_rows(job_t *proto, const uint16_t *B, int64_t n_rows, const int64_t *rows,
                    int32_t n_threads) {
  const int64_t L = proto->L, M = proto->M, N = proto->N, K = proto->K;
  int64_t total = rows ? n_rows : L * M;
  int nt = default_threads(n_threads);
  for (int64_t t = 0; t < total; ++t) {
    int64_t r = rows ? rows[t] : t;
    if (r < 0 || r >= L * M) return ORC_BAD_ARGS;
  }
  int64_t *brow = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
  int64_t *bpos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
  double *Bd = (double *)malloc(sizeof(double) * (size_t)(K * N));
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
  job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nt);
  decode_job_t *djobs = (decode_job_t *)malloc(sizeof(decode_job_t) * (size_t)nt);
  int status = ORC_OK;
  if (!brow || !bpos || !Bd || !th || !jobs || !djobs) {
    status = ORC_NO_MEM;
    goto done;
  }
  for (int64_t l = 0; l < L && status == ORC_OK; ++l) {
    int64_t cnt = 0;
    for (int64_t t = 0; t < total; ++t) {
      int64_t r = rows ? rows[t] : t;
      if (r / M == l) {
        brow[cnt] = r;
        bpos[cnt] = t;
        ++cnt;
      }
    }
    if (cnt == 0) continue;
    /* decode B[l] */
    const uint16_t *Bl = B + l * K * N;
    for (int w = 0; w < nt; ++w) {
      djobs[w].B = Bl;
      djobs[w].Bd = Bd;
      djobs[w].type = proto->ab_type;
      djobs[w].N = N;
      djobs[w].k0 = K * w / nt;
      djobs[w].k1 = K * (w + 1) / nt;
      pthread_create(&th[w], NULL, decode_worker, &djobs[w]);
    }
    for (int w = 0; w < nt; ++w) pthread_join(th[w], NULL);
    /* rows of batch l */
    int used = 0;
    for (int w = 0; w < nt; ++w) {
      int64_t a = cnt * w / nt, b = cnt * (w + 1) / nt;
      if (b <= a) continue;
      jobs[used] = *proto;
      jobs[used].Bd = Bd;
      jobs[used].batch = l;
      jobs[used].rows = brow + a;
      jobs[used].pos = bpos + a;
      jobs[used].count = b - a;
      jobs[used].status = ORC_OK;
      pthread_create(&th[used], NULL, row_worker, &jobs[used]);
      ++used;
    }
    for (int w = 0; w < used; ++w) {
      pthread_join(th[w], NULL);
      if (jobs[w].status != ORC_OK) status = jobs[w].status;
    }
  }
done:
  free(brow);
  free(bpos);
  free(Bd);
  free(th);
  free(jobs);
  free(djobs);
  return status;
}

int orc_gemm_epilogue(int64_t L, int64_t M, int64_t N, int64_t K, int32_t ab_type,
                      const uint16_t *A, const uint16_t *B, int32_t n_aux,
                      const int32_t *aux_type, const void *const *aux, int32_t n_scalar,
                      const double *scalars, int32_t n_nodes, const orc_node *nodes,
                      int32_t n_out, const int32_t *out_type, void *const *outs,
                      double *const *pre, int64_t n_rows, const int64_t *rows,
                      int32_t n_threads) {
  if (L <= 0 || M <= 0 || N <= 0 || K <= 0 || !A || !B) return ORC_BAD_ARGS;
  if (ab_type != ORC_F16 && ab_type != ORC_BF16) return ORC_BAD_ARGS;
  if (n_aux < 0 || n_scalar < 0 || n_out <= 0 || !out_type || !outs) return ORC_BAD_ARGS;
  if (n_aux > 0 && (!aux || !aux_type)) return ORC_BAD_ARGS;
  if (n_scalar > 0 && !scalars) return ORC_BAD_ARGS;
  for (int32_t s = 0; s < n_aux; ++s)
    if (!check_type(aux_type[s]) || !aux[s]) return ORC_BAD_ARGS;
  for (int32_t o = 0; o < n_out; ++o)
    if (!check_type(out_type[o]) || !outs[o]) return ORC_BAD_ARGS;
  int st = validate_dag(n_nodes, nodes, n_aux, n_scalar, n_out);
  if (st != ORC_OK) return st;
  job_t proto;
  memset(&proto, 0, sizeof(proto));
  proto.L = L;
  proto.M = M;
  proto.N = N;
  proto.K = K;
  proto.ab_type = ab_type;
  proto.A = A;
  proto.n_aux = n_aux;
  proto.aux_type = aux_type;
  proto.aux = aux;
  proto.scalars = scalars;
  proto.n_nodes = n_nodes;
  proto.nodes = nodes;
  proto.out_type = out_type;
  proto.outs = outs;
  proto.pre = pre;
  proto.n_out = n_out;
  return run_rows(&proto, B, n_rows, rows, n_threads);
}

int orc_gemm_accum(int64_t L, int64_t M, int64_t N, int64_t K, int32_t ab_type,
                   const uint16_t *A, const uint16_t *B, double *acc, int64_t n_rows,
                   const int64_t *rows, int32_t n_threads) {
  if (L <= 0 || M <= 0 || N <= 0 || K <= 0 || !A || !B || !acc) return ORC_BAD_ARGS;
  if (ab_type != ORC_F16 && ab_type != ORC_BF16) return ORC_BAD_ARGS;
  job_t proto;
  memset(&proto, 0, sizeof(proto));
  proto.L = L;
  proto.M = M;
  proto.N = N;
  proto.K = K;
  proto.ab_type = ab_type;
  proto.A = A;
  proto.acc_rows = acc;
  return run_rows(&proto, B, n_rows, rows, n_threads);
}
