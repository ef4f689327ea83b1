/*
 * CPU fp64 attention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the checker, not the product.  Only the test suite, the smoke
 * entry point and the CPU-baseline / reference legs of the benchmark load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (plain definition, fp64 throughout, no intermediate
 * rounding).  For batch b, query head h, query row i, with G = Hq / Hkv and
 * kv head g = floor(h / G):
 *
 *   s_j   = scale * sum_d Q[b,h,i,d] * K[b,g,j,d]      for j in V(i)
 *   V(i)  = {0 .. Nk-1}                  (non-causal)
 *         = {0 .. min(i, Nk-1)}          (causal, aligned at row 0)
 *   M     = max_j s_j,   Z = sum_j exp(s_j - M)
 *   LSE   = M + ln Z                      (natural log, scale included)
 *   O[d]  = sum_j exp(s_j - M) / Z * V[b,g,j,d]
 *
 * Sources: "FlashAttention-3 vs Triton Kernels" (dailyaiworld), intro -- the
 * FlashAttention result is the softmax attention output, computed without
 * materialising the N x N score matrix, i.e. the same numbers as the plain
 * definition; the (batch, heads, seq, head_dim) layout comes from the
 * benchmark listing in its "Benchmarking Triton vs FlashAttention-3" section.
 * The smzdm digest, section 5 ("Attention cannot be split like GEMM") fixes
 * how partial results over key shards recombine: each shard carries its
 * output and an lse_i state and the combine renormalises through them; adding
 * raw partial outputs is wrong because the softmax denominators differ.
 * The PyTorch autoWS design note, "How the compiler does it", names the
 * "correction" role, i.e. the running max / sum rescale of online softmax.
 *
 * Inputs are bf16 bit patterns (uint16).  bf16 is the top half of an IEEE
 * binary32, so widening to double is exact.
 *
 * Three formulations are provided:
 *   oracle_attn_rows         the two-pass definition above (what GPU results
 *                            are compared against);
 *   oracle_attn_rows_online  running max / sum with rescale over key blocks
 *                            (the online-softmax recurrence), fp64;
 *   oracle_attn_rows_split   key axis cut into nsplit chunks, each giving a
 *                            normalised partial O_c and lse_c, recombined by
 *                            log-sum-exp weights.
 * The last two exist to pin the algebra of the method against the first.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const uint16_t *q, *k, *v;
  int64_t B, Hq, Hkv, Nq, Nk, D;
  int causal;
  double scale;
  const int64_t *rows;
  int64_t nrows;
  double *out_o, *out_lse;
  /* formulation selector and its parameter */
  int mode; /* 0 two-pass, 1 online, 2 split, 3 split partials only */
  int64_t param;
  double *part_o, *part_lse; /* mode 3 outputs [nrows, nsplit, D] and [nrows, nsplit] */
  int64_t row_begin, row_end;
  int status;
} job_t;

static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Number of keys visible to query row i. */
static int64_t visible_keys(const job_t *jb, int64_t i) {
  if (!jb->causal) return jb->Nk;
  return (i + 1 < jb->Nk) ? (i + 1) : jb->Nk;
}

/* Scores s_j = scale * <q_i, k_j> for j in [0, n).  q is the widened row. */
static void scores(const job_t *jb, const double *qrow, const uint16_t *kbase, int64_t n,
                   double *s) {
  const int64_t D = jb->D;
  for (int64_t j = 0; j < n; ++j) {
    const uint16_t *kr = kbase + j * D;
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d) acc += qrow[d] * bf16_to_double(kr[d]);
    s[j] = jb->scale * acc;
  }
}

/* Two-pass definition over keys [j0, j1): returns lse and writes the
 * normalised output into o (length D).  Empty range -> lse = -inf, o = 0. */
static double two_pass_range(const job_t *jb, const double *s, const uint16_t *vbase, int64_t j0,
                             int64_t j1, double *o) {
  const int64_t D = jb->D;
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  if (j1 <= j0) return -INFINITY;
  double M = -INFINITY;
  for (int64_t j = j0; j < j1; ++j)
    if (s[j] > M) M = s[j];
  double Z = 0.0;
  for (int64_t j = j0; j < j1; ++j) Z += exp(s[j] - M);
  for (int64_t j = j0; j < j1; ++j) {
    const double w = exp(s[j] - M) / Z;
    const uint16_t *vr = vbase + j * D;
    for (int64_t d = 0; d < D; ++d) o[d] += w * bf16_to_double(vr[d]);
  }
  return M + log(Z);
}

/* Online softmax: keys visited in blocks of `block`; running max m, running
 * denominator l and unnormalised accumulator acc are rescaled by
 * exp(m_old - m_new) whenever the max grows. */
static double online_range(const job_t *jb, const double *s, const uint16_t *vbase, int64_t n,
                           int64_t block, double *o, double *acc) {
  const int64_t D = jb->D;
  double m = -INFINITY, l = 0.0;
  for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
  for (int64_t j0 = 0; j0 < n; j0 += block) {
    const int64_t j1 = (j0 + block < n) ? (j0 + block) : n;
    double bm = -INFINITY;
    for (int64_t j = j0; j < j1; ++j)
      if (s[j] > bm) bm = s[j];
    const double m_new = (bm > m) ? bm : m;
    const double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
    l *= alpha;
    for (int64_t d = 0; d < D; ++d) acc[d] *= alpha;
    for (int64_t j = j0; j < j1; ++j) {
      const double p = exp(s[j] - m_new);
      l += p;
      const uint16_t *vr = vbase + j * D;
      for (int64_t d = 0; d < D; ++d) acc[d] += p * bf16_to_double(vr[d]);
    }
    m = m_new;
  }
  for (int64_t d = 0; d < D; ++d) o[d] = acc[d] / l;
  return m + log(l);
}

/* Log-sum-exp recombination of nsplit normalised partial states. */
static double combine_states(const double *po, const double *plse, int64_t nsplit, int64_t D,
                             double *o) {
  double mx = -INFINITY;
  for (int64_t c = 0; c < nsplit; ++c)
    if (plse[c] > mx) mx = plse[c];
  double sum = 0.0;
  for (int64_t c = 0; c < nsplit; ++c)
    if (plse[c] != -INFINITY) sum += exp(plse[c] - mx);
  const double L = mx + log(sum);
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int64_t c = 0; c < nsplit; ++c) {
    if (plse[c] == -INFINITY) continue;
    const double w = exp(plse[c] - L);
    for (int64_t d = 0; d < D; ++d) o[d] += w * po[c * D + d];
  }
  return L;
}

static void *worker(void *arg) {
  job_t *jb = (job_t *)arg;
  const int64_t D = jb->D, Nk = jb->Nk, Nq = jb->Nq, Hq = jb->Hq, Hkv = jb->Hkv;
  const int64_t G = Hq / Hkv;
  double *qrow = (double *)malloc(sizeof(double) * D);
  double *s = (double *)malloc(sizeof(double) * (Nk > 0 ? Nk : 1));
  double *tmp = (double *)malloc(sizeof(double) * D);
  const int64_t nsplit = (jb->mode >= 2) ? jb->param : 1;
  double *po = (double *)malloc(sizeof(double) * D * nsplit);
  double *plse = (double *)malloc(sizeof(double) * nsplit);
  if (!qrow || !s || !tmp || !po || !plse) {
    jb->status = -1;
    goto done;
  }
  for (int64_t r = jb->row_begin; r < jb->row_end; ++r) {
    const int64_t flat = jb->rows[r];
    const int64_t i = flat % Nq;
    const int64_t bh = flat / Nq;
    const int64_t h = bh % Hq;
    const int64_t b = bh / Hq;
    const int64_t g = h / G;
    const uint16_t *qr = jb->q + flat * D;
    for (int64_t d = 0; d < D; ++d) qrow[d] = bf16_to_double(qr[d]);
    const uint16_t *kbase = jb->k + (b * Hkv + g) * Nk * D;
    const uint16_t *vbase = jb->v + (b * Hkv + g) * Nk * D;
    const int64_t n = visible_keys(jb, i);
    scores(jb, qrow, kbase, n, s);
    double *o = (jb->mode == 3) ? tmp : jb->out_o + r * D;
    double lse;
    if (jb->mode == 0) {
      lse = two_pass_range(jb, s, vbase, 0, n, o);
    } else if (jb->mode == 1) {
      lse = online_range(jb, s, vbase, n, jb->param, o, tmp);
    } else {
      /* chunk c covers keys [c*C, (c+1)*C) of the full key axis, C = ceil(Nk/nsplit),
       * intersected with the visible set V(i). */
      const int64_t C = (Nk + nsplit - 1) / nsplit;
      for (int64_t c = 0; c < nsplit; ++c) {
        int64_t j0 = c * C, j1 = (c + 1) * C;
        if (j1 > n) j1 = n;
        if (j0 > n) j0 = n;
        plse[c] = two_pass_range(jb, s, vbase, j0, j1, po + c * D);
      }
      if (jb->mode == 3) {
        memcpy(jb->part_o + r * nsplit * D, po, sizeof(double) * nsplit * D);
        memcpy(jb->part_lse + r * nsplit, plse, sizeof(double) * nsplit);
        lse = 0.0;
      } else {
        lse = combine_states(po, plse, nsplit, D, o);
      }
    }
    if (jb->out_lse) jb->out_lse[r] = lse;
  }
done:
  free(qrow);
  free(s);
  free(tmp);
  free(po);
  free(plse);
  return NULL;
}

static int run(job_t proto, int nthreads) {
  if (!proto.q || !proto.k || !proto.v || !proto.rows) return -1;
  if (proto.mode != 3 && (!proto.out_o || !proto.out_lse)) return -1;
  if (proto.B <= 0 || proto.Hq <= 0 || proto.Hkv <= 0 || proto.Nq <= 0 || proto.Nk <= 0 ||
      proto.D <= 0 || proto.Hq % proto.Hkv != 0)
    return -2;
  for (int64_t r = 0; r < proto.nrows; ++r)
    if (proto.rows[r] < 0 || proto.rows[r] >= proto.B * proto.Hq * proto.Nq) return -3;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > proto.nrows) nthreads = proto.nrows > 0 ? (int)proto.nrows : 1;
  job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return -4;
  }
  const int64_t per = (proto.nrows + nthreads - 1) / nthreads;
  int rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].row_begin = t * per < proto.nrows ? t * per : proto.nrows;
    jobs[t].row_end = (t + 1) * per < proto.nrows ? (t + 1) * per : proto.nrows;
    jobs[t].status = 0;
    if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) {
      worker(&jobs[t]);
      tids[t] = 0;
    }
  }
  for (int t = 0; t < nthreads; ++t) {
    if (tids[t]) pthread_join(tids[t], NULL);
    if (jobs[t].status) rc = jobs[t].status;
  }
  free(jobs);
  free(tids);
  return rc;
}

#define PROTO_INIT                                                                              \
  job_t p;                                                                                      \
  memset(&p, 0, sizeof p);                                                                      \
  p.q = q; p.k = k; p.v = v; p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = Nq; p.Nk = Nk; p.D = D;    \
  p.causal = causal; p.scale = scale; p.rows = rows; p.nrows = nrows; p.out_o = out_o;          \
  p.out_lse = out_lse;

/* Two-pass definition for the listed query rows.  rows[r] is the flat index
 * (b*Hq + h)*Nq + i; out_o is [nrows, D], out_lse is [nrows]. */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                     int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D, int causal,
                     double scale, const int64_t *rows, int64_t nrows, double *out_o,
                     double *out_lse, int nthreads) {
  PROTO_INIT
  p.mode = 0;
  return run(p, nthreads);
}

/* Online-softmax formulation, keys visited in blocks of `block`. */
int oracle_attn_rows_online(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                            int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                            int causal, double scale, const int64_t *rows, int64_t nrows,
                            int64_t block, double *out_o, double *out_lse, int nthreads) {
  if (block < 1) return -2;
  PROTO_INIT
  p.mode = 1;
  p.param = block;
  return run(p, nthreads);
}

/* Split-KV formulation: nsplit chunks of ceil(Nk/nsplit) keys, recombined
 * through their log-sum-exp states. */
int oracle_attn_rows_split(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                           int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D, int causal,
                           double scale, const int64_t *rows, int64_t nrows, int64_t nsplit,
                           double *out_o, double *out_lse, int nthreads) {
  if (nsplit < 1) return -2;
  PROTO_INIT
  p.mode = 2;
  p.param = nsplit;
  return run(p, nthreads);
}

/* The per-chunk partial states of the split formulation, without combining:
 * part_o [nrows, nsplit, D] (each normalised by its own denominator) and
 * part_lse [nrows, nsplit] (-inf for a chunk with no visible key). */
int oracle_attn_rows_partials(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                              int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                              int causal, double scale, const int64_t *rows, int64_t nrows,
                              int64_t nsplit, double *part_o, double *part_lse, int nthreads) {
  if (nsplit < 1 || !part_o || !part_lse) return -2;
  double *out_o = NULL, *out_lse = NULL;
  PROTO_INIT
  p.mode = 3;
  p.param = nsplit;
  p.part_o = part_o;
  p.part_lse = part_lse;
  return run(p, nthreads);
}

/* FP8 E4M3 ("fn" flavour of the OCP 8-bit floating-point format, the
 * low-precision tensor-core input the FlashAttention-3 page names):
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
 * holds subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN.  Every such
 * value has at most 4 significant bits and an exponent in [-9, 8], so it is
 * exactly a bf16 value: out[i] gets those bf16 bits.  Returns -3 (and stops)
 * at a NaN code, 0 otherwise. */
int oracle_e4m3_to_bf16(const uint8_t *in, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    const unsigned sign = in[i] >> 7, e = (in[i] >> 3) & 15u, m = in[i] & 7u;
    if (e == 15u && m == 7u) return -3;
    const double mag = (e == 0u) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    const float f = (float)(sign ? -mag : mag);
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    out[i] = (uint16_t)(u >> 16);
  }
  return 0;
}

/* Log-sum-exp combine of partial states: part_o [nrows, nsplit, D],
 * part_lse [nrows, nsplit] -> out_o [nrows, D], out_lse [nrows]. */
int oracle_combine(const double *part_o, const double *part_lse, int64_t nrows, int64_t nsplit,
                   int64_t D, double *out_o, double *out_lse) {
  if (!part_o || !part_lse || !out_o || !out_lse || nsplit < 1 || D < 1) return -2;
  for (int64_t r = 0; r < nrows; ++r)
    out_lse[r] = combine_states(part_o + r * nsplit * D, part_lse + r * nsplit, nsplit, D,
                                out_o + r * D);
  return 0;
}
