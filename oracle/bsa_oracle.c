/*
 * CPU oracle for block-sparse FP8 attention prefill over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, call or load this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Plain, slow and written to be checked by eye against the two pages it restates:
 *
 *   [QBSA]  "Quant Block Sparse Attention" (CANNBotDSL sample README)
 *             - 算子介绍: the formula  Q^_i = Q_i^fp8 * q_descale_i,  K^_j = K_j^fp8 * k_descale_j,
 *               V^_j = V_j^fp8 * v_descale_head(j),
 *               O_i = sum_{j in Omega_i} softmax_{j in Omega_i}(Q^_i K^_j^T * softmax_scale + mask_ij) V^_j
 *             - feature table: FP8 E4M3FN inputs, BF16 output, FP32 LSE, D = 128, block 128,
 *               mask_mode 3 = right-context causal, GQA with N1 % N2 == 0
 *             - 稀疏索引与 PA 页表: only the first sparse_seq_len indices are valid, logical
 *               blocks map through block_table to physical pages, a KV tail block shorter
 *               than 128 excludes its padding, an empty task gives O = 0 and LSE = -FLT_MAX
 *   [HPC]   "hpc-ops Block-Sparse FP8 Attention" (article)
 *             - 块稀疏调度: block_mask [B, N1, Qb, Kb], 128-token Q and KV tiles, 1 = compute
 *             - 活跃 tile 列表: the active KV tiles of a Q tile, written in order
 *             - 固定 P-scale 量化技巧: P is multiplied by a fixed scale (256) and quantised to
 *               e4m3 before the PV product; the epilogue undoes the scale together with the
 *               V descale; scores past the causal edge are -inf
 *
 * Two modes:
 *   ORACLE_EXACT (0): the formula itself in fp64 over the dequantised inputs.
 *   ORACLE_PEMU  (1): the tiled online softmax, one 128-token KV tile at a time in ascending
 *                     order, with P rounded to e4m3 at the fixed P-scale before the PV sum;
 *                     optionally two list tiles per step (the 256-wide macro block of
 *                     [QBSA]'s kernel description) or the list in slices merged by LSE.
 *
 * Readings taken where the pages leave a step open (each is listed in the design notes):
 *   causal edge j <= i + (kv_len - q_len); KV head of query head h is h / (N1/N2);
 *   pages are [P, N2, page_size, 128]; per-token K descale is [P, N2, page_size];
 *   a row with no visible key gets O = 0 and LSE = -FLT_MAX; LSE = natural log of the sum of
 *   exp over the scaled logits; P -> e4m3 rounds to nearest even and saturates to +-448;
 *   the running sum l uses the unrounded p.
 *
 * Parity pins live in tests/test_oracle_pins.py (brute-force dense attention, closed forms,
 * invariants, the exhaustive e4m3 table).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define TILE 128
#define HEAD_DIM 128

#define ORACLE_EXACT 0
#define ORACLE_PEMU 1

#define SCALE_PER_TENSOR 0
#define SCALE_PER_TOKEN_HEAD 1
#define SCALE_PER_HEAD 2

/* descale rules of the quantise step */
#define ORACLE_DESCALE_AMAX 0    /* amax / 448 */
#define ORACLE_DESCALE_UE8M0 1   /* amax / 448 rounded up to a power of two */

/* error codes returned by the oracle (data the pages call invalid) */
#define ORACLE_OK 0
#define ORACLE_BAD_INDEX 1       /* sparse index outside [0, Kb) or sparse_seq_len outside [0, Kb] */
#define ORACLE_BAD_PAGE 2        /* block_table entry outside [0, num_pages) for a needed token */
#define ORACLE_BAD_ARG 4

typedef struct {
  int B, N1, N2, D, page_size, max_q_len, max_kv_len, num_pages, max_pages_per_seq, total_q;
  int k_scale_kind, v_scale_kind, causal;
} oracle_dims_t;

typedef struct {
  const uint8_t *q;            /* [T, N1, 128] e4m3 */
  const uint8_t *k_pages;      /* [P, N2, ps, 128] e4m3 */
  const uint8_t *v_pages;      /* [P, N2, ps, 128] e4m3 */
  const float *q_descale;      /* [T, N1] */
  const float *k_descale;      /* [1] or [P, N2, ps] */
  const float *v_descale;      /* [1] or [N2] */
  const int *cu_seqlens_q;     /* [B + 1] */
  const int *seqused_kv;       /* [B] or NULL (kv_len = q_len) */
  const int *block_table;      /* [B, L] */
  const uint8_t *block_mask;   /* [B, N1, Qb, Kb] or NULL */
  const int *sparse_indices;   /* [B, N1, Qb, Kb] or NULL */
  const int *sparse_seq_len;   /* [B, N1, Qb] or NULL */
  double softmax_scale;
  double p_scale;
} oracle_inputs_t;

/* ------------------------------------------------------------------------------------
 * E4M3FN (OCP 8-bit floating point specification, v1.0): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448.
 * ------------------------------------------------------------------------------------ */
double oracle_e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 3) & 15;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);                /* subnormal: m/8 * 2^(1-7) */
  else
    v = ldexp(8.0 + (double)m, e - 10);      /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* Round-to-nearest-even with saturation to +-448 (NaN stays NaN). */
uint8_t oracle_e4m3_encode(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal quantum 2^-9; a result of 8 quanta is the smallest normal, code 0x08 */
    double r = nearbyint(ldexp(a, 9));
    return sign | (uint8_t)r;
  }
  int e;
  frexp(a, &e);                    /* a = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
  int ue = e - 1;
  double r = nearbyint(ldexp(a, 3 - ue));   /* in [8, 16] */
  if (r >= 16.0) { r = 8.0; ue += 1; }
  if (ue + 7 > 15 || (ue + 7 == 15 && r - 8.0 > 6.0)) return sign | 0x7E;
  return sign | (uint8_t)(((ue + 7) << 3) | ((int)r - 8));
}

/* ------------------------------------------------------------------------------------
 * Sequence geometry.
 * ------------------------------------------------------------------------------------ */
static int q_len_of(const oracle_inputs_t *in, int b) {
  return in->cu_seqlens_q[b + 1] - in->cu_seqlens_q[b];
}
static int kv_len_of(const oracle_inputs_t *in, int b) {
  return in->seqused_kv ? in->seqused_kv[b] : q_len_of(in, b);
}
static int cdiv(int a, int b) { return (a + b - 1) / b; }

/* Number of KV tiles that can hold a visible key for some row of Q tile qt: tiles at or past
 * it contribute exactly zero (causal edge, or past kv_len), so they are not in the list. */
int oracle_kend(const oracle_dims_t *d, const oracle_inputs_t *in, int b, int qt) {
  int ql = q_len_of(in, b), kl = kv_len_of(in, b);
  int Kb = cdiv(d->max_kv_len, TILE);
  if (qt * TILE >= ql) return 0;
  long lim = kl;                                          /* keys j < kv_len */
  if (d->causal) {
    int last_row = (qt * TILE + TILE < ql ? qt * TILE + TILE : ql) - 1;
    long c = (long)last_row + (kl - ql) + 1;              /* keys j <= last_row + off */
    if (c < lim) lim = c;
  }
  if (lim < 0) lim = 0;
  int ke = (int)((lim + TILE - 1) / TILE);
  return ke < Kb ? ke : Kb;
}

/* Canonical active-tile list of task (b, h, qt): ascending, no repeats, every tile < kend.
 * [HPC] 块稀疏调度 / 活跃 tile 列表; [QBSA] 稀疏索引与 PA 页表.
 * Returns the count, writes the tiles to list[0..count), and ORs data errors into *err. */
int oracle_active_tiles(const oracle_dims_t *d, const oracle_inputs_t *in, int b, int h, int qt,
                        int *list, int *err) {
  int Qb = cdiv(d->max_q_len, TILE);
  int Kb = cdiv(d->max_kv_len, TILE);
  int kend = oracle_kend(d, in, b, qt);
  int n = 0;
  size_t row = (((size_t)b * d->N1 + h) * Qb + qt) * (size_t)Kb;
  if (in->block_mask) {
    for (int t = 0; t < kend; ++t)
      if (in->block_mask[row + t] != 0) list[n++] = t;
  } else if (in->sparse_indices) {
    int len = in->sparse_seq_len[((size_t)b * d->N1 + h) * Qb + qt];
    if (len < 0 || len > Kb) { *err |= ORACLE_BAD_INDEX; len = len < 0 ? 0 : Kb; }
    char *sel = (char *)calloc((size_t)Kb + 1, 1);
    for (int e = 0; e < len; ++e) {
      int t = in->sparse_indices[row + e];
      if (t < 0 || t >= Kb) { *err |= ORACLE_BAD_INDEX; continue; }
      sel[t] = 1;
    }
    for (int t = 0; t < kend; ++t)
      if (sel[t]) list[n++] = t;
    free(sel);
  } else {
    for (int t = 0; t < kend; ++t) list[n++] = t;     /* dense path: no mask given */
  }
  return n;
}

/* All tasks at once: lists [B, N1, Qb, Kb] (entries past the count are -1), counts [B, N1, Qb]. */
int oracle_all_lists(const oracle_dims_t *d, const oracle_inputs_t *in, int *lists, int *counts) {
  int Qb = cdiv(d->max_q_len, TILE);
  int Kb = cdiv(d->max_kv_len, TILE);
  int err = 0;
  for (int b = 0; b < d->B; ++b)
    for (int h = 0; h < d->N1; ++h)
      for (int qt = 0; qt < Qb; ++qt) {
        size_t task = ((size_t)b * d->N1 + h) * Qb + qt;
        int *l = lists + task * Kb;
        for (int t = 0; t < Kb; ++t) l[t] = -1;
        counts[task] = oracle_active_tiles(d, in, b, h, qt, l, &err);
      }
  return err;
}

/* ------------------------------------------------------------------------------------
 * Dequantised operands ([QBSA] 算子介绍).
 * ------------------------------------------------------------------------------------ */
static int page_of(const oracle_dims_t *d, const oracle_inputs_t *in, int b, int j, int *err) {
  int pg = in->block_table[(size_t)b * d->max_pages_per_seq + j / d->page_size];
  if (pg < 0 || pg >= d->num_pages) { *err |= ORACLE_BAD_PAGE; return -1; }
  return pg;
}

static void dequant_q(const oracle_dims_t *d, const oracle_inputs_t *in, int tok, int h, double *qh) {
  const uint8_t *src = in->q + ((size_t)tok * d->N1 + h) * HEAD_DIM;
  double s = in->q_descale[(size_t)tok * d->N1 + h];
  for (int k = 0; k < HEAD_DIM; ++k) qh[k] = oracle_e4m3_decode(src[k]) * s;
}

static double k_descale_of(const oracle_dims_t *d, const oracle_inputs_t *in, int pg, int g, int slot) {
  if (d->k_scale_kind == SCALE_PER_TOKEN_HEAD)
    return in->k_descale[((size_t)pg * d->N2 + g) * d->page_size + slot];
  return in->k_descale[0];
}

static double v_descale_of(const oracle_dims_t *d, const oracle_inputs_t *in, int g) {
  return d->v_scale_kind == SCALE_PER_HEAD ? in->v_descale[g] : in->v_descale[0];
}

static const uint8_t *kv_row(const oracle_dims_t *d, const uint8_t *pages, int pg, int g, int slot) {
  return pages + (((size_t)pg * d->N2 + g) * d->page_size + slot) * HEAD_DIM;
}

/* ------------------------------------------------------------------------------------
 * The P-emulating online softmax over the active tiles tiles[t_lo .. t_hi) of one row, in
 * order, `group` consecutive list tiles per step (1: one 128-token tile at a time, [HPC]
 * 固定 P-scale; 2: the 256-wide macro block of [QBSA]'s kernel description, two sparse
 * 128-token blocks per step, an odd last tile alone): per step the running max m, alpha =
 * exp(m_old - m), p = exp(x - m) in fp32, l from the unrounded p, P * p_scale rounded to
 * e4m3 for the P.V sum.  keys [na] are the row's allowed keys in ascending order and s their
 * logits.  Returns (m, l, acc) with acc the un-normalised sum in P-scale units; m = -inf and
 * l = 0 when nothing is visible.
 * ------------------------------------------------------------------------------------ */
static int pemu_slice(const oracle_dims_t *d, const oracle_inputs_t *in, int b, int g,
                      const int *tiles, int t_lo, int t_hi, int group, const int *keys,
                      const double *s, int na, double *m_out, double *l_out, double *acc) {
  int err = 0;
  double m = -INFINITY, l = 0.0;
  for (int k = 0; k < HEAD_DIM; ++k) acc[k] = 0.0;
  int a = 0;
  for (int ti = t_lo; ti < t_hi; ti += group) {
    int t0 = tiles[ti] * TILE;
    int tl = tiles[(ti + group < t_hi ? ti + group : t_hi) - 1] * TILE;  /* the step's last tile */
    while (a < na && keys[a] < t0) ++a;              /* skip keys of earlier slices */
    int a0 = a;
    while (a < na && keys[a] < tl + TILE) ++a;       /* keys of this step's tiles: [a0, a) */
    double mt = -INFINITY;
    for (int e = a0; e < a; ++e) {
      double x = (double)(float)s[e];                /* the logit as a 32-bit float */
      if (x > mt) mt = x;
    }
    double mn = m > mt ? m : mt;
    if (mn == -INFINITY) continue;                   /* nothing visible yet */
    double alpha = (m == -INFINITY) ? 0.0 : exp(m - mn);
    double psum = 0.0;
    double tile_acc[HEAD_DIM];
    for (int k = 0; k < HEAD_DIM; ++k) tile_acc[k] = 0.0;
    for (int e = a0; e < a; ++e) {
      double x = (double)(float)s[e];
      double p = (double)(float)exp(x - mn);
      psum += p;
      uint8_t p8 = oracle_e4m3_encode((double)(float)(p * in->p_scale));
      double pq = oracle_e4m3_decode(p8);
      int j = keys[e];
      int pg = page_of(d, in, b, j, &err);
      if (pg < 0) continue;
      const uint8_t *vr = kv_row(d, in->v_pages, pg, g, j % d->page_size);
      for (int k = 0; k < HEAD_DIM; ++k) tile_acc[k] += pq * oracle_e4m3_decode(vr[k]);
    }
    l = alpha * l + psum;
    for (int k = 0; k < HEAD_DIM; ++k) acc[k] = alpha * acc[k] + tile_acc[k];
    m = mn;
  }
  *m_out = m;
  *l_out = l;
  return err;
}

/* ------------------------------------------------------------------------------------
 * One output row (token tok of sequence b, query head h).
 * ------------------------------------------------------------------------------------ */
static int one_row(const oracle_dims_t *d, const oracle_inputs_t *in, int mode, int splits,
                   int group, int tok, int h, double *o, double *lse) {
  int err = 0;
  int b = 0;
  while (b + 1 < d->B && in->cu_seqlens_q[b + 1] <= tok) ++b;
  int ql = q_len_of(in, b), kl = kv_len_of(in, b);
  int i = tok - in->cu_seqlens_q[b];                 /* row inside the sequence */
  int off = kl - ql;                                 /* right-context causal offset */
  int G = d->N1 / d->N2;
  int g = h / G;                                     /* KV head of query head h */
  int Kb = cdiv(d->max_kv_len, TILE);
  int qt = i / TILE;

  double qh[HEAD_DIM], kh[HEAD_DIM];
  dequant_q(d, in, tok, h, qh);
  double vd = v_descale_of(d, in, g);

  /* Omega: KV tiles enabled for this row's Q tile, in ascending order */
  int *tiles = (int *)malloc(sizeof(int) * (size_t)(Kb + 1));
  int nt = oracle_active_tiles(d, in, b, h, qt, tiles, &err);

  /* allowed keys A_i: j in an enabled tile, j < kv_len, j <= i + off (causal) */
  int nkeys = 0;
  for (int a = 0; a < nt; ++a) nkeys += TILE;
  int *keys = (int *)malloc(sizeof(int) * (size_t)(nkeys + 1));
  double *s = (double *)malloc(sizeof(double) * (size_t)(nkeys + 1));
  int na = 0;
  for (int a = 0; a < nt; ++a)
    for (int c = 0; c < TILE; ++c) {
      int j = tiles[a] * TILE + c;
      if (j >= kl) continue;
      if (d->causal && j > i + off) continue;
      keys[na++] = j;
    }

  /* s_ij = softmax_scale * <Q^_i, K^_j> */
  for (int a = 0; a < na; ++a) {
    int j = keys[a];
    int pg = page_of(d, in, b, j, &err);
    if (pg < 0) { s[a] = 0.0; continue; }
    const uint8_t *kr = kv_row(d, in->k_pages, pg, g, j % d->page_size);
    double kd = k_descale_of(d, in, pg, g, j % d->page_size);
    for (int k = 0; k < HEAD_DIM; ++k) kh[k] = oracle_e4m3_decode(kr[k]) * kd;
    double dot = 0.0;
    for (int k = 0; k < HEAD_DIM; ++k) dot += qh[k] * kh[k];
    s[a] = in->softmax_scale * dot;
  }

  for (int k = 0; k < HEAD_DIM; ++k) o[k] = 0.0;
  if (na == 0) {
    *lse = -FLT_MAX;                                 /* empty set: O = 0, LSE = -FLT_MAX */
  } else if (mode == ORACLE_EXACT) {
    double M = -INFINITY;
    for (int a = 0; a < na; ++a) if (s[a] > M) M = s[a];
    double l = 0.0;
    for (int a = 0; a < na; ++a) {
      int j = keys[a];
      int pg = page_of(d, in, b, j, &err);
      double w = exp(s[a] - M);
      l += w;
      if (pg < 0) continue;
      const uint8_t *vr = kv_row(d, in->v_pages, pg, g, j % d->page_size);
      for (int k = 0; k < HEAD_DIM; ++k) o[k] += w * oracle_e4m3_decode(vr[k]) * vd;
    }
    for (int k = 0; k < HEAD_DIM; ++k) o[k] /= l;
    *lse = M + log(l);
  } else {
    /* Tiled online softmax with P rounded to e4m3 at the fixed P-scale ([HPC] 固定 P-scale),
     * over the whole list, or over `splits` consecutive slices of it, each from m = -inf,
     * merged by their log-sum-exp weights (the split-KV step). */
    double m = -INFINITY, l = 0.0;
    double acc[HEAD_DIM];
    for (int k = 0; k < HEAD_DIM; ++k) acc[k] = 0.0;
    int ns = splits < 1 ? 1 : splits;
    for (int c = 0; c < ns; ++c) {
      double mc, lc, accc[HEAD_DIM];
      err |= pemu_slice(d, in, b, g, tiles, (int)((long)c * nt / ns), (int)((long)(c + 1) * nt / ns),
                        group, keys, s, na, &mc, &lc, accc);
      if (lc == 0.0 || mc == -INFINITY) continue;    /* an empty slice adds nothing */
      double mn = m > mc ? m : mc;
      double wo = (m == -INFINITY) ? 0.0 : exp(m - mn), wc = exp(mc - mn);
      l = wo * l + wc * lc;
      for (int k = 0; k < HEAD_DIM; ++k) acc[k] = wo * acc[k] + wc * accc[k];
      m = mn;
    }
    if (l == 0.0 || m == -INFINITY) {
      *lse = -FLT_MAX;
    } else {
      for (int k = 0; k < HEAD_DIM; ++k) o[k] = acc[k] * vd / (in->p_scale * l);
      *lse = m + log(l);
    }
  }
  free(tiles);
  free(keys);
  free(s);
  return err;
}

/* Rows given as (token, head) pairs; o [nrows, 128], lse [nrows].  In the P-emulating mode
 * the list is cut into `splits` slices and each slice steps `group` list tiles at a time.
 * Returns the OR of the data errors met.  nthreads <= 0 means the OpenMP default. */
int oracle_attention_rows_grouped(const oracle_dims_t *d, const oracle_inputs_t *in, int mode,
                                  int splits, int group, const int *rows, long nrows, double *o,
                                  double *lse, int nthreads) {
  if (!d || !in || d->D != HEAD_DIM || d->N2 <= 0 || d->N1 % d->N2 != 0) return ORACLE_BAD_ARG;
  if (mode == ORACLE_PEMU && !(in->p_scale > 0.0)) return ORACLE_BAD_ARG;
  if (group < 1) return ORACLE_BAD_ARG;
  int err = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16) reduction(| : err)
#endif
  for (long r = 0; r < nrows; ++r)
    err |= one_row(d, in, mode, splits, group, rows[2 * r], rows[2 * r + 1], o + r * HEAD_DIM,
                   lse + r);
  (void)nthreads;
  return err;
}

/* One 128-token tile per step. */
int oracle_attention_rows_split(const oracle_dims_t *d, const oracle_inputs_t *in, int mode,
                                int splits, const int *rows, long nrows, double *o, double *lse,
                                int nthreads) {
  return oracle_attention_rows_grouped(d, in, mode, splits, 1, rows, nrows, o, lse, nthreads);
}

/* The whole active list in one online softmax (splits = 1). */
int oracle_attention_rows(const oracle_dims_t *d, const oracle_inputs_t *in, int mode,
                          const int *rows, long nrows, double *o, double *lse, int nthreads) {
  return oracle_attention_rows_split(d, in, mode, 1, rows, nrows, o, lse, nthreads);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------------------
 * Quantisation into the attention inputs (the step before the attention call).
 *
 * The FlashMLA page (section 量化 / 解量化的源码实现) states the rule for one 128-element
 * tile: the scale is the tile's largest absolute value over 448 (the largest finite e4m3)
 * and the stored value is e4m3(x / scale).  The attention pages give Q per token per head,
 * K per token per head (or per tensor) and V per head (or per tensor) descales, i.e. the
 * same rule applied to each 128-element row of Q and K.  Readings: by default the scale is
 * not rounded (ORACLE_DESCALE_AMAX); with ORACLE_DESCALE_UE8M0 it is rounded up to a power of
 * two, FlashMLA's cast of the scale to UE8M0 (the same section: the smallest 2^k not below
 * amax / 448, so that multiplying a code by the scale is exact); an all-zero row gets descale
 * 1 and zero codes under either rule; both divisions are fp32 divisions (the precision of the
 * inputs' consumers); e4m3 rounds to nearest even and saturates (oracle_e4m3_encode).
 * ------------------------------------------------------------------------------------ */
static float bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* The smallest power of two not below x (x > 0, finite): frexpf writes x = m * 2^e with m in
 * [0.5, 1), so x is itself a power of two exactly when m = 0.5, and otherwise 2^e is the next
 * one up.  Subnormal x are handled by frexpf like any other. */
static float pow2_ceil(float x) {
  int e;
  float m = frexpf(x, &e);
  return m == 0.5f ? x : ldexpf(1.0f, e);
}

/* One row of 128 bf16 values -> 128 codes; returns the row's descale. */
static float quantize_row(const uint16_t *x, uint8_t *codes, int rule) {
  float amax = 0.0f;
  for (int i = 0; i < HEAD_DIM; ++i) {
    float a = fabsf(bf16_value(x[i]));
    if (a > amax) amax = a;
  }
  float descale = amax > 0.0f ? amax / 448.0f : 1.0f;
  if (rule == ORACLE_DESCALE_UE8M0 && amax > 0.0f) descale = pow2_ceil(descale);
  for (int i = 0; i < HEAD_DIM; ++i) {
    float v = bf16_value(x[i]) / descale;
    codes[i] = oracle_e4m3_encode((double)v);
  }
  return descale;
}

/* x [rows, 128] bf16 -> codes [rows, 128] e4m3, descale [rows] (Q [T, N1, 128] gives the
 * q_descale layout [T, N1] directly); rule = ORACLE_DESCALE_AMAX or ORACLE_DESCALE_UE8M0. */
void oracle_quantize_rows(const uint16_t *x, long rows, int rule, uint8_t *codes,
                          float *descale) {
  for (long r = 0; r < rows; ++r)
    descale[r] = quantize_row(x + r * HEAD_DIM, codes + r * HEAD_DIM, rule);
}

/* Writes new K/V tokens into the paged cache.  Token i of sequence b (rows cu_new[b] + i of
 * k_new / v_new [T_new, N2, 128] bf16) lands at logical position pos = cache_len[b] + i, i.e.
 * page block_table[b, pos / page_size], slot pos % page_size of [P, N2, page_size, 128].
 * K: with SCALE_PER_TOKEN_HEAD each (token, head) row is quantised as above (under
 * k_descale_rule) and its descale stored in k_descale [P, N2, page_size]; with
 * SCALE_PER_TENSOR the codes are e4m3(x / k_scale)
 * with the caller's k_scale.  V: e4m3(x / v_scale[head]) (SCALE_PER_HEAD) or / v_scale[0].
 * A token whose page is missing or outside [0, num_pages) is skipped and reported. */
int oracle_append_kv(int B, int N2, int page_size, int num_pages, int max_pages_per_seq,
                     int k_scale_kind, int v_scale_kind, int k_descale_rule,
                     const uint16_t *k_new,
                     const uint16_t *v_new, const int *cu_new, const int *cache_len,
                     const int *block_table, const float *k_scale, const float *v_scale,
                     uint8_t *k_pages, uint8_t *v_pages, float *k_descale) {
  int err = 0;
  for (int b = 0; b < B; ++b) {
    int n = cu_new[b + 1] - cu_new[b];
    for (int i = 0; i < n; ++i) {
      long pos = (long)cache_len[b] + i;
      long lp = pos / page_size;
      int slot = (int)(pos % page_size);
      int pg = lp < max_pages_per_seq ? block_table[(size_t)b * max_pages_per_seq + lp] : -1;
      if (pg < 0 || pg >= num_pages) {
        err |= ORACLE_BAD_PAGE;
        continue;
      }
      for (int g = 0; g < N2; ++g) {
        size_t src = ((size_t)(cu_new[b] + i) * N2 + g) * HEAD_DIM;
        size_t row = ((size_t)pg * N2 + g) * page_size + slot;
        if (k_scale_kind == SCALE_PER_TOKEN_HEAD) {
          k_descale[row] = quantize_row(k_new + src, k_pages + row * HEAD_DIM, k_descale_rule);
        } else {
          for (int e = 0; e < HEAD_DIM; ++e)
            k_pages[row * HEAD_DIM + e] =
                oracle_e4m3_encode((double)(bf16_value(k_new[src + e]) / k_scale[0]));
        }
        float vs = v_scale_kind == SCALE_PER_HEAD ? v_scale[g] : v_scale[0];
        for (int e = 0; e < HEAD_DIM; ++e)
          v_pages[row * HEAD_DIM + e] = oracle_e4m3_encode((double)(bf16_value(v_new[src + e]) / vs));
      }
    }
  }
  return err;
}
