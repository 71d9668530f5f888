/*
 * CPU oracle for the low-bit draft head -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow statement of what the draft head computes, written from the module docstring
 * and code of "radiance_drafthead.py" (the 2-bit MTP draft head page). Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg load this library; the product path never
 * does. It shares no code, header, table or helper with the CUDA library.
 *
 * Precision: the quantiser is fp32 exactly as the page evaluates it (torch eager fp32 ops,
 * torch.round = half-to-even, bf16 casts round to nearest even); everything after it is fp64.
 * Build with -ffp-contract=off so no multiply-add is fused.
 *
 * Steps, each following the page:
 *   orc_quantize_pack   asymmetric min/max quantiser, quarter-split (int2) or half-split (int4)
 *   orc_quantize_pack_f32  the same on fp32 rows (an FP8 head's scaled e4m3 values)
 *                       packing, premultiplied scale S and zero term ZS
 *                       (the load-time quantiser; module docstring on the quarter-split packing).
 *   orc_coarse          c[m,n] = sum_gi ( S*P_gi - ZS*XS_gi ), P_gi = sum_k x_k (1 + v_k/beta),
 *                       XS_gi = sum_k x_k  (module docstring on the hoisted bit-pattern dequant,
 *                       and the int2 coarse kernel), beta = 4 (int2) or 16 (int4).
 *   orc_coarse_dequant  the same value written as a dot with dequantised weights,
 *                       sum_k x_k ((S/beta) v_k - (ZS - S)), used as a self-check of the fold.
 *   orc_block_topk      per 64-row block, the KCAND largest coarse values (block candidate emission).
 *   orc_global_topr     the R largest of a row's block candidates (head application).
 *   orc_rerank          exact logit sum_k x_k W[n,k] for the selected rows (exact rerank).
 *   orc_argmax          the argmax the caller takes over the reranked logits.
 *   orc_exact_logits    brute force: the exact logit of every vocab row.
 * Ties: selections order by (value descending, row id ascending); the argmax takes the lowest id.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BLOCK 64 /* BLOCK_N: width of one candidate block */

/* ---- bf16 <-> fp32 -------------------------------------------------------------------- */
static float bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* fp32 -> bf16, round to nearest, ties to even (what .to(torch.bfloat16) does). */
static uint16_t float_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* ---- a tiny thread pool: split [0, n) into contiguous ranges ----------------------------- */
typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct {
  range_fn fn;
  void* ctx;
  int64_t lo, hi;
} range_job;

static void* range_trampoline(void* p) {
  range_job* j = (range_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < nthreads) nthreads = (int)(n > 0 ? n : 1);
  if (nthreads == 1) {
    fn(ctx, 0, n);
    return;
  }
  pthread_t th[256];
  range_job jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t lo = (int64_t)t * per, hi = lo + per;
    if (hi > n) hi = n;
    jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].lo = lo; jobs[t].hi = hi < lo ? lo : hi;
    if (pthread_create(&th[t], NULL, range_trampoline, &jobs[t]) != 0) {
      fn(ctx, jobs[t].lo, jobs[t].hi); /* run inline if a thread cannot start */
      jobs[t].fn = NULL;
    } else {
      ++started;
    }
  }
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].fn) pthread_join(th[t], NULL);
  (void)started;
}

/* ---- quantise + pack ------------------------------------------------------------------ */
/*
 * Per vocab row n and group gi (k in [gi*G, gi*G+G)), with w = float(W[n,k]):
 *   lo, hi = min, max over the group
 *   sc = (hi - lo) / lv, then sc = max(sc, 1e-8)           lv = 2^bits - 1
 *   zp = round(-lo / sc) clamped to [0, lv]                round = half to even
 *   q  = round(w / sc + zp) clamped to [0, lv]
 *   S  = bf16(bias * sc),  ZS = bf16(bias * sc + zp * sc)  bias = 4 (int2) or 16 (int4)
 * Packing, int2 (Q = K/4): byte j = q[j] | q[Q+j] << 2 | q[2Q+j] << 4 | q[3Q+j] << 6.
 * Packing, int4 (H = K/2): byte j = q[j] | q[H+j] << 4.
 */
typedef struct {
  const uint16_t* W; /* bf16 rows, or */
  const float* Wf;   /* fp32 rows (an FP8 head's e4m3 values times the row scale) */
  int64_t K;
  int G, bits;
  uint8_t* packed;
  uint16_t *S, *ZS;
} quant_ctx;

static float wval(const quant_ctx* c, int64_t n, int64_t k) {
  return c->Wf ? c->Wf[n * c->K + k] : bf16_to_float(c->W[n * c->K + k]);
}

static void quant_rows(void* p, int64_t lo_row, int64_t hi_row) {
  quant_ctx* c = (quant_ctx*)p;
  const int64_t K = c->K;
  const int G = c->G;
  const int64_t ng = K / G;
  const float lv = (float)((1 << c->bits) - 1);
  const float bias = c->bits == 2 ? 4.0f : 16.0f;
  uint8_t* q = (uint8_t*)malloc((size_t)K);
  if (!q) return;
  for (int64_t n = lo_row; n < hi_row; ++n) {
    for (int64_t gi = 0; gi < ng; ++gi) {
      float lo = wval(c, n, gi * G), hi = lo;
      for (int t = 1; t < G; ++t) {
        float v = wval(c, n, gi * G + t);
        if (v < lo) lo = v;
        if (v > hi) hi = v;
      }
      float sc = (hi - lo) / lv;
      if (sc < 1e-8f) sc = 1e-8f; /* clamp(min=1e-8) */
      float zp = rintf(-lo / sc);
      if (zp < 0.0f) zp = 0.0f;
      if (zp > lv) zp = lv;
      for (int t = 0; t < G; ++t) {
        float v = wval(c, n, gi * G + t);
        float r = rintf(v / sc + zp);
        if (r < 0.0f) r = 0.0f;
        if (r > lv) r = lv;
        q[gi * G + t] = (uint8_t)r;
      }
      float s4 = bias * sc;
      float zs = zp * sc;
      c->S[n * ng + gi] = float_to_bf16(s4);
      c->ZS[n * ng + gi] = float_to_bf16(s4 + zs);
    }
    if (c->bits == 2) {
      const int64_t Q = K / 4;
      uint8_t* out = c->packed + n * Q;
      for (int64_t j = 0; j < Q; ++j)
        out[j] = (uint8_t)(q[j] | (q[Q + j] << 2) | (q[2 * Q + j] << 4) | (q[3 * Q + j] << 6));
    } else {
      const int64_t H = K / 2;
      uint8_t* out = c->packed + n * H;
      for (int64_t j = 0; j < H; ++j) out[j] = (uint8_t)(q[j] | (q[H + j] << 4));
    }
  }
  free(q);
}

int orc_quantize_pack(const uint16_t* W, int64_t N, int64_t K, int G, int bits, uint8_t* packed,
                      uint16_t* S, uint16_t* ZS, int nthreads) {
  if (!W || !packed || !S || !ZS) return -1;
  if (N <= 0 || K <= 0 || G <= 0 || (bits != 2 && bits != 4)) return -2;
  if (K % G) return -2;
  if (K % (8 / bits)) return -2;
  quant_ctx c = {W, NULL, K, G, bits, packed, S, ZS};
  parallel_for(N, nthreads, quant_rows, &c);
  return 0;
}

/* The same quantiser on fp32 rows: an FP8 head's values e4m3(b) * row_scale (page
 * "radiance_drafthead.py", the load-time quantiser on the FP8 head: the e4m3 values widened to
 * fp32 and multiplied by the row's scale, one fp32 multiply, done by the caller). */
int orc_quantize_pack_f32(const float* Wf, int64_t N, int64_t K, int G, int bits,
                          uint8_t* packed, uint16_t* S, uint16_t* ZS, int nthreads) {
  if (!Wf || !packed || !S || !ZS) return -1;
  if (N <= 0 || K <= 0 || G <= 0 || (bits != 2 && bits != 4)) return -2;
  if (K % G) return -2;
  if (K % (8 / bits)) return -2;
  quant_ctx c = {NULL, Wf, K, G, bits, packed, S, ZS};
  parallel_for(N, nthreads, quant_rows, &c);
  return 0;
}

/* ---- unpacking (the layout above, read back) ------------------------------------------- */
/* Code v of element k of a packed row. */
static int code_at(const uint8_t* row, int64_t K, int bits, int64_t k) {
  if (bits == 2) {
    const int64_t Q = K / 4;
    return (row[k % Q] >> (2 * (int)(k / Q))) & 3;
  }
  const int64_t H = K / 2;
  return (row[k % H] >> (4 * (int)(k / H))) & 15;
}

int orc_unpack_codes(const uint8_t* packed, int64_t N, int64_t K, int bits, uint8_t* codes) {
  if (!packed || !codes) return -1;
  if (bits != 2 && bits != 4) return -2;
  const int64_t rb = K * bits / 8;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) codes[n * K + k] = (uint8_t)code_at(packed + n * rb, K, bits, k);
  return 0;
}

/* ---- coarse value ----------------------------------------------------------------------- */
typedef struct {
  const uint16_t* x;
  int64_t M, K;
  const uint8_t* packed;
  const uint16_t *S, *ZS;
  int64_t N;
  int G, bits;
  double* out;
  int dequant_form;
} coarse_ctx;

static void coarse_rows(void* p, int64_t lo_row, int64_t hi_row) {
  coarse_ctx* c = (coarse_ctx*)p;
  const int64_t K = c->K, M = c->M, N = c->N;
  const int G = c->G;
  const int64_t ng = K / G;
  const int64_t rb = K * c->bits / 8;
  const double beta = c->bits == 2 ? 4.0 : 16.0;
  double* d = (double*)malloc(sizeof(double) * (size_t)K);  /* 1 + v/beta */
  int* v = (int*)malloc(sizeof(int) * (size_t)K);
  double* xv = (double*)malloc(sizeof(double) * (size_t)K);
  if (!d || !v || !xv) { free(d); free(v); free(xv); return; }
  for (int64_t n = lo_row; n < hi_row; ++n) {
    const uint8_t* row = c->packed + n * rb;
    for (int64_t k = 0; k < K; ++k) {
      v[k] = code_at(row, K, c->bits, k);
      d[k] = 1.0 + (double)v[k] / beta;
    }
    for (int64_t m = 0; m < M; ++m) {
      for (int64_t k = 0; k < K; ++k) xv[k] = (double)bf16_to_float(c->x[m * K + k]);
      double acc = 0.0;
      for (int64_t gi = 0; gi < ng; ++gi) {
        const double s = (double)bf16_to_float(c->S[n * ng + gi]);
        const double zs = (double)bf16_to_float(c->ZS[n * ng + gi]);
        if (c->dequant_form) {
          double dv = 0.0;
          for (int64_t k = gi * G; k < gi * G + G; ++k)
            dv += xv[k] * ((s / beta) * (double)v[k] - (zs - s));
          acc += dv;
        } else {
          double pg = 0.0, xs = 0.0;
          for (int64_t k = gi * G; k < gi * G + G; ++k) {
            pg += xv[k] * d[k];
            xs += xv[k];
          }
          acc += s * pg - zs * xs;
        }
      }
      c->out[m * N + n] = acc;
    }
  }
  free(d); free(v); free(xv);
}

static int coarse_common(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                         const uint16_t* S, const uint16_t* ZS, int64_t N, int G, int bits,
                         double* out, int nthreads, int dequant_form) {
  if (!x || !packed || !S || !ZS || !out) return -1;
  if (M <= 0 || N <= 0 || K <= 0 || G <= 0 || (bits != 2 && bits != 4) || K % G) return -2;
  coarse_ctx c = {x, M, K, packed, S, ZS, N, G, bits, out, dequant_form};
  parallel_for(N, nthreads, coarse_rows, &c);
  return 0;
}

int orc_coarse(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed, const uint16_t* S,
               const uint16_t* ZS, int64_t N, int G, int bits, double* out, int nthreads) {
  return coarse_common(x, M, K, packed, S, ZS, N, G, bits, out, nthreads, 0);
}

int orc_coarse_dequant(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                       const uint16_t* S, const uint16_t* ZS, int64_t N, int G, int bits,
                       double* out, int nthreads) {
  return coarse_common(x, M, K, packed, S, ZS, N, G, bits, out, nthreads, 1);
}

/* ---- selections ------------------------------------------------------------------------- */
typedef struct {
  double v;
  int32_t id;
} scored;

/* value descending, then id ascending */
static int by_value_then_id(const void* a, const void* b) {
  const scored* x = (const scored*)a;
  const scored* y = (const scored*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

/* Per row m and 64-row block b: the kcand largest c[m, n] for n in the block, descending.
 * Slots beyond the block's valid rows hold (-inf, -1). */
int orc_block_topk(const double* c, int64_t M, int64_t N, int kcand, double* cand_val,
                   int32_t* cand_id) {
  if (!c || !cand_val || !cand_id) return -1;
  if (M <= 0 || N <= 0 || kcand < 1 || kcand > ORC_BLOCK) return -2;
  const int64_t nblk = (N + ORC_BLOCK - 1) / ORC_BLOCK;
  scored buf[ORC_BLOCK];
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t b = 0; b < nblk; ++b) {
      int cnt = 0;
      for (int64_t n = b * ORC_BLOCK; n < N && n < (b + 1) * ORC_BLOCK; ++n) {
        buf[cnt].v = c[m * N + n];
        buf[cnt].id = (int32_t)n;
        ++cnt;
      }
      qsort(buf, (size_t)cnt, sizeof(scored), by_value_then_id);
      for (int s = 0; s < kcand; ++s) {
        const int64_t o = m * nblk * kcand + b * kcand + s;
        cand_val[o] = s < cnt ? buf[s].v : -INFINITY;
        cand_id[o] = s < cnt ? buf[s].id : -1;
      }
    }
  }
  return 0;
}

/* The R largest of each row's ncand candidates, descending (value, then id ascending). */
int orc_global_topr(const double* cand_val, const int32_t* cand_id, int64_t M, int64_t ncand,
                    int R, int32_t* rr_id, double* rr_val) {
  if (!cand_val || !cand_id || !rr_id || !rr_val) return -1;
  if (M <= 0 || ncand <= 0 || R < 1 || R > ncand) return -2;
  scored* buf = (scored*)malloc(sizeof(scored) * (size_t)ncand);
  if (!buf) return -1;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t i = 0; i < ncand; ++i) {
      buf[i].v = cand_val[m * ncand + i];
      buf[i].id = cand_id[m * ncand + i];
    }
    qsort(buf, (size_t)ncand, sizeof(scored), by_value_then_id);
    for (int j = 0; j < R; ++j) {
      rr_id[m * R + j] = buf[j].id;
      rr_val[m * R + j] = buf[j].v;
    }
  }
  free(buf);
  return 0;
}

/* ---- exact logits ----------------------------------------------------------------------- */
static double exact_dot(const uint16_t* xr, const uint16_t* wr, int64_t K) {
  double s = 0.0;
  for (int64_t k = 0; k < K; ++k) s += (double)bf16_to_float(xr[k]) * (double)bf16_to_float(wr[k]);
  return s;
}

/* e[m, j] = sum_k x[m,k] W[ids[m,j], k]; an id < 0 (an empty slot) scores -inf. */
int orc_rerank(const uint16_t* x, int64_t M, int64_t K, const uint16_t* W, int64_t N,
               const int32_t* ids, int R, double* e) {
  if (!x || !W || !ids || !e) return -1;
  if (M <= 0 || K <= 0 || N <= 0 || R < 1) return -2;
  for (int64_t m = 0; m < M; ++m)
    for (int j = 0; j < R; ++j) {
      const int32_t n = ids[m * R + j];
      if (n >= N) return -2;
      e[m * R + j] = n < 0 ? -INFINITY : exact_dot(x + m * K, W + (int64_t)n * K, K);
    }
  return 0;
}

/* out[m] = ids[m, j*] with e[m, j*] maximal; equal maxima go to the lowest id. */
int orc_argmax(const double* e, const int32_t* ids, int64_t M, int R, int32_t* out) {
  if (!e || !ids || !out) return -1;
  if (M <= 0 || R < 1) return -2;
  for (int64_t m = 0; m < M; ++m) {
    int best = -1;
    for (int j = 0; j < R; ++j) {
      if (ids[m * R + j] < 0) continue;
      if (best < 0 || e[m * R + j] > e[m * R + best] ||
          (e[m * R + j] == e[m * R + best] && ids[m * R + j] < ids[m * R + best]))
        best = j;
    }
    out[m] = best < 0 ? -1 : ids[m * R + best];
  }
  return 0;
}

typedef struct {
  const uint16_t* x;
  int64_t M, K;
  const uint16_t* W;
  int64_t N;
  double* out;
} exact_ctx;

static void exact_rows(void* p, int64_t lo, int64_t hi) {
  exact_ctx* c = (exact_ctx*)p;
  for (int64_t n = lo; n < hi; ++n)
    for (int64_t m = 0; m < c->M; ++m)
      c->out[m * c->N + n] = exact_dot(c->x + m * c->K, c->W + n * c->K, c->K);
}

/* Brute force: the exact logit of every vocab row. */
int orc_exact_logits(const uint16_t* x, int64_t M, int64_t K, const uint16_t* W, int64_t N,
                     double* out, int nthreads) {
  if (!x || !W || !out) return -1;
  if (M <= 0 || K <= 0 || N <= 0) return -2;
  exact_ctx c = {x, M, K, W, N, out};
  parallel_for(N, nthreads, exact_rows, &c);
  return 0;
}
