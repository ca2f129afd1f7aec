/*
 * CPU oracle for the tensor-parallel overlap GEMMs.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this file's library.  It shares no code, header or table with the CUDA path.
 *
 * Everything here is the plain definition, written out as loops in double
 * precision over the already-rounded inputs (bf16 or e4m3 values widened
 * exactly to double):
 *
 *  - ring arrival order.  In TransformerEngine's atomic_gemm_overlap_ag
 *    (issue "curious about atomic_gemm_overlap_ag", the C++ listing of
 *    CommOverlapP2PBase::atomic_gemm_overlap_ag) every ring step sends a chunk
 *    to the next rank and receives one from the previous rank.  A rank
 *    therefore holds its own chunk at step 0 and, at step s, the chunk that
 *    started on rank (self - s) mod tp.
 *  - all-gather.  The gathered buffer is the row concatenation of the ranks'
 *    chunks in rank order (the listing's comment: the all-gather output must be
 *    contiguous in every rank after the ring exchanges).
 *  - AG+GEMM.  Y = G . W^T with G the gathered rows (the listing's TN GEMM of
 *    the gathered buffer against the weight, m = output features, n = gathered
 *    rows); for FP8 inputs the product carries both per-tensor scale_inv
 *    factors (the gathered input keeps B.scale_inv()).
 *  - GEMM+reduce-scatter / row-parallel linear + all-reduce.  Each rank holds a
 *    K-slice X_r, W_r; the result is sum_r X_r . W_r^T (nvFuser PR "Reference
 *    implementation for Linear+Allreduce with overlapping": a matmul of each
 *    input chunk with the weight shard transposed followed by an all-reduce
 *    SUM; TransformerEngine PR "Comm+GEMM overlap API updated to support
 *    cuBlasMp backend": GEMM followed by reduce-scatter).  Reduce-scatter hands
 *    rank b the row block b of that sum.
 *  - the same sum as a bf16 ring carries it.  The nvFuser PR's nsys trace runs
 *    the all-reduce as NCCL's bf16 ring kernel (AllReduce_Sum_bf16_RING_LL):
 *    every rank's partial X_r . W_r^T travels as bf16, and each hop adds the
 *    bf16 value it receives to its own bf16 partial in fp32 and sends the sum
 *    on rounded to bf16.  The ring visits the ranks of a row block in a fixed
 *    order that ends at the rank the block belongs to (reduce-scatter: block
 *    b sums ranks b+1, ..., b; the all-reduce of one row chunk is a
 *    reduce-scatter of its tp parts, part i ending at rank i).  Rounding is
 *    round-to-nearest-even throughout.
 *
 * The summation order inside the double loops is irrelevant at the tolerances
 * used: every product of two bf16 (or two e4m3) values is exact in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- decoding */

/* bf16: the upper 16 bits of an IEEE binary32. */
double oracle_decode_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* OCP FP8 E4M3 ("E4M3FN"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * subnormals at exponent 0, S.1111.111 is NaN, no infinities. */
double oracle_decode_e4m3(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 15;
  int f = c & 7;
  double v;
  if (e == 15 && f == 7) return NAN;
  if (e == 0)
    v = ldexp((double)f, -9); /* f/8 * 2^(1-7) */
  else
    v = ldexp(8.0 + f, e - 10); /* (1 + f/8) * 2^(e-7) */
  return sign ? -v : v;
}

static double g_e4m3[256];
static pthread_once_t g_once = PTHREAD_ONCE_INIT;
static void init_tables(void) {
  for (int i = 0; i < 256; ++i) g_e4m3[i] = oracle_decode_e4m3((uint8_t)i);
}

/* dtype codes: 0 = bf16 (uint16 bit patterns), 1 = e4m3 (uint8 codes) */
static inline double elem(int dtype, const void* base, int64_t idx) {
  if (dtype == 0) return oracle_decode_bf16(((const uint16_t*)base)[idx]);
  return g_e4m3[((const uint8_t*)base)[idx]];
}

/* ------------------------------------------------------------ ring, gather */

/* Order in which rank `self` comes to hold the tp chunks: step s -> rank. */
int oracle_ring_order(int tp, int self, int* out) {
  if (tp < 1 || self < 0 || self >= tp) return 1;
  for (int s = 0; s < tp; ++s) out[s] = ((self - s) % tp + tp) % tp;
  return 0;
}

/* Row concatenation of the tp chunks (each rows_per_rank x row_bytes bytes). */
int oracle_gather(int tp, int64_t rows_per_rank, int64_t row_bytes, const void* const* x, void* out) {
  if (tp < 1) return 1;
  int64_t chunk = rows_per_rank * row_bytes;
  for (int r = 0; r < tp; ++r)
    for (int64_t i = 0; i < chunk; ++i) ((uint8_t*)out)[(int64_t)r * chunk + i] = ((const uint8_t*)x[r])[i];
  return 0;
}

/* The gathered buffer as rank `self` holds it after ring step `step`:
 * chunks of the ranks reached at steps 0..step sit in their rank-order slot,
 * every other byte keeps the value `sentinel`. */
int oracle_staging_after_step(int tp, int self, int step, int64_t rows_per_rank, int64_t row_bytes,
                              const void* const* x, uint8_t sentinel, void* out) {
  if (tp < 1 || self < 0 || self >= tp || step < -1 || step >= tp) return 1;
  int64_t chunk = rows_per_rank * row_bytes;
  memset(out, sentinel, (size_t)(chunk * tp));
  int order[64];
  if (tp > 64 || oracle_ring_order(tp, self, order)) return 1;
  for (int s = 0; s <= step; ++s) {
    int r = order[s];
    memcpy((uint8_t*)out + (int64_t)r * chunk, x[r], (size_t)chunk);
  }
  return 0;
}

/* ------------------------------------------------------------- products */

typedef struct {
  int kind;            /* 0: AG product, 1: K-split sum */
  int dtype;
  int tp;
  int64_t k;           /* AG: contraction length; K-split: per-rank slice length */
  int64_t m;
  const void* g;       /* AG: gathered X [n, k] */
  const void* w;       /* AG: W [m, k] */
  const void* const* xs; /* K-split: tp x [n, k] */
  const void* const* ws; /* K-split: tp x [m, k] */
  double scale;        /* AG FP8: sx * sw; else 1 */
  int64_t ntiles, th, tw;
  const int64_t* r0;
  const int64_t* c0;
  double* out;         /* ntiles x th x tw */
  int64_t next;        /* work counter (tile-row items) */
  pthread_mutex_t mu;
} work_t;

static void do_item(work_t* w, int64_t item) {
  int64_t t = item / w->th, rr = item % w->th;
  int64_t i = w->r0[t] + rr;
  double* o = w->out + (t * w->th + rr) * w->tw;
  for (int64_t cc = 0; cc < w->tw; ++cc) {
    int64_t c = w->c0[t] + cc;
    double acc = 0.0;
    if (w->kind == 0) {
      for (int64_t q = 0; q < w->k; ++q)
        acc += elem(w->dtype, w->g, i * w->k + q) * elem(w->dtype, w->w, c * w->k + q);
      acc *= w->scale;
    } else {
      for (int r = 0; r < w->tp; ++r)
        for (int64_t q = 0; q < w->k; ++q)
          acc += elem(w->dtype, w->xs[r], i * w->k + q) * elem(w->dtype, w->ws[r], c * w->k + q);
      acc *= w->scale;
    }
    o[cc] = acc;
  }
}

static void* worker(void* p) {
  work_t* w = (work_t*)p;
  int64_t total = w->ntiles * w->th;
  for (;;) {
    pthread_mutex_lock(&w->mu);
    int64_t item = w->next;
    w->next += 16;
    pthread_mutex_unlock(&w->mu);
    if (item >= total) break;
    int64_t end = item + 16 < total ? item + 16 : total;
    for (; item < end; ++item) do_item(w, item);
  }
  return NULL;
}

static int run(work_t* w, int nthreads) {
  pthread_once(&g_once, init_tables);
  pthread_mutex_init(&w->mu, NULL);
  w->next = 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int t = 1; t < nthreads; ++t)
    if (pthread_create(&th[started], NULL, worker, w) == 0) ++started;
  worker(w);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&w->mu);
  return 0;
}

/* AG+GEMM reference on a list of th x tw output tiles:
 * out[t][a][b] = scale * sum_q G[r0[t]+a, q] * W[c0[t]+b, q]. */
int oracle_ag_tiles(int dtype, int64_t k, int64_t m, const void* g, const void* w, double sx, double sw,
                    int64_t ntiles, const int64_t* r0, const int64_t* c0, int64_t th, int64_t tw,
                    double* out, int nthreads) {
  if ((dtype != 0 && dtype != 1) || k < 1 || m < 1) return 1;
  work_t wk;
  memset(&wk, 0, sizeof(wk));
  wk.kind = 0; wk.dtype = dtype; wk.k = k; wk.m = m; wk.g = g; wk.w = w;
  wk.scale = (dtype == 1) ? sx * sw : 1.0;
  wk.ntiles = ntiles; wk.th = th; wk.tw = tw; wk.r0 = r0; wk.c0 = c0; wk.out = out;
  return run(&wk, nthreads);
}

/* K-split sum reference on a list of tiles:
 * out[t][a][b] = scale * sum_r sum_q X_r[r0[t]+a, q] * W_r[c0[t]+b, q], q < kr,
 * scale = sx * sw for e4m3 inputs (one scale_inv for all X_r, one for all
 * W_r, the per-tensor scaling the gathered input carries in the AG listing,
 * applied to the K-split case), 1 for bf16. */
int oracle_ksplit_tiles(int dtype, int tp, int64_t kr, int64_t m, const void* const* xs, const void* const* ws,
                        double sx, double sw, int64_t ntiles, const int64_t* r0, const int64_t* c0, int64_t th,
                        int64_t tw, double* out, int nthreads) {
  if ((dtype != 0 && dtype != 1) || tp < 1 || kr < 1 || m < 1) return 1;
  work_t wk;
  memset(&wk, 0, sizeof(wk));
  wk.kind = 1; wk.dtype = dtype; wk.tp = tp; wk.k = kr; wk.m = m; wk.xs = xs; wk.ws = ws;
  wk.scale = (dtype == 1) ? sx * sw : 1.0;
  wk.ntiles = ntiles; wk.th = th; wk.tw = tw; wk.r0 = r0; wk.c0 = c0; wk.out = out;
  return run(&wk, nthreads);
}

/* ------------------------------------------------------- bf16 ring (wire) */

/* Round a double to the nearest bf16 value, ties to even, from the format's
 * definition: 8 significant bits, binary32's exponent range (normal numbers
 * from 2^-126, subnormals spaced 2^-133), magnitudes that round to 2^128 or
 * more become infinity.  Zeros, infinities and NaNs pass through. */
double oracle_round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  double a = fabs(v);
  int e;
  frexp(a, &e);                     /* a = f * 2^e, 0.5 <= f < 1: a lies in [2^(e-1), 2^e) */
  int q = e - 8;                    /* spacing of 8 significant bits in that binade */
  if (q < -133) q = -133;           /* below 2^-126: the subnormal spacing */
  double h = ldexp(1.0, q);
  double r = rint(a / h) * h;       /* a / h is exact; rint rounds half to even */
  if (r >= ldexp(1.0, 128)) r = INFINITY;
  return copysign(r, v);
}

/* Test hook: a deliberately wrong variant of the ring arithmetic, compiled
 * only into the oracle copies the pin tests build to show that the golden
 * cases catch each mistake.  1: partials not rounded to bf16; 2: running sums
 * kept in fp32 and rounded once at the end; 3: ring starting at the owner. */
#ifndef ORACLE_WIRE_PLANT
#define ORACLE_WIRE_PLANT 0
#endif

/* Rank whose row block (reduce-scatter) or ring-order part of a row chunk
 * (all-reduce, n_chunks chunks) contains output row i. */
static int row_owner(int op_ar, int tp, int64_t n, int n_chunks, int64_t i) {
  if (!op_ar) return (int)(i / (n / tp));
  int64_t rows_chunk = n / n_chunks;
  return (int)((i % rows_chunk) / (rows_chunk / tp));
}

typedef struct {
  int dtype, tp, op_ar, n_chunks;
  int64_t kr, m, n;
  const void* const* xs;
  const void* const* ws;
  double scale;
  int64_t ntiles, th, tw;
  const int64_t* r0;
  const int64_t* c0;
  double* out;
  int64_t next;
  pthread_mutex_t mu;
} wire_t;

static double wire_element(const wire_t* w, int64_t i, int64_t c) {
  int owner = row_owner(w->op_ar, w->tp, w->n, w->n_chunks, i);
  double s = 0.0;
  for (int j = 0; j < w->tp; ++j) {
    int r = ((ORACLE_WIRE_PLANT == 3 ? owner : owner + 1) + j) % w->tp;
    double part = 0.0;                        /* rank r's partial, exact in double */
    for (int64_t q = 0; q < w->kr; ++q)
      part += elem(w->dtype, w->xs[r], i * w->kr + q) * elem(w->dtype, w->ws[r], c * w->kr + q);
    part *= w->scale;
    double p = (ORACLE_WIRE_PLANT == 1) ? (double)(float)part : oracle_round_bf16(part);  /* sent as bf16 */
    if (j == 0) {
      s = p;
    } else {
      float sum = (float)s + (float)p;         /* the hop's fp32 addition */
      s = (ORACLE_WIRE_PLANT == 2) ? (double)sum : oracle_round_bf16((double)sum);  /* sent on as bf16 */
    }
  }
  return (ORACLE_WIRE_PLANT == 1 || ORACLE_WIRE_PLANT == 2) ? oracle_round_bf16(s) : s;
}

static void* wire_worker(void* arg) {
  wire_t* w = (wire_t*)arg;
  int64_t total = w->ntiles * w->th;
  for (;;) {
    pthread_mutex_lock(&w->mu);
    int64_t item = w->next;
    w->next += 16;
    pthread_mutex_unlock(&w->mu);
    if (item >= total) break;
    int64_t end = item + 16 < total ? item + 16 : total;
    for (; item < end; ++item) {
      int64_t t = item / w->th, rr = item % w->th;
      double* o = w->out + (t * w->th + rr) * w->tw;
      for (int64_t cc = 0; cc < w->tw; ++cc) o[cc] = wire_element(w, w->r0[t] + rr, w->c0[t] + cc);
    }
  }
  return NULL;
}

/* The K-split sum of every listed th x tw output tile as a bf16 ring computes
 * it: out[t][a][b] = the ring sum of element (r0[t]+a, c0[t]+b) over the
 * ranks' partials sum_q X_r[i, q] * W_r[c, q] * scale (q < kr; scale = sx * sw
 * for e4m3 inputs, 1 for bf16), each partial rounded to bf16, each hop's fp32
 * sum rounded to bf16, in the ring order of the row's owner.  op_ar = 0:
 * reduce-scatter (owner = row block of n / tp rows); op_ar = 1: all-reduce in
 * n_chunks row chunks of tp ring-order parts each. */
int oracle_ksplit_wire_bf16_tiles(int dtype, int tp, int64_t kr, int64_t m, int64_t n, int op_ar, int n_chunks,
                                  const void* const* xs, const void* const* ws, double sx, double sw,
                                  int64_t ntiles, const int64_t* r0, const int64_t* c0, int64_t th, int64_t tw,
                                  double* out, int nthreads) {
  if ((dtype != 0 && dtype != 1) || tp < 1 || kr < 1 || m < 1 || n < 1 || n % tp != 0) return 1;
  if (op_ar && (n_chunks < 1 || n % ((int64_t)n_chunks * tp) != 0)) return 1;
  pthread_once(&g_once, init_tables);
  wire_t w;
  memset(&w, 0, sizeof(w));
  w.dtype = dtype; w.tp = tp; w.op_ar = op_ar; w.n_chunks = op_ar ? n_chunks : 1;
  w.kr = kr; w.m = m; w.n = n; w.xs = xs; w.ws = ws;
  w.scale = (dtype == 1) ? sx * sw : 1.0;
  w.ntiles = ntiles; w.th = th; w.tw = tw; w.r0 = r0; w.c0 = c0; w.out = out;
  pthread_mutex_init(&w.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th_[256];
  int started = 0;
  for (int k = 1; k < nthreads; ++k)
    if (pthread_create(&th_[started], NULL, wire_worker, &w) == 0) ++started;
  wire_worker(&w);
  for (int k = 0; k < started; ++k) pthread_join(th_[k], NULL);
  pthread_mutex_destroy(&w.mu);
  return 0;
}
