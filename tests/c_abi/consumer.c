/*
 * A plain C program that uses libtpoverlap through its header only: the C ABI
 * as a C caller sees it, with no Python in between.  Test infrastructure: it
 * links the CPU oracle (oracle/oracle.c) for the expected values and the
 * seeded input generator (tensor_comm_gemm_gb300/gen/tpo_synth.c) for the
 * inputs.
 *
 * Cases (all bf16, uniform inputs in [-1, 1)):
 *   AG+GEMM      tp=3, n=768, k=320, m=264 (a partial column tile)
 *   GEMM+RS      tp=2, n=512, k=2x192, m=256
 *   GEMM+AR      tp=2, n=512, k=2x128, m=264, two row chunks
 *   no-allocation AG on the AG case: bit-identical to the context's result
 *   argument errors: TPO_ERR_INVALID_ARG with a message, nothing launched
 * Every output element is compared with the oracle at the parity tests' bar:
 * |y - ref| <= 1e-2 (|ref| + 1), relative Frobenius error <= 5e-3.
 * Exit status 0 when every check passes; the failures are printed.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "tpoverlap.h"

/* seeded generator (its own module, shared by the tests and the oracle's inputs) */
int tpo_synth_uniform_bf16(uint64_t key, int64_t count, uint16_t* out, int nthreads);
/* CPU oracle */
double oracle_decode_bf16(uint16_t b);
int oracle_gather(int tp, int64_t rows_per_rank, int64_t row_bytes, const void* const* x, void* out);
int oracle_ag_tiles(int dtype, int64_t k, int64_t m, const void* g, const void* w, double sx, double sw,
                    int64_t ntiles, const int64_t* r0, const int64_t* c0, int64_t th, int64_t tw, double* out,
                    int nthreads);
int oracle_ksplit_tiles(int dtype, int tp, int64_t kr, int64_t m, const void* const* xs, const void* const* ws,
                        double sx, double sw, int64_t ntiles, const int64_t* r0, const int64_t* c0, int64_t th,
                        int64_t tw, double* out, int nthreads);

static int failures = 0;

#define CHECK(cond, ...)                        \
  do {                                          \
    if (!(cond)) {                              \
      fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
      fprintf(stderr, __VA_ARGS__);             \
      fprintf(stderr, "\n");                    \
      ++failures;                               \
    }                                           \
  } while (0)

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
  if (cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

static uint16_t* host_bf16(uint64_t key, int64_t count) {
  uint16_t* h = (uint16_t*)malloc((size_t)count * 2);
  tpo_synth_uniform_bf16(key, count, h, 4);
  return h;
}

/* Compares n x m bf16 outputs (row-major, row stride m) with the oracle's doubles. */
static void compare(const char* what, const uint16_t* y, const double* ref, int64_t n, int64_t m) {
  double num = 0, den = 0, worst = 0;
  int64_t bad = 0;
  for (int64_t i = 0; i < n * m; ++i) {
    const double g = oracle_decode_bf16(y[i]), r = ref[i];
    const double d = fabs(g - r);
    num += d * d;
    den += r * r;
    if (!(d <= 1e-2 * (fabs(r) + 1.0))) {
      ++bad;
      if (d > worst) worst = d;
    }
  }
  const double rel = sqrt(num) / (den > 0 ? sqrt(den) : 1e-300);
  CHECK(bad == 0, "%s: %lld elements outside the bar (worst |err| %.3e)", what, (long long)bad, worst);
  CHECK(rel <= 5e-3, "%s: relative Frobenius error %.3e", what, rel);
  printf("%s: %lld x %lld outputs, relative Frobenius error %.3e\n", what, (long long)n, (long long)m, rel);
}

static void case_ag(void) {
  const int tp = 3;
  const int64_t n = 768, k = 320, m = 264, rows = n / tp;
  uint16_t* hx[3];
  const void* dx[3];
  for (int r = 0; r < tp; ++r) {
    hx[r] = host_bf16(0xA600 + r, rows * k);
    dx[r] = dev_copy(hx[r], (size_t)(rows * k * 2));
  }
  uint16_t* hw = host_bf16(0xA6FF, m * k);
  void* dw = dev_copy(hw, (size_t)(m * k * 2));
  void* dy = NULL;
  cudaMalloc(&dy, (size_t)(n * m * 2));
  cudaStream_t s;
  cudaStreamCreate(&s);

  tpo_ctx* ctx = tpo_ctx_create(tp, n, k, m, TPO_BF16);
  CHECK(ctx != NULL, "tpo_ctx_create: %s", tpo_last_error());
  if (!ctx) return;
  tpo_status st = tpo_ag_gemm(ctx, dx, dw, dy, NULL, NULL, s);
  CHECK(st == TPO_OK, "tpo_ag_gemm: %d %s", (int)st, tpo_last_error());
  st = tpo_sync_status(ctx);
  CHECK(st == TPO_OK, "tpo_sync_status after AG: %d %s", (int)st, tpo_last_error());
  uint16_t* y = (uint16_t*)malloc((size_t)(n * m * 2));
  cudaMemcpy(y, dy, (size_t)(n * m * 2), cudaMemcpyDeviceToHost);

  uint16_t* g = (uint16_t*)malloc((size_t)(n * k * 2));
  oracle_gather(tp, rows, k * 2, (const void* const*)hx, g);
  double* ref = (double*)malloc((size_t)(n * m) * sizeof(double));
  const int64_t r0[1] = {0}, c0[1] = {0};  /* one tile: the whole output */
  CHECK(oracle_ag_tiles(0, k, m, g, hw, 1.0, 1.0, 1, r0, c0, n, m, ref, 4) == 0, "oracle_ag_tiles");
  compare("AG+GEMM tp=3 768x320x264", y, ref, n, m);

  /* the entry point without allocation on the same inputs: the same bits */
  void* dy2 = NULL;
  cudaMalloc(&dy2, (size_t)(n * m * 2));
  cudaMemset(dy2, 0xFF, (size_t)(n * m * 2));
  st = tpo_ag_gemm_noalloc(tp, n, k, m, TPO_BF16, dx, dw, dy2, NULL, NULL, s);
  CHECK(st == TPO_OK, "tpo_ag_gemm_noalloc: %d %s", (int)st, tpo_last_error());
  uint16_t* y2 = (uint16_t*)malloc((size_t)(n * m * 2));
  cudaMemcpy(y2, dy2, (size_t)(n * m * 2), cudaMemcpyDeviceToHost);
  CHECK(memcmp(y, y2, (size_t)(n * m * 2)) == 0, "no-allocation AG differs from the context's result");
  printf("AG+GEMM without allocation: %s\n", memcmp(y, y2, (size_t)(n * m * 2)) == 0 ? "bit-identical" : "DIFFERENT");

  /* argument errors are caught before any launch */
  st = tpo_ag_gemm(ctx, NULL, dw, dy, NULL, NULL, s);
  CHECK(st == TPO_ERR_INVALID_ARG && strlen(tpo_last_error()) > 0, "NULL x: %d", (int)st);
  const void* bad[3] = {dx[0], (const char*)dx[1] + 2, dx[2]};
  st = tpo_ag_gemm(ctx, bad, dw, dy, NULL, NULL, s);
  CHECK(st == TPO_ERR_INVALID_ARG, "misaligned x[1]: %d", (int)st);
  st = tpo_sync_status(ctx);
  CHECK(st == TPO_OK, "tpo_sync_status after argument errors: %d", (int)st);
  CHECK(tpo_ctx_destroy(ctx) == TPO_OK, "tpo_ctx_destroy");
  CHECK(tpo_ctx_destroy(NULL) == TPO_OK, "tpo_ctx_destroy(NULL)");

  for (int r = 0; r < tp; ++r) {
    cudaFree((void*)dx[r]);
    free(hx[r]);
  }
  cudaFree(dw);
  cudaFree(dy);
  cudaFree(dy2);
  cudaStreamDestroy(s);
  free(hw);
  free(y);
  free(y2);
  free(g);
  free(ref);
}

/* GEMM+RS (op 0) or row-parallel GEMM+AR (op 1) over tp K-slices. */
static void case_ksplit(int op, int tp, int64_t n, int64_t k, int64_t m, int chunks) {
  const int64_t kr = k / tp;
  uint16_t* hx[2];
  uint16_t* hw[2];
  const void* dx[2];
  const void* dw[2];
  for (int r = 0; r < tp; ++r) {
    hx[r] = host_bf16(0xB500 + 16 * op + r, n * kr);
    hw[r] = host_bf16(0xB580 + 16 * op + r, m * kr);
    dx[r] = dev_copy(hx[r], (size_t)(n * kr * 2));
    dw[r] = dev_copy(hw[r], (size_t)(m * kr * 2));
  }
  tpo_ctx* ctx = tpo_ctx_create(tp, n, k, m, TPO_BF16);
  CHECK(ctx != NULL, "tpo_ctx_create: %s", tpo_last_error());
  if (!ctx) return;
  uint16_t* y = (uint16_t*)malloc((size_t)(n * m * 2));
  void* dy = NULL;
  void* yb[2] = {NULL, NULL};
  tpo_status st;
  if (op == 0) {  /* rank b's block: rows [b n/tp, (b+1) n/tp) */
    for (int b = 0; b < tp; ++b) cudaMalloc(&yb[b], (size_t)(n / tp * m * 2));
    st = tpo_gemm_rs(ctx, dx, dw, yb, NULL);
  } else {
    cudaMalloc(&dy, (size_t)(n * m * 2));
    st = tpo_gemm_ar(ctx, dx, dw, dy, chunks, NULL);
  }
  CHECK(st == TPO_OK, "%s: %d %s", op == 0 ? "tpo_gemm_rs" : "tpo_gemm_ar", (int)st, tpo_last_error());
  st = tpo_sync_status(ctx);
  CHECK(st == TPO_OK, "tpo_sync_status: %d %s", (int)st, tpo_last_error());
  if (op == 0)
    for (int b = 0; b < tp; ++b)
      cudaMemcpy(y + (size_t)(b * (n / tp) * m), yb[b], (size_t)(n / tp * m * 2), cudaMemcpyDeviceToHost);
  else
    cudaMemcpy(y, dy, (size_t)(n * m * 2), cudaMemcpyDeviceToHost);

  double* ref = (double*)malloc((size_t)(n * m) * sizeof(double));
  const int64_t r0[1] = {0}, c0[1] = {0};  /* one tile: the whole output */
  CHECK(oracle_ksplit_tiles(0, tp, kr, m, (const void* const*)hx, (const void* const*)hw, 1.0, 1.0, 1, r0, c0, n, m,
                            ref, 4) == 0,
        "oracle_ksplit_tiles");
  char what[96];
  snprintf(what, sizeof(what), "%s tp=%d %lldx%lldx%lld", op == 0 ? "GEMM+RS" : "GEMM+AR", tp, (long long)n,
           (long long)k, (long long)m);
  compare(what, y, ref, n, m);
  CHECK(tpo_ctx_destroy(ctx) == TPO_OK, "tpo_ctx_destroy");
  for (int r = 0; r < tp; ++r) {
    cudaFree((void*)dx[r]);
    cudaFree((void*)dw[r]);
    free(hx[r]);
    free(hw[r]);
  }
  for (int b = 0; b < 2; ++b)
    if (yb[b]) cudaFree(yb[b]);
  if (dy) cudaFree(dy);
  free(y);
  free(ref);
}

int main(void) {
  int dev_count = 0;
  if (cudaGetDeviceCount(&dev_count) != cudaSuccess || dev_count < 1) {
    fprintf(stderr, "no CUDA device\n");
    return 2;
  }
  printf("%s\n", tpo_version());
  case_ag();
  case_ksplit(0, 2, 512, 384, 256, 1);
  case_ksplit(1, 2, 512, 256, 264, 2);
  if (failures) {
    fprintf(stderr, "%d check(s) failed\n", failures);
    return 1;
  }
  printf("all C ABI checks passed\n");
  return 0;
}
