// AG+GEMM entry point that allocates nothing (tpo_ag_gemm_noalloc).
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// an inference server that reserved all device memory for its own pool up
// front, a runtime whose allocator forbids raw device allocations after
// start-up (so that memory use stays fixed and predictable), or an embedding
// that only owns the input and output buffers it is handed.  Such callers
// cannot create a context, because tpo_ctx_create allocates the staging buffer
// and the counters.  This file gives them the overlapped AG+GEMM with its
// scratch (staging buffer, chunk counters, error word) in a file-scope static
// device array: it is part of the library image, so every GPU that loads the
// library holds it, from the library's first use on that GPU until the process
// exits, and no call allocates anything.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>

#include "schedule.h"
#include "tpo_params.h"
#include "tpoverlap.h"

namespace {

// Staging buffer of up to TPO_NOALLOC_MAX_STAGING_BYTES, followed by the
// counters and error word of the kernel.
constexpr size_t kWordsBytes = (sizeof(tpo::DevWords) + 255) / 256 * 256;
static_assert(kWordsBytes == TPO_NOALLOC_WORDS_BYTES, "the header states the size of the word block");
static __device__ __align__(256) uint8_t g_noalloc_scratch[TPO_NOALLOC_MAX_STAGING_BYTES + kWordsBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool done = false;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  int max_coop_grid = 0;
  int max_pairs = 0;           // co-resident CTA pairs of the 2-SM variant (0: single-SM tiles only)
  long long shape[5] = {-1, -1, -1, -1, -1};  // the latest call's (tp, n, k, m, dtype)
  int producers = 0;           // and its producer CTA count from the schedule model
};

std::mutex g_mu;
DeviceSetup g_setup[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;
tpo_status fail(tpo_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  tpo::set_last_error(buf);  // the message tpo_last_error returns on this thread
  return s;
}

tpo_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TPO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One-time set-up of device `dev` (which must be current): the device address
// of the static array, the kernel's shared-memory opt-in and occupancy, and the
// tensor-map encoder.  Runs under g_mu.
tpo_status setup_device(int dev, DeviceSetup** out) {
  DeviceSetup& s = g_setup[dev];
  if (!s.done) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch array");
    int major = 0, minor = 0, sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device attributes");
    if (major != 10 || minor != 3) return fail(TPO_ERR_UNSUPPORTED, "libtpoverlap is compiled for sm_103a only (device is sm_%d%d)",
                                               major, minor);
    e = tpo::configure_kernel();
    if (e == cudaSuccess) e = tpo::max_blocks_per_sm(&per_sm);
    if (e != cudaSuccess) return cuda_fail(e, "kernel configuration");
    if (!g_encode_fn) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess)
        return fail(TPO_ERR_CUDA, "driver entry point cuTensorMapEncodeTiled unavailable");
      g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    int pairs = 0;
    if (tpo::max_active_pairs(&pairs) != cudaSuccess) {
      cudaGetLastError();
      pairs = 0;  // pairs cannot be placed: single-SM tiles serve every call
    }
    s.scratch = static_cast<uint8_t*>(ptr);
    s.num_sms = sms;
    s.max_coop_grid = per_sm * sms;
    s.max_pairs = pairs;
    s.done = true;
  }
  *out = &s;
  return TPO_OK;
}

bool encode(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem, uint64_t inner, uint64_t outer,
            uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode_fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [inner, rows, slots] view of `slots` consecutive [rows, inner] blocks.
bool encode3(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem, uint64_t inner, uint64_t rows,
             uint64_t slots, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  cuuint64_t dims[3] = {inner, rows, slots};
  cuuint64_t strides[2] = {inner * static_cast<uint64_t>(elem), inner * static_cast<uint64_t>(elem) * rows};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode_fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" tpo_status tpo_ag_gemm_noalloc(int tp, int64_t n, int64_t k, int64_t m, int dtype,
                                          const void* const* x, const void* w, void* y,
                                          const float* d_scale_inv_x, const float* d_scale_inv_w, void* stream) {
  // ---- arguments (the same rules as tpo_ctx_create + tpo_ag_gemm)
  if (tp < 1 || tp > TPO_MAX_TP) return fail(TPO_ERR_INVALID_ARG, "tp=%d out of range [1, %d]", tp, TPO_MAX_TP);
  if (dtype != TPO_BF16 && dtype != TPO_FP8_E4M3) return fail(TPO_ERR_INVALID_ARG, "dtype=%d unknown", dtype);
  if (n <= 0 || k <= 0 || m <= 0 || n > (1ll << 30) || k > (1ll << 30) || m > (1ll << 30))
    return fail(TPO_ERR_INVALID_ARG, "sizes must be in [1, 2^30]");
  if (n % tp != 0) return fail(TPO_ERR_UNSUPPORTED, "n=%lld must be a multiple of tp=%d", (long long)n, tp);
  if (m % 8 != 0) return fail(TPO_ERR_UNSUPPORTED, "m=%lld must be a multiple of 8", (long long)m);
  const bool fp8 = dtype == TPO_FP8_E4M3;
  const int elem = fp8 ? 1 : 2;
  if (k % (fp8 ? 16 : 8) != 0) return fail(TPO_ERR_UNSUPPORTED, "k=%lld not a multiple of %d", (long long)k,
                                            fp8 ? 16 : 8);
  const uint64_t staging_bytes = static_cast<uint64_t>(n) * static_cast<uint64_t>(k) * elem;
  if (staging_bytes > TPO_NOALLOC_MAX_STAGING_BYTES)
    return fail(TPO_ERR_INVALID_ARG,
                "gathered input of %llu bytes (n*k*element size) exceeds the no-allocation limit of %llu bytes; "
                "use tpo_ctx_create/tpo_ag_gemm for this size",
                (unsigned long long)staging_bytes, (unsigned long long)TPO_NOALLOC_MAX_STAGING_BYTES);
  if (!x) return fail(TPO_ERR_INVALID_ARG, "x must be an array of tp device pointers");
  for (int r = 0; r < tp; ++r)
    if (!aligned16(x[r])) return fail(TPO_ERR_INVALID_ARG, "x[%d] must be non-NULL and 16-byte aligned", r);
  if (!aligned16(w) || !aligned16(y)) return fail(TPO_ERR_INVALID_ARG, "w and y must be non-NULL, 16-byte aligned");
  if (fp8 && (!d_scale_inv_x || !d_scale_inv_w))
    return fail(TPO_ERR_INVALID_ARG, "e4m3 inputs need both scale_inv device pointers");
  if (!fp8 && (d_scale_inv_x || d_scale_inv_w))
    return fail(TPO_ERR_INVALID_ARG, "bf16 inputs take no scale_inv pointers (pass NULL)");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "no usable CUDA device");
  if (dev < 0 || dev >= kMaxDevices) return fail(TPO_ERR_UNSUPPORTED, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_mu);  // calls share the array: one at a time per process
  DeviceSetup* s = nullptr;
  tpo_status st = setup_device(dev, &s);
  if (st != TPO_OK) return st;

  uint8_t* staging = s->scratch;
  tpo::DevWords* words = reinterpret_cast<tpo::DevWords*>(s->scratch + TPO_NOALLOC_MAX_STAGING_BYTES);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  // ---- launch parameters: overlapped schedule, observer rank 0; CTA pairs
  // (2-SM MMA) wherever every 256-row tile lies in one slot, as tpo_ag_gemm
  tpo::Params p;
  tpo::init_params(p);
  const int64_t rows = n / tp;
  const int cg = (rows % (2 * tpo::BM) == 0 && s->max_pairs >= 1) ? 2 : 1;
  const int kel = tpo::BK_BYTES / elem;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!(encode3(&p.mapA[0], staging, dt, elem, k, rows, tp, kel, tpo::BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode3(&p.mapA[1], x[0], dt, elem, k, rows, 1, kel, tpo::BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode(&p.mapB[0], w, dt, elem, k, m, kel, tpo::BN / cg, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode3(&p.mapY[0], y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, m, rows, tp, tpo::EPI_COLS, 32,
                CU_TENSOR_MAP_SWIZZLE_64B)))
    return fail(TPO_ERR_INVALID_ARG, "tensor map encoding failed (pointer or size not TMA-compatible)");
  for (int r = 0; r < tp; ++r) p.src[r] = static_cast<const uint8_t*>(x[r]);
  p.staging = staging;
  p.words = words;
  p.scale_x = d_scale_inv_x;
  p.scale_w = d_scale_inv_w;
  p.chunk_bytes = rows * k * elem;
  p.timeout_ns = 2000ull * 1000000ull;
  p.op = tpo::OP_AG;
  p.fp8 = fp8 ? 1 : 0;
  p.tp = tp;
  p.self_rank = 0;
  p.cta_group = cg;
  p.rows_per_group = static_cast<int>(rows);
  p.row_tiles = static_cast<int>((rows + tpo::BM * cg - 1) / (tpo::BM * cg));
  p.m = static_cast<int>(m);
  p.y_rows = static_cast<int>(rows);
  p.num_groups = tp;
  p.kb_per_seg = static_cast<int>((k * elem + tpo::BK_BYTES - 1) / tpo::BK_BYTES);
  p.num_segs = 1;
  p.gate = 1;
  // the automatic column plan of tpo_ag_gemm (more, narrower tiles for launches of few tiles)
  tpo::auto_columns(p, m, std::min((s->num_sms - tpo::AUTO_COLS_PRODUCERS) / cg, cg == 2 ? s->max_pairs : s->num_sms));
  // producer CTAs from the library's schedule model (kept for the latest shape on this device)
  const long long shape[5] = {tp, n, k, m, dtype};
  if (std::memcmp(shape, s->shape, sizeof(shape)) != 0) {
    s->producers = tpo::model_producers(p, cg, tp, s->num_sms, s->max_pairs);
    std::memcpy(s->shape, shape, sizeof(shape));
  }
  const int P = s->producers;
  const int tiles = p.total_tiles;
  int G = (cg == 1) ? std::min(s->num_sms - P, tiles)
                    : 2 * std::min(std::min((s->num_sms - P) / 2, s->max_pairs - P / 2), tiles);
  if (P < 1 || G < cg || P + G > s->max_coop_grid) return fail(TPO_ERR_UNSUPPORTED, "device too small");
  for (int r = 0; r < TPO_MAX_TP; ++r) p.target[r] = static_cast<uint32_t>(P);  // counters start at zero
  p.num_producers = P;
  p.num_gemm = G;
  // dynamic tiles for launches of at least 8 rounds, as tpo_ag_gemm's default; the claim counter
  // starts at zero with the other words
  p.dyn = (tiles >= 8 * (G / cg)) ? 1 : 0;
  p.sched_base = 0;

  // The array keeps the previous call's contents: the counters and the error
  // word must start at zero (the staging buffer is fully rewritten).
  e = cudaMemsetAsync(words, 0, offsetof(tpo::DevWords, pad), cs);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the counters");
  // a plain launch: the grid never exceeds the co-resident CTA count
  e = tpo::launch_fused(p, P + G, false, cs);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");

  // Wait for the call and read its error word (16 bytes into host memory).
  // On a failure here the kernel may still be running: wait for the stream
  // before the lock is released, so that the next call's clearing of the
  // counters cannot overtake it.
  uint32_t err[4] = {0, 0, 0, 0};
  e = cudaMemcpyAsync(err, words->err, sizeof(err), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) {
    cudaStreamSynchronize(cs);
    return cuda_fail(e, "waiting for the call");
  }
  if (err[0] != tpo::DEV_OK)
    return fail(TPO_ERR_TIMEOUT, "device wait timed out (site %u, block %u, extra %u)", err[1], err[2], err[3]);
  return TPO_OK;
}
