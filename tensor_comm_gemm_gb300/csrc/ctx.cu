// Host side of libtpoverlap: context, argument validation, tensor maps and the
// launch schedule of each operation.  See include/tpoverlap.h for the contract.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cctype>
#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "schedule.h"
#include "tpo_params.h"
#include "tpoverlap.h"

using tpo::Params;

namespace {

thread_local std::string g_err;

tpo_status fail(tpo_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

tpo_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TPO_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D row-major tensor [outer, inner] of `elem` bytes per element.
bool encode2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [inner, rows, slots] view of `slots` consecutive row-major [rows, inner]
// blocks; a box never crosses from one block into the next (rows past a
// block's end load as zeros and are clipped on stores).
bool encode3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem, uint64_t inner, uint64_t rows,
              uint64_t slots, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  cuuint64_t dims[3] = {inner, rows, slots};
  cuuint64_t strides[2] = {inner * static_cast<uint64_t>(elem), inner * static_cast<uint64_t>(elem) * rows};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

struct tpo_ctx {
  int tp = 0;
  int64_t n = 0, k = 0, m = 0;
  int dtype = 0;
  int device = 0;
  int num_sms = 0;
  int max_coop_grid = 0;
  int max_pairs = 0;             // co-resident CTA pairs of the 2-SM variant
  bool coop_clusters = true;     // cooperative launches accept cluster dimensions
  // options
  int64_t producer_sms = 0, gemm_ctas = 0, mode = 0, seq_copy_ctas = 0, self_rank = 0, wait_timeout_ms = 2000,
          trace = 0, debug_skip_chunk = -1, debug_delay_ns = 0, debug_last_step = -1, cta_group = 0,
          cooperative = 0, reduce = 0, tail_split = 0, debug_skip_partial = -1, stage_kblocks = 1,
          col_split = 0, pdl = 1, sched = 0;
  // device memory
  uint8_t* staging = nullptr;
  size_t staging_bytes = 0;
  float* ws = nullptr;  // epilogue-reduction running sums, one BM x BN fp32 block per SM
  tpo::TailDesc* tail_dev = nullptr;               // AG tail split: per-group schedules (device)
  tpo::TailDesc tail_host[tpo::MAX_GEMM_CTAS] = {};  // and their host copy
  int64_t tail_key[11] = {};                       // the plan the device table holds
  tpo::DevWords* words = nullptr;
  uint32_t target[TPO_MAX_TP] = {};  // per slot: counter value once the latest call published it
  uint32_t done_target = 0;  // RS/AR done-counter value after the latest call
  int done_op = -1;          // operation and output-group count the done counters follow
  int done_groups = 0;
  cudaStream_t aux = nullptr;
  cudaStream_t copy = nullptr;             // split mode: chunk copies run here
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_copy[TPO_MAX_TP] = {};
  cudaEvent_t last = nullptr;
  bool has_last = false;
  uint32_t last_dev_err[4] = {0, 0, 0, 0};
  const float* ks_scale_x = nullptr;  // e4m3 RS/AR scale_inv pointers (tpo_set_fp8_scales)
  const float* ks_scale_w = nullptr;
  int64_t last_producers = 0, last_gemm_ctas = 0, last_cta_group = 0;  // shape of the latest kernel launch
  int64_t last_kps = 0;          // K blocks per pipeline stage of the latest kernel launch
  int64_t last_split_tiles = 0;  // tail tiles of the latest kernel launch (AG tail split)
  int64_t pc_key[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};  // the last AG launch shape (see producer_count)
  int pc_val = 0;                // its producer count
  int64_t last_col_plan = 0;     // packed extra column tiles of the latest kernel launch (col_split encoding)
  int64_t last_late_groups = 0;  // producer CTA groups that joined its GEMM
  int64_t last_dyn = 0;          // 1 when the latest kernel launch claimed its tiles dynamically
  uint32_t sched_base = 0;       // value of the device's tile-claim counter after the launches so far
  uint32_t part_epoch = 0;       // launches with the AG tail split so far (part_ready value of this launch)
  // tensor-map cache: the maps of the latest kCacheWays pointer sets of each op
  static constexpr int kCacheWays = 4;
  struct MapSet {
    CUtensorMap a[TPO_MAX_TP], b[TPO_MAX_TP], y[TPO_MAX_TP];
  };
  MapSet cache[3][kCacheWays];
  const void* cache_key[3][kCacheWays][3 * TPO_MAX_TP + 2];
  bool cache_valid[3][kCacheWays] = {};
  int cache_next[3] = {0, 0, 0};
};

namespace {

int64_t* opt_slot(tpo_ctx* c, const char* key, int64_t* lo, int64_t* hi) {
  using Field = int64_t tpo_ctx::*;
  struct E {
    const char* k;
    Field f;
    int64_t lo, hi;
  };
  const E table[] = {
      {"producer_sms", &tpo_ctx::producer_sms, 0, 1024},
      {"gemm_ctas", &tpo_ctx::gemm_ctas, 0, 1 << 20},
      {"mode", &tpo_ctx::mode, 0, 4},
      {"seq_copy_ctas", &tpo_ctx::seq_copy_ctas, 0, 1 << 20},
      {"self_rank", &tpo_ctx::self_rank, 0, TPO_MAX_TP - 1},
      {"wait_timeout_ms", &tpo_ctx::wait_timeout_ms, 1, 600000},
      {"trace", &tpo_ctx::trace, 0, 1},
      {"debug_skip_chunk", &tpo_ctx::debug_skip_chunk, -1, TPO_MAX_TP - 1},
      {"debug_delay_ns", &tpo_ctx::debug_delay_ns, 0, 1000000000},
      {"debug_last_step", &tpo_ctx::debug_last_step, -1, TPO_MAX_TP - 1},
      {"cta_group", &tpo_ctx::cta_group, 0, 2},
      {"cooperative", &tpo_ctx::cooperative, 0, 1},
      {"reduce", &tpo_ctx::reduce, 0, 2},
      {"tail_split", &tpo_ctx::tail_split, 0, 3},
      {"debug_skip_partial", &tpo_ctx::debug_skip_partial, -1, tpo::MAX_GEMM_CTAS - 1},
      {"stage_kblocks", &tpo_ctx::stage_kblocks, 1, 2},
      {"col_split", &tpo_ctx::col_split, -1, INT64_MAX},
      {"pdl", &tpo_ctx::pdl, 0, 1},
      {"sched", &tpo_ctx::sched, 0, 2},
  };
  for (const E& e : table)
    if (std::strcmp(e.k, key) == 0) {
      *lo = e.lo;
      *hi = e.hi;
      if (std::strcmp(key, "self_rank") == 0 || std::strcmp(key, "debug_skip_chunk") == 0 ||
          std::strcmp(key, "debug_last_step") == 0)
        *hi = c->tp - 1;
      return &(c->*(e.f));
    }
  return nullptr;
}

const char* kOptKeys[] = {"producer_sms",     "gemm_ctas",      "mode",           "seq_copy_ctas",
                          "self_rank",        "wait_timeout_ms", "trace",          "debug_skip_chunk",
                          "debug_delay_ns",   "debug_last_step", "cta_group",      "cooperative",
                          "reduce",           "tail_split",     "debug_skip_partial", "stage_kblocks",
                          "col_split",        "pdl",           "sched"};

void destroy_all(tpo_ctx* c) {
  if (!c) return;
  if (c->has_last) cudaEventSynchronize(c->last);
  if (c->aux) cudaStreamSynchronize(c->aux);
  if (c->staging) cudaFree(c->staging);
  if (c->ws) cudaFree(c->ws);
  if (c->tail_dev) cudaFree(c->tail_dev);
  if (c->words) cudaFree(c->words);
  if (c->copy) cudaStreamSynchronize(c->copy);
  if (c->last) cudaEventDestroy(c->last);
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->ev_join) cudaEventDestroy(c->ev_join);
  for (cudaEvent_t e : c->ev_copy)
    if (e) cudaEventDestroy(e);
  if (c->copy) cudaStreamDestroy(c->copy);
  if (c->aux) cudaStreamDestroy(c->aux);
  delete c;
}

// Fill the fields common to every launch.
void base_params(const tpo_ctx* c, Params& p) {
  p.words = c->words;
  p.staging = c->staging;
  p.timeout_ns = static_cast<unsigned long long>(c->wait_timeout_ms) * 1000000ull;
  p.delay_ns = static_cast<unsigned long long>(c->debug_delay_ns);
  p.skip_slot = static_cast<int>(c->debug_skip_chunk);
  p.last_step = static_cast<int>(c->debug_last_step);
  p.trace_on = static_cast<int>(c->trace);
  p.self_rank = static_cast<int>(c->self_rank);
  p.tp = c->tp;
  p.fp8 = c->dtype == TPO_FP8_E4M3;
  p.pdl = static_cast<int>(c->pdl);
}

tpo_status reset_trace(tpo_ctx* c, cudaStream_t s) {
  if (!c->trace) return TPO_OK;
  unsigned long long* tr = c->words->trace;
  cudaError_t e = cudaMemsetAsync(tr, 0, sizeof(unsigned long long) * TPO_TRACE_WORDS, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(tr + TPO_TRACE_START, 0xFF, sizeof(unsigned long long), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(tr + TPO_TRACE_ACQUIRE, 0xFF, sizeof(unsigned long long) * TPO_MAX_TP, s);
  return e == cudaSuccess ? TPO_OK : cuda_fail(e, "trace reset");
}

int64_t packed_columns(const Params& p);

// Dynamic tiles (option sched: 0 automatic, 1 round robin, 2 dynamic) for a
// GEMM launch of `groups` CTA groups: automatic takes them for launches of at
// least 8 rounds, where the groups' speeds drift apart over a round-robin
// schedule.  The tail-split build keeps its own schedule.
bool want_dynamic(const tpo_ctx* c, const Params& p, int groups) {
  if (groups <= 0 || p.tail_split || p.late_groups || c->sched == 1) return false;
  return c->sched == 2 || p.total_tiles >= 8 * groups;
}

tpo_status launch(tpo_ctx* c, Params& p, int grid, bool coop, cudaStream_t s) {
  const int groups = p.cta_group > 0 ? p.num_gemm / p.cta_group : 0;
  p.dyn = want_dynamic(c, p, groups) ? 1 : 0;
  p.sched_base = c->sched_base;
  c->last_dyn = p.dyn;
  c->last_producers = p.num_producers;
  c->last_gemm_ctas = p.num_gemm;
  c->last_cta_group = p.cta_group;
  c->last_kps = p.kps;
  c->last_split_tiles = 0;
  c->last_late_groups = p.late_groups;
  c->last_col_plan = packed_columns(p);
  if (p.tail_split && p.num_gemm > 0)
    c->last_split_tiles = p.total_tiles - p.split_full * (p.num_gemm / p.cta_group);
  if (coop && (!c->cooperative || (p.cta_group == 2 && !c->coop_clusters))) coop = false;
  cudaError_t e = tpo::launch_fused(p, grid, coop, s);
  if (e != cudaSuccess && coop && p.cta_group == 2) {
    // Cooperative launches of clusters are not accepted here: launch without the
    // attribute.  The grid never exceeds the co-resident pair count, so every
    // CTA is still placed at once (and every wait stays bounded regardless).
    cudaGetLastError();
    c->coop_clusters = false;
    e = tpo::launch_fused(p, grid, false, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  if (p.dyn) c->sched_base += static_cast<uint32_t>(p.total_tiles + groups);  // every group's claims, one past the end each
  e = cudaEventRecord(c->last, s);
  if (e != cudaSuccess) return cuda_fail(e, "event record");
  c->has_last = true;
  return TPO_OK;
}

bool cache_lookup(tpo_ctx* c, int op, const void* const* key, int nkey, Params& p) {
  for (int way = 0; way < tpo_ctx::kCacheWays; ++way) {
    if (!c->cache_valid[op][way]) continue;
    bool hit = true;
    for (int i = 0; i < nkey && hit; ++i) hit = c->cache_key[op][way][i] == key[i];
    if (!hit) continue;
    const tpo_ctx::MapSet& m = c->cache[op][way];
    std::memcpy(p.mapA, m.a, sizeof(p.mapA));
    std::memcpy(p.mapB, m.b, sizeof(p.mapB));
    std::memcpy(p.mapY, m.y, sizeof(p.mapY));
    return true;
  }
  return false;
}

void cache_store(tpo_ctx* c, int op, const void* const* key, int nkey, const Params& p) {
  const int way = c->cache_next[op];
  c->cache_next[op] = (way + 1) % tpo_ctx::kCacheWays;
  for (int i = 0; i < nkey; ++i) c->cache_key[op][way][i] = key[i];
  tpo_ctx::MapSet& m = c->cache[op][way];
  std::memcpy(m.a, p.mapA, sizeof(p.mapA));
  std::memcpy(m.b, p.mapB, sizeof(p.mapB));
  std::memcpy(m.y, p.mapY, sizeof(p.mapY));
  c->cache_valid[op][way] = true;
}

// Advance the expected counter value of every slot this call's producer is
// meant to publish (all slots, or those of ring steps 0..debug_last_step) by
// the number of producer CTAs, and copy the targets into the launch.
void advance_targets(tpo_ctx* c, Params& p, int producers) {
  for (int step = 0; step < c->tp; ++step) {
    if (c->debug_last_step >= 0 && step > c->debug_last_step) continue;
    const int slot = static_cast<int>(((c->self_rank - step) % c->tp + c->tp) % c->tp);
    c->target[slot] += static_cast<uint32_t>(producers);
  }
  std::memcpy(p.target, c->target, sizeof(p.target));
}

int clamp_grid(int64_t want, int total_tiles) {
  if (want > total_tiles) want = total_tiles;
  return static_cast<int>(want < 1 ? 1 : want);
}

// Single-SM (1) or CTA-pair (2) MMA variant for a call whose tile groups are
// `rows_per_group` rows and, for AR, whose ring-order parts are `part_rows`.
// Pairs need every 256-row tile inside one group (and one part).
int choose_cg(const tpo_ctx* c, int64_t rows_per_group, int64_t part_rows) {
  const bool fits = c->max_pairs >= 1 && rows_per_group % (2 * tpo::BM) == 0 && part_rows % (2 * tpo::BM) == 0;
  if (c->cta_group == 1) return 1;
  if (c->cta_group == 2) return fits ? 2 : -1;
  return fits ? 2 : 1;
}

// GEMM CTAs for a launch of `tiles` tiles with `producers` producer CTAs.
int gemm_grid(const tpo_ctx* c, int cg, int64_t want, int producers, int tiles) {
  if (cg == 1) return clamp_grid(want, tiles);
  int64_t pairs = want / 2;
  const int64_t room = c->max_pairs - producers / 2;
  if (pairs > room) pairs = room;
  if (pairs > tiles) pairs = tiles;
  if (pairs < 1) pairs = 1;
  return static_cast<int>(2 * pairs);
}

// ---------------------------------------------------------------- schedule model
//
// The host's model of a whole-tile launch: its G CTA groups take tiles round
// robin, each group one tile after another, in the kernel's tile order; a
// tile of AG ring step g waits until that step's chunk has landed
// (ready_us[g]).  A tile costs nkb 128-byte K blocks of kKbUs x (0.91 + 0.09
// w / 8) microseconds for w 32-column strips: measured on 256-row tile pairs
// while the MMAs were issued from a single thread, when a K block of a tile
// 128 to 256 columns wide cost 559 to 585 SM cycles whatever its width.
// Issued from a converged warp, narrower tiles now cost somewhat less (a
// 192-column tile's K block ~0.86 of a 256-column one's; the operand loads
// then bound it); the model keeps the older figures, which shape only the
// producer count and column plan of launches with narrow tiles.
constexpr double kKbUs = 0.33;

template <int TILE_M>
double tiles_end_t(const Params& p, int G, const double* ready_us, int nkb) {
  std::vector<double> ends(static_cast<size_t>(G), 0.0);
  const double kb = nkb * kKbUs;
  for (int t = 0; t < p.total_tiles; ++t) {
    const tpo::TileIndex ti = tpo::tile_index<TILE_M>(p, t);
    const int cols = tpo::group_cols_of(p, ti.group);
    const int w = tpo::tile_strip0(p, cols, ti.c + 1) - tpo::tile_strip0(p, cols, ti.c);
    double& e = ends[static_cast<size_t>(t % G)];
    e = std::max(e, ready_us ? ready_us[ti.group] : 0.0) + kb * (0.91 + 0.09 * w / tpo::MAX_TILE_STRIPS);
  }
  double end = 0;
  for (double v : ends) end = std::max(end, v);
  return end;
}

double tiles_end(const Params& p, int cg, int G, const double* ready_us, int nkb) {
  return cg == 2 ? tiles_end_t<2 * tpo::BM>(p, G, ready_us, nkb) : tiles_end_t<tpo::BM>(p, G, ready_us, nkb);
}

// Column tiles of each group (sets p's column fields) for option col_split:
// 0 (the default) gives every group the fewest tiles that are at most BN
// wide; other values give group g (g < 16) ((v >> 4g) & 15) extra tiles,
// splitting its strips evenly into narrower tiles.
void plan_columns(const tpo_ctx* c, Params& p) {
  if (c->col_split == 0) {  // automatic: the GEMM CTA groups a launch of this op can have
    int64_t groups = (p.op == tpo::OP_AG ? c->num_sms - tpo::AUTO_COLS_PRODUCERS : c->num_sms) / p.cta_group;
    if (c->gemm_ctas > 0) groups = std::min<int64_t>(groups, c->gemm_ctas / p.cta_group);
    if (p.cta_group == 2) groups = std::min<int64_t>(groups, c->max_pairs);
    tpo::auto_columns(p, c->m, static_cast<int>(std::max<int64_t>(groups, 1)));
    return;
  }
  tpo::set_columns(p, c->m, nullptr);
  if (c->col_split < 0) return;
  int extra[tpo::MAX_GROUPS] = {};
  const int most = std::min(p.strips, p.uniform_cols + 15);
  for (int g = 0; g < p.num_groups && g < 16; ++g)
    extra[g] = std::min(static_cast<int>((c->col_split >> (4 * g)) & 15), most - p.uniform_cols);
  tpo::set_columns(p, c->m, extra);
}

// Packed extra column tiles of the first 16 groups (the col_split encoding).
int64_t packed_columns(const Params& p) {
  int64_t v = 0;
  if (p.uniform_cols > 0) return 0;
  const int base = (p.strips + tpo::MAX_TILE_STRIPS - 1) / tpo::MAX_TILE_STRIPS;
  for (int g = 0; g < p.num_groups && g < 16; ++g)
    v |= static_cast<int64_t>(std::min(15, p.group_cols[g] - base)) << (4 * g);
  return v;
}

// The fewest producer CTAs (even for CTA pairs; up to 32) whose modelled end
// is within 0.5 % of the best, for an overlapped AG launch whose tiles (and
// column tiles) p describes: grid_of(P) gives the GEMM's CTA groups next to P
// producer CTAs; a producer CTA moves up to 37 GB/s of chunk data beside a
// running GEMM and all of them together up to 705 GB/s, both taken 1.25
// times slower for margin; ring step g's chunk is ready at g tau and the
// launch lasts until the GEMM's end and the copy of all tp chunks.
template <class GridOf>
int best_producers(const Params& p, int cg, int tp, int num_sms, int nkb, int64_t chunk_bytes, GridOf grid_of) {
  double ends[33] = {};
  double best_end = 0;
  double ready[TPO_MAX_TP];
  for (int P = cg; P <= 32 && P <= num_sms - 2 * cg; P += cg) {
    const double rate = std::min(37e9, 705e9 / P) / 1.25;
    const double tau_us = static_cast<double>(chunk_bytes) / (P * rate) * 1e6;
    for (int g = 0; g < tp; ++g) ready[g] = g * tau_us;
    ends[P] = std::max(tp * tau_us, tiles_end(p, cg, grid_of(P), ready, nkb));
    if (best_end == 0 || ends[P] < best_end) best_end = ends[P];
  }
  for (int P = cg; P <= 32 && P <= num_sms - 2 * cg; P += cg)
    if (ends[P] <= best_end * 1.005) return P;
  return 8;
}

// Producer CTAs of an overlapped AG call, and the column tiles of its GEMM
// (set in p).  An explicit producer_sms option wins.  `split` is the tail-split
// schedule (0 none): its launches keep the fewest column tiles.
//
// With the tail split's schedule 1 every GEMM group shortens the GEMM, so the
// count is the smallest (from 4) that keeps the copy ahead of it.
// Each gathered chunk must land before the GEMM reaches its first tile, with
// 15% to spare, and the whole staging copy (own chunk last) within 90% of the
// GEMM.  The model: a producer CTA moves about 47 GB/s of chunk data (94 GB/s
// of HBM reads and writes, whatever its depth of copies in flight), and a CTA
// group spends about 0.3 us per 128-byte K block of a tile.
//
// Without it, the schedule model decides for every producer count (even for
// CTA pairs) up to 32: the GEMM grid that remains, a chunk copy time tau (a
// producer CTA moves up to 37 GB/s of chunk data beside a running GEMM and all
// of them together up to 705 GB/s, both taken 1.25 times slower for margin),
// ring step g's chunk ready at g tau, and the launch lasting until the GEMM's
// end and the copy of all tp chunks (the observer's own chunk last).  The fewest producers whose end is within 0.5 %
// of the best win: fewer copy SMs disturb the GEMM's loads less.  Computed
// once per launch shape and kept in the context.
int producer_count(tpo_ctx* c, Params& p, int cg, int tiles, int nkb, int split) {
  const int64_t chunk_bytes = p.chunk_bytes;
  auto grid_of = [&](int P) {
    return gemm_grid(c, cg, c->gemm_ctas ? c->gemm_ctas : c->num_sms - P, P, tiles) / cg;
  };
  // the launch's column tiles (the tail split keeps the fewest)
  auto set_cols = [&]() {
    if (split)
      tpo::set_columns(p, c->m, nullptr);
    else
      plan_columns(c, p);
  };
  if (split == 1 && c->producer_sms <= 0) {
    tpo::set_columns(p, c->m, nullptr);
    const double rate = 47e9, t_tile = nkb * 0.3e-6;
    const int per_group = tiles / c->tp;
    for (int P = 4; P <= 32 && P < c->num_sms - 2 * cg; P += cg) {
      const int G = gemm_grid(c, cg, c->num_sms - P, P, tiles) / cg;
      const int R = tiles % G, gt = R ? std::min(G, tpo::TAIL_SPLIT * R) : 0;
      const double tau = static_cast<double>(chunk_bytes) / (P * rate);
      bool ok = c->tp * tau <= 0.9 * (static_cast<double>(tiles) / G) * t_tile;
      for (int j = 1; j < c->tp && ok; ++j) {  // ring step j's chunk: first tile j * per_group
        const int f = j * per_group;
        if (f < R) {
          ok = false;  // a split tile, needed from the start
          break;
        }
        // whole round r after the split tiles; groups with split work start it R / gt tiles late
        const int r = (f - R) / G, sl = (f - R) % G;
        const double start = r + ((gt > 0 && sl >= G - gt) ? static_cast<double>(R) / gt : 0.0);
        ok = j * tau <= 0.85 * start * t_tile;
      }
      if (ok) return P;
    }
  }
  const int64_t key[9] = {cg, c->gemm_ctas, c->producer_sms, c->col_split, tiles, nkb, chunk_bytes, c->m, split};
  set_cols();
  if (std::memcmp(key, c->pc_key, sizeof(key)) == 0) return c->pc_val;
  const int best = (c->producer_sms > 0)
                       ? static_cast<int>(c->producer_sms) + ((cg == 2) ? static_cast<int>(c->producer_sms & 1) : 0)
                       : best_producers(p, cg, c->tp, c->num_sms, nkb, chunk_bytes, grid_of);
  std::memcpy(c->pc_key, key, sizeof(key));
  c->pc_val = best;
  return best;
}

// Tail-split plan of an AG GEMM launch (see SegIter in the kernel) with G GEMM
// groups and L producer groups that join once their copy is done.
//
// With L > 0 the plan expects the copy of all tp chunks to end after
// tp * chunk_bytes / (P * 31 GB/s) plus 3 us (a producer CTA's copy rate next
// to a running GEMM), plans for 1.2 times that, and counts 0.36 us per
// 128-byte K block of a tile: from these, the work is cut so that GEMM and
// late groups end together.  A late start planned too early would make the
// late groups end last, hence the margin; planned too late, they idle at the
// end instead.  The plan only moves time: any plan gives exact tiles.
//
// With L == 0 (or no time for the late groups) the R = T mod G leftover tiles
// are shared among min(G, TAIL_SPLIT R) GEMM groups, first (schedule 1) or
// after the whole rounds (`last`, schedule 3: the operands are then warm in
// L2, where split parts that start at different K offsets find them).
void plan_split(const tpo_ctx* c, Params& p, int tiles, int G, int L, bool last) {
  const long long kbu = p.kb_per_seg / p.kps;  // K units of a tile (AG: one K segment)
  p.tail_split = 0;
  p.late_groups = 0;
  if (G < 1 || kbu < 1) return;
  if (L > 0) {
    const int P = L * p.cta_group;
    const double t_copy = c->tp * static_cast<double>(p.chunk_bytes) / (P * 31e9) + 3e-6;
    const double late = 1.2 * t_copy / (p.kps * 0.36e-6);  // planned late start, in K units
    const double E = (static_cast<double>(tiles) * kbu + L * late) / (G + L);  // units per GEMM group
    if (E > late + 1.0) {
      int full = static_cast<int>(E / kbu);
      if (full > tiles / G) full = tiles / G;
      const long long wt = static_cast<long long>(tiles - full * G) * kbu;
      long long sm = static_cast<long long>(E - static_cast<double>(full) * kbu);
      if (sm < 0) sm = 0;
      if (sm * G > wt) sm = wt / G;
      if (wt - sm * G > 0) {
        p.tail_split = 1;
        p.split_tail_first = 0;
        p.split_full = full;
        p.split_ga = G;
        p.split_wa = sm * G;
        p.split_gb = L;
        p.split_wb = wt - sm * G;
        p.late_groups = L;
        return;
      }
    }
  }
  const int full = tiles / G, R = tiles - full * G;
  if (R == 0) return;
  p.tail_split = 1;
  p.split_tail_first = last ? 0 : 1;
  p.split_full = full;
  p.split_ga = std::min(G, tpo::TAIL_SPLIT * R);
  p.split_wa = static_cast<long long>(R) * kbu;
  p.split_gb = 0;
  p.split_wb = 0;
}

// The schedule of CTA group g under the plan in `p` (see TailDesc), in the
// 32-bit arithmetic the plan's bounds allow.
tpo::TailDesc make_tail(const Params& p, int g, int G, int T, int kbu_i) {
  tpo::TailDesc d{};
  const uint32_t kbu = static_cast<uint32_t>(kbu_i);
  const uint32_t ga = static_cast<uint32_t>(p.split_ga), gb = static_cast<uint32_t>(p.split_gb);
  const uint32_t wa = static_cast<uint32_t>(p.split_wa), wb = static_cast<uint32_t>(p.split_wb);
  auto start_of = [&](uint32_t w) -> uint32_t {  // first tail unit of group w (w <= ga + gb)
    if (w <= ga) return ga > 0 ? wa * w / ga : 0u;
    return wa + wb * (w - ga) / gb;
  };
  d.first = p.split_tail_first != 0;
  d.nfull = g < G ? p.split_full : 0;
  if (d.first) {
    d.whole_base = T - p.split_full * G;
    d.slot = (g - static_cast<int>(ga) + G) % G;
  } else {
    d.slot = g;
    d.tail_base = p.split_full * G;
  }
  const uint32_t ug = static_cast<uint32_t>(g);
  if (ug >= ga + gb) return d;
  const uint32_t pos = start_of(ug), end = start_of(ug + 1);
  uint32_t p2 = pos;
  if (pos < end && pos % kbu != 0) {  // the range starts inside a tile: a later part of it
    const uint32_t t0 = pos / kbu;
    d.wr_lo = static_cast<int>(pos - t0 * kbu);
    d.wr_hi = static_cast<int>(std::min(kbu, static_cast<uint32_t>(d.wr_lo) + (end - pos)));
    d.wr_t = static_cast<int>(t0);
    d.has_wr = 1;
    p2 = pos + static_cast<uint32_t>(d.wr_hi - d.wr_lo);
  }
  if (p2 < end) {  // from a tile boundary: whole tiles, then perhaps the first part of one more
    d.tw0 = static_cast<int>(p2 / kbu);
    d.tw1 = static_cast<int>(end / kbu);
    const uint32_t rem = end - static_cast<uint32_t>(d.tw1) * kbu;
    if (rem > 0) {
      d.has_fin = 1;
      d.fin_t = d.tw1;
      d.fin_hi = static_cast<int>(rem);
      d.fin_w0 = g + 1;
      const uint32_t tile_end = static_cast<uint32_t>(d.tw1 + 1) * kbu;
      for (uint32_t w = ug + 1; w < ga + gb && start_of(w) < tile_end; ++w) ++d.fin_nw;
    }
  }
  return d;
}

// Fill the device table of per-group schedules for the plan in `p` (copied
// only when the plan changed) and point the launch at it.
tpo_status upload_tails(tpo_ctx* c, Params& p, int T, int G, cudaStream_t s) {
  const int groups = G + p.late_groups, kbu = p.kb_per_seg / p.kps;
  const int64_t key[11] = {p.split_tail_first, p.split_full, p.split_ga, p.split_gb, p.split_wa,
                           p.split_wb, T, G, groups, kbu, p.kps};
  p.tail_tab = c->tail_dev;
  if (std::memcmp(key, c->tail_key, sizeof(key)) == 0) return TPO_OK;
  if (groups > tpo::MAX_GEMM_CTAS) return fail(TPO_ERR_INVALID_ARG, "too many CTA groups for the tail split");
  for (int g = 0; g < groups; ++g) c->tail_host[g] = make_tail(p, g, G, T, kbu);
  cudaError_t e = cudaMemcpyAsync(c->tail_dev, c->tail_host, sizeof(tpo::TailDesc) * groups, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "tail table upload");
  std::memcpy(c->tail_key, key, sizeof(key));
  return TPO_OK;
}

// Validation shared by RS and AR.
tpo_status check_ksplit(tpo_ctx* c, const void* const* x, const void* const* w) {
  const int kq = c->dtype == TPO_BF16 ? 8 : 16;
  if (c->k % c->tp != 0 || (c->k / c->tp) % kq != 0)
    return fail(TPO_ERR_UNSUPPORTED, "k/tp must be an integer multiple of %d (16-byte rows; k=%lld, tp=%d)", kq,
                (long long)c->k, c->tp);
  if (c->dtype == TPO_FP8_E4M3 && (!c->ks_scale_x || !c->ks_scale_w))
    return fail(TPO_ERR_INVALID_ARG, "e4m3 GEMM+RS/AR needs tpo_set_fp8_scales first");
  if (!x || !w) return fail(TPO_ERR_INVALID_ARG, "x and w must be arrays of tp device pointers");
  for (int r = 0; r < c->tp; ++r)
    if (!aligned16(x[r]) || !aligned16(w[r]))
      return fail(TPO_ERR_INVALID_ARG, "x[%d] / w[%d] must be non-NULL and 16-byte aligned", r, r);
  return TPO_OK;
}

}  // namespace

namespace tpo {
void set_last_error(const char* msg) { g_err = msg; }

void auto_columns(Params& p, long long m, int gemm_groups) {
  set_columns(p, m, nullptr);
  const int per_col = p.num_groups * p.row_tiles;  // tiles per column tile of every group
  if (per_col <= 0 || 2 * p.total_tiles > gemm_groups) return;
  const int cols = std::min(p.strips, gemm_groups / per_col);
  if (cols <= p.uniform_cols) return;
  int extra[MAX_GROUPS];
  for (int g = 0; g < p.num_groups; ++g) extra[g] = cols - p.uniform_cols;
  set_columns(p, m, extra);
}

int model_producers(const Params& p, int cg, int tp, int num_sms, int max_pairs) {
  const int tiles = p.total_tiles;
  auto grid_of = [&](int P) {
    if (cg == 1) return std::max(1, std::min(num_sms - P, tiles));
    return std::max(1, std::min(std::min((num_sms - P) / 2, max_pairs - P / 2), tiles));
  };
  return best_producers(p, cg, tp, num_sms, p.kb_per_seg, p.chunk_bytes, grid_of);
}
}  // namespace tpo

extern "C" {

const char* tpo_last_error(void) { return g_err.c_str(); }

const char* tpo_version(void) {
  static char v[128];
  std::snprintf(v, sizeof(v), "libtpoverlap 0.1 (nvcc %d.%d, sm_103a, tcgen05)", __CUDACC_VER_MAJOR__,
                __CUDACC_VER_MINOR__);
  return v;
}

tpo_ctx* tpo_ctx_create(int tp, int64_t n, int64_t k, int64_t m, int dtype) {
  if (tp < 1 || tp > TPO_MAX_TP) {
    fail(TPO_ERR_INVALID_ARG, "tp=%d out of range [1, %d]", tp, TPO_MAX_TP);
    return nullptr;
  }
  if (dtype != TPO_BF16 && dtype != TPO_FP8_E4M3) {
    fail(TPO_ERR_INVALID_ARG, "dtype=%d is neither TPO_BF16 (0) nor TPO_FP8_E4M3 (1)", dtype);
    return nullptr;
  }
  if (n <= 0 || k <= 0 || m <= 0 || n > (1ll << 30) || k > (1ll << 30) || m > (1ll << 30)) {
    fail(TPO_ERR_INVALID_ARG, "sizes must be in [1, 2^30] (n=%lld k=%lld m=%lld)", (long long)n, (long long)k,
         (long long)m);
    return nullptr;
  }
  // Any size works with the tiling (partial tiles load zeros and clip their
  // stores); what remains are equal chunks per rank and 16-byte row pitches.
  if (n % tp != 0) {
    fail(TPO_ERR_UNSUPPORTED, "n=%lld must be a multiple of tp=%d (equal row chunks per rank)", (long long)n, tp);
    return nullptr;
  }
  if (m % 8 != 0) {
    fail(TPO_ERR_UNSUPPORTED, "m=%lld must be a multiple of 8 (16-byte rows of the bf16 output)", (long long)m);
    return nullptr;
  }
  const int kq = dtype == TPO_BF16 ? 8 : 16;
  if (k % kq != 0) {
    fail(TPO_ERR_UNSUPPORTED, "k=%lld must be a multiple of %d for this dtype (16-byte rows)", (long long)k, kq);
    return nullptr;
  }
  tpo_ctx* c = new tpo_ctx();
  c->tp = tp;
  c->n = n;
  c->k = k;
  c->m = m;
  c->dtype = dtype;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e != cudaSuccess) {
    cuda_fail(e, "no usable CUDA device");
    destroy_all(c);
    return nullptr;
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, c->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, c->device);
  if (major != 10 || minor != 3) {
    fail(TPO_ERR_UNSUPPORTED, "libtpoverlap is compiled for sm_103a only; device is sm_%d%d", major, minor);
    destroy_all(c);
    return nullptr;
  }
  if (!load_encode()) {
    fail(TPO_ERR_CUDA, "driver entry point cuTensorMapEncodeTiled unavailable");
    destroy_all(c);
    return nullptr;
  }
  int per_sm = 0;
  e = tpo::configure_kernel();
  if (e == cudaSuccess) e = tpo::max_blocks_per_sm(&per_sm);
  if (e != cudaSuccess || per_sm < 1) {
    if (e != cudaSuccess)
      cuda_fail(e, "kernel configuration");
    else
      fail(TPO_ERR_CUDA, "kernel does not fit on an SM");
    destroy_all(c);
    return nullptr;
  }
  c->max_coop_grid = per_sm * c->num_sms;
  if (tpo::max_active_pairs(&c->max_pairs) != cudaSuccess) {
    cudaGetLastError();
    c->max_pairs = 0;  // pairs cannot be placed: the single-SM variant serves every call
  }
  const int elem = dtype == TPO_BF16 ? 2 : 1;
  c->staging_bytes = static_cast<size_t>(n) * static_cast<size_t>(k) * elem;
  e = cudaMalloc(&c->staging, c->staging_bytes);
  if (e != cudaSuccess) {
    fail(TPO_ERR_OOM, "staging buffer of %zu bytes: %s", c->staging_bytes, cudaGetErrorString(e));
    cudaGetLastError();
    destroy_all(c);
    return nullptr;
  }
  e = cudaMalloc(&c->words, sizeof(tpo::DevWords));
  if (e == cudaSuccess)
    e = cudaMalloc(&c->ws, static_cast<size_t>(c->num_sms) * tpo::BM * tpo::BN * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&c->tail_dev, sizeof(c->tail_host));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->aux, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->last, cudaEventDisableTiming);
  if (e == cudaSuccess) {
    int lo = 0, hi = 0;
    cudaDeviceGetStreamPriorityRange(&lo, &hi);
    e = cudaStreamCreateWithPriority(&c->copy, cudaStreamNonBlocking, hi);  // copies first when SMs free up
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming);
  for (int r = 0; r < TPO_MAX_TP && e == cudaSuccess; ++r)
    e = cudaEventCreateWithFlags(&c->ev_copy[r], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->words, 0, sizeof(tpo::DevWords), c->aux);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->aux);
  if (e != cudaSuccess) {
    cuda_fail(e, "context set-up");
    destroy_all(c);
    return nullptr;
  }
  // environment overrides of the option defaults
  for (const char* key : kOptKeys) {
    char env[64] = "TPO_";
    size_t j = 4;
    for (const char* s = key; *s && j + 1 < sizeof(env); ++s) env[j++] = static_cast<char>(std::toupper(*s));
    env[j] = 0;
    if (const char* v = std::getenv(env)) {
      if (tpo_set_opt(c, key, std::strtoll(v, nullptr, 10)) != TPO_OK) {
        destroy_all(c);
        return nullptr;
      }
    }
  }
  return c;
}

tpo_status tpo_ctx_destroy(tpo_ctx* c) {
  destroy_all(c);
  return TPO_OK;
}

tpo_status tpo_set_opt(tpo_ctx* c, const char* key, int64_t value) {
  if (!c || !key) return fail(TPO_ERR_INVALID_ARG, "NULL context or key");
  int64_t lo, hi;
  int64_t* f = opt_slot(c, key, &lo, &hi);
  if (!f) return fail(TPO_ERR_INVALID_ARG, "unknown option '%s'", key);
  if (value < lo || value > hi)
    return fail(TPO_ERR_INVALID_ARG, "option '%s'=%lld outside [%lld, %lld]", key, (long long)value, (long long)lo,
                (long long)hi);
  *f = value;
  return TPO_OK;
}

tpo_status tpo_get_opt(tpo_ctx* c, const char* key, int64_t* value) {
  if (!c || !key || !value) return fail(TPO_ERR_INVALID_ARG, "NULL argument");
  if (std::strcmp(key, "last_producer_ctas") == 0) return *value = c->last_producers, TPO_OK;
  if (std::strcmp(key, "last_gemm_ctas") == 0) return *value = c->last_gemm_ctas, TPO_OK;
  if (std::strcmp(key, "last_cta_group") == 0) return *value = c->last_cta_group, TPO_OK;
  if (std::strcmp(key, "last_stage_kblocks") == 0) return *value = c->last_kps, TPO_OK;
  if (std::strcmp(key, "last_split_tiles") == 0) return *value = c->last_split_tiles, TPO_OK;
  if (std::strcmp(key, "last_late_groups") == 0) return *value = c->last_late_groups, TPO_OK;
  if (std::strcmp(key, "last_col_plan") == 0) return *value = c->last_col_plan, TPO_OK;
  if (std::strcmp(key, "last_sched") == 0) return *value = c->last_dyn ? 2 : 1, TPO_OK;
  if (std::strcmp(key, "coop_clusters") == 0) return *value = c->coop_clusters ? 1 : 0, TPO_OK;
  if (std::strcmp(key, "tp") == 0) return *value = c->tp, TPO_OK;
  if (std::strcmp(key, "n") == 0) return *value = c->n, TPO_OK;
  if (std::strcmp(key, "k") == 0) return *value = c->k, TPO_OK;
  if (std::strcmp(key, "m") == 0) return *value = c->m, TPO_OK;
  if (std::strcmp(key, "dtype") == 0) return *value = c->dtype, TPO_OK;
  int64_t lo, hi;
  int64_t* f = opt_slot(c, key, &lo, &hi);
  if (!f) return fail(TPO_ERR_INVALID_ARG, "unknown option '%s'", key);
  *value = *f;
  return TPO_OK;
}

tpo_status tpo_ag_gemm(tpo_ctx* c, const void* const* x, const void* w, void* y, const float* d_scale_inv_x,
                       const float* d_scale_inv_w, void* stream) {
  if (!c) return fail(TPO_ERR_INVALID_ARG, "NULL context");
  if (!x) return fail(TPO_ERR_INVALID_ARG, "x must be an array of tp device pointers");
  for (int r = 0; r < c->tp; ++r)
    if (!aligned16(x[r])) return fail(TPO_ERR_INVALID_ARG, "x[%d] must be non-NULL and 16-byte aligned", r);
  if (!aligned16(w) || !aligned16(y)) return fail(TPO_ERR_INVALID_ARG, "w and y must be non-NULL, 16-byte aligned");
  const bool fp8 = c->dtype == TPO_FP8_E4M3;
  if (fp8 && (!d_scale_inv_x || !d_scale_inv_w))
    return fail(TPO_ERR_INVALID_ARG, "e4m3 contexts need both scale_inv device pointers");
  if (!fp8 && (d_scale_inv_x || d_scale_inv_w))
    return fail(TPO_ERR_INVALID_ARG, "bf16 contexts take no scale_inv pointers (pass NULL)");
  if (c->self_rank >= c->tp) return fail(TPO_ERR_INVALID_ARG, "self_rank >= tp");
  if (c->debug_last_step >= 0 && c->mode != 3)
    return fail(TPO_ERR_INVALID_ARG, "debug_last_step applies to mode 3 (producer only)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int elem = fp8 ? 1 : 2;
  const int kel = tpo::BK_BYTES / elem;
  const int64_t rows = c->n / c->tp;

  const int cg = choose_cg(c, rows, rows);
  if (cg < 0) return fail(TPO_ERR_UNSUPPORTED, "cta_group=2 needs n/tp a multiple of 256 and placeable CTA pairs");

  Params p;
  tpo::init_params(p);
  base_params(c, p);
  p.op = tpo::OP_AG;
  p.cta_group = cg;
  p.ws = c->ws;
  p.skip_part = static_cast<int>(c->debug_skip_partial);
  const void* key[5] = {c->staging, x[c->self_rank], w, y, reinterpret_cast<const void*>(static_cast<intptr_t>(cg))};
  if (!cache_lookup(c, tpo::OP_AG, key, 5, p)) {
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    bool ok =
        encode3d(&p.mapA[0], c->staging, dt, elem, c->k, rows, c->tp, kel, tpo::BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode3d(&p.mapA[1], x[c->self_rank], dt, elem, c->k, rows, 1, kel, tpo::BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode2d(&p.mapB[0], w, dt, elem, c->k, c->m, kel, tpo::BN / cg, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode3d(&p.mapY[0], y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->m, rows, c->tp, tpo::EPI_COLS, 32,
                 CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return fail(TPO_ERR_INVALID_ARG, "tensor map encoding failed (pointer or size not TMA-compatible)");
    cache_store(c, tpo::OP_AG, key, 5, p);
  }
  for (int r = 0; r < c->tp; ++r) p.src[r] = static_cast<const uint8_t*>(x[r]);
  p.scale_x = d_scale_inv_x;
  p.scale_w = d_scale_inv_w;
  p.chunk_bytes = rows * c->k * elem;
  p.rows_per_group = static_cast<int>(rows);
  p.row_tiles = static_cast<int>(ceil_div(rows, tpo::BM * cg));
  p.m = static_cast<int>(c->m);
  p.y_rows = static_cast<int>(rows);
  p.num_groups = c->tp;
  p.kb_per_seg = static_cast<int>(ceil_div(c->k * elem, tpo::BK_BYTES));
  p.num_segs = 1;
  p.gate = 1;
  // K blocks per pipeline stage: one (six stages) unless two are asked for (pairs, when they divide)
  p.kps = (cg == 2 && c->stage_kblocks == 2 && p.kb_per_seg % 2 == 0) ? 2 : 1;
  tpo::set_columns(p, c->m, nullptr);
  const int tiles_fewest = p.total_tiles;  // the split mode's per-slot launches keep the fewest column tiles

  tpo_status st = reset_trace(c, s);
  if (st != TPO_OK) return st;
  const int64_t gemm_want = c->gemm_ctas ? c->gemm_ctas : c->num_sms;
  // The tail split (modes 0, 1, 2) stores partials in the workspace (one block
  // per GEMM CTA).  Its sums depend on the launch shape and the plan, so modes
  // 1 and 2 run the GEMM with mode 0's groups and plan (the producer CTAs
  // then skip the copy and run their share at once): all three give the same
  // bits.
  const int split = (c->mode == 0 || c->mode == 1 || c->mode == 2) ? static_cast<int>(c->tail_split) : 0;
  if (!split) plan_columns(c, p);  // the tail split keeps the fewest column tiles
  const int tiles = p.total_tiles;  // the GEMM grid follows the launch's tile count
  const int nkb = p.kb_per_seg;
  // producer count, GEMM grid and column plan of the overlapped launch
  auto overlap_grid = [&](int* P, int* G) {
    *P = producer_count(c, p, cg, tiles, nkb, split);  // even for CTA pairs: clusters of two
    *G = gemm_grid(c, cg, c->gemm_ctas ? c->gemm_ctas : c->num_sms - *P, *P, tiles);
  };
  // The GEMM launch of modes 0-2 with G GEMM CTAs and P producer CTAs.
  auto gemm_launch = [&](int P, int G, bool copy, bool coop) {
    p.num_producers = P;
    p.num_gemm = G;
    p.copy_on = copy ? 1 : 0;
    if (split && P + G <= c->num_sms && P + G <= tpo::MAX_GEMM_CTAS)
      plan_split(c, p, tiles, G / cg, split == 2 ? P / cg : 0, split == 3);
    // the kernel's tail arithmetic is 32-bit: units times groups must stay below 2^31
    if (p.tail_split && (p.split_wa * (p.split_ga + 1) >= (1ll << 31) || p.split_wb * (p.split_gb + 1) >= (1ll << 31) ||
                         static_cast<long long>(tiles) * (p.kb_per_seg / p.kps) >= (1ll << 31)))
      p.tail_split = p.late_groups = 0;
    if (p.tail_split) {
      p.part_target = ++c->part_epoch;
      const tpo_status ts = upload_tails(c, p, tiles, G / cg, s);
      if (ts != TPO_OK) return ts;
    }
    if (!copy && !p.late_groups) p.num_producers = 0;  // nothing for the producer CTAs to do
    const int grid = p.num_producers + p.num_gemm;
    return launch(c, p, grid, coop || p.tail_split != 0, s);  // split tiles: every CTA co-resident
  };
  switch (c->mode) {
    case 0: {  // overlapped: one cooperative launch, producer and GEMM co-resident
      int P, G;
      overlap_grid(&P, &G);
      if (P < 1 || c->num_sms - P < cg || P + G > c->max_coop_grid)
        return fail(TPO_ERR_INVALID_ARG, "producer_sms=%d + gemm CTAs=%d exceed the %d co-resident CTAs", P, G,
                    c->max_coop_grid);
      advance_targets(c, p, P);
      return gemm_launch(P, G, true, true);
    }
    case 1: {  // sequential: the copy to completion, then the same GEMM
      const int Pc = static_cast<int>(c->seq_copy_ctas ? c->seq_copy_ctas : c->num_sms);
      advance_targets(c, p, Pc);
      p.num_producers = Pc;
      p.num_gemm = 0;
      p.cta_group = 1;  // a producer-only launch needs no CTA pairs
      st = launch(c, p, Pc, false, s);
      if (st != TPO_OK) return st;
      p.cta_group = cg;
      int P = 0, G = gemm_grid(c, cg, gemm_want, 0, tiles);
      if (split)
        overlap_grid(&P, &G);
      else
        plan_columns(c, p);
      return gemm_launch(P, G, false, false);
    }
    case 2: {  // GEMM only: chunks published by an earlier call
      std::memcpy(p.target, c->target, sizeof(p.target));
      int P = 0, G = gemm_grid(c, cg, gemm_want, 0, tiles);
      if (split)
        overlap_grid(&P, &G);
      else
        plan_columns(c, p);
      return gemm_launch(P, G, false, false);
    }
    case 4: {  // split: per ring step a chunk copy, then a GEMM launch over that slot
      const int P = producer_count(c, p, cg, tiles, nkb, 0);
      const int G = gemm_grid(c, cg, c->gemm_ctas ? c->gemm_ctas : c->num_sms - P, P, tiles_fewest / c->tp);
      cudaError_t e = cudaEventRecord(c->ev_fork, s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(c->copy, c->ev_fork, 0);
      if (e != cudaSuccess) return cuda_fail(e, "split fork");
      Params cp = p;  // copies: one producer launch per ring step, arrival order, own chunk last
      cp.cta_group = 1;
      cp.num_producers = P;
      cp.num_gemm = 0;
      for (int si = 0; si < c->tp; ++si) {
        const int step = (si + 1) % c->tp;
        const int slot = static_cast<int>(((c->self_rank - step) % c->tp + c->tp) % c->tp);
        cp.only_step = step;
        c->target[slot] += static_cast<uint32_t>(P);  // counters stay consistent for later modes
        std::memcpy(cp.target, c->target, sizeof(cp.target));
        st = launch(c, cp, P, false, c->copy);
        if (st != TPO_OK) return st;
        e = cudaEventRecord(c->ev_copy[slot], c->copy);
        if (e != cudaSuccess) return cuda_fail(e, "split copy event");
      }
      // GEMMs: the observer's own chunk first (in place), then each slot once copied
      Params gp = p;
      gp.gate = 0;
      gp.num_groups = 1;
      tpo::set_columns(gp, c->m, nullptr);  // one slot per launch, fewest column tiles
      gp.num_producers = 0;
      gp.num_gemm = G;
      const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      for (int step = 0; step < c->tp; ++step) {
        const int slot = static_cast<int>(((c->self_rank - step) % c->tp + c->tp) % c->tp);
        gp.self_rank = slot;  // group 0 of a one-group launch is this slot
        if (step > 0) {
          if (!encode3d(&gp.mapA[1], c->staging + static_cast<size_t>(slot) * p.chunk_bytes, dt, elem, c->k, rows,
                        1, kel, tpo::BM, CU_TENSOR_MAP_SWIZZLE_128B))
            return fail(TPO_ERR_INVALID_ARG, "tensor map encoding failed");
          e = cudaStreamWaitEvent(s, c->ev_copy[slot], 0);
          if (e != cudaSuccess) return cuda_fail(e, "split wait");
        }
        st = launch(c, gp, G, false, s);
        if (st != TPO_OK) return st;
      }
      e = cudaEventRecord(c->ev_join, c->copy);  // the staging buffer is complete when the call ends
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->ev_join, 0);
      if (e == cudaSuccess) e = cudaEventRecord(c->last, s);
      return e == cudaSuccess ? TPO_OK : cuda_fail(e, "split join");
    }
    default: {  // producer only
      const int P = producer_count(c, p, cg, tiles, nkb, static_cast<int>(c->tail_split));
      if (P > c->max_coop_grid) return fail(TPO_ERR_INVALID_ARG, "producer_sms too large");
      advance_targets(c, p, P);
      p.num_producers = P;
      p.num_gemm = 0;
      p.cta_group = 1;
      return launch(c, p, P, false, s);
    }
  }
}

static tpo_status ksplit_common(tpo_ctx* c, int op, const void* const* x, const void* const* w,
                                void* const* yb, void* y, int n_chunks, cudaStream_t s) {
  const int64_t kr = c->k / c->tp;
  const int groups = (op == tpo::OP_RS) ? c->tp : n_chunks;
  const int64_t rows_per_group = c->n / groups;
  const int64_t part_rows = (op == tpo::OP_AR) ? rows_per_group / c->tp : rows_per_group;
  const int cg = choose_cg(c, rows_per_group, part_rows);
  if (cg < 0) return fail(TPO_ERR_UNSUPPORTED, "cta_group=2 needs 256-row tile groups and placeable CTA pairs");
  Params p;
  tpo::init_params(p);
  base_params(c, p);
  p.op = op;
  p.cta_group = cg;
  const void* key[3 * TPO_MAX_TP + 2];
  int nkey = 0;
  for (int r = 0; r < c->tp; ++r) {
    key[nkey++] = x[r];
    key[nkey++] = w[r];
    key[nkey++] = (op == tpo::OP_RS) ? yb[r] : nullptr;
  }
  key[nkey++] = y;
  // the MMA variant sets the W box; the AR output map's part rows follow the chunk count
  key[nkey++] = reinterpret_cast<const void*>(static_cast<intptr_t>(cg * 1000 + groups));
  const bool fp8 = c->dtype == TPO_FP8_E4M3;
  const int elem = fp8 ? 1 : 2;
  const int kel = tpo::BK_BYTES / elem;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!cache_lookup(c, op, key, nkey, p)) {
    bool ok = true;
    for (int r = 0; r < c->tp && ok; ++r) {
      ok = encode3d(&p.mapA[r], x[r], dt, elem, kr, c->n, 1, kel, tpo::BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode2d(&p.mapB[r], w[r], dt, elem, kr, c->m, kel, tpo::BN / cg, CU_TENSOR_MAP_SWIZZLE_128B);
      if (ok && op == tpo::OP_RS)
        ok = encode3d(&p.mapY[r], yb[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->m, c->n / c->tp, 1,
                      tpo::EPI_COLS, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    }
    if (ok && op == tpo::OP_AR)  // one map slot per ring-order part of every row chunk
      ok = encode3d(&p.mapY[0], y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c->m, part_rows,
                    static_cast<uint64_t>(groups) * c->tp, tpo::EPI_COLS, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return fail(TPO_ERR_INVALID_ARG, "tensor map encoding failed (pointer or size not TMA-compatible)");
    cache_store(c, op, key, nkey, p);
  }
  p.rows_per_group = static_cast<int>(rows_per_group);
  p.part_rows = static_cast<int>(part_rows);
  p.tiles_per_part = static_cast<int>(ceil_div(part_rows, tpo::BM * cg));
  p.row_tiles = (op == tpo::OP_AR) ? c->tp * p.tiles_per_part : p.tiles_per_part;
  p.m = static_cast<int>(c->m);
  p.y_rows = static_cast<int>(part_rows);
  p.num_groups = groups;
  p.kb_per_seg = static_cast<int>(ceil_div(kr * elem, tpo::BK_BYTES));
  p.num_segs = c->tp;
  p.gate = 0;
  p.scale_x = c->ks_scale_x;
  p.scale_w = c->ks_scale_w;
  p.reduce_mode = static_cast<int>(c->reduce);
  p.ws = c->ws;
  // pairs with stage_kblocks 2: two K blocks per stage when every accumulation unit has an even count
  p.kps = (cg == 2 && c->stage_kblocks == 2 &&
           (p.reduce_mode ? p.kb_per_seg : p.num_segs * p.kb_per_seg) % 2 == 0) ? 2 : 1;
  plan_columns(c, p);  // automatic or explicit column plan
  const int tiles = p.total_tiles;  // the GEMM grid follows the plan's tile count
  tpo_status st = reset_trace(c, s);
  if (st != TPO_OK) return st;
  {
    // one done counter per output group (RS owner block, AR row chunk), all on
    // the same target: restart them when the operation or the group count changes
    if (op != c->done_op || groups != c->done_groups) {
      cudaError_t e = cudaMemsetAsync(c->words->done, 0, sizeof(c->words->done), s);
      if (e != cudaSuccess) return cuda_fail(e, "done-counter reset");
      c->done_target = 0;
      c->done_op = op;
      c->done_groups = groups;
    }
    // every epilogue warp of every CTA adds its tile's strip count: per group,
    // row tiles x CTAs x strips x warps, whatever the group's column tiling
    c->done_target += static_cast<uint32_t>(p.row_tiles * cg * p.strips * tpo::EPI_WARPS);
    p.done_target = c->done_target;
  }
  p.num_producers = 0;
  p.num_gemm = gemm_grid(c, cg, c->gemm_ctas ? c->gemm_ctas : c->num_sms, 0, tiles);
  // the running-sum workspace has one block per SM: at most one GEMM CTA per SM
  if (p.reduce_mode && p.num_gemm > c->num_sms) p.num_gemm = c->num_sms - c->num_sms % cg;
  return launch(c, p, p.num_gemm, false, s);
}

tpo_status tpo_gemm_rs(tpo_ctx* c, const void* const* x, const void* const* w, void* const* y, void* stream) {
  if (!c) return fail(TPO_ERR_INVALID_ARG, "NULL context");
  tpo_status st = check_ksplit(c, x, w);
  if (st != TPO_OK) return st;
  if (!y) return fail(TPO_ERR_INVALID_ARG, "y must be an array of tp device pointers");
  for (int r = 0; r < c->tp; ++r)
    if (!aligned16(y[r])) return fail(TPO_ERR_INVALID_ARG, "y[%d] must be non-NULL and 16-byte aligned", r);
  return ksplit_common(c, tpo::OP_RS, x, w, y, nullptr, c->tp, static_cast<cudaStream_t>(stream));
}

tpo_status tpo_gemm_ar(tpo_ctx* c, const void* const* x, const void* const* w, void* y, int n_row_chunks,
                       void* stream) {
  if (!c) return fail(TPO_ERR_INVALID_ARG, "NULL context");
  tpo_status st = check_ksplit(c, x, w);
  if (st != TPO_OK) return st;
  if (!aligned16(y)) return fail(TPO_ERR_INVALID_ARG, "y must be non-NULL and 16-byte aligned");
  if (n_row_chunks < 1 || n_row_chunks > TPO_MAX_ROW_CHUNKS)
    return fail(TPO_ERR_INVALID_ARG, "n_row_chunks=%d outside [1, %d]", n_row_chunks, TPO_MAX_ROW_CHUNKS);
  if (c->n % (static_cast<int64_t>(n_row_chunks) * c->tp) != 0)
    return fail(TPO_ERR_UNSUPPORTED, "n=%lld must be a multiple of n_row_chunks*tp (equal ring-order parts)",
                (long long)c->n);
  return ksplit_common(c, tpo::OP_AR, x, w, nullptr, y, n_row_chunks, static_cast<cudaStream_t>(stream));
}

tpo_status tpo_set_fp8_scales(tpo_ctx* c, const float* d_scale_inv_x, const float* d_scale_inv_w) {
  if (!c) return fail(TPO_ERR_INVALID_ARG, "NULL context");
  if (c->dtype != TPO_FP8_E4M3) return fail(TPO_ERR_INVALID_ARG, "scales apply to e4m3 contexts only");
  if (!d_scale_inv_x || !d_scale_inv_w) return fail(TPO_ERR_INVALID_ARG, "scale pointers must be non-NULL");
  c->ks_scale_x = d_scale_inv_x;
  c->ks_scale_w = d_scale_inv_w;
  return TPO_OK;
}

tpo_status tpo_sync_status(tpo_ctx* c) {
  if (!c) return fail(TPO_ERR_INVALID_ARG, "NULL context");
  cudaError_t e = cudaSuccess;
  if (c->has_last) e = cudaEventSynchronize(c->last);
  if (e != cudaSuccess) return cuda_fail(e, "synchronise");
  uint32_t err[4];
  e = cudaMemcpyAsync(err, c->words->err, sizeof(err), cudaMemcpyDeviceToHost, c->aux);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->aux);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (err[0] == tpo::DEV_OK) return TPO_OK;
  std::memcpy(c->last_dev_err, err, sizeof(err));
  // make the context usable again: counters and error word back to zero
  e = cudaMemsetAsync(c->words, 0, offsetof(tpo::DevWords, pad), c->aux);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->aux);
  if (e != cudaSuccess) return cuda_fail(e, "reset after device failure");
  std::memset(c->target, 0, sizeof(c->target));
  c->part_epoch = 0;
  c->done_target = 0;
  c->done_op = -1;
  c->done_groups = 0;
  c->sched_base = 0;
  return fail(TPO_ERR_TIMEOUT, "device wait timed out (site %u, block %u, extra %u)", err[1], err[2], err[3]);
}

tpo_status tpo_last_device_error(tpo_ctx* c, uint32_t out[4]) {
  if (!c || !out) return fail(TPO_ERR_INVALID_ARG, "NULL argument");
  std::memcpy(out, c->last_dev_err, sizeof(c->last_dev_err));
  return TPO_OK;
}

const void* tpo_staging_ptr(tpo_ctx* c) { return c ? c->staging : nullptr; }

const uint32_t* tpo_done_counters(tpo_ctx* c, uint32_t* target) {
  if (!c) return nullptr;
  if (target) *target = c->done_target;
  return c->words->done;
}

tpo_status tpo_read_trace(tpo_ctx* c, uint64_t* out, int cap) {
  if (!c || !out || cap < 1) return fail(TPO_ERR_INVALID_ARG, "bad arguments");
  if (c->has_last) {
    cudaError_t e = cudaEventSynchronize(c->last);
    if (e != cudaSuccess) return cuda_fail(e, "synchronise");
  }
  const int nw = cap < TPO_TRACE_WORDS ? cap : TPO_TRACE_WORDS;
  cudaError_t e = cudaMemcpyAsync(out, c->words->trace, sizeof(uint64_t) * nw, cudaMemcpyDeviceToHost, c->aux);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->aux);
  return e == cudaSuccess ? TPO_OK : cuda_fail(e, "read trace");
}

}  // extern "C"
