// Launch parameters shared by the host launcher (ctx.cu) and the fused kernel
// (kernels.cu).  Private to libtpoverlap.
#pragma once

#include <cuda.h>
#include <stdint.h>
#include <string.h>

#include "tpoverlap.h"

namespace tpo {

// Tile shape.  A CTA owns BM rows of a BN-column output tile.  With the
// single-SM MMA (CG = 1) one CTA computes a BM x BN tile; with the 2-SM MMA
// (tcgen05 cta_group::2, CG = 2) a CTA pair computes a 2*BM x BN tile, each CTA
// loading its own BM rows of A and half (BN/2 rows) of the B tile.  Every
// pipeline stage holds 128-byte K slices (64 bf16 or 128 e4m3 contraction
// elements), the width of one 128-byte swizzle row.
constexpr int BM = TPO_BLOCK_M;
constexpr int BN = TPO_BLOCK_N;
constexpr int BK_BYTES = 128;
constexpr int A_STAGE_BYTES = BM * BK_BYTES;  // 16 KiB
constexpr int STAGE_AREA = 196608;            // 192 KiB of pipeline stages
template <int CG>
struct Pipe {
  static constexpr int B_ROWS = BN / CG;                  // B rows one CTA loads per K block
  static constexpr int B_STAGE_BYTES = B_ROWS * BK_BYTES;  // 32 or 16 KiB per K block
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;  // one K block of A and B
  static constexpr int STAGES = STAGE_AREA / STAGE_BYTES;  // 4 or 6 stages of one K block
  static constexpr int TILE_M = BM * CG;                  // output rows of one tile
};
// A stage may hold kps K blocks (A blocks first, then B blocks); the stage
// count follows: STAGE_AREA / (kps * Pipe<CG>::STAGE_BYTES).
constexpr int MAX_STAGES = 6;
constexpr int NUM_THREADS = 192;              // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int EPI_WARPS = 4;
constexpr int EPI_COLS = 32;                  // columns per epilogue store box
// Tile widths are whole 32-column strips (one epilogue store box each): a
// group's strips across m are split evenly into its column tiles, each of
// MIN_TILE_STRIPS .. BN / STRIP strips.
constexpr int STRIP = EPI_COLS;
constexpr int MAX_TILE_STRIPS = BN / STRIP;   // 8: a full BN-column tile
constexpr int MIN_TILE_STRIPS = 4;            // narrowest tile a column plan may choose (128 columns)
constexpr int MAX_GROUPS = TPO_MAX_ROW_CHUNKS;  // tile groups of one launch (AG slots, RS blocks, AR chunks)
constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 2;  // 32 rows x 32 bf16
constexpr int TMEM_COLS = 512;                // two BN-column fp32 accumulators

// Producer (chunk copy) role: bulk copies through a ring of shared buffers.
constexpr int COPY_PIECE = 16384;
constexpr int COPY_BUFS = 12;
constexpr int COPY_LAG = 6;

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int SMEM_STAGES = 0;
constexpr int SMEM_EPI = SMEM_STAGES + STAGE_AREA;                      // 196608
constexpr int SMEM_BARS = SMEM_EPI + EPI_WARPS * 2 * EPI_BUF_BYTES;     // 212992
// barriers: full[MAX_STAGES], empty[MAX_STAGES], tmem_full[2], tmem_empty[2],
// drain, copy[COPY_BUFS], part[EPI_WARPS] (split-tile finishers' bulk copies),
// tile_full[TQ_DEPTH], tile_empty[TQ_DEPTH] (the dynamic tiles' index ring)
constexpr int TQ_DEPTH = 4;  // tile indices a CTA group's claiming thread may run ahead of its slowest role
constexpr int BAR_FULL = 0, BAR_EMPTY = MAX_STAGES, BAR_TFULL = 2 * MAX_STAGES, BAR_TEMPTY = BAR_TFULL + 2,
              BAR_DRAIN = BAR_TEMPTY + 2, BAR_COPY = BAR_DRAIN + 1, BAR_PART = BAR_COPY + COPY_BUFS,
              BAR_TQ_FULL = BAR_PART + EPI_WARPS, BAR_TQ_EMPTY = BAR_TQ_FULL + TQ_DEPTH;
constexpr int NUM_BARS = BAR_TQ_EMPTY + TQ_DEPTH;
constexpr int SMEM_TMEM_SLOT = SMEM_BARS + NUM_BARS * 8;
constexpr int SMEM_TAIL = SMEM_TMEM_SLOT + 16;   // split builds: the CTA group's schedule (64 bytes)
constexpr int SMEM_TQ = SMEM_TAIL + 64;          // dynamic tiles: the ring of claimed tile indices
constexpr int SMEM_USED = SMEM_TQ + 4 * TQ_DEPTH;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for aligning the base
static_assert(COPY_BUFS * COPY_PIECE <= STAGE_AREA, "copy ring must fit the stage area");
static_assert(Pipe<1>::STAGES * Pipe<1>::STAGE_BYTES <= STAGE_AREA && Pipe<2>::STAGES <= MAX_STAGES, "stages");
static_assert(SMEM_ALLOC <= 232448, "exceeds the per-CTA shared memory limit");

enum Op : int { OP_AG = 0, OP_RS = 1, OP_AR = 2 };

constexpr int MAX_GEMM_CTAS = 256;  // GEMM CTAs of one launch (at most one per SM)
// AG tail split: the tiles left over after the whole rounds are divided along
// K among at most TAIL_SPLIT x (leftover tiles) CTA groups.
constexpr int TAIL_SPLIT = 2;

// Device error word layout: [0] code, [1] site, [2] block, [3] slot/extra.
enum DevErr : uint32_t { DEV_OK = 0, DEV_TIMEOUT = 1 };
enum Site : uint32_t {
  SITE_COUNTER = 1,    // GEMM TMA thread waiting on a chunk counter
  SITE_EMPTY = 2,      // TMA thread waiting for a free stage
  SITE_FULL = 3,       // MMA warp waiting for a loaded stage
  SITE_TMEM_EMPTY = 4, // MMA warp waiting for a drained accumulator
  SITE_TMEM_FULL = 5,  // epilogue waiting for a finished accumulator
  SITE_COPY = 6,       // producer waiting for a bulk load
  SITE_DRAIN = 7,      // clean-up waits after a failure
  SITE_PARTIAL = 8,    // epilogue waiting for a split tile's partial
  SITE_TILE = 9        // a role waiting for its pair's next tile index (dynamic tiles)
};

// A CTA group's schedule with the AG tail split (see SegIter in the kernel),
// worked out on the host once per plan and read by each CTA during its
// set-up.  The tail range is a later part of one tile (K units [wr_lo,
// wr_hi)), whole tiles [tw0, tw1), then the first part of one more tile (K
// units [0, fin_hi), whose later parts the groups fin_w0 .. fin_w0+fin_nw-1
// hold); whole rounds (nfull tiles from whole_base + slot, stride G) come
// after the tail range (first) or before it.
struct TailDesc {
  int first, nfull, whole_base, slot, tail_base;
  int has_wr, wr_t, wr_lo, wr_hi, tw0, tw1, has_fin, fin_t, fin_hi, fin_w0, fin_nw;
};
static_assert(sizeof(TailDesc) == 64, "one 64-byte line per group");

// Per-context device words (one allocation).
struct DevWords {
  uint32_t counters[TPO_MAX_TP];        // per-slot chunk counters (monotonic)
  uint32_t err[4];
  uint32_t done[TPO_MAX_ROW_CHUNKS];    // per output group done counters (RS owner block, AR row chunk; monotonic)
  uint32_t part_ready[MAX_GEMM_CTAS * 4];  // per GEMM CTA and epilogue warp: launch number of its last stored partial
  uint32_t sched;                        // dynamic tiles: claims of every launch so far (monotonic)
  uint32_t pad[11];
  unsigned long long trace[TPO_TRACE_WORDS];
};

struct Params {
  // Tensor maps.  A and Y maps are 3-D [inner, rows, slot] so that tiles clip at
  // slot edges; B maps are 2-D [k, m].
  CUtensorMap mapA[TPO_MAX_TP];  // AG: [0] staging [k, n/tp, tp], [1] X_self [k, n/tp, 1]; RS/AR: X_r [k/tp, n, 1]
  CUtensorMap mapB[TPO_MAX_TP];  // AG: [0] W; RS/AR: W_r
  CUtensorMap mapY[TPO_MAX_TP];  // AG: [0] Y [m, n/tp, tp]; RS: y[b] [m, n/tp, 1]; AR: [0] Y [m, part rows, parts]
  const uint8_t* src[TPO_MAX_TP];  // producer sources X_r
  uint8_t* staging;
  float* ws;              // RS/AR epilogue-reduction modes: a BM x BN fp32 running sum per GEMM CTA
  const TailDesc* tail_tab;  // AG tail split: one TailDesc per CTA group
  DevWords* words;
  const float* scale_x;
  const float* scale_w;
  long long chunk_bytes;
  unsigned long long timeout_ns;
  unsigned long long delay_ns;
  uint32_t target[TPO_MAX_TP];  // per slot: counter value once this call has published it
  uint32_t done_target;   // RS/AR done-counter value once this call stored the whole group
  uint32_t part_target;   // AG tail split: this launch's number (part_ready value of a stored partial)
  uint32_t sched_base;    // dynamic tiles: words->sched at this launch's start (claims minus this = tile index)
  int op;
  int fp8;
  int tp;
  int self_rank;
  int num_producers;      // CTAs [0, num_producers) run the producer role
  int num_gemm;           // CTAs [num_producers, +num_gemm) run the GEMM role
  int rows_per_group;     // AG: rows per slot; RS: rows per block; AR: rows per chunk
  int row_tiles;          // row tiles per group (the last one may be partial)
  int strips;             // 32-column strips across m (the last one may be partial)
  int uniform_cols;       // > 0: every group has this many column tiles (group_cols unused)
  int total_tiles;        // tiles of the launch over all groups
  int group_cols[MAX_GROUPS];      // column tiles of each group (strips split evenly among them)
  int group_base[MAX_GROUPS + 1];  // first tile of each group
  int part_rows;          // AR: rows of one ring-order part of a chunk (rows_per_group / tp)
  int tiles_per_part;     // AR: row tiles per part
  int m;                  // output columns
  int y_rows;             // rows of one slot of the output map (store boxes starting past it are skipped)
  int num_groups;         // AG: tp slots; RS: tp blocks; AR: row chunks
  int kb_per_seg;         // 128-byte K blocks per segment
  int num_segs;           // AG: 1; RS/AR: tp
  int gate;               // 1: wait on chunk counters before loading a slot
  int skip_slot;          // debug: never publish this slot (-1 off)
  int last_step;          // debug: producer stops after this ring step (-1 all)
  int only_step;          // producer copies this ring step only (-1: every step)
  int kps;                // 128-byte K blocks per pipeline stage (1, or 2 for CTA pairs)
  int reduce_mode;        // RS/AR: 0 chain the ranks' K-slices in one accumulator, 1 add per-rank
                          // partials in the epilogue (fp32), 2 as 1 with bf16 rounding of every
                          // partial and running sum (a bf16 ring's wire format)
  int trace_on;
  int cta_group;          // 1: single-SM MMA, 2: CTA pairs (cluster of 2) with the 2-SM MMA
  int tail_split;         // AG: split tail tiles along K (see SegIter in the kernel)
  int split_tail_first;   // tail tiles first (1) or after split_full whole rounds (0)
  int split_full;         // whole rounds of the GEMM groups
  int split_ga, split_gb; // groups of the two tail bands
  long long split_wa, split_wb;  // tail K units of the two bands
  int late_groups;        // producer CTA groups that join the GEMM after their copy
  int copy_on;            // producer CTAs copy (0: they only run as late GEMM groups)
  int skip_part;          // test hook: this GEMM CTA never publishes its partial (-1: none)
  int pdl;                // host side: launch with programmatic dependent launch (set-up overlaps the launch before)
  int dyn;                // builds without the split: each CTA group claims its next tile from words->sched
                          // (1) instead of taking tiles g, g+G, ... (0)
};

// Column tiling of a launch with p.num_groups groups of p.row_tiles row tiles
// over m columns.  extra[g] (or all zero if extra is null) adds column tiles
// to group g beyond the fewest that keep every tile at most BN wide; the
// caller keeps each group within [ceil(strips / 8), strips] tiles.
inline void set_columns(Params& p, long long m, const int* extra) {
  p.strips = static_cast<int>((m + STRIP - 1) / STRIP);
  const int base = (p.strips + MAX_TILE_STRIPS - 1) / MAX_TILE_STRIPS;
  bool uniform = true;
  p.group_base[0] = 0;
  for (int g = 0; g < p.num_groups; ++g) {
    p.group_cols[g] = base + (extra ? extra[g] : 0);
    uniform = uniform && p.group_cols[g] == base;
    p.group_base[g + 1] = p.group_base[g] + p.row_tiles * p.group_cols[g];
  }
  p.uniform_cols = uniform ? base : 0;
  p.total_tiles = p.group_base[p.num_groups];
}

// A tile of the launch (see tile_at in the kernel): its group, its column
// index inside the group's column sweep and its row tile.  Host and device
// share this arithmetic, so that the host's schedule model walks the tiles
// the kernel computes.
struct TileIndex {
  int group, c, r;
};
template <int TILE_M>
__host__ __device__ __forceinline__ TileIndex tile_index(const Params& p, int t) {
  constexpr int RB = 2048 / TILE_M;  // row tiles per swept block
  int grp, cols, rem;
  if (p.uniform_cols > 0) {
    const int per_group = p.row_tiles * p.uniform_cols;
    grp = t / per_group;
    rem = t - grp * per_group;
    cols = p.uniform_cols;
  } else {
    grp = 0;
    while (grp + 1 < p.num_groups && t >= p.group_base[grp + 1]) ++grp;
    rem = t - p.group_base[grp];
    cols = p.group_cols[grp];
  }
  const int full = p.row_tiles / RB;  // whole blocks of RB row tiles
  TileIndex ti;
  ti.group = grp;
  if (rem < full * RB * cols) {
    const int b = rem / (RB * cols), w = rem - b * RB * cols;
    ti.c = w / RB;
    ti.r = b * RB + (w - ti.c * RB);
  } else {  // the last, shorter block
    const int h = p.row_tiles - full * RB, w = rem - full * RB * cols;
    ti.c = w / h;
    ti.r = full * RB + (w - ti.c * h);
  }
  return ti;
}
// First strip of column tile c of a group with `cols` column tiles.
__host__ __device__ __forceinline__ int tile_strip0(const Params& p, int cols, int c) {
  return static_cast<int>(static_cast<long long>(c) * p.strips / cols);
}
__host__ __device__ __forceinline__ int group_cols_of(const Params& p, int grp) {
  return p.uniform_cols > 0 ? p.uniform_cols : p.group_cols[grp];
}

// Zeroes a launch description and sets every field whose "off" value is not 0.
inline void init_params(Params& p) {
  memset(&p, 0, sizeof(p));
  p.skip_slot = -1;
  p.last_step = -1;
  p.only_step = -1;
  p.skip_part = -1;
  p.copy_on = 1;
  p.cta_group = 1;
  p.kps = 1;
}

// Host-side launch helpers defined next to the kernel (kernels.cu).
cudaError_t configure_kernel();
cudaError_t max_blocks_per_sm(int* n);
// Largest number of co-resident CTA pairs of the 2-SM variant (0 if pairs cannot be placed).
cudaError_t max_active_pairs(int* n);
// Launches the variant p.cta_group selects; pair launches use clusters of 2.
cudaError_t launch_fused(const Params& p, int grid, bool cooperative, cudaStream_t stream);

// Sets the thread-local message returned by tpo_last_error (ctx.cu).
void set_last_error(const char* msg);

}  // namespace tpo
