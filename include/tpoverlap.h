/*
 * libtpoverlap -- tensor-parallel linear layers whose GEMM overlaps the movement
 * of its operand or result chunks, on one GB300 (sm_103a).
 *
 * The tp "ranks" of a tensor-parallel group are simulated as tp chunk buffers in
 * one GPU's memory.  Three operations are provided:
 *
 *   AG+GEMM   Y = allgather_rows(X_0 .. X_tp-1) . W^T, rows in rank order.
 *             TransformerEngine issue "curious about atomic_gemm_overlap_ag",
 *             listing of CommOverlapP2PBase::atomic_gemm_overlap_ag: a ring of
 *             chunk send/recv steps fills the gathered buffer, a per-chunk
 *             producer counter marks each chunk ready, and one GEMM consumes
 *             the chunks as their counters flip.
 *   GEMM+RS   Y = sum_r X_r . W_r^T, rank b receives row block b.
 *             TransformerEngine PR "Comm+GEMM overlap API updated to support
 *             cuBlasMp backend", sequence diagram, GEMM + reduce-scatter path.
 *   GEMM+AR   Y = sum_r X_r . W_r^T in full, produced in row chunks.
 *             nvFuser PR "Reference implementation for Linear+Allreduce with
 *             overlapping": row-parallel linear, per-chunk matmul then
 *             all-reduce SUM.
 *
 * Conventions (TN layout, as the listing's transa/transb and m/n naming):
 *   n  rows of Y (tokens), m  columns of Y (output features),
 *   k  the GLOBAL contraction length.  For AG every X_r is [n/tp, k]; for RS and
 *      AR every rank holds a K-slice, X_r [n, k/tp] and W_r [m, k/tp].
 *   All matrices are dense row-major; X and W are "K-major" (the contraction
 *   index is contiguous); Y is always bf16.
 *   bf16 buffers hold IEEE bfloat16, e4m3 buffers OCP FP8 E4M3 codes.
 *
 * Ownership: the caller owns every X, W, Y buffer and the stream.  The context
 * owns the staging buffer (the gathered X), the per-chunk counters, the device
 * error word and the trace buffer; all are allocated by tpo_ctx_create and
 * nothing is allocated by the per-call entry points.
 *
 * Calls are stream-ordered and asynchronous: they validate their arguments on
 * the host, enqueue work on `stream` (a cudaStream_t passed as void*, NULL for
 * the legacy default stream) and return.  Inputs must stay valid until the
 * stream reaches the call.  Argument errors are reported synchronously before
 * anything is enqueued.  A device-side failure (a bounded wait that ran out) is
 * recorded in the context's error word and reported by the next
 * tpo_sync_status; until then the word is sticky and later calls on the
 * context abort early.  Every entry point sets a thread-local message readable
 * through tpo_last_error when it fails.
 *
 * A context is not thread-safe: calls on one context must come from one host
 * thread at a time.  Calls that overlap on the GPU (different streams) must use
 * different contexts.
 */
#ifndef TPOVERLAP_H
#define TPOVERLAP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tpo_ctx tpo_ctx; /* opaque */

/* Input element type (Y is always bf16). */
typedef enum { TPO_BF16 = 0, TPO_FP8_E4M3 = 1 } tpo_dtype;

typedef enum {
  TPO_OK = 0,
  TPO_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or option */
  TPO_ERR_UNSUPPORTED = 2, /* valid request outside what the library supports */
  TPO_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  TPO_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out */
  TPO_ERR_OOM = 5          /* device allocation failed in tpo_ctx_create */
} tpo_status;

/* Operation limits of the library. */
#define TPO_MAX_TP 16
#define TPO_MAX_ROW_CHUNKS 64
#define TPO_BLOCK_M 128 /* rows of one output tile */
#define TPO_BLOCK_N 256 /* columns of one output tile */
/* Sizes need not be multiples of the tile: the last tile of a slot, block or
 * part loads zeros past its edge and stores only the rows and columns that
 * exist.  Row pitches must be multiples of 16 bytes. */

/*
 * Create a context for one problem size on the current CUDA device.
 *   tp     number of simulated ranks, 1..16
 *   n      rows of Y, a multiple of tp (every rank holds n/tp rows)
 *   k      global contraction length: a multiple of 8 (bf16) or 16 (e4m3);
 *          for RS/AR also k % tp == 0 and k/tp a multiple of 8 (16 for e4m3)
 *   m      columns of Y, a multiple of 8
 *   dtype  a tpo_dtype value
 * Allocates the staging buffer (n*k elements), counters, error word and trace
 * buffer on the current device.  Returns NULL on any error (no half-built
 * context is ever returned); tpo_last_error says why.
 * The signature follows the context-handle pattern of the cuBLASMp backend in
 * TransformerEngine PR "Comm+GEMM overlap API updated to support cuBlasMp
 * backend" (nvte_comm_gemm_ctx_create ... nvte_comm_gemm_ctx_destroy).
 */
tpo_ctx* tpo_ctx_create(int tp, int64_t n, int64_t k, int64_t m, int dtype);

/* Release everything the context owns (synchronises with its pending work).
 * tpo_ctx_destroy(NULL) is a no-op returning TPO_OK. */
tpo_status tpo_ctx_destroy(tpo_ctx* ctx);

/*
 * AG+GEMM: Y[n, m] = gather(X_0..X_tp-1)[n, k] . W[m, k]^T, Y rows in rank order.
 *   x      host array of tp device pointers; x[r] is rank r's chunk [n/tp, k]
 *   w      device pointer, [m, k]
 *   y      device pointer, [n, m] bf16
 *   d_scale_inv_x, d_scale_inv_w
 *          e4m3 contexts: device pointers to one fp32 each (the per-tensor
 *          scale_inv of all X_r together and of W); the product is multiplied
 *          by both in fp32 before rounding.  bf16 contexts: must be NULL.
 *   stream cudaStream_t
 * Semantics (listing of atomic_gemm_overlap_ag): the observer rank `self_rank`
 * (option, default 0) holds its own chunk and receives the others in ring
 * order self-1, self-2, ... (mod tp).  A producer role copies each arriving
 * chunk into its rank-order slot of the staging buffer and publishes the
 * slot's counter with release semantics; the GEMM role acquire-waits on that
 * counter before its first tensor-memory load of the slot.  Y is written in
 * rank order directly (no rotation buffer).  All pointers 16-byte aligned.
 * The result is bit-identical in every mode (option "mode").
 */
tpo_status tpo_ag_gemm(tpo_ctx* ctx, const void* const* x, const void* w, void* y,
                       const float* d_scale_inv_x, const float* d_scale_inv_w, void* stream);

/*
 * GEMM+RS: y[b] = rows [b*n/tp, (b+1)*n/tp) of sum_r X_r . W_r^T.
 *   x   host array of tp device pointers, X_r [n, k/tp]
 *   w   host array of tp device pointers, W_r [m, k/tp]
 *   y   host array of tp device pointers, y[b] [n/tp, m] bf16
 * The partial products are summed in a fixed ring order inside one GEMM:
 * the output rows owned by rank b accumulate ranks b+1, b+2, ..., b (mod tp),
 * the order of a ring reduce-scatter that ends at the owner, in fp32, with a
 * single rounding to bf16 in the epilogue.  e4m3 contexts take their scales
 * from tpo_set_fp8_scales.  Blocks are produced in order (block 0 first);
 * after every tile of block b is stored, block b's done counter (see
 * tpo_done_counters) reaches its target with release semantics.
 */
tpo_status tpo_gemm_rs(tpo_ctx* ctx, const void* const* x, const void* const* w, void* const* y,
                       void* stream);

/*
 * GEMM+AR (row-parallel linear): Y[n, m] = sum_r X_r . W_r^T.
 *   x, w          as tpo_gemm_rs
 *   y             device pointer [n, m] bf16
 *   n_row_chunks  1..64; n must be a multiple of n_row_chunks*tp
 * Output tiles are produced chunk by chunk (row chunk 0 first).  Inside row
 * chunk c, the rows of the chunk's i-th of tp equal parts sum ranks i+1, ...,
 * i (mod tp), the per-part order of a ring all-reduce of that chunk.  After
 * every tile of chunk c is stored, the chunk's done counter (see
 * tpo_done_counters) reaches its target with release semantics.  e4m3
 * contexts as tpo_gemm_rs.
 */
tpo_status tpo_gemm_ar(tpo_ctx* ctx, const void* const* x, const void* const* w, void* y,
                       int n_row_chunks, void* stream);

/*
 * Scales for GEMM+RS / GEMM+AR on an e4m3 context: device pointers to one fp32
 * each, the scale_inv shared by all X_r and the one shared by all W_r (one
 * per-tensor scale across the ranks' K-slices, as the gathered AG input
 * carries one).  The accumulated sum is multiplied by both in fp32 before the
 * bf16 rounding.  The pointers are read by every later RS/AR call (they must
 * stay valid); required before the first RS/AR call of an e4m3 context;
 * TPO_ERR_INVALID_ARG on a bf16 context or NULL pointers.
 */
tpo_status tpo_set_fp8_scales(tpo_ctx* ctx, const float* d_scale_inv_x, const float* d_scale_inv_w);

/*
 * Options (integers).  Keys:
 *   "producer_sms"     CTAs given to the chunk producer in overlapped AG; 0 (the
 *                      default) picks, from a model of the copy and GEMM rates
 *                      and the round-robin tile schedule, the fewest CTAs
 *                      whose copy does not delay the GEMM (at most 32; even
 *                      for pairs); with tail_split 1, the smallest count from
 *                      4 whose copy stays ahead of the split schedule; an odd
 *                      count for pairs is rounded up
 *   "gemm_ctas"        CTAs given to the GEMM (0 = all SMs not producing)
 *   "tail_split"       AG, modes 0-2 (default 0: whole tiles only, and every
 *                      grid, mode and producer count gives the same bits).
 *                      1: the tiles left over after the GEMM CTAs' whole
 *                      rounds go first and are divided along K among them;
 *                      2: the producer CTAs join the GEMM once their copy is
 *                      done, and the last tiles are divided along K between
 *                      the GEMM CTAs (a short share each) and them (the rest),
 *                      sized from a model of both rates; 3: as 1 but the
 *                      leftover tiles come after the whole rounds.  Each later K part of
 *                      a split tile is an fp32 partial in the context's
 *                      workspace, added in K order to the first part before
 *                      the bf16 rounding, so the result depends on the plan:
 *                      modes 1 and 2 then run mode 0's launch shape and plan
 *                      (same bits in all three); other producer counts,
 *                      gemm_ctas values and mode 4 (never split) may round
 *                      split tiles differently.
 *   "mode"             AG schedule: 0 overlapped (one launch, producer and GEMM
 *                      co-resident), 1 sequential (copy to completion, then the
 *                      same GEMM), 2 GEMM only (staging and counters must hold a
 *                      previous call's chunks), 3 producer only (no GEMM; y is
 *                      not written), 4 split: per ring step one chunk copy on a
 *                      side stream and one GEMM launch over that slot after it
 *                      (no counters; the multi-launch design of the split
 *                      all-gather overlap in TransformerEngine PR "Comm+GEMM
 *                      overlap API updated to support cuBlasMp backend" and the
 *                      ring decomposition of nvFuser PR "Ring-based
 *                      decomposition for Allgather+GEMM overlap ATen
 *                      implementation"), for comparison
 *   "seq_copy_ctas"    CTAs of the copy in sequential mode (0 = all SMs)
 *   "self_rank"        observer rank for the ring order, 0..tp-1
 *   "wait_timeout_ms"  bound of every device-side wait (default 2000)
 *   "trace"            1 = record device timestamps (tpo_read_trace)
 *   "debug_skip_chunk" slot whose counter the producer never publishes (-1 off)
 *   "debug_delay_ns"   producer spin before each publish
 *   "debug_last_step"  mode 3 only: the producer stops after this ring step
 *                      (-1 = all steps)
 *   "debug_skip_partial" GEMM CTA (index among the GEMM CTAs) that never
 *                      publishes its split-tile partial (-1 off): the tile's
 *                      finisher times out
 *   "stage_kblocks"    128-byte K blocks per shared-memory pipeline stage of
 *                      the CTA-pair variant: 1 (default; six stages of one
 *                      K block, each released as soon as its MMAs are done)
 *                      or 2 (three stages of two, one barrier test per eight
 *                      MMAs; used only where every accumulation unit has an
 *                      even number of K blocks).  Results are identical; one
 *                      block per stage measured 1.4-2.6 % faster on 4096^3.
 *   "col_split"        column tiles per tile group (AG ring step, RS owner
 *                      block, AR row chunk), the group's 32-column strips
 *                      split evenly among them: -1 the fewest tiles of at
 *                      most 256 columns; 0 (default) automatic: the fewest,
 *                      unless the launch has at most half as many tiles as
 *                      it can have GEMM CTA groups (the SMs, less 32 for the
 *                      AG producers, per MMA variant), then as many narrower
 *                      tiles per group (down to 32 columns) as still fit in
 *                      one round; otherwise 4 bits per group g < 16
 *                      ((v >> 4g) & 15) of extra tiles.  The GEMM grid
 *                      follows the plan's tile count.  Results are identical
 *                      (the MMA computes every output element the same way
 *                      whatever the tile width).  A K block of a narrower
 *                      tile costs less, but not in proportion (at 192
 *                      columns ~0.86 of a 256-column one: the operand loads
 *                      bound it), so more tiles pay only where they all fit
 *                      in one round: each tile's epilogue is then shorter.
 *   "sched"            which CTA group computes which tile: 1 round robin
 *                      (group g takes tiles g, g+G, g+2G, ...); 2 dynamic
 *                      (each group claims its next tile from a launch-wide
 *                      counter, so that faster groups take more tiles and
 *                      the tiles in flight stay a contiguous run of the tile
 *                      order); 0 (default) automatic: dynamic for launches of
 *                      at least 8 rounds, round robin otherwise and with the
 *                      AG tail split.  Results are identical either way.
 *   "cta_group"        MMA variant: 0 automatic, 1 single-SM 128x256 tiles,
 *                      2 CTA pairs (2-SM MMA, 256x256 tiles; needs every tile
 *                      group a multiple of 256 rows).  Results are identical.
 *   "cooperative"      0 (default): overlapped AG is a plain launch whose grid
 *                      never exceeds the co-resident CTA count, so once no
 *                      other work holds SMs every producer and GEMM CTA runs at
 *                      once (if other work does, a GEMM CTA's wait for a chunk
 *                      is bounded: TPO_ERR_TIMEOUT, never a hang); 1: a
 *                      cooperative launch, whose co-residency the driver
 *                      guarantees, but which cannot start before the launch
 *                      ahead of it has ended (no "pdl" overlap)
 *   "pdl"              1 (default): every kernel launch is marked for
 *                      programmatic dependent launch: its CTAs may start their
 *                      set-up (barriers, tensor memory) on SMs the previous
 *                      launch on the stream has left and wait (griddepcontrol)
 *                      for that launch's completion before touching global
 *                      memory.  Measured on back-to-back 4096^3 AG calls:
 *                      2.8-3.6 % faster.  0: ordinary stream order.
 *   "reduce"           GEMM+RS / GEMM+AR sum of the ranks' partial products:
 *                      0 (default) chain every rank's K-slice, in ring order,
 *                      into one fp32 accumulator; 1 compute each rank's partial
 *                      on its own and add the partials in ring order in the
 *                      epilogue (fp32); 2 as 1 but round every partial and
 *                      every running sum to bf16, the arithmetic of a bf16
 *                      ring reduce-scatter such as the bf16 ring all-reduce in
 *                      nvFuser PR "Reference implementation for Linear+Allreduce
 *                      with overlapping".  In modes 1 and 2 each rank's
 *                      partial takes one of the two tensor-memory accumulators
 *                      and the running sum lives in a context-owned workspace
 *                      (one 128 x 256 block per SM, fp32 in mode 1, bf16 in
 *                      mode 2), so the MMAs never wait for the additions.
 * Read-only keys for tpo_get_opt: "last_producer_ctas", "last_gemm_ctas",
 * "last_cta_group", "last_stage_kblocks", "last_split_tiles",
 * "last_late_groups", "last_col_plan", "last_sched" (shape of the context's latest kernel
 * launch: producer CTAs, GEMM CTAs, 1 or 2 CTAs per MMA, K blocks per
 * pipeline stage, tiles split along K, producer CTA groups that joined the
 * GEMM, extra column tiles per group in the col_split encoding, each
 * group's count capped at 15 in the report, 1 round robin or 2 dynamic tiles),
 * "coop_clusters" (0 once the driver refused a cooperative cluster launch),
 * "tp", "n", "k", "m", "dtype" (the sizes the context was created for).
 * Environment variables TPO_<KEY in upper case> override the defaults at
 * create time.  Unknown keys or out-of-range values: TPO_ERR_INVALID_ARG.
 */
tpo_status tpo_set_opt(tpo_ctx* ctx, const char* key, int64_t value);
tpo_status tpo_get_opt(tpo_ctx* ctx, const char* key, int64_t* value);

/* Wait for all work this context enqueued, read and clear the device error
 * word.  Returns TPO_OK or the recorded failure (TPO_ERR_TIMEOUT); after a
 * failure the counters are re-zeroed so the context is usable again. */
tpo_status tpo_sync_status(tpo_ctx* ctx);

/* Details of the last device failure seen by tpo_sync_status: code, site,
 * block index, slot (4 words). */
tpo_status tpo_last_device_error(tpo_ctx* ctx, uint32_t out[4]);

/* Thread-local message of the last failing call on this thread ("" if none). */
const char* tpo_last_error(void);

/* Read-only device pointer to the staging buffer [n, k] (the gathered X in rank
 * order), for inspection after a synchronised AG call. */
const void* tpo_staging_ptr(tpo_ctx* ctx);

/* Device pointer to the done counters (TPO_MAX_ROW_CHUNKS uint32 words), one
 * per output group of the latest tpo_gemm_rs (group b = owner block y[b]) or
 * tpo_gemm_ar (group c = row chunk c) call, and the value every group's counter
 * reaches once that call has stored all of the group's rows.  The GEMM raises
 * them with release semantics as it finishes each tile, so a consumer that
 * acquire-loads a counter equal to *target may read the group's rows while
 * the rest of the output is still being computed: the signal the
 * communication side of an atomic GEMM+RS (or of a chunked all-reduce) waits
 * on.  The counters restart from zero when the operation or the group count
 * changes between calls. */
const uint32_t* tpo_done_counters(tpo_ctx* ctx, uint32_t* target);

/* Trace words (uint64 nanoseconds of the device global timer), valid after
 * tpo_sync_status when option "trace" was 1; reset by each traced call. */
#define TPO_TRACE_START 0      /* earliest CTA start */
#define TPO_TRACE_END 1        /* latest CTA end */
#define TPO_TRACE_PUBLISH 2    /* + slot: latest producer publish of the slot */
#define TPO_TRACE_ACQUIRE 18   /* + slot: earliest GEMM acquire of the slot */
#define TPO_TRACE_WAIT_NS 34   /* total ns GEMM CTAs spent waiting on counters */
#define TPO_TRACE_CHUNK_DONE 35 /* + group: completion time of an RS block / AR row chunk */
/* Pipeline diagnosis (SM clock cycles summed over GEMM CTAs): */
#define TPO_TRACE_CYC_TMA_EMPTY 100  /* TMA issuer blocked on a free stage */
#define TPO_TRACE_CYC_MMA_FULL 101   /* MMA issuer blocked on a loaded stage */
#define TPO_TRACE_CYC_MMA_TEMPTY 102 /* MMA issuer blocked on a drained accumulator */
#define TPO_TRACE_CYC_EPI_TFULL 103  /* epilogue warps blocked on a finished accumulator */
#define TPO_TRACE_CYC_GEMM 104       /* GEMM CTAs' total cycles (set-up to tear-down) */
#define TPO_TRACE_KBLOCKS 105        /* 128-byte K blocks issued to the tensor cores */
#define TPO_TRACE_WORDS 128
tpo_status tpo_read_trace(tpo_ctx* ctx, uint64_t* out, int cap);

/* Library build string (compiler, target architecture). */
const char* tpo_version(void);

/*
 * AG+GEMM that allocates no device memory.  The pages have no counterpart of
 * this entry point; it exists for callers that cannot call cudaMalloc when they
 * run the layer: a serving process that reserved all device memory for its own
 * pool at start-up, a runtime whose allocator forbids raw device allocations
 * after initialisation so that its memory use stays fixed, or any code that
 * only owns the buffers it is handed.  tpo_ctx_create allocates, so these
 * callers cannot hold a context.
 *
 * Computes what tpo_ag_gemm computes for observer rank 0 in one overlapped
 * launch with the launch shape tpo_ag_gemm picks under default options (CTA
 * pairs wherever n/tp is a multiple of 256, the automatic column plan, the
 * schedule model's producer count, 2 s wait bound).  The result is
 * bit-identical to tpo_ag_gemm's whenever that call computes whole
 * tiles (option tail_split 0, the default), in any mode and with either MMA
 * variant; the tail-split schedules (tail_split 1 to 3) add K-split partials
 * in an order that depends on their launch shape and agree with it only
 * within the parity tolerance.  Arguments as tpo_ctx_create (tp, n, k, m,
 * dtype) plus tpo_ag_gemm (x, w, y, scale_inv pointers, stream).
 *
 * Scratch (the gathered staging buffer, the chunk counters and the error word)
 * lives in a static device array of the library: TPO_NOALLOC_MAX_STAGING_BYTES
 * plus TPO_NOALLOC_WORDS_BYTES (the kernel's word block rounded up to 256
 * bytes), held by every GPU that loads the library until the process exits.
 * n*k*element size above TPO_NOALLOC_MAX_STAGING_BYTES is rejected with
 * TPO_ERR_INVALID_ARG and a message naming the limit.
 * The first call on a device sets that device up (looks up the array's device
 * address, configures the kernel); make it before any stream capture.
 * Every call shares the array and clears its counters and error word on
 * `stream` first; calls whose GPU work could overlap (other streams, other host
 * threads) race on the array.  The call blocks until its work on `stream` has
 * finished, then returns TPO_OK or TPO_ERR_TIMEOUT if a device wait ran out.
 * If it returns TPO_ERR_CUDA after its launch (the error word could not be
 * read back), it first tries to wait for `stream`; should that fail as well,
 * the kernel may still be running and the array's contents stay undefined
 * until the device is reset.
 */
#define TPO_NOALLOC_MAX_STAGING_BYTES (32ull << 20) /* 32 MiB */
#define TPO_NOALLOC_WORDS_BYTES 5632ull             /* counters, error word, trace: 5.5 KiB */
tpo_status tpo_ag_gemm_noalloc(int tp, int64_t n, int64_t k, int64_t m, int dtype, const void* const* x,
                               const void* w, void* y, const float* d_scale_inv_x,
                               const float* d_scale_inv_w, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TPOVERLAP_H */
