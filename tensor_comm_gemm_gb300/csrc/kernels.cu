// Fused persistent kernel of libtpoverlap (sm_103a).
//
// One launch carries two roles, split by block index:
//
//  * producer CTAs [0, num_producers): the ring-order chunk producer.  Each
//    arriving rank chunk is a contiguous byte range; every producer CTA moves
//    its share with bulk asynchronous copies (global -> shared -> global, 16 KiB
//    pieces through a ring of shared buffers, full-line coalesced writes) and
//    then adds 1 to the slot's counter with release semantics.  This is the role
//    of userbuffers_send/recv plus producer() in TransformerEngine's
//    atomic_gemm_overlap_ag listing (issue "curious about
//    atomic_gemm_overlap_ag"), with the copy moved onto a few SMs.
//
//  * GEMM CTAs: a persistent tcgen05 GEMM.  Warp 0 issues TMA loads (after an
//    acquire-wait on the slot's counter for gathered rows), warp 1 issues
//    tcgen05.mma (one elected lane of the converged warp) into a double-
//    buffered fp32 accumulator in tensor memory, warps 2..5 drain the accumulator (tcgen05.ld), round to
//    bf16 and TMA-store the tile.  In the pair variant (CG = 2) two CTAs of a
//    cluster share one 256 x 256 tile through the 2-SM MMA: each loads its own
//    128 rows of A and half of the B tile, the even CTA issues the MMAs, and
//    each CTA's tensor memory receives its own 128 rows of the result.  This
//    replaces the counter-gated cuBLAS atomic GEMM of the same listing.  For
//    GEMM+RS / GEMM+AR the K loop of a tile walks the ranks' K-slices in a
//    fixed ring order into one accumulator.
//
// The kernel is built three times per tile variant: fused_kernel<CG, false,
// false> (round-robin tiles), fused_kernel<CG, false, true> (dynamic tiles,
// claimed from a launch-wide counter) and fused_kernel<CG, true, false> with
// the optional AG tail split (K-split tiles, fp32 partials, producer CTAs
// joining the GEMM), each launched only when a call asks for its schedule, so
// no build carries the others' code.
//
// Every wait (mbarrier, chunk counter) is bounded by the device global timer.
// On expiry the waiting thread records the failure in the context's error word
// and the CTA winds down: it waits for its own copies in flight, lets issued
// MMAs finish, frees its tensor memory and exits.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "tpo_params.h"

namespace tpo {

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool aborted(const Params& p) {
  return *reinterpret_cast<volatile uint32_t*>(&p.words->err[0]) != 0u;
}

__device__ void raise_error(const Params& p, uint32_t code, uint32_t site, uint32_t extra) {
  if (atomicCAS(&p.words->err[0], 0u, code) == 0u) {
    p.words->err[1] = site;
    p.words->err[2] = blockIdx.x;
    p.words->err[3] = extra;
    __threadfence();
  }
}

// ------------------------------------------------------------------ launch order

// Programmatic dependent launch: a launch that the host marks may begin its
// set-up (barriers, tensor memory) while the launch before it on the stream is
// still running; griddepcontrol.wait then holds the thread until that launch
// has completed and its memory is visible, so nothing before it touches global
// memory.  Without the mark both instructions return at once.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Bounded wait for the phase of parity `parity` to complete.  With
// `honor_abort`, a failure recorded by any CTA also ends the wait (false).
__device__ bool mbar_wait(const Params& p, uint32_t bar, uint32_t parity, uint32_t site, bool honor_abort) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 15u) == 0u) {
      if (honor_abort && aborted(p)) return false;
      if (gtime() - t0 > p.timeout_ns) {
        raise_error(p, DEV_TIMEOUT, site, blockIdx.x);
        return false;
      }
    }
  }
}
// mbar_wait whose completion acquires at cluster scope: arrivals from the
// other CTA of a pair (with release at cluster scope) order that CTA's earlier
// writes before this thread's later accesses.
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}
__device__ bool mbar_wait_cluster(const Params& p, uint32_t bar, uint32_t parity, uint32_t site) {
  if (mbar_test_cluster(bar, parity)) return true;
  const unsigned long long t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_cluster(bar, parity)) return true;
    if ((i & 15u) == 0u) {
      if (aborted(p)) return false;
      if (gtime() - t0 > p.timeout_ns) {
        raise_error(p, DEV_TIMEOUT, site, blockIdx.x);
        return false;
      }
    }
  }
}
// mbar_wait that adds the SM cycles spent blocked to *cycles (trace runs only).
__device__ __forceinline__ bool mbar_wait_timed(const Params& p, uint32_t bar, uint32_t parity, uint32_t site,
                                                bool honor_abort, unsigned long long* cycles) {
  if (!p.trace_on) return mbar_wait(p, bar, parity, site, honor_abort);
  if (mbar_test(bar, parity)) return true;
  const long long c0 = clock64();
  const bool ok = mbar_wait(p, bar, parity, site, honor_abort);
  *cycles += static_cast<unsigned long long>(clock64() - c0);
  return ok;
}
// mbar_wait for all 32 lanes of a converged warp: the same result in every
// lane (the slow path runs in lane 0; afterwards every lane observes the
// completed phase itself).
__device__ __forceinline__ bool mbar_wait_warp(const Params& p, uint32_t bar, uint32_t parity, uint32_t site,
                                               unsigned long long* cycles) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_timed(p, bar, parity, site, true, cycles) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)mbar_test(bar, parity);
  return ok != 0;
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ------------------------------------------------------------------ bulk copies / TMA

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// A operands: [inner K, rows, slot] maps, so a tile's rows never run into the
// next slot (rows past a slot's end read as zeros).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Outputs: [m, rows, slot] maps; the store writes only the part of the box
// inside the slot and inside m.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 16-byte global accesses under an L2 cache policy.
__device__ __forceinline__ void st_global_v4_keep(uint4* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                  uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void ld_global_v4_keep(const uint4* p, uint32_t (&h)[4], uint64_t pol) {
  asm volatile("ld.global.L2::cache_hint.v4.b32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
               : "l"(p), "l"(pol)
               : "memory");
}

// ------------------------------------------------------------------ release / acquire

__device__ __forceinline__ void red_add_release(uint32_t* ptr, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_release(uint32_t* ptr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_release(uint32_t* ptr, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with
// the 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);  // start address, 16-byte units
  d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride byte offset: one 8-row atom
  d |= static_cast<uint64_t>(1) << 46;                 // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                 // swizzle mode: 128 bytes
  return d;
}

// Instruction descriptor: dense, fp32 accumulator, K-major A and B,
// A/B bf16 (kind::f16) or e4m3 (kind::f8f6f4), M = tile rows; the tile's
// width N (a multiple of 32 up to BN) is added per tile with idesc_n.
__host__ __device__ constexpr uint32_t make_idesc(bool fp8, int m) {
  return (1u << 4) | ((fp8 ? 0u : 1u) << 7) | ((fp8 ? 0u : 1u) << 10) | (static_cast<uint32_t>(m >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_n(uint32_t idesc, int n) {
  return idesc | (static_cast<uint32_t>(n >> 3) << 17);
}

// Loads 32 columns of the warp's 32 tensor-memory lanes and waits for them in
// one statement: the compiler never sees the registers before the data landed
// (a separate wait would let it copy them while the load is still in flight).
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}


__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }


// ------------------------------------------------------------------ clusters (CTA pairs)

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA load whose completion is signalled on a barrier that may live in the peer CTA.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_alloc_cg(uint32_t slot_smem, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish_cg() {
  if constexpr (CG == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc_cg(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// The MMA issuer is a whole converged warp; inside each asm statement
// elect.sync picks the one lane that issues.  (Issued from one thread of a
// diverged warp, a tcgen05.mma took ~53 cycles of that thread and a K block's
// four ~213, against ~73 for the four from a converged warp: with the stage
// test and commit around them the single thread needed ~450 cycles per K
// block, more than the tensor core's 384 at N = 192 or 256 at N = 128.)
#define TPO_MMA_KBLOCK(CGS, KIND)                                                                         \
  asm volatile("{\n\t.reg .pred E, A, T;\n\t.reg .b32 r;\n\t"                                              \
               "setp.ne.b32 A, %4, 0;\n\tsetp.ne.b32 T, %5, 0;\n\t"                                        \
               "elect.sync r|E, 0xffffffff;\n\t"                                                          \
               "@E tcgen05.mma.cta_group::" CGS ".kind::" KIND " [%0], %1, %2, %3, A;\n\t"                 \
               "@E tcgen05.mma.cta_group::" CGS ".kind::" KIND " [%0], %6, %7, %3, T;\n\t"                 \
               "@E tcgen05.mma.cta_group::" CGS ".kind::" KIND " [%0], %8, %9, %3, T;\n\t"                 \
               "@E tcgen05.mma.cta_group::" CGS ".kind::" KIND " [%0], %10, %11, %3, T;\n\t}" ::"r"(d),    \
               "l"(a), "l"(b), "r"(idesc), "r"(acc0), "r"(1u), "l"(a + 2u), "l"(b + 2u), "l"(a + 4u),     \
               "l"(b + 4u), "l"(a + 6u), "l"(b + 6u))
// One 128-byte K block: four MMAs of K = 32 bytes (descriptor start addresses
// 32 bytes apart); acc0 = 0 overwrites the accumulator with the first.
// CG = 2 issues the 2-SM form (M = 256 over the pair).
template <int CG, bool FP8>
__device__ __forceinline__ void mma_kblock(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
  if constexpr (CG == 1) {
    if constexpr (FP8)
      TPO_MMA_KBLOCK("1", "f8f6f4");
    else
      TPO_MMA_KBLOCK("1", "f16");
  } else {
    if constexpr (FP8)
      TPO_MMA_KBLOCK("2", "f8f6f4");
    else
      TPO_MMA_KBLOCK("2", "f16");
  }
}
#undef TPO_MMA_KBLOCK
// Arrive on `bar` (same offset in every CTA of the group) once all prior MMAs
// completed; a whole converged warp executes it, one elected lane commits.
template <int CG>
__device__ __forceinline__ void mma_commit_cg(uint32_t bar) {
  if constexpr (CG == 1) {
    asm volatile(
        "{\n\t.reg .pred E;\n\t.reg .b32 r;\n\telect.sync r|E, 0xffffffff;\n\t"
        "@E tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
  } else {
    const uint16_t mask = 0x3;
    asm volatile(
        "{\n\t.reg .pred E;\n\t.reg .b32 r;\n\telect.sync r|E, 0xffffffff;\n\t"
        "@E tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
            bar),
        "h"(mask)
        : "memory");
  }
}
// Commit that arrives on this CTA's barrier only (whole warp, one elected lane).
template <int CG>
__device__ __forceinline__ void mma_commit_local_cg(uint32_t bar) {
  if constexpr (CG == 1)
    mma_commit_cg<1>(bar);
  else
    asm volatile(
        "{\n\t.reg .pred E;\n\t.reg .b32 r;\n\telect.sync r|E, 0xffffffff;\n\t"
        "@E tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// ------------------------------------------------------------------ tile schedule

struct Tile {
  int a_map;  // AG: 0 staging, 1 X_self
  int a_row;  // row coordinate of the A tile in its map
  int a_z;    // slot coordinate of the A tile in its map
  int gate;   // slot whose counter gates the A loads, or -1
  int y_map;  // output map index
  int y_row;  // row coordinate of the output tile in its map
  int y_z;    // slot coordinate of the output tile in its map
  int col;    // first output column (= first W row)
  int ncols;  // tile width: a multiple of 32 up to BN (may reach past m at the right edge)
  int seg0;   // RS/AR: rank of the first K segment
  int group;  // AR: row chunk
};

// Tiles are ordered group by group (AG: ring step, RS: owner block, AR: row
// chunk).  Inside a group, blocks of up to 2048 rows are swept column tile by
// column tile, rows fastest: consecutive CTAs share a W tile, and a block's
// rows of X stay in L2 while its sweep passes over all of W (a group with
// more rows would otherwise stream X from memory once per column tile).  A
// group's column tiles split its 32-column strips evenly (widths differ by at
// most one strip); groups may have different column-tile counts, which the
// host chooses so that the round-robin rounds come out even.
// Every role of a CTA walks the same sequence t = g, g+G, ...
template <int TILE_M>
__device__ __forceinline__ Tile tile_at(const Params& p, int t) {
  const TileIndex ti = tile_index<TILE_M>(p, t);
  const int grp = ti.group, r = ti.r;
  const int cols = group_cols_of(p, grp);
  const int s0 = tile_strip0(p, cols, ti.c), s1 = tile_strip0(p, cols, ti.c + 1);
  Tile T;
  T.col = s0 * STRIP;
  T.ncols = (s1 - s0) * STRIP;
  T.group = grp;
  if (p.op == OP_AG) {
    const int slot = ((p.self_rank - grp) % p.tp + p.tp) % p.tp;
    // ring step 0 is the observer's own chunk: read in place, nothing to wait on
    T.a_map = (grp == 0) ? 1 : 0;
    T.a_row = r * TILE_M;
    T.a_z = (grp == 0) ? 0 : slot;
    T.gate = (grp == 0 || !p.gate) ? -1 : slot;
    T.y_map = 0;
    T.y_row = r * TILE_M;
    T.y_z = slot;
    T.seg0 = 0;
  } else if (p.op == OP_RS) {
    // rows past the block's end (a ragged last tile) are computed but never stored
    T.a_map = -1;
    T.a_row = grp * p.rows_per_group + r * TILE_M;
    T.a_z = 0;
    T.gate = -1;
    T.y_map = grp;
    T.y_row = r * TILE_M;
    T.y_z = 0;
    T.seg0 = (grp + 1) % p.tp;  // ring reduce-scatter: the owner's own slice comes last
  } else {
    // a row chunk is tp ring-order parts (part i sums ranks i+1, ..., i), each
    // tiled on its own so that no tile mixes two summation orders
    const int part = r / p.tiles_per_part, rr = r - part * p.tiles_per_part;
    T.a_map = -1;
    T.a_row = grp * p.rows_per_group + part * p.part_rows + rr * TILE_M;
    T.a_z = 0;
    T.gate = -1;
    T.y_map = 0;
    T.y_row = rr * TILE_M;
    T.y_z = grp * p.tp + part;
    T.seg0 = (part + 1) % p.tp;
  }
  return T;
}

// The work of CTA group g (a CTA, or a pair of them).  Groups 0 .. G-1 are
// the GEMM CTAs; with late groups (p.late_groups > 0) the producer CTAs join
// as groups G, G+1, ... once their copy is done.
//
// Without the tail split: tiles t = g, g+G, g+2G, ... in rounds.
//
// With it (AG), some tiles are "tail" tiles whose K units (kps K blocks each)
// are laid end to end and cut into consecutive ranges, one per group, in two
// bands: groups [0, ga) share the first wa units evenly, groups [ga, ga+gb)
// the next wb units.  A range holds at most a later part of one tile first
// (SEG_WRITE: stored as an fp32 partial to the group's workspace block), then
// whole tiles, and at most the first part of one more tile last (SEG_FINISH:
// its accumulator plus the later parts' partials in K order, then the
// output).  A finisher only ever waits for higher groups' first tail segment,
// which waits for nothing the finisher holds.
//
//  * tail first (schedule 1): the R = T mod G leftover tiles are the first
//    tiles (the observer's own chunk, readable at once), shared by
//    ga = min(G, TAIL_SPLIT R) groups; the whole rounds follow from tile R,
//    the groups without tail work taking each round's lowest tiles.
//  * tail last: the GEMM groups first take p.split_full whole rounds; the
//    remaining tiles are shared either by ga = min(G, TAIL_SPLIT R) GEMM
//    groups (schedule 3), or by the GEMM groups (band a, a short range each)
//    and the late groups (band b, the rest; schedule 2), sized on the host
//    so that both end together given when the copy should finish.
// The host works each group's ranges out once per plan (a TailDesc per
// group in a device table); the kernel only steps through them.
enum SegKind : int { SEG_WHOLE = 0, SEG_FINISH = 1, SEG_WRITE = 2 };
struct Seg {
  int t, kb_lo, kb_hi, kind;
  int w0, nw;  // SEG_FINISH: the groups w0, ..., w0 + nw - 1 hold the tile's later parts
  bool last;   // SEG_FINISH: no tile of this CTA group follows (its pipeline stages are then idle)
};
// Dynamic tiles (builds without the split, p.dyn): instead of the fixed round
// robin, a CTA group's TMA thread (the even CTA's, for pairs) claims each next
// tile with an atomic add on a launch-wide counter, so that groups that run
// faster take more tiles and the tiles in flight stay a contiguous run of the
// tile order (their shared operands stay in L2 together).  It passes every
// index to the group's other roles (its MMA warp, the epilogue warps and,
// for pairs, the odd CTA's TMA thread and epilogue warps) through a ring of
// TQ_DEPTH shared-memory words: a full barrier per slot in each CTA (one
// arrival from the claiming thread) and an empty barrier per slot in the even
// CTA (one arrival from every reading thread or warp).  A claim at or past
// the launch's tile count ends the group's work; each group makes exactly one
// such claim, so a launch advances the counter by tiles + groups.
struct DynTiles {  // the dynamic instantiation's ring state (role 1 the claiming thread, 2 a reading thread, 3 a reading warp)
  int dyn, T, cg;
  uint32_t q, ring, full0, empty0, peer_ring, peer_full0, rank, pre;
  const Params* pp;
};
struct NoDynTiles {};
// SPLIT: the build with the tail split; DYN: the build with dynamic tiles
// (kernels built without either take the round robin only).
template <bool SPLIT, bool DYN = false>
struct SegIter : std::conditional_t<DYN, DynTiles, NoDynTiles> {
  int g, s, nfull, G, whole_base, slot, kbu, kps;
  bool first;
  int tail_base, ts, wr_t, wr_lo, wr_hi, tw0, tw1, fin_t, fin_hi, fin_w0, fin_nw;
  bool has_wr, has_fin;
  // `tail`: the CTA's TailDesc in shared memory (split builds with the split on)
  __device__ SegIter(const Params& p, int g_, int G_, int T, int nkb, const TailDesc* tail)
      : g(g_), s(0), G(G_), kps(p.kps) {
    kbu = nkb / kps;
    first = true;
    has_wr = has_fin = false;
    tail_base = ts = wr_t = wr_lo = wr_hi = tw0 = tw1 = fin_t = fin_hi = fin_w0 = fin_nw = 0;
    if (!SPLIT || !p.tail_split) {
      nfull = g < T && g < G ? (T - g + G - 1) / G : 0;
      whole_base = 0;
      slot = g;
      return;
    }
    const TailDesc d = *tail;
    first = d.first != 0;
    nfull = d.nfull;
    whole_base = d.whole_base;
    slot = d.slot;
    tail_base = d.tail_base;
    has_wr = d.has_wr != 0;
    wr_t = d.wr_t;
    wr_lo = d.wr_lo;
    wr_hi = d.wr_hi;
    tw0 = d.tw0;
    tw1 = d.tw1;
    has_fin = d.has_fin != 0;
    fin_t = d.fin_t;
    fin_hi = d.fin_hi;
    fin_w0 = d.fin_w0;
    fin_nw = d.fin_nw;
  }
  // Switches this iterator to dynamic tiles in role `role` (see above) for a
  // CTA of group size cg_ whose shared memory starts at sbase.
  __device__ void set_dynamic(const Params& p, int role, uint32_t sbase, uint32_t rank_, int cg_, int T_) {
    auto& d = *static_cast<DynTiles*>(this);
    d.dyn = role;
    d.pp = &p;
    d.T = T_;
    d.cg = cg_;
    d.rank = rank_;
    d.q = d.pre = 0;
    d.ring = sbase + SMEM_TQ;
    d.full0 = sbase + SMEM_BARS + 8u * BAR_TQ_FULL;
    d.empty0 = sbase + SMEM_BARS + 8u * BAR_TQ_EMPTY;
    d.peer_ring = d.peer_full0 = 0;
    if (d.cg == 2) {
      d.peer_ring = map_to_rank(d.ring, 1);
      d.peer_full0 = map_to_rank(d.full0, 1);
      if (d.rank != 0) d.empty0 = map_to_rank(d.empty0, 0);  // the odd CTA's readers arrive on the even CTA's barrier
    }
  }
  __device__ bool dyn_next(Seg& o) {
    auto& d = *static_cast<DynTiles*>(this);
    const Params& p = *d.pp;
    const int dyn = d.dyn, T = d.T, cg = d.cg;
    const uint32_t q = d.q, ring = d.ring, full0 = d.full0, empty0 = d.empty0, rank = d.rank;
    const uint32_t slot_q = q % TQ_DEPTH, par = (q / TQ_DEPTH) & 1u;
    uint32_t t = 0;
    if (dyn == 1) {
      // the slot's previous index has been read by every role of the group
      // (cluster-scope acquire: the odd CTA's reads of the slot come before the overwrite below)
      if (q >= TQ_DEPTH && !mbar_wait_cluster(p, empty0 + 8u * slot_q, par ^ 1u, SITE_TILE)) return false;
      // The claim for the tile after this one goes out now and is read at the
      // next call, so its round trip overlaps this tile's work.
      if (q == 0) d.pre = atomicAdd(&p.words->sched, 1u) - p.sched_base;
      t = d.pre < static_cast<uint32_t>(T) ? d.pre : static_cast<uint32_t>(T);
      if (t < static_cast<uint32_t>(T)) d.pre = atomicAdd(&p.words->sched, 1u) - p.sched_base;
      st_shared_u32(ring + 4u * slot_q, t);
      mbar_arrive(full0 + 8u * slot_q);
      if (cg == 2) {
        st_shared_cluster_u32(d.peer_ring + 4u * slot_q, t);
        mbar_arrive_cluster(d.peer_full0 + 8u * slot_q);  // release: the index is visible first
      }
    } else {
      const int lane = threadIdx.x & 31;
      int ok = 1;
      if (dyn == 2 || lane == 0) {
        // (in the odd CTA the index was written from the even CTA: cluster-scope acquire)
        ok = (rank != 0 ? mbar_wait_cluster(p, full0 + 8u * slot_q, par, SITE_TILE)
                        : mbar_wait(p, full0 + 8u * slot_q, par, SITE_TILE, true)) ? 1 : 0;
        if (ok) {
          t = ld_shared_u32(ring + 4u * slot_q);
          if (rank != 0)
            mbar_arrive_cluster(empty0 + 8u * slot_q);
          else
            mbar_arrive(empty0 + 8u * slot_q);
        }
      }
      if (dyn == 3) {
        ok = __shfl_sync(0xffffffffu, ok, 0);
        t = __shfl_sync(0xffffffffu, t, 0);
      }
      if (!ok) return false;
    }
    d.q = q + 1;
    if (t >= static_cast<uint32_t>(T)) return false;
    o.t = static_cast<int>(t);
    o.kb_lo = 0;
    o.kb_hi = kbu * kps;
    o.kind = SEG_WHOLE;
    o.w0 = o.nw = 0;
    o.last = false;
    return true;
  }
  __device__ bool tail_next(Seg& o) {
    if (ts == 0) {
      ts = 1;
      if (has_wr) {
        o.t = tail_base + wr_t;
        o.kb_lo = wr_lo * kps;
        o.kb_hi = wr_hi * kps;
        o.kind = SEG_WRITE;
        return true;
      }
    }
    if (ts == 1) {
      if (tw0 < tw1) {
        o.t = tail_base + tw0++;
        o.kb_lo = 0;
        o.kb_hi = kbu * kps;
        o.kind = SEG_WHOLE;
        return true;
      }
      ts = 2;
    }
    if (ts == 2) {
      ts = 3;
      if (has_fin) {
        o.t = tail_base + fin_t;
        o.kb_lo = 0;
        o.kb_hi = fin_hi * kps;
        o.kind = SEG_FINISH;
        o.w0 = fin_w0;
        o.nw = fin_nw;
        o.last = !first || nfull == 0;
        return true;
      }
    }
    return false;
  }
  __device__ bool next(Seg& o) {
    if constexpr (DYN) return dyn_next(o);
    if constexpr (SPLIT) {
      o.w0 = o.nw = 0;
      o.last = false;
      if (first && tail_next(o)) return true;
    }
    if (s < nfull) {
      o.t = whole_base + slot + s * G;
      o.kb_lo = 0;
      o.kb_hi = kbu * kps;
      o.kind = SEG_WHOLE;
      ++s;
      return true;
    }
    if constexpr (SPLIT) return !first && tail_next(o);
    return false;
  }
};

// ------------------------------------------------------------------ producer role

__device__ __forceinline__ uint32_t piece_bytes(const Params& p, long long piece) {
  const long long rem = p.chunk_bytes - piece * COPY_PIECE;
  return static_cast<uint32_t>(rem < COPY_PIECE ? rem : COPY_PIECE);
}

// Copy pieces [lo, hi) of one chunk; `seq` numbers this CTA's loads across
// chunks (buffer = seq % COPY_BUFS, phase parity = (seq / COPY_BUFS) & 1).
__device__ bool copy_pieces(const Params& p, const uint8_t* src, uint8_t* dst, long long lo, long long hi,
                            uint32_t sbase, uint32_t bars, unsigned long long seq) {
  const long long np = hi - lo;
  constexpr long long AHEAD = COPY_BUFS - COPY_LAG;
  auto issue = [&](long long i) {
    const unsigned long long s = seq + i;
    const uint32_t b = static_cast<uint32_t>(s % COPY_BUFS);
    const uint32_t bytes = piece_bytes(p, lo + i);
    mbar_expect_tx(bars + 8u * b, bytes);
    bulk_load(sbase + b * COPY_PIECE, src + (lo + i) * COPY_PIECE, bytes, bars + 8u * b);
  };
  for (long long i = 0; i < np && i < AHEAD; ++i) issue(i);
  for (long long i = 0; i < np; ++i) {
    const unsigned long long s = seq + i;
    const uint32_t b = static_cast<uint32_t>(s % COPY_BUFS);
    if (!mbar_wait(p, bars + 8u * b, static_cast<uint32_t>((s / COPY_BUFS) & 1u), SITE_COPY, true)) {
      for (long long j = i; j < np && j < i + AHEAD; ++j) {  // loads still in flight
        const unsigned long long sj = seq + j;
        mbar_wait(p, bars + 8u * static_cast<uint32_t>(sj % COPY_BUFS),
                  static_cast<uint32_t>((sj / COPY_BUFS) & 1u), SITE_DRAIN, false);
      }
      bulk_wait<0>();
      return false;
    }
    bulk_store(dst + (lo + i) * COPY_PIECE, sbase + b * COPY_PIECE, piece_bytes(p, lo + i));
    bulk_commit();
    if (i + AHEAD < np) {
      bulk_wait_read<COPY_LAG>();  // the store that last read buffer (i + AHEAD) % COPY_BUFS is done
      issue(i + AHEAD);
    }
  }
  return true;
}

__device__ void producer_role(const Params& p, uint8_t* smem) {
  if (threadIdx.x != 0) return;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + SMEM_BARS + 8u * BAR_COPY;
  for (int b = 0; b < COPY_BUFS; ++b) mbar_init(bars + 8u * b, 1);
  fence_barrier_init();
  grid_dep_wait();  // the sources may come from the launch before
  if (p.trace_on) atomicMin(&p.words->trace[TPO_TRACE_START], gtime());

  const long long pieces = (p.chunk_bytes + COPY_PIECE - 1) / COPY_PIECE;
  const long long P = p.num_producers, pid = blockIdx.x;
  const long long lo = pieces * pid / P, hi = pieces * (pid + 1) / P;
  unsigned long long seq = 0;
  // Ring steps 1 .. tp-1 in arrival order, then step 0 (the observer's own
  // chunk, which the GEMM reads in place, copied last into its slot).
  for (int si = 0; si < p.tp; ++si) {
    const int step = (si + 1) % p.tp;
    if (p.last_step >= 0 && step > p.last_step) continue;
    if (p.only_step >= 0 && step != p.only_step) continue;
    const int slot = ((p.self_rank - step) % p.tp + p.tp) % p.tp;
    const uint8_t* src = p.src[slot];
    uint8_t* dst = p.staging + static_cast<long long>(slot) * p.chunk_bytes;
    if (!copy_pieces(p, src, dst, lo, hi, sbase, bars, seq)) return;
    seq += static_cast<unsigned long long>(hi - lo);
    bulk_wait<0>();  // this CTA's writes of the chunk are complete
    fence_proxy_async_global();
    if (p.delay_ns) {
      const unsigned long long t0 = gtime();
      while (gtime() - t0 < p.delay_ns) __nanosleep(256);
    }
    if (slot != p.skip_slot) red_add_release(&p.words->counters[slot], 1u);
    if (p.trace_on) atomicMax(&p.words->trace[TPO_TRACE_PUBLISH + slot], gtime());
  }
}

// ------------------------------------------------------------------ GEMM role

__device__ bool wait_counter(const Params& p, int slot) {
  const uint32_t* c = &p.words->counters[slot];
  const unsigned long long t0 = gtime();
  bool waited = false;
  while (static_cast<int>(ld_acquire(c) - p.target[slot]) < 0) {
    waited = true;
    if (aborted(p)) return false;
    if (gtime() - t0 > p.timeout_ns) {
      raise_error(p, DEV_TIMEOUT, SITE_COUNTER, static_cast<uint32_t>(slot));
      return false;
    }
    __nanosleep(64);
  }
  fence_proxy_async_global();  // order the acquire before the tensor (async-proxy) loads
  if (p.trace_on) {
    const unsigned long long t1 = gtime();
    atomicMin(&p.words->trace[TPO_TRACE_ACQUIRE + slot], t1);
    if (waited) atomicAdd(&p.words->trace[TPO_TRACE_WAIT_NS], t1 - t0);
  }
  return true;
}

// Bounded wait (every lane of a warp) until a split tile's partial of this
// launch is in the workspace; the acquire orders the lane's later loads.
__device__ bool wait_partial(const Params& p, const uint32_t* flag) {
  const unsigned long long t0 = gtime();
  while (static_cast<int>(ld_acquire(flag) - p.part_target) < 0) {
    if (aborted(p)) return false;
    if (gtime() - t0 > p.timeout_ns) {
      raise_error(p, DEV_TIMEOUT, SITE_PARTIAL, static_cast<uint32_t>(flag - p.words->part_ready));
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

struct Bars {
  uint32_t full0, empty0, tfull0, tempty0, drain;
};

// The TMA issuer: one thread keeps every stage of the pipeline in flight.  Like
// the MMA issuer it runs from registers only (tensor-map addresses, ring
// position, stage and phase), so that refills follow stage releases closely.
template <int CG, bool AG, bool SPLIT, int KPS, bool DYN>
__device__ void tma_loop(const Params& p, uint32_t sbase, const Bars& B, uint32_t rank, int g, int G,
                         int total_tiles, int nkb, bool trace, const TailDesc* tail) {
  using PP = Pipe<CG>;
  const uint64_t mapA0 = reinterpret_cast<uint64_t>(&p.mapA[0]);
  const uint64_t mapB0 = reinterpret_cast<uint64_t>(&p.mapB[0]);
  constexpr uint64_t kMap = sizeof(CUtensorMap);
  const int tp = p.tp, kb_per_seg = p.kb_per_seg;
  const int kelems = p.fp8 ? BK_BYTES : BK_BYTES / 2;
  const uint32_t full0 = B.full0, empty0 = B.empty0;
  const uint32_t full0_leader = (CG == 2) ? map_to_rank(full0, 0) : full0;
  const int a_off = BM * static_cast<int>(rank);
  constexpr uint32_t kps = KPS;
  constexpr uint32_t stage_bytes = kps * PP::STAGE_BYTES;
  constexpr uint32_t nstages = STAGE_AREA / stage_bytes;
  uint32_t ready = 0, stage = 0, phase = 0, armed = 0;
  bool ok = true;
  unsigned long long cyc_empty = 0;
  SegIter<SPLIT, DYN> it(p, g, G, total_tiles, nkb, tail);
  if constexpr (DYN) it.set_dynamic(p, (CG == 1 || rank == 0) ? 1 : 2, sbase, rank, CG, total_tiles);
  Seg sg;
  while (ok && it.next(sg)) {
    const Tile T = tile_at<PP::TILE_M>(p, sg.t);
    if (AG && T.gate >= 0 && !((ready >> T.gate) & 1u)) {
      if (!wait_counter(p, T.gate)) {
        ok = false;
        break;
      }
      ready |= 1u << T.gate;
    }
    int r = AG ? T.a_map : T.seg0;  // tensor map of the current K segment
    int kk = sg.kb_lo;               // (RS/AR segments always start at K block 0)
    // each CTA of a pair loads half of the tile's B rows (its box may reach
    // into the next tile's rows, which the MMA does not read)
    const int a_row = T.a_row + a_off, a_z = T.a_z, b_row = T.col + (CG == 2 ? (T.ncols >> 1) * static_cast<int>(rank) : 0);
    for (int i = sg.kb_lo; i < sg.kb_hi; i += KPS) {  // one stage of KPS K blocks per pass
      const uint32_t sbase_stage = sbase + SMEM_STAGES + stage * stage_bytes;
      // wait until the MMAs released the stage, then arm its barrier
      const uint32_t eb = empty0 + 8u * stage;
      if (!mbar_test(eb, phase ^ 1u) && !mbar_wait_timed(p, eb, phase ^ 1u, SITE_EMPTY, true, &cyc_empty)) {
        ok = false;
        break;
      }
      if (CG == 1 || rank == 0) mbar_expect_tx(full0 + 8u * stage, CG * stage_bytes);
      ++armed;
#pragma unroll
      for (int blk = 0; blk < KPS; ++blk) {
        const CUtensorMap* ma = reinterpret_cast<const CUtensorMap*>(mapA0 + kMap * static_cast<uint64_t>(r));
        const CUtensorMap* mb = reinterpret_cast<const CUtensorMap*>(mapB0 + kMap * static_cast<uint64_t>(AG ? 0 : r));
        const uint32_t sa = sbase_stage + blk * A_STAGE_BYTES;
        const uint32_t sb = sbase_stage + kps * A_STAGE_BYTES + blk * PP::B_STAGE_BYTES;
        const int kx = kk * kelems;
        if constexpr (CG == 1) {
          const uint32_t fb = full0 + 8u * stage;
          tma_load_3d(sa, ma, fb, kx, a_row, a_z);
          tma_load_2d(sb, mb, fb, kx, b_row);
        } else {
          // both halves complete on the even CTA's barrier, which expects the pair's bytes
          const uint32_t fl = full0_leader + 8u * stage;
          tma_load_3d_pair(sa, ma, fl, kx, a_row, a_z);
          tma_load_2d_pair(sb, mb, fl, kx, b_row);
        }
        if (++kk == kb_per_seg) {  // next K segment: the next rank in ring order
          kk = 0;
          if (!AG && ++r == tp) r = 0;
        }
      }
      if (++stage == nstages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok) {  // loads already issued must land before the CTA releases its shared memory
    if (CG == 1 || rank == 0) {
      const uint32_t first = armed > nstages ? armed - nstages : 0u;
      for (uint32_t j = first; j < armed; ++j)
        mbar_wait(p, full0 + 8u * (j % nstages), (j / nstages) & 1u, SITE_DRAIN, false);
    } else if (armed > 0) {
      // the odd CTA's loads signal the even CTA's barrier: give them time to land
      const unsigned long long t0 = gtime();
      while (gtime() - t0 < 200000ull) __nanosleep(1000);
    }
  }
  if (trace) atomicAdd(&p.words->trace[TPO_TRACE_CYC_TMA_EMPTY], cyc_empty);
}

template <int CG, bool SPLIT, bool DYN>
__device__ void tma_role(const Params& p, uint32_t sbase, const Bars& B, uint32_t rank, int g, int G,
                         int total_tiles, int nkb, const TailDesc* tail) {
  const bool trace = p.trace_on != 0;
  if (p.op == OP_AG)
    (CG == 2 && p.kps == 2) ? tma_loop<CG, true, SPLIT, 2, DYN>(p, sbase, B, rank, g, G, total_tiles, nkb, trace, tail)
                            : tma_loop<CG, true, SPLIT, 1, DYN>(p, sbase, B, rank, g, G, total_tiles, nkb, trace, tail);
  else
    (CG == 2 && p.kps == 2) ? tma_loop<CG, false, false, 2, DYN>(p, sbase, B, rank, g, G, total_tiles, nkb, trace, tail)
                            : tma_loop<CG, false, false, 1, DYN>(p, sbase, B, rank, g, G, total_tiles, nkb, trace, tail);
}

// The MMA issuer: the whole of warp 1 of the group's even CTA, converged (one
// elected lane issues each MMA and commit).  tcgen05.mma issue returns only
// once the tensor core can take the instruction, so only a few MMAs are ever
// queued: every cycle the issuer spends between two MMAs is tensor-pipe idle
// time.  The loop therefore keeps all state in registers (no parameter
// reloads), tests each stage's barrier inline (a warp vote, so that every
// branch is uniform) and only falls back to the bounded wait when it is not
// ready.  KPS: K blocks per pipeline stage (p.kps), fixed at compile time so
// that a stage's MMAs issue back to back with no per-block bookkeeping.
template <int CG, bool FP8, bool SPLIT, int KPS, bool DYN>
__device__ void mma_loop(const Params& p, uint32_t sbase, uint32_t tmem, const Bars& B, int g, int G,
                         int total_tiles, int nkb, bool trace, const TailDesc* tail) {
  using PP = Pipe<CG>;
  constexpr uint32_t idesc0 = make_idesc(FP8, PP::TILE_M);
  constexpr uint32_t kps = KPS;
  const uint32_t stage_bytes = kps * PP::STAGE_BYTES;
  const uint32_t nstages = STAGE_AREA / stage_bytes;
  const uint64_t kStageDesc = static_cast<uint64_t>(stage_bytes >> 4);  // stage step in the address field
  constexpr uint64_t kBlkA = static_cast<uint64_t>(A_STAGE_BYTES >> 4), kBlkB = static_cast<uint64_t>(PP::B_STAGE_BYTES >> 4);
  const uint64_t da0 = smem_desc_sw128(sbase + SMEM_STAGES);
  const uint64_t db0 = smem_desc_sw128(sbase + SMEM_STAGES + kps * A_STAGE_BYTES);
  const uint32_t full0 = B.full0, empty0 = B.empty0, tfull0 = B.tfull0, tempty0 = B.tempty0;
  // Accumulation units: a whole tile (K-slices chained in one accumulator), or
  // in the epilogue-reduction modes one rank's K-slice.  Units alternate
  // between the two accumulators, so the epilogue drains one while the MMAs
  // fill the other.
  const bool per_rank = p.reduce_mode != 0;
  const int units = per_rank ? p.num_segs : 1;
  const int kpu = per_rank ? p.kb_per_seg : nkb;
  uint32_t stage = 0, phase = 0, ul = 0, issued = 0;
  bool ok = true;
  unsigned long long cyc_full = 0, cyc_tempty = 0;
  SegIter<SPLIT, DYN> it(p, g, G, total_tiles, nkb, tail);
  if constexpr (DYN) it.set_dynamic(p, 3, sbase, 0, CG, total_tiles);
  Seg sg;
  while (ok && it.next(sg)) {
   const uint32_t idesc = idesc_n(idesc0, tile_at<PP::TILE_M>(p, sg.t).ncols);
   for (int u = 0; u < units; ++u, ++ul) {
    const uint32_t acc = ul & 1u;
    const uint32_t te = tempty0 + 8u * acc;
    const uint32_t tpar = ((ul >> 1) & 1u) ^ 1u;
    if (!mbar_wait_warp(p, te, tpar, SITE_TMEM_EMPTY, &cyc_tempty)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d = tmem + acc * BN;
    const int nk = per_rank ? kpu : sg.kb_hi - sg.kb_lo;  // a multiple of KPS
    for (int i = 0; i < nk; i += KPS) {
      const uint32_t fb = full0 + 8u * stage;
      if (!mbar_wait_warp(p, fb, phase, SITE_FULL, &cyc_full)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t das = da0 + kStageDesc * stage, dbs = db0 + kStageDesc * stage;
#pragma unroll
      for (int b = 0; b < KPS; ++b)
        mma_kblock<CG, FP8>(d, das + kBlkA * b, dbs + kBlkB * b, idesc, (i + b) > 0 ? 1u : 0u);
      issued += KPS;
      mma_commit_cg<CG>(empty0 + 8u * stage);  // frees the stage (in both CTAs) once read
      if (++stage == nstages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    mma_commit_cg<CG>(tfull0 + 8u * acc);  // accumulator ready for the epilogue(s)
   }
  }
  if (!ok) {  // every MMA issued so far must complete before tensor memory is freed
    mma_commit_local_cg<CG>(B.drain);
    if ((threadIdx.x & 31) == 0) mbar_wait(p, B.drain, 0u, SITE_DRAIN, false);
    __syncwarp();
  }
  if (trace && (threadIdx.x & 31) == 0) {
    atomicAdd(&p.words->trace[TPO_TRACE_CYC_MMA_FULL], cyc_full);
    atomicAdd(&p.words->trace[TPO_TRACE_CYC_MMA_TEMPTY], cyc_tempty);
    atomicAdd(&p.words->trace[TPO_TRACE_KBLOCKS], static_cast<unsigned long long>(issued));
  }
}

template <int CG, bool SPLIT, bool DYN>
__device__ void mma_role(const Params& p, uint32_t sbase, uint32_t tmem, const Bars& B, int g, int G,
                         int total_tiles, int nkb, const TailDesc* tail) {
  const bool trace = p.trace_on != 0;
  if (CG == 2 && p.kps == 2) {
    if (p.fp8)
      mma_loop<CG, true, SPLIT, 2, DYN>(p, sbase, tmem, B, g, G, total_tiles, nkb, trace, tail);
    else
      mma_loop<CG, false, SPLIT, 2, DYN>(p, sbase, tmem, B, g, G, total_tiles, nkb, trace, tail);
  } else {
    if (p.fp8)
      mma_loop<CG, true, SPLIT, 1, DYN>(p, sbase, tmem, B, g, G, total_tiles, nkb, trace, tail);
    else
      mma_loop<CG, false, SPLIT, 1, DYN>(p, sbase, tmem, B, g, G, total_tiles, nkb, trace, tail);
  }
}

template <int CG, bool SPLIT, bool DYN>
__device__ void epilogue_role(const Params& p, uint8_t* smem, uint32_t tmem, const Bars& B, uint32_t rank, int g,
                              int G, int total_tiles, const TailDesc* tail) {
  using PP = Pipe<CG>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;  // tensor-memory lanes this warp may read: [32*quad, 32*quad+32)
  const uint32_t sbase_smem = smem_u32(smem);
  const uint32_t ebase = smem_u32(smem + SMEM_EPI + (warp - 2) * 2 * EPI_BUF_BYTES);
  const float scale = p.fp8 ? (__ldg(p.scale_x) * __ldg(p.scale_w)) : 1.0f;
  const int row_off = BM * static_cast<int>(rank);
  const int rmode = p.reduce_mode;
  const int units = rmode ? p.num_segs : 1;
  // Epilogue-reduction modes: the running sum of the CTA's 128 x 256 tile lives
  // in its own workspace block, laid out [column chunk][16-byte group][row] so
  // that a warp's access is one contiguous 512 bytes, and marked to stay in L2
  // while the operand streams pass through.
  uint4* const ws_row = rmode ? reinterpret_cast<uint4*>(p.ws) +
                                    static_cast<size_t>(blockIdx.x - p.num_producers) * (BM * BN / 4) + quad * 32 + lane
                              : nullptr;
  uint64_t ws_pol = 0;
  if (rmode || SPLIT) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(ws_pol));
  // Split tiles (AG tail split): a CTA's partial of a later part of a tile sits
  // in its own workspace block, unscaled fp32, laid out warp by warp: each
  // epilogue warp's 32 rows are one contiguous 32 KiB run of [32-column chunk]
  // [16-byte group][row] (512 coalesced bytes per chunk and group).
  const int cta = g * CG + static_cast<int>(rank);  // workspace block and partial flags of this CTA
  auto part_at = [&](int blk, int c, int v) -> uint4* {
    return reinterpret_cast<uint4*>(p.ws) + static_cast<size_t>(blk) * (BM * BN / 4) + quad * (32 * BN / 4) +
           (c * 8 + v) * 32 + lane;
  };
  uint32_t ul = 0, nst = 0, pphase = 0;
  unsigned long long cyc_tfull = 0;
  bool ok_all = true;
  // A part of a split tile, on its own path so that whole tiles run the same
  // code as in the build without the split.  A later part (SEG_WRITE) goes to
  // this CTA's workspace block as unscaled fp32 and is published per warp; the
  // first part (SEG_FINISH) waits for the later parts' flags, adds them in K
  // order and stores the tile like a whole one.  When the finished tile is
  // the CTA group's last (its MMAs and loads are over, so the pipeline stages
  // are idle), each warp first copies its rows of the later parts into its
  // quarter of the stage area with bulk copies, a few round trips in all;
  // otherwise it reads them from global memory one chunk ahead.
  auto split_part = [&](const Tile& T, const Seg& sg, uint32_t ul_) -> bool {
    const bool write = sg.kind == SEG_WRITE;
    const int nch = T.ncols / EPI_COLS;
    if (!write)
      for (int j = 0; j < sg.nw; ++j)
        if (!wait_partial(p, &p.words->part_ready[((sg.w0 + j) * CG + static_cast<int>(rank)) * EPI_WARPS + quad]))
          return false;
    const uint32_t acc = ul_ & 1u;
    const uint32_t bar = B.tfull0 + 8u * acc, par = (ul_ >> 1) & 1u;
    int okw = (lane == 0) ? (mbar_wait_timed(p, bar, par, SITE_TMEM_FULL, true, &cyc_tfull) ? 1 : 0) : 0;
    if (!__shfl_sync(0xffffffffu, okw, 0)) return false;
    mbar_wait(p, bar, par, SITE_TMEM_FULL, false);
    tc_fence_after();
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
    auto add_part = [&](uint32_t(&r)[32], const uint32_t(&h)[32]) {
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(h[e]));
    };
    // staged path: this warp's quarter of the stage area holds `span` chunks of every later part
    constexpr int kWarpArea = STAGE_AREA / EPI_WARPS;   // 48 KiB
    constexpr int kChunkBytes = 32 * EPI_COLS * 4;      // one warp's 32 rows x 32 columns, fp32
    const bool staged = !write && sg.nw > 0 && sg.last && sg.nw * kChunkBytes <= kWarpArea;
    const int span = staged ? kWarpArea / (sg.nw * kChunkBytes) : 0;
    const uint32_t pbuf = sbase_smem + SMEM_STAGES + static_cast<uint32_t>((warp - 2) * kWarpArea);
    const uint32_t pbar = sbase_smem + SMEM_BARS + 8u * static_cast<uint32_t>(BAR_PART + (warp - 2));
    int c_lo = 0, c_hi = 0;  // chunks now in shared memory
    auto stage = [&](int c0) -> bool {  // bulk-copy chunks [c0, c0 + span) of every later part
      const int cnt = min(span, nch - c0);
      __syncwarp();  // every lane is done reading the previous range
      if (lane == 0) {
        if (c0 == 0)
          fence_proxy_async_global();  // the acquired partials, read through the async proxy
        else
          fence_proxy_async_smem();    // the previous range's reads come before its overwrite
        mbar_expect_tx(pbar, static_cast<uint32_t>(sg.nw * cnt * kChunkBytes));
        for (int j = 0; j < sg.nw; ++j)
          bulk_load(pbuf + static_cast<uint32_t>(j * span * kChunkBytes),
                    reinterpret_cast<const uint8_t*>(p.ws) +
                        (static_cast<size_t>((sg.w0 + j) * CG + static_cast<int>(rank)) * (BM * BN) +
                         static_cast<size_t>(quad) * (32 * BN) + static_cast<size_t>(c0) * (32 * EPI_COLS)) * 4,
                    static_cast<uint32_t>(cnt * kChunkBytes), pbar);
      }
      int okb = (lane == 0) ? (mbar_wait(p, pbar, pphase, SITE_PARTIAL, true) ? 1 : 0) : 0;
      if (!__shfl_sync(0xffffffffu, okb, 0)) {
        if (lane == 0) mbar_wait(p, pbar, pphase, SITE_DRAIN, false);  // copies in flight land first
        return false;
      }
      mbar_wait(p, pbar, pphase, SITE_PARTIAL, false);  // every lane observes the completed phase
      pphase ^= 1u;
      c_lo = c0;
      c_hi = c0 + cnt;
      return true;
    };
    auto load_part = [&](int j, int c, uint32_t(&h)[32]) {
      if (staged) {
        const uint32_t a = pbuf + static_cast<uint32_t>((j * span + (c - c_lo)) * kChunkBytes) + lane * 16u;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint32_t x0, x1, x2, x3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3) : "r"(a + v * 512u) : "memory");
          h[4 * v] = x0;
          h[4 * v + 1] = x1;
          h[4 * v + 2] = x2;
          h[4 * v + 3] = x3;
        }
        return;
      }
      const int blk = (sg.w0 + j) * CG + static_cast<int>(rank);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        uint32_t x[4];
        ld_global_v4_keep(part_at(blk, c, v), x, ws_pol);
        h[4 * v] = x[0];
        h[4 * v + 1] = x[1];
        h[4 * v + 2] = x[2];
        h[4 * v + 3] = x[3];
      }
    };
    uint32_t pa[32];
    if (!write && sg.nw > 0 && !staged) load_part(0, 0, pa);
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      uint32_t pn[32];
      if (!write && sg.nw > 0) {
        if (staged) {  // the chunk's later parts from shared memory, a new range when needed
          if (c >= c_hi && !stage(c)) return false;
          load_part(0, c, pa);
        } else if (c + 1 < nch) {  // from global memory, one chunk ahead
          load_part(0, c + 1, pn);
        }
      }
      uint32_t r[32];
      tmem_ld32_sync(taddr + c * EPI_COLS, r);
      if (c == nch - 1) {  // accumulator fully read: hand it back to the MMA issuer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 1)
            mbar_arrive(B.tempty0 + 8u * acc);
          else
            mbar_arrive_cluster(map_to_rank(B.tempty0 + 8u * acc, 0));
        }
      }
      if (write) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          st_global_v4_keep(part_at(cta, c, v), r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3], ws_pol);
        continue;
      }
      if (sg.nw > 0) add_part(r, pa);  // the later parts in K order
      for (int j = 1; j < sg.nw; ++j) {
        uint32_t h[32];
        load_part(j, c, h);
        add_part(r, h);
      }
      if (!staged) {
#pragma unroll
        for (int e = 0; e < 32; ++e) pa[e] = pn[e];
      }
      const int ox = T.col + c * EPI_COLS, oy = T.y_row + row_off + quad * 32;
      if (ox >= p.m || oy >= p.y_rows) continue;  // wholly past the output's edge: no buffer, no store
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * j]) * scale,
                                                       __uint_as_float(r[2 * j + 1]) * scale);
        packed[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      const uint32_t buf = ebase + (nst & 1u) * EPI_BUF_BYTES;
      ++nst;
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const uint32_t addr = buf + lane * 64 + (static_cast<uint32_t>(ch ^ ((lane >> 1) & 3)) << 4);
        st_shared_v4(addr, packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&p.mapY[T.y_map], buf, ox, oy, T.y_z);
        bulk_commit();
      }
    }
    if (write) {  // this warp's rows of the partial are stored: publish them
      __syncwarp();
      if (lane == 0 && cta != p.skip_part) {
        __threadfence();
        st_release(&p.words->part_ready[cta * EPI_WARPS + quad], p.part_target);
      }
    }
    return true;
  };
  SegIter<SPLIT, DYN> it(p, g, G, total_tiles, p.num_segs * p.kb_per_seg, tail);
  if constexpr (DYN) it.set_dynamic(p, 3, sbase_smem, rank, CG, total_tiles);
  Seg sg;
  while (ok_all && it.next(sg)) {
    const Tile T = tile_at<PP::TILE_M>(p, sg.t);
    if constexpr (SPLIT) {
      if (sg.kind != SEG_WHOLE) {  // a part of a split tile (AG: one accumulation unit)
        ok_all = split_part(T, sg, ul);
        ++ul;
        continue;
      }
    }
    for (int u = 0; u < units; ++u, ++ul) {
      const uint32_t acc = ul & 1u;
      const uint32_t bar = B.tfull0 + 8u * acc, par = (ul >> 1) & 1u;
      int ok = (lane == 0) ? (mbar_wait_timed(p, bar, par, SITE_TMEM_FULL, true, &cyc_tfull) ? 1 : 0) : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        ok_all = false;
        break;
      }
      mbar_wait(p, bar, par, SITE_TMEM_FULL, false);  // already complete: gives every lane its ordering
      tc_fence_after();
      const bool last = (u == units - 1);
      const int nch = T.ncols / EPI_COLS;  // 32-column chunks of this tile
      const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t taddr = tmem + lanes + acc * BN;
      // The running sum of this thread's row, 32 columns per chunk: fp32 in
      // mode 1; in mode 2 every running sum is a bf16 value, kept as bf16.
      auto store_sum = [&](int c, const uint32_t(&r)[32]) {
        if (rmode == 2) {
          uint4* w4 = reinterpret_cast<uint4*>(ws_row) + c * 4 * BM;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = (r[8 * v + 2 * i] >> 16) | (r[8 * v + 2 * i + 1] & 0xffff0000u);
            st_global_v4_keep(w4 + v * BM, h[0], h[1], h[2], h[3], ws_pol);
          }
        } else {
          uint4* w4 = reinterpret_cast<uint4*>(ws_row) + c * 8 * BM;
#pragma unroll
          for (int v = 0; v < 8; ++v) st_global_v4_keep(w4 + v * BM, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3], ws_pol);
        }
      };
      auto load_sum = [&](int c, uint32_t(&q)[32]) {
        if (rmode == 2) {
          const uint4* w4 = reinterpret_cast<const uint4*>(ws_row) + c * 4 * BM;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t h[4];
            ld_global_v4_keep(w4 + v * BM, h, ws_pol);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              q[8 * v + 2 * i] = h[i] << 16;
              q[8 * v + 2 * i + 1] = h[i] & 0xffff0000u;
            }
          }
        } else {
          const uint4* w4 = reinterpret_cast<const uint4*>(ws_row) + c * 8 * BM;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            uint32_t h[4];
            ld_global_v4_keep(w4 + v * BM, h, ws_pol);
            q[4 * v] = h[0];
            q[4 * v + 1] = h[1];
            q[4 * v + 2] = h[2];
            q[4 * v + 3] = h[3];
          }
        }
      };
      // One 32-column chunk: read it from tensor memory (handing the accumulator
      // back after the last chunk), add it to the running sum `q` in the
      // epilogue-reduction modes, and either keep the sum in the workspace or
      // round the result to bf16 and store it.
      auto chunk = [&](int c, const uint32_t(&q)[32], bool have_q) {
        uint32_t r[32];
        tmem_ld32_sync(taddr + c * EPI_COLS, r);
        if (c == nch - 1) {  // accumulator fully read: hand it back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (CG == 1)
              mbar_arrive(B.tempty0 + 8u * acc);
            else
              mbar_arrive_cluster(map_to_rank(B.tempty0 + 8u * acc, 0));
          }
        }
        float out_scale = scale;
        if (rmode) {
          // this rank's partial, added in ring order to the running sum
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float part = __uint_as_float(r[j]);
            float v;
            if (rmode == 2) {  // bf16 on the wire: the partial and every running sum are rounded
              part = round_bf16(part * scale);
              v = have_q ? round_bf16(__uint_as_float(q[j]) + part) : part;
            } else {
              v = have_q ? __uint_as_float(q[j]) + part : part;
            }
            r[j] = __float_as_uint(v);
          }
          if (rmode == 2) out_scale = 1.0f;
          if (!last) {
            store_sum(c, r);
            return;
          }
        }
        // A box wholly past the output's edge is neither staged nor stored.  It
        // must not take a staging buffer either: the wait below counts issued
        // stores, so a buffer may only alternate with boxes that were stored.
        const int ox = T.col + c * EPI_COLS, oy = T.y_row + row_off + quad * 32;
        if (ox >= p.m || oy >= p.y_rows) return;
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * j]) * out_scale,
                                                         __uint_as_float(r[2 * j + 1]) * out_scale);
          packed[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        const uint32_t buf = ebase + (nst & 1u) * EPI_BUF_BYTES;
        ++nst;
        if (lane == 0) bulk_wait_read<1>();  // the store that used this buffer (the one before last) has read it
        __syncwarp();
        // row `lane` of a 32 x 64-byte box in the 64-byte swizzle layout the
        // output tensor map expects (16-byte chunk index XOR (row / 2) % 4)
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t addr = buf + lane * 64 + (static_cast<uint32_t>(ch ^ ((lane >> 1) & 3)) << 4);
          st_shared_v4(addr, packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&p.mapY[T.y_map], buf, ox, oy, T.y_z);
          bulk_commit();
        }
      };
      if (rmode && u > 0) {
        // the running sum of the next chunk is fetched while this chunk is processed
        uint32_t qa[32], qb[32];
        load_sum(0, qa);
#pragma unroll 1
        for (int c = 0; c < nch; c += 2) {
          const bool two = c + 1 < nch;
          if (two) load_sum(c + 1, qb);
          chunk(c, qa, true);
          if (c + 2 < nch) load_sum(c + 2, qa);
          if (two) chunk(c + 1, qb, true);
        }
      } else {
        const uint32_t none[32] = {};
#pragma unroll 1
        for (int c = 0; c < nch; ++c) chunk(c, none, false);
      }
    }
    if (ok_all && p.op != OP_AG && lane == 0) {  // this warp's rows of the tile are in memory: count them
      // one count per 32-column strip, so that every group's count ends at the
      // same target whatever its column tiling
      bulk_wait<0>();
      fence_proxy_async_global();
      const uint32_t add = static_cast<uint32_t>(T.ncols / EPI_COLS);
      const uint32_t old = atom_add_release(&p.words->done[T.group], add);
      if (p.trace_on && old + add == p.done_target) p.words->trace[TPO_TRACE_CHUNK_DONE + T.group] = gtime();
    }
  }
  if (lane == 0) bulk_wait<0>();
  if (p.trace_on && lane == 0) atomicAdd(&p.words->trace[TPO_TRACE_CYC_EPI_TFULL], cyc_tfull);
  __syncwarp();
}

template <int CG, bool SPLIT, bool DYN>
__device__ void gemm_role(const Params& p, uint8_t* smem) {
  using PP = Pipe<CG>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long cyc_start = clock64();
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = (CG == 2) ? cluster_rank() : 0u;
  Bars B;
  B.full0 = sbase + SMEM_BARS + 8u * BAR_FULL;
  B.empty0 = sbase + SMEM_BARS + 8u * BAR_EMPTY;
  B.tfull0 = sbase + SMEM_BARS + 8u * BAR_TFULL;
  B.tempty0 = sbase + SMEM_BARS + 8u * BAR_TEMPTY;
  B.drain = sbase + SMEM_BARS + 8u * BAR_DRAIN;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SMEM_TMEM_SLOT);
  TailDesc* tail = reinterpret_cast<TailDesc*>(smem + SMEM_TAIL);
  // GEMM CTAs are groups 0 .. G-1; producer CTAs that join afterwards follow
  const int bid = static_cast<int>(blockIdx.x), G = p.num_gemm / CG;
  const int g = bid >= p.num_producers ? (bid - p.num_producers) / CG : G + bid / CG;
  const int total_tiles = p.total_tiles;
  const int nkb = p.num_segs * p.kb_per_seg;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(B.full0 + 8u * s, 1);
      mbar_init(B.empty0 + 8u * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(B.tfull0 + 8u * a, 1);
      mbar_init(B.tempty0 + 8u * a, CG * EPI_WARPS);  // one arrival per epilogue warp of the group
    }
    mbar_init(B.drain, 1);
    if constexpr (DYN)
      for (int s = 0; s < TQ_DEPTH; ++s) {  // the tile index ring's barriers
        mbar_init(sbase + SMEM_BARS + 8u * (BAR_TQ_FULL + s), 1);
        mbar_init(sbase + SMEM_BARS + 8u * (BAR_TQ_EMPTY + s), CG * (1 + EPI_WARPS));
      }
    if constexpr (SPLIT)
      for (int w = 0; w < EPI_WARPS; ++w) mbar_init(B.full0 + 8u * (BAR_PART - BAR_FULL + w), 1);
    fence_barrier_init();
  }
  __syncwarp();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers exist before anyone signals them
  if (warp == 1) {
    tmem_alloc_cg<CG>(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_cg<CG>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  grid_dep_wait();  // set-up done: from here on global memory may depend on the launch before
  if (p.trace_on && threadIdx.x == 0) atomicMin(&p.words->trace[TPO_TRACE_START], gtime());
  if constexpr (SPLIT) {  // the group's schedule (host-built)
    if (warp == 2 && lane < 16 && p.tail_split)
      reinterpret_cast<int*>(tail)[lane] = __ldg(reinterpret_cast<const int*>(p.tail_tab + g) + lane);
    __syncthreads();
  }

  if (warp == 0) {
    if (lane == 0) tma_role<CG, SPLIT, DYN>(p, sbase, B, rank, g, G, total_tiles, nkb, tail);
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) mma_role<CG, SPLIT, DYN>(p, sbase, tmem, B, g, G, total_tiles, nkb, tail);  // the whole warp
    __syncwarp();
  } else {
    epilogue_role<CG, SPLIT, DYN>(p, smem, tmem, B, rank, g, G, total_tiles, tail);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // neither CTA leaves while its peer may still use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg<CG>(tmem, TMEM_COLS);
  }
  if (p.trace_on && threadIdx.x == 0)
    atomicAdd(&p.words->trace[TPO_TRACE_CYC_GEMM], static_cast<unsigned long long>(clock64() - cyc_start));
}

// SPLIT: the build with the AG tail split (launched only when p.tail_split is
// set); the default build carries none of its code.
template <int CG, bool SPLIT, bool DYN>
__global__ void __launch_bounds__(NUM_THREADS, 1) fused_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  grid_dep_launch();  // the next launch may set up on SMs this one leaves
  if (static_cast<int>(blockIdx.x) < p.num_producers) {
    if (p.copy_on) producer_role(p, smem);
    if constexpr (SPLIT) {
      if (p.late_groups > 0) {  // the copy is done: join the GEMM (its ring buffers are free)
        __syncthreads();
        gemm_role<CG, SPLIT, DYN>(p, smem);
      }
    }
  } else if (static_cast<int>(blockIdx.x) < p.num_producers + p.num_gemm) {
    gemm_role<CG, SPLIT, DYN>(p, smem);
  }
  if (p.trace_on && threadIdx.x == 0) atomicMax(&p.words->trace[TPO_TRACE_END], gtime());
}

// ------------------------------------------------------------------ host side launch

cudaError_t configure_kernel() {
  cudaError_t e = cudaFuncSetAttribute(fused_kernel<1, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_kernel<2, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_kernel<1, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_kernel<2, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_kernel<1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_kernel<2, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  return e;
}

cudaError_t max_blocks_per_sm(int* n) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, fused_kernel<1, false, false>, NUM_THREADS, SMEM_ALLOC);
}

cudaError_t max_active_pairs(int* n) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_ALLOC;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, fused_kernel<2, false, false>, &cfg);
}

cudaError_t launch_fused(const Params& p, int grid, bool cooperative, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  int na = 0;
  if (p.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  if (p.cta_group == 2) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (p.tail_split) {
    if (p.cta_group == 2) return cudaLaunchKernelEx(&cfg, fused_kernel<2, true, false>, p);
    return cudaLaunchKernelEx(&cfg, fused_kernel<1, true, false>, p);
  }
  if (p.dyn) {
    if (p.cta_group == 2) return cudaLaunchKernelEx(&cfg, fused_kernel<2, false, true>, p);
    return cudaLaunchKernelEx(&cfg, fused_kernel<1, false, true>, p);
  }
  if (p.cta_group == 2) return cudaLaunchKernelEx(&cfg, fused_kernel<2, false, false>, p);
  return cudaLaunchKernelEx(&cfg, fused_kernel<1, false, false>, p);
}

}  // namespace tpo
