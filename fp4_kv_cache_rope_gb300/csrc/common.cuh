// Shared device-side building blocks of the CSA2 kernels (sm_103a):
// PTX wrappers for mbarriers, TMA / bulk copies, tcgen05 MMA and tensor
// memory, bounded waits, and the workspace layout shared by the launchers.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kGroup = 16;                  // channels per E4M3 scale
constexpr int kBlock = CSA2_BLOCK;          // positions per pool block
constexpr int kPoolBlocks = CSA2_POOL_BLOCKS;
constexpr int kMaxTopk = CSA2_MAX_TOPK;
constexpr int kPoolPositions = kPoolBlocks * kBlock;   // 16,384 candidates
constexpr int kMaxSplits = 8;               // attention split-K limit (one cluster per query row)
constexpr uint64_t kWaitNs = 2000000000ull; // default limit of a bounded on-chip wait (~2 s)

// ------------------------------------------------------------------ workspace
// The workspace is carved into 256-byte aligned regions in this order.
struct WsLayout {
  size_t status;       // uint32 status word
  size_t row_len;      // int32 [max_rows]  visible length per query row
  size_t tile_prefix;  // int32 [max_rows+1] prefix sum of 128-position tiles
  size_t scores;       // fp32 [max_rows, score_stride]
  size_t blockmax;     // fp32 [max_rows, bm_stride]
  size_t cand;         // fp32 [max_rows, kPoolPositions] Reindex candidate scores
  size_t total;
  int64_t score_stride, bm_stride;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t max_len, int64_t max_rows) {
  WsLayout L{};
  L.score_stride = (max_len + 127) / 128 * 128;
  L.bm_stride = (L.score_stride / kBlock + 31) / 32 * 32;
  size_t off = 0;
  L.status = off; off = align256(off + 256);
  L.row_len = off; off = align256(off + 4 * max_rows);
  L.tile_prefix = off; off = align256(off + 4 * (max_rows + 1));
  L.scores = off; off = align256(off + 4 * (size_t)max_rows * L.score_stride);
  L.blockmax = off; off = align256(off + 4 * (size_t)max_rows * L.bm_stride);
  L.cand = off; off = align256(off + 4 * (size_t)max_rows * kPoolPositions);
  L.total = off;
  return L;
}

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void set_status(uint32_t* st, uint32_t bits) {
  if (st) atomicOr(st, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ clusters
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ int cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return (int)r;
}
// Barrier over every thread of the cluster; orders shared-memory writes
// before it with reads after it across the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Load from the same shared-memory variable of CTA `rank` of the cluster.
// Ordering with the peer's writes comes from the cluster barrier between
// them, so independent loads may be in flight together.
__device__ __forceinline__ uint32_t peer_u32(const void* p, int rank) {
  uint32_t a = smem_u32(p), r, v;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(r));
  return v;
}

__device__ __forceinline__ uint4 peer_u32x4(const void* p, int rank) {
  uint32_t a = smem_u32(p), r;
  uint4 v;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(r));
  return v;
}

__device__ __forceinline__ float4 peer_f32x4(const void* p, int rank) {
  uint32_t a = smem_u32(p), r;
  float4 v;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(r));
  return v;
}
__device__ __forceinline__ float peer_f32(const void* p, int rank) {
  return __uint_as_float(peer_u32(p, rank));
}

// Physical cache row of (sequence b, position t); -1 when the page id is bad.
// Positions are below max_len (an int32), so page arithmetic runs in 32 bits:
// a shift for power-of-two page sizes, one unsigned division otherwise (a
// 64-bit division is a long software sequence on the GPU).
struct RowMap {
  const int32_t* page_table;
  int32_t page_size, max_pages_per_seq, max_len, num_pages;
  int32_t page_shift;  // log2(page_size) when it is a power of two, else -1
  __device__ __forceinline__ uint32_t page_of(uint32_t t) const {
    return page_shift >= 0 ? t >> page_shift : t / (uint32_t)page_size;
  }
  __device__ __forceinline__ uint32_t in_page(uint32_t t) const {
    return page_shift >= 0 ? t & (uint32_t)(page_size - 1) : t % (uint32_t)page_size;
  }
  __device__ __forceinline__ int64_t row(int b, int64_t t) const {
    if (page_size == 0) return (int64_t)b * max_len + t;
    const uint32_t pg = page_of((uint32_t)t);
    int32_t phys = page_table[(int64_t)b * max_pages_per_seq + pg];
    if (phys < 0 || phys >= num_pages) return -1;
    return (int64_t)phys * page_size + in_page((uint32_t)t);
  }
};
inline RowMap row_map_of(const csa2_cache& c) {
  int32_t shift = -1;
  if (c.page_size > 0 && (c.page_size & (c.page_size - 1)) == 0)
    for (shift = 0; (1 << shift) < c.page_size; ++shift) {
    }
  return RowMap{c.page_table, c.page_size, c.max_pages_per_seq, c.max_len, c.num_pages, shift};
}

// ------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Raises the barrier's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Limit of the pipeline waits below, per translation unit (each kernel file
// has its own copy); kWaitNs unless csa2_set_wait_limit changed it.
static __device__ unsigned long long g_wait_ns = kWaitNs;

// Waits for the phase with the given parity to complete.  Gives up after
// g_wait_ns or when *abort is set by another thread; returns false then and
// the caller records CSA2_DEV_TIMEOUT and winds down.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t lim = g_wait_ns;
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 7) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > lim) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Wait used while winding down: for copies and MMAs this CTA issued, which
// complete on their own.  It ignores the abort flag and the settable limit
// (a CTA must not exit, or free tensor memory, while one is in flight) and
// gives up only after the fixed kWaitNs.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && globaltimer() - t0 > kWaitNs) return false;
  }
}

// Waits until every copy armed on a ring of n mbarriers has landed.  Arm i
// (i = 0 .. armed-1) went to barrier i % n in phase i / n; phases of one
// barrier complete in order, so waiting for the last armed phase of each
// barrier covers all of them.
__device__ __forceinline__ void drain_armed(uint64_t* bars, int n, int armed) {
  for (int s = 0; s < n && s < armed; ++s) {
    const int last = s + n * ((armed - 1 - s) / n);
    mbar_wait_drain(bars + s, (uint32_t)((last / n) & 1));
  }
}

// Sets this translation unit's wait limit (host side).
static inline cudaError_t set_wait_limit_here(unsigned long long ns) {
  return cudaMemcpyToSymbol(g_wait_ns, &ns, sizeof(ns));
}

// ---------------------------------------------- programmatic dependent launch
// The step's kernels are launched with programmatic stream serialisation, so a
// kernel's CTAs may start while the previous kernel of the stream finishes.
// Before touching anything that kernel writes (or reads and this one
// overwrites) a kernel waits here: the wait returns once the previous grid has
// completed and its memory operations are visible.  Without the launch
// attribute it returns at once.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel of the stream start launching; its CTAs still wait in
// griddep_wait until this grid has completed.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ async copies
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// 16-byte global -> shared copy through the load/store path (L1 bypassed).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
// Arrives on `bar` once every cp.async this thread issued so far has landed
// (the arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, FP8 E4M3 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// D[tmem] (+)= A[smem] * B[smem]^T, f16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// D[tmem] (+)= (A * 2^(sa-127)) (B * 2^(sb-127))^T, block-scaled with one E8M0
// scale per 32 K-elements (kind::mxf8f6f4, scale_vec::1X).  Scale of A row m:
// tensor-memory lane m, column sfa + m/32, byte "A scale id" of idesc; scale
// of B column n: lane 32*(m/32) + n%32 (every lane quadrant holds a copy),
// column sfb + n/32, byte "B scale id".
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate));
}
// Copies a 32-row x 16-byte shared-memory matrix (descriptor `src`) into
// tensor-memory columns taddr .. taddr+3 of every lane quadrant: lane 32q + r,
// column taddr + j receives bytes 4j..4j+3 of row r.  Asynchronous, ordered
// before later tcgen05.mma of the same thread.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t src) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src)
               : "memory");
}
// Arrives on `bar` once all previously issued MMAs of this thread completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns; lane i of the warp reads TMEM lane
// (base lane + i).  Values are valid only after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t v0, uint32_t v1) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(v0),
               "r"(v1)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Keeps the compiler from moving uses of r above the preceding wait.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

// Shared-memory matrix descriptor of tcgen05 (K-major or MN-major canonical
// layouts).  swizzle: 0 none, 2 = 128 B, 4 = 64 B, 6 = 32 B.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of sm_100-class MMAs
  d |= (uint64_t)(swizzle & 7) << 61;
  return d;
}

// Instruction descriptor: fp32 accumulator, operand formats a/b, majorness,
// M and N.  kind::f16: 0 = f16, 1 = bf16.  kind::f8f6f4: 0 = E4M3.
// Instruction descriptor of kind::mxf8f6f4 with E8M0 scales (both operands
// K-major): A/B formats (E4M3 0, E2M1 5), N/8 at bit 17, the E8M0 scale type
// at bit 23, M/16 at bit 24; the B and A scale ids (bits 4 and 29) are OR-ed
// in per K step.
__host__ __device__ constexpr uint32_t instr_desc_mx(uint32_t afmt, uint32_t bfmt, int m, int n) {
  return (afmt << 7) | (bfmt << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
         ((uint32_t)(m >> 4) << 24);
}
__host__ __device__ constexpr uint32_t mx_scale_ids(uint32_t a_id, uint32_t b_id) {
  return (a_id << 29) | (b_id << 4);
}
__host__ __device__ constexpr uint32_t instr_desc(uint32_t afmt, uint32_t bfmt, bool a_mn,
                                                  bool b_mn, int m, int n) {
  return (1u << 4) | (afmt << 7) | (bfmt << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Order-preserving map of fp32 onto uint32 (larger float -> larger key);
// -0.0 is mapped like +0.0.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------ launchers
struct IndexLaunch;  // defined in indexer.cu
}  // namespace csa2
