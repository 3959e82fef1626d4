// Steps 4-5 of the path: gather the selected FP4 rows (and the FP8 window
// rows), dequantise them, and run one softmax over all of them per head.
//
//   o_h = sum_j softmax_j(scale * q_h . x_j) x_j,   K = V = x_j (width D)
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" knowledge
// note: section "FP4 main KV: trade precision for bytes, not for a new GEMM"
// (dequantise before the attention arithmetic, SWA kept in FP8) and "Putting
// It Together" steps 7-8 (sparse attention with the local window).
//
// Exactness of the operand conversion: an E2M1 value times an E4M3 scale has
// at most 5 significant bits and lies in [2^-10, 2688]; an E4M3 window value
// lies in [2^-9, 448]: both are exact in f16.  Queries (bf16) are scaled per
// head by a power of two so that the largest magnitude fits f16, which keeps
// every bf16 value whose exponent is within f16's normal range exact.  The
// softmax weights are rounded to f16 before the P.V product and the same
// rounded weights are summed for the normaliser.
//
// Work split.  The keys of one query row (its selected entries, then its
// window rows) are cut into `splits` contiguous shares, one CTA each; the
// CTAs of a row form one thread-block cluster and merge their partial
// outputs through distributed shared memory at the end.  A CTA walks its
// share in tiles of up to 112 keys, all of them resident at once:
//
//   S^T[keys x heads] = X . Q^T      tcgen05.mma M = 128 (the tile's keys;
//                                    rows 112-127 are not used), N = 64
//                                    heads, K = D in steps of 16;
//   O^T[D x heads]  += X^T . P^T     M = 128 channels per accumulator tile,
//                                    N = 64 heads, K = the tile's keys.
//
// With the keys as M the QK product runs at the M = 128 rate of the tensor
// core (64 heads as M would run at the M = 64 rate), and each softmax thread
// owns one key, so it writes its row of P^T (the PV product's B operand,
// heads contiguous) without any exchange.  Tiles of 112 keys (not 128) make
// X (126 KB), Q (72 KB) and P^T (14 KB) fit in shared memory together.
//
// Warps (320 threads):
//   0-7  compute: dequantise tile i+1 into the X slabs while the tensor core
//        runs PV of tile i (slab pair by slab pair, as each PV accumulator
//        tile finishes with it), then the softmax of tile i+1 once its QK
//        product lands: thread (key j = 32 (warp % 4) + lane, heads
//        32 (warp / 4) .. +32).  The running maximum per head is raised
//        lazily: only when a logit exceeds it by more than 2^8 (then O^T
//        and the sums are rescaled in place).  A tile's raw bytes are read
//        (from L2) when its dequantisation starts, while PV of the previous
//        tile still holds the first slab pair.
//   8    MMA issuer (lane 0) and tensor-memory owner.
//   9    index warp: turns the tile's index entries into cache rows (page
//        table, bounds checks) up to four tiles ahead and prefetches those
//        rows from HBM into L2, so the compute warps' reads hit L2.
#include "codec.cuh"
#include "launch.h"

namespace csa2 {

constexpr int kTile = 112;          // keys per tile
constexpr int kAttnThreads = 320;
constexpr int kComputeThreads = 256;
constexpr int kKtSlots = 4;         // key-table ring (tiles resolved ahead)

template <int NSLAB>
struct AttnCfg {
  static constexpr int D = NSLAB * 64;
  static constexpr int NT = (NSLAB + 1) / 2;     // O^T accumulator tiles of 128 channels
  static constexpr int kXSlab = kTile * 128;     // [112 keys x 64 channels] f16, 128-byte rows
  static constexpr int kQSlab = 64 * 128;        // [64 heads x 64 channels] f16
  static constexpr int kXOff = 0;
  // Q directly after X: QK reads 128 rows of each X slab, and rows 112-127
  // of the last slab fall on Q (finite values; those S^T rows are unused)
  static constexpr int kQOff = NSLAB * kXSlab;
  static constexpr int kPOff = kQOff + NSLAB * kQSlab;
  static constexpr int kMiscOff = kPOff + kTile * 128;
  // misc area (byte offsets)
  static constexpr int kBars = 0;                // 32 mbarriers
  static constexpr int kFlags = 256;             // abort flag, tensor-memory address
  static constexpr int kQmul = 512;              // f32 [64] logit factor per head (log2 domain)
  static constexpr int kMrow = 768;              // f32 [64] running maximum per head
  static constexpr int kLrow = 1024;             // f32 [64] softmax denominator per head
  static constexpr int kFw = 1280;               // f32 [64] merge factor per head
  static constexpr int kLsum = 1536;             // f32 [4][64] per-quadrant partial sums
  static constexpr int kTmax = 2560;             // f32 [4][64] per-quadrant tile maxima
  static constexpr int kKtab = 3584;             // int32 [kKtSlots][kTile] key table
  static constexpr int kMiscBytes = kKtab + kKtSlots * kTile * 4;
  static constexpr int kSmem = kMiscOff + kMiscBytes;
  // Dequantisation items (key, 64-channel slab), laid out so that the 32
  // lanes of a warp take kSG consecutive slabs of 32/kSG consecutive keys:
  // each key's lanes read contiguous bytes of its row (few L1 wavefronts per
  // load), and the 16-byte stores into the swizzled slabs hit every bank
  // group equally.  Slabs past the last full group of kSG are taken 32 keys
  // at a time.
  static constexpr int kSG = NSLAB >= 4 ? 4 : NSLAB;
  static constexpr int kKPG = 32 / kSG;                       // keys per group
  static constexpr int kNFull = NSLAB / kSG;                  // full slab groups
  static constexpr int kKG = kTile / kKPG;                    // key groups
  static constexpr int kFullItems = kNFull * kKG * 32;
  static constexpr int kAllItems = kFullItems + (NSLAB - kNFull * kSG) * 128;
  static constexpr int kItems = (kAllItems + kComputeThreads - 1) / kComputeThreads;
  static_assert(kTile % kKPG == 0 && kTile <= 128, "item layout");
  // tensor memory: S^T x2 (128 columns), then O^T (64 NT)
  static constexpr int kTmemCols = 128 + 64 * NT <= 256 ? 256 : 512;
  static_assert(kSmem <= 227 * 1024, "attention: shared memory");
  static_assert((kXSlab % 1024) == 0 && (kQOff % 1024) == 0 && (kPOff % 1024) == 0,
                "128-byte swizzle atoms need 1024-byte aligned slabs");
  static_assert(NSLAB * kXSlab >= 64 * D * 2, "the X slabs hold the staged bf16 query");
  static_assert(7 + 2 * NT + 2 * kKtSlots <= 32, "mbarrier area");
};

struct AttnParams {
  // per layer (the layers of one call share the selection and the cache):
  // queries, window rows and outputs
  const uint16_t* q[CSA2_MAX_ATTN_LAYERS];
  const uint8_t* swa[CSA2_MAX_ATTN_LAYERS];
  float* out[CSA2_MAX_ATTN_LAYERS];
  int32_t n_layers;
  int32_t heads, n_rows, tq, batch;
  const int32_t* q_pos;
  const int32_t* idx;
  const int32_t* cnt;
  int32_t kcap;
  const int32_t* swa_cnt;
  int32_t window;
  float scale_log2;  // softmax scale * log2(e)
  int32_t splits;    // CTAs per query row (the cluster size)
  const uint8_t* codes;
  const uint8_t* scales;
  int64_t code_stride, scale_stride;
  const int32_t* seq_len;
  RowMap map;
  uint32_t* status;
};

struct RowKeys {
  int b, n_global, n_swa, vis;
  const uint8_t* swa0;  // first window row of this query
};

__device__ __forceinline__ RowKeys row_keys(const AttnParams& p, int row, int D,
                                            const uint8_t* swa) {
  RowKeys r;
  const int b = row / p.tq, tq = row % p.tq;
  r.b = b;
  int c = p.cnt[row];
  r.n_global = c < 0 ? 0 : (c > p.kcap ? p.kcap : c);
  int vis = p.seq_len[b];
  if (p.q_pos) {
    const int lim = p.q_pos[row] + 1;
    vis = lim < vis ? lim : vis;
  }
  r.vis = vis;
  if (p.q_pos == nullptr) {
    int w = p.swa_cnt ? p.swa_cnt[b] : p.window;
    r.n_swa = w < 0 ? 0 : (w > p.window ? p.window : w);
    r.swa0 = swa + (int64_t)b * p.window * D;
  } else {
    // band row r holds position q_pos[b][0] - (W - 1) + r; query tq sees band
    // rows tq .. tq + W - 1 with a position >= 0
    const int p0 = p.q_pos[(int64_t)b * p.tq];
    int lo = (p.window - 1) - p0;
    lo = lo > tq ? lo : tq;
    const int hi = tq + p.window;  // exclusive
    r.n_swa = hi > lo ? hi - lo : 0;
    r.swa0 = swa + ((int64_t)b * (p.tq + p.window - 1) + lo) * D;
  }
  return r;
}

// This CTA's share of the row's keys: selected entries [g0, g0+ng) of the
// index list and window rows [w0, w0+nw); local key l < ng is entry g0 + l,
// else window row w0 + l - ng.  Tiles hold ts keys (a multiple of 16, at most
// kTile), the last one the remainder (never empty).
struct CtaKeys {
  int g0, ng, w0, nw, n, ntile, ts;
  __device__ __forceinline__ int tile_keys(int i) const {
    const int r = n - i * ts;
    return r < ts ? r : ts;
  }
};

__device__ __forceinline__ CtaKeys cta_keys(const RowKeys& rk, int split, int splits) {
  CtaKeys k;
  k.g0 = (int)((int64_t)rk.n_global * split / splits);
  k.ng = (int)((int64_t)rk.n_global * (split + 1) / splits) - k.g0;
  k.w0 = (int)((int64_t)rk.n_swa * split / splits);
  k.nw = (int)((int64_t)rk.n_swa * (split + 1) / splits) - k.w0;
  k.n = k.ng + k.nw;
  k.ntile = (k.n + kTile - 1) / kTile;
  k.ts = k.ntile ? ((k.n + k.ntile - 1) / k.ntile + 15) / 16 * 16 : 0;
  return k;
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, %2, %3, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// Largest value over the 32 lanes of the warp.
__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// 2^x with the hardware approximation (relative error about 2^-22; the
// weights are rounded to f16 afterwards).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte store of f16x8 into row `row` (128-byte rows, 128-byte swizzle) of
// a slab at chunk position c (0..7).
__device__ __forceinline__ void st_swz(uint8_t* slab, int row, int c, uint4 v) {
  *reinterpret_cast<uint4*>(slab + row * 128 + ((c ^ (row & 7)) << 4)) = v;
}

// 32 tensor-memory lanes x 32 consecutive 32-bit columns: lane i of the warp
// reads TMEM lane (base lane + i).  Valid after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

// Brings [p, p + bytes) from HBM into L2, one prefetch per 64 bytes (the
// L2's fetch unit from HBM), each at an address inside the range (fire and
// forget: nothing waits for them).
__device__ __forceinline__ void prefetch_l2(const uint8_t* p, uint32_t bytes) {
  for (uint32_t o = 0; o < bytes; o += 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + o));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p + bytes - 1));
}

__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(const void* p, int rank) {
  uint32_t r;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// f16 copy of the query rows [heads x D] (bf16, staged row-major in shared
// memory at qs) into the swizzled Q slabs by the compute threads (thread t of
// 256), assuming no head needs scaling; returns, over the compute warps,
// whether some |q| >= 2^14 (then the copy is redone with a power-of-two scale
// per head).  Rows past `heads` are zero.
template <int NSLAB>
__device__ __forceinline__ bool convert_query(const uint8_t* qs, uint8_t* sq, int t, int heads) {
  constexpr int D = NSLAB * 64;
  constexpr int kChunks = D / 8;     // 16-byte chunks per head row
  constexpr int kAll = 64 * kChunks;
  constexpr int kQSlab = 64 * 128;
  constexpr int n = kComputeThreads;
  constexpr int kBatch = 6;            // loads in flight per thread and round
  bool big = false;
  for (int i0 = t; i0 < kAll; i0 += kBatch * n) {
    constexpr int kPer = kBatch;
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = i0 + n * u;
      v[u] = (i < kAll && i / kChunks < heads) ? reinterpret_cast<const uint4*>(qs)[i]
                                               : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = i0 + n * u;
      if (i >= kAll) break;
      const int h = i / kChunks, c = i - h * kChunks;
      const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t r[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        big |= ((w4[q] & 0x7F80u) >= (141u << 7)) | (((w4[q] >> 16) & 0x7F80u) >= (141u << 7));
        __half2 h2 = __floats2half2_rn(__uint_as_float(w4[q] << 16),
                                       __uint_as_float(w4[q] & 0xFFFF0000u));
        r[q] = *reinterpret_cast<uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(sq + (c >> 3) * kQSlab + h * 128 + (((c & 7) ^ (h & 7)) << 4)) =
          make_uint4(r[0], r[1], r[2], r[3]);
    }
  }
  return named_sync_or(1, kComputeThreads, big);
}

// Raises the running maximum of every head to cover the current tile (the
// softmax warps' rare path; uniform over them): the tile's maximum per head
// from this thread's logits sr (key slot of lane, heads 32 hf ..) through the
// warps' maxima in tmax, the sums l and, past the first tile, the O^T columns
// rescaled by 2^(m_old - m_new) once PV of the previous tile is complete,
// and the new maxima written to mrow.
template <int NT>
__device__ __noinline__ void raise_running_max(const uint32_t* sr, float* l, bool valid, int i,
                                               const float* qmul, float* mrow, float* tmax, int quad,
                                               int hf, int lane, uint32_t tO, uint32_t lane_base,
                                               uint64_t* pvt, volatile int* abort_flag, bool& ok) {
  const int hh = 32 * hf + lane;   // the head this lane publishes
  float mine = -INFINITY;
#pragma unroll
  for (int h = 0; h < 32; ++h) {
    const float x = valid ? __uint_as_float(sr[h]) * qmul[32 * hf + h] : -INFINITY;
    const float r = warp_max(x);
    mine = lane == h ? r : mine;
  }
  tmax[quad * 64 + hh] = mine;
  named_sync(3, kComputeThreads);
  const float m_old = mrow[hh];
  const float m_new = fmaxf(fmaxf(m_old, fmaxf(tmax[hh], tmax[64 + hh])),
                            fmaxf(tmax[128 + hh], tmax[192 + hh]));
  const float alpha = m_old == -INFINITY ? (m_new == -INFINITY ? 1.0f : 0.0f)
                                         : fast_exp2(m_old - m_new);
#pragma unroll
  for (int h = 0; h < 32; ++h) l[h] *= __shfl_sync(0xffffffffu, alpha, h);
  if (i > 0) {
    // O^T *= alpha per head column, once PV of tile i-1 is complete (PV of
    // this tile waits for the softmax warps' p_full arrivals)
    if (ok && !mbar_wait(pvt + NT - 1, (i - 1) & 1, abort_flag)) ok = false;
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
#pragma unroll 1
      for (int t2 = 0; t2 < 2 * NT; ++t2) {
        uint32_t v[16];
        const int hb = 16 * (t2 & 1);
        const uint32_t a = tO + lane_base + 64 * (t2 >> 1) + 32 * hf + hb;
        tmem_ld16(a, v);
        tmem_ld_wait();
        reg_fence(v);
#pragma unroll
        for (int h = 0; h < 16; ++h)
          v[h] = __float_as_uint(__uint_as_float(v[h]) * __shfl_sync(0xffffffffu, alpha, hb + h));
        tmem_st16(a, v);
      }
      tmem_st_wait();
    }
  }
  named_sync(3, kComputeThreads);   // every thread has read mrow and tmax
  if (quad == 0) mrow[hh] = m_new;
  named_sync(3, kComputeThreads);   // the new maxima are in mrow
}

// Key slot jj and slab s of dequantisation item `it` (see AttnCfg); false
// for the unused slots of the last partial group.
template <int NSLAB>
__device__ __forceinline__ bool item_of(int it, int& jj, int& s) {
  using C = AttnCfg<NSLAB>;
  if (it < C::kFullItems) {
    const int g = it >> 5, l = it & 31;
    const int kg = g % C::kKG, sg = g / C::kKG;
    jj = C::kKPG * kg + l % C::kKPG;
    s = C::kSG * sg + l / C::kKPG;
    return true;
  }
  const int it2 = it - C::kFullItems;
  jj = it2 & 127;
  s = C::kNFull * C::kSG + (it2 >> 7);
  return it2 < C::kAllItems - C::kFullItems && jj < kTile;
}

// Raw bytes of one (key, 64-channel slab) item: FP4 codes (32 B in a, b) and
// the slab's four scale bytes (c.x), or an FP8 window row's 64 bytes.
struct RawItem {
  uint4 a, b, c, d;
};

template <int NSLAB>
__global__ void __launch_bounds__(kAttnThreads, 1) attention_kernel(AttnParams p) {
  using C = AttnCfg<NSLAB>;
  constexpr int D = C::D;
  constexpr int NT = C::NT;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sx = smem + C::kXOff;
  uint8_t* sq = smem + C::kQOff;
  uint8_t* sp = smem + C::kPOff;
  uint8_t* misc = smem + C::kMiscOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + C::kBars);
  uint64_t* s_full = bars + 0;             // [2] QK of the tile landed (commit)
  uint64_t* p_full = bars + 2;             // softmax weights written (8 warps)
  uint64_t* q_ready = bars + 4;            // f16 query slabs written (8 warps)
  uint64_t* drain = bars + 5;
  uint64_t* xg = bars + 6;                 // [NT] X slab pair t of the tile written (8 warps)
  uint64_t* pvt = bars + 6 + NT;           // [NT] PV accumulator tile t done (commit)
  uint64_t* kt_full = bars + 6 + 2 * NT;   // [kKtSlots] key table written (index warp)
  uint64_t* kt_empty = kt_full + kKtSlots; // [kKtSlots] key table consumed (8 warps)
  uint64_t* q_land = kt_empty + kKtSlots;  // the query row's bulk copy landed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + C::kFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + C::kFlags + 4);
  float* qmul = reinterpret_cast<float*>(misc + C::kQmul);
  float* mrow = reinterpret_cast<float*>(misc + C::kMrow);
  float* lrow = reinterpret_cast<float*>(misc + C::kLrow);
  float* fw = reinterpret_cast<float*>(misc + C::kFw);
  float* lsum = reinterpret_cast<float*>(misc + C::kLsum);
  float* tmax = reinterpret_cast<float*>(misc + C::kTmax);
  int32_t* ktab = reinterpret_cast<int32_t*>(misc + C::kKtab);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_status(p.status, CSA2_DEV_BAD_ALIGN);
    return;
  }
  const int split = blockIdx.x;
  const int layer = (int)blockIdx.y / p.n_rows;  // grid rows: layer-major, then query row
  const int row = (int)blockIdx.y - layer * p.n_rows;
  const uint16_t* q_l = p.q[0];
  const uint8_t* swa_l = p.swa[0];
  float* out_l = p.out[0];
#pragma unroll
  for (int l = 1; l < CSA2_MAX_ATTN_LAYERS; ++l)
    if (l == layer) {
      q_l = p.q[l];
      swa_l = p.swa[l];
      out_l = p.out[l];
    }

  if (tid == 0) {
    mbar_init(s_full + 0, 1);
    mbar_init(s_full + 1, 1);
    mbar_init(p_full, 8);
    mbar_init(q_ready, 8);
    mbar_init(drain, 1);
    for (int t = 0; t < NT; ++t) {
      mbar_init(xg + t, 8);
      mbar_init(pvt + t, 1);
    }
    for (int s = 0; s < kKtSlots; ++s) {
      mbar_init(kt_full + s, 1);
      mbar_init(kt_empty + s, 8);
    }
    mbar_init(q_land, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (tid < 64) mrow[tid] = -INFINITY;
  if (warp == 8) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 128;  // O^T tile t at columns 128 + 64 t
  bool ok = true;  // this thread's view: false once a wait gave up
  // ---- Before the dependency wait: the query, which the selection does not
  // produce (the kernels ahead of the one this launch depends on have all
  // completed when it starts), so its copy and conversion overlap the tail
  // of the selection.  One bulk copy per 32 KB brings the row (bf16
  // [heads x D], contiguous and 16-byte aligned) into the X slabs.
  if (warp == 9 && lane == 1) {
    // the output row's first and last lines (their address translation is
    // then ready when the merge writes them)
    const float* o0 = out_l + (int64_t)row * p.heads * D;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(o0));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(o0 + (int64_t)p.heads * D - 1));
  }
  if (warp == 9 && lane == 0) {
    const uint8_t* qg = reinterpret_cast<const uint8_t*>(q_l + (int64_t)row * p.heads * D);
    const uint32_t qbytes = (uint32_t)p.heads * D * 2;
    mbar_arrive_expect_tx(q_land, qbytes);
    for (uint32_t o = 0; o < qbytes; o += 32768u)
      bulk_load(sx + o, qg + o, qbytes - o < 32768u ? qbytes - o : 32768u, q_land);
  }
  if (warp < 8) {
    const int ct = tid;
    // ---- query: f16 copy of the bf16 rows, staged in the X slabs by the
    // bulk copy above.  When some |q| >= 2^14, each head is redone scaled by
    // a power of two so that its f16 copy stays exact (the logit factor
    // absorbs the power).
    const uint8_t* qs = sx;
    if (!mbar_wait(q_land, 0, abort_flag)) ok = false;
    ok = __all_sync(0xffffffffu, ok);
    if (!convert_query<NSLAB>(qs, sq, ct, p.heads)) {
      if (ct < 64) qmul[ct] = ct < p.heads ? p.scale_log2 : 0.0f;
    } else {
      constexpr int kChunks = D / 8;
      constexpr int kPer = (kChunks + 31) / 32;
      for (int hh = 0; hh < 8; ++hh) {
        const int h = 8 * warp + hh;
        uint4 v[kPer];
        float mx = 0.0f;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int c = lane + 32 * i;
          v[i] = make_uint4(0, 0, 0, 0);
          if (h < p.heads && c < kChunks)
            v[i] = *reinterpret_cast<const uint4*>(qs + (h * D + c * 8) * 2);
          const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            mx = fmaxf(mx, fabsf(__uint_as_float(w4[u] << 16)));
            mx = fmaxf(mx, fabsf(__uint_as_float(w4[u] & 0xFFFF0000u)));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e = 0;
        if (mx > 16384.0f) e = (int)ceilf(log2f(mx)) - 14;
        const float inv = exp2f((float)-e);
        if (lane == 0) qmul[h] = h < p.heads ? p.scale_log2 * exp2f((float)e) : 0.0f;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int c = lane + 32 * i;
          if (c < kChunks) {
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              __half2 h2 = __floats2half2_rn(__uint_as_float(w4[u] << 16) * inv,
                                             __uint_as_float(w4[u] & 0xFFFF0000u) * inv);
              o[u] = *reinterpret_cast<uint32_t*>(&h2);
            }
            st_swz(sq + (c >> 3) * C::kQSlab, h, c & 7, make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
      }
    }
    fence_async_smem();
    named_sync(1, kComputeThreads);  // Q slabs and qmul written; the staged rows are free
    if (lane == 0) mbar_arrive(q_ready);
  }
  // everything read from here on may come from the previous kernels (the
  // selection and seq_len)
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 9) {
    // this CTA's share of the index list requested into L1 before the row's
    // counts are known, its start taken for a full selection (a shorter one
    // only makes part of the prefetch miss)
    const int g0s = (int)((int64_t)p.kcap * split / p.splits);
    const int g1s = (int)((int64_t)p.kcap * (split + 1) / p.splits);
    for (int e = g0s + 32 * lane; e < g1s; e += 32 * 32)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(p.idx + (int64_t)row * p.kcap + e));
  }
  const RowKeys rk = row_keys(p, row, D, swa_l);
  const CtaKeys ck = cta_keys(rk, split, p.splits);

  if (warp < 8) {
    // ============================================================ compute warps
    const int ct = tid;               // 0..255
    const int quad = warp & 3, hf = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const int j = 32 * quad + lane;   // softmax: this thread's key slot
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      if (ok && !mbar_wait(bar, parity, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
    };
    // raw bytes of tile i's keys for this thread's items
    auto load_raw = [&](int i, RawItem (&raw)[C::kItems], uint32_t& kinds) {
      const int32_t* tab = ktab + (i % kKtSlots) * kTile;
      const int nk = ck.tile_keys(i);
      kinds = 0;
#pragma unroll
      for (int u = 0; u < C::kItems; ++u) {
        int jj, s;
        if (ok && item_of<NSLAB>(ct + kComputeThreads * u, jj, s)) {
          const int v = jj < nk ? tab[jj] : -1;
          if (v >= 0) {
            const uint8_t* cp = p.codes + (int64_t)v * p.code_stride + s * 32;
            raw[u].a = __ldg(reinterpret_cast<const uint4*>(cp));
            raw[u].b = __ldg(reinterpret_cast<const uint4*>(cp + 16));
            raw[u].c.x = __ldg(reinterpret_cast<const uint32_t*>(p.scales + (int64_t)v * p.scale_stride + s * 4));
            kinds |= 1u << (2 * u);
          } else if (v <= -2) {
            const uint4* wp = reinterpret_cast<const uint4*>(rk.swa0 + (int64_t)(-2 - v) * D + s * 64);
            raw[u].a = __ldg(wp);
            raw[u].b = __ldg(wp + 1);
            raw[u].c = __ldg(wp + 2);
            raw[u].d = __ldg(wp + 3);
            kinds |= 2u << (2 * u);
          }
        }
      }
    };

    float l[32];  // partial softmax denominators: this key slot, heads 32 hf + h
#pragma unroll
    for (int h = 0; h < 32; ++h) l[h] = 0.0f;

    // Raw bytes of the tile to dequantise next, loaded one tile ahead (right
    // after the previous dequantisation), so that their latency is hidden
    // behind that tile's QK product, softmax and PV product.
    RawItem raw[C::kItems];
    uint32_t kinds = 0;
    if (ck.ntile > 0) {
      wait_all(kt_full, 0);
      load_raw(0, raw, kinds);
    }

    for (int i = 0; i < ck.ntile; ++i) {
      const int nk = ck.tile_keys(i);
      // ---- dequantise tile i, four slabs at a time (a warp's items cover
      // four consecutive slabs): slabs 4q .. 4q+3 are free once PV of tile
      // i-1 has finished with accumulator tiles 2q and 2q+1
      for (int q = 0; 2 * q < NT; ++q) {
        const bool two = 2 * q + 1 < NT;
        if (i > 0) {
          wait_all(pvt + 2 * q, (i - 1) & 1);
          if (two) wait_all(pvt + 2 * q + 1, (i - 1) & 1);
        }
        if (ok) {
#pragma unroll
          for (int u = 0; u < C::kItems; ++u) {
            int jj, s;
            if (!item_of<NSLAB>(ct + kComputeThreads * u, jj, s) || (s >> 2) != q) continue;
            uint8_t* slab = sx + s * C::kXSlab;
            const uint32_t kind = (kinds >> (2 * u)) & 3u;
            if (kind == 1) {
              const uint32_t cw[8] = {raw[u].a.x, raw[u].a.y, raw[u].a.z, raw[u].a.w,
                                      raw[u].b.x, raw[u].b.y, raw[u].b.z, raw[u].b.w};
#pragma unroll
              for (int c = 0; c < 8; ++c) {  // 8 channels = 4 code bytes, group c/2
                const uint32_t sb = (raw[u].c.x >> (8 * (c >> 1))) & 0xFFu;
                const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
                const __half2 sh = *reinterpret_cast<const __half2*>(&s2);
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const uint32_t v2 = e2m1x2_to_f16x2((cw[c] >> (8 * q)) & 0xFFu);
                  __half2 r2 = __hmul2(*reinterpret_cast<const __half2*>(&v2), sh);
                  o[q] = *reinterpret_cast<uint32_t*>(&r2);
                }
                st_swz(slab, jj, c, make_uint4(o[0], o[1], o[2], o[3]));
              }
            } else if (kind == 2) {
              const uint4 w[4] = {raw[u].a, raw[u].b, raw[u].c, raw[u].d};
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint32_t lo = (c & 1) ? w[c >> 1].z : w[c >> 1].x;
                const uint32_t hi = (c & 1) ? w[c >> 1].w : w[c >> 1].y;
                st_swz(slab, jj, c,
                       make_uint4(e4m3x2_to_f16x2(lo & 0xFFFFu), e4m3x2_to_f16x2(lo >> 16),
                                  e4m3x2_to_f16x2(hi & 0xFFFFu), e4m3x2_to_f16x2(hi >> 16)));
              }
            } else {
#pragma unroll
              for (int c = 0; c < 8; ++c) st_swz(slab, jj, c, make_uint4(0, 0, 0, 0));
            }
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(xg + 2 * q);
          if (two) mbar_arrive(xg + 2 * q + 1);
        }
      }
      // ---- the next tile's raw bytes
      if (i + 1 < ck.ntile) {
        wait_all(kt_full + ((i + 1) % kKtSlots), ((i + 1) / kKtSlots) & 1);
        load_raw(i + 1, raw, kinds);
      }
      // ---- softmax of tile i
      wait_all(s_full + (i & 1), (i >> 1) & 1);
      tc_fence_after();
      uint32_t sr[32];
      if (ok) {
        tmem_ld32(tmem + lane_base + 64 * (i & 1) + 32 * hf, sr);
        tmem_ld_wait();
        reg_fence32(sr);
      }
      const int32_t* tab = ktab + (i % kKtSlots) * kTile;
      const bool valid = ok && j < nk && tab[j] != -1;
      const float4* qm4 = reinterpret_cast<const float4*>(qmul + 32 * hf);
      const float4* mr4 = reinterpret_cast<const float4*>(mrow + 32 * hf);
      float vmax = -INFINITY;
#pragma unroll
      for (int h4 = 0; h4 < 8; ++h4) {
        const float4 q = qm4[h4], m = mr4[h4];
        vmax = fmaxf(vmax, __uint_as_float(sr[4 * h4]) * q.x - m.x);
        vmax = fmaxf(vmax, __uint_as_float(sr[4 * h4 + 1]) * q.y - m.y);
        vmax = fmaxf(vmax, __uint_as_float(sr[4 * h4 + 2]) * q.z - m.z);
        vmax = fmaxf(vmax, __uint_as_float(sr[4 * h4 + 3]) * q.w - m.w);
      }
      if (!valid) vmax = -INFINITY;
      // raise the running maximum when a logit exceeds it by more than 2^8
      // (always on the first tile); uniform over the compute warps.  On that
      // rare path S^T is read again from tensor memory afterwards, so that
      // its registers are free while O^T and the sums are rescaled.
      if (named_sync_or(2, kComputeThreads, vmax > 8.0f)) {
        // (out of line, so that the rare path's registers do not weigh on
        // the main loop; S^T is read again afterwards)
        float lt[32];   // copies: only these have their address taken
        uint32_t st[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          lt[h] = l[h];
          st[h] = sr[h];
        }
        raise_running_max<NT>(st, lt, valid, i, qmul, mrow, tmax, quad, hf, lane, tO, lane_base,
                              pvt, abort_flag, ok);
#pragma unroll
        for (int h = 0; h < 32; ++h) l[h] = lt[h];
        tc_fence_after();
        if (ok) {
          tmem_ld32(tmem + lane_base + 64 * (i & 1) + 32 * hf, sr);
          tmem_ld_wait();
          reg_fence32(sr);
        }
      }
      // weights p = 2^(logit - m), rounded to f16, summed as rounded; this
      // key's row of P^T, 8 heads (16 bytes) at a time
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t pk[4];
        const float4 qa = qm4[2 * u], qb = qm4[2 * u + 1], ma = mr4[2 * u], mb = mr4[2 * u + 1];
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const float mv[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 8 * u + 2 * e;
          const float x0 = __uint_as_float(sr[h]) * qv[2 * e] - mv[2 * e];
          const float x1 = __uint_as_float(sr[h + 1]) * qv[2 * e + 1] - mv[2 * e + 1];
          const float e0 = valid ? fast_exp2(x0) : 0.0f;
          const float e1 = valid ? fast_exp2(x1) : 0.0f;
          const __half2 ph = __floats2half2_rn(e0, e1);
          const float2 pf = __half22float2(ph);
          l[h] += pf.x;
          l[h + 1] += pf.y;
          pk[e] = *reinterpret_cast<const uint32_t*>(&ph);
        }
        if (j < kTile) st_swz(sp, j, 4 * hf + u, make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(p_full);
        mbar_arrive(kt_empty + (i % kKtSlots));
      }
    }
    // ---- after the last tile: per-head denominators (sum over the key slots)
    if (ck.ntile > 0) wait_all(pvt + NT - 1, (ck.ntile - 1) & 1);
    tc_fence_after();
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int h = 0; h < off; ++h) {
        const float send = upper ? l[h] : l[h + off];
        const float keep = upper ? l[h + off] : l[h];
        l[h] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    lsum[quad * 64 + 32 * hf + lane] = l[0];   // lane holds head 32 hf + lane
    named_sync(1, kComputeThreads);
    if (ct < 64) {
      const float s = (lsum[ct] + lsum[64 + ct]) + (lsum[128 + ct] + lsum[192 + ct]);
      const bool any = ck.ntile > 0 && ok;
      lrow[ct] = any ? s : 0.0f;
      if (!any) mrow[ct] = -INFINITY;
    }
  } else if (warp == 8) {
    // ================================================================ MMA warp
    if (lane == 0 && ck.ntile > 0) {
      constexpr uint32_t idesc_qk = instr_desc(0, 0, false, false, 128, 64);
      constexpr uint32_t idesc_pv = instr_desc(0, 0, true, true, 128, 64);
      // Descriptors are built once; an operand's descriptor at a byte offset
      // o from its base is the base descriptor plus o/16 (the start-address
      // field holds address/16 in its low 14 bits, and shared-memory
      // addresses stay below 2^18).  This keeps the issue loop to one add
      // per operand: the issuing thread shares its scheduler with two busy
      // compute warps, and each MMA takes only ~50 cycles of tensor time.
      const uint64_t qk_a = smem_desc(smem_u32(sx), 16, 1024, 2);
      const uint64_t qk_b = smem_desc(smem_u32(sq), 16, 1024, 2);
      const uint64_t pv_a = smem_desc(smem_u32(sx), C::kXSlab, 1024, 2);
      const uint64_t pv_b = smem_desc(smem_u32(sp), C::kXSlab, 1024, 2);
      bool issued = false;
      ok = mbar_wait(q_ready, 0, abort_flag);
      for (int i = 0; ok && i < ck.ntile; ++i) {
        const uint32_t sd = tmem + 64 * (i & 1);
        for (int t = 0; t < NT; ++t) {
          if (!mbar_wait(xg + t, i & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t a_t = qk_a + (uint64_t)(t * (2 * C::kXSlab / 16));
          const uint64_t b_t = qk_b + (uint64_t)(t * (2 * C::kQSlab / 16));
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            if (2 * t + s2 >= NSLAB) break;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16(sd, a_t + (uint64_t)((s2 * C::kXSlab + kk * 32) / 16),
                      b_t + (uint64_t)((s2 * C::kQSlab + kk * 32) / 16), idesc_qk,
                      (t | s2 | kk) != 0 ? 1u : 0u);
          }
          issued = true;
        }
        if (!ok) break;
        mma_commit(s_full + (i & 1));
        if (!mbar_wait(p_full, i & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const int nks = (ck.tile_keys(i) + 15) / 16;
        const uint32_t acc0 = i > 0 ? 1u : 0u;
        for (int t = 0; t < NT; ++t) {
          // A = X^T read channel-major: channels of slabs 2t, 2t+1 (for an odd
          // slab count the last tile's upper half falls on Q: unused rows)
          const uint64_t a_t = pv_a + (uint64_t)(t * (2 * C::kXSlab / 16));
          const uint32_t d_t = tO + 64 * t;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            if (kk < nks)
              mma_f16(d_t, a_t + (uint64_t)(kk * 2048 / 16), pv_b + (uint64_t)(kk * 2048 / 16),
                      idesc_pv, kk > 0 ? 1u : acc0);
          mma_commit(pvt + t);
        }
      }
      if (issued) {  // let every issued MMA land before tensor memory is freed
        mma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ============================================================== index warp
    constexpr uint32_t kCodeBytes = D / 2;
    constexpr uint32_t kScaleBytes = D / 16;
    for (int i = 0; i < ck.ntile; ++i) {
      const int slot = i % kKtSlots;
      if (i >= kKtSlots) {
        if (ok && !mbar_wait(kt_empty + slot, ((i / kKtSlots) - 1) & 1, abort_flag)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      int32_t* tab = ktab + slot * kTile;
      const int base = i * ck.ts;
      const int nk = ck.tile_keys(i);
      constexpr int kPer = (kTile + 31) / 32;
      int pos[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {  // index entries first, all in flight
        const int jj = lane + 32 * u;
        const int l = base + jj;
        pos[u] = (jj < nk && l < ck.ng) ? __ldg(p.idx + (int64_t)row * p.kcap + ck.g0 + l) : 0;
      }
      int vv[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int jj = lane + 32 * u;
        const int l = base + jj;
        int v = -1;
        if (jj < nk) {
          if (l < ck.ng) {
            if (pos[u] >= 0 && pos[u] < rk.vis) {
              const int64_t r = p.map.row(rk.b, pos[u]);
              if (r >= 0) v = (int)r;
              else set_status(p.status, CSA2_DEV_BAD_PAGE);
            } else {
              set_status(p.status, CSA2_DEV_BAD_INDEX);
            }
          } else {
            v = -2 - (ck.w0 + l - ck.ng);
          }
        }
        vv[u] = v;
        if (jj < kTile) tab[jj] = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(kt_full + slot);
      // the tile's rows into L2 once its table is out (the compute warps
      // read them from there; tile 0's reads may already be under way)
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        if (vv[u] >= 0) {
          prefetch_l2(p.codes + (int64_t)vv[u] * p.code_stride, kCodeBytes);
          prefetch_l2(p.scales + (int64_t)vv[u] * p.scale_stride, kScaleBytes);
        } else if (vv[u] <= -2) {
          prefetch_l2(rk.swa0 + (int64_t)(-2 - vv[u]) * D, (uint32_t)D);
        }
      }
    }
    // the CTA must not exit while the query copy may still write its shared
    // memory (the compute warps stop waiting for it after a timeout)
    if (lane == 0) mbar_wait_drain(q_land, 0);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool any = ck.ntile > 0 && !*abort_flag;

  if (p.splits == 1) {
    // ---- output: o[h][c] = O^T[c][h] / l_h
    if (warp < 8) {
      const int quad = warp & 3, hf = warp >> 2;
#pragma unroll 1
      for (int t = 0; t < NT; ++t) {
        const int c = 128 * t + 32 * quad + lane;
        if (128 * t + 32 * quad >= D) continue;   // warp-uniform: channels past D
        uint32_t v[32];
        if (any) {
          tmem_ld32(tO + ((uint32_t)(32 * quad) << 16) + 64 * t + 32 * hf, v);
          tmem_ld_wait();
          reg_fence32(v);
        }
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const int head = 32 * hf + h;
          if (head < p.heads) {
            const float lh = lrow[head];
            const float o = (any && lh > 0.0f) ? __uint_as_float(v[h]) / lh : 0.0f;
            out_l[((int64_t)row * p.heads + head) * D + c] = o;
          }
        }
      }
    }
  } else {
    // ---- split-K merge over the cluster of the row:
    //   o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s  per head,
    // M the largest m_s with l_s > 0.  Each CTA scales its own O^T by its
    // factor 2^(m_s - M) / den and stores it straight into the shared memory
    // of the CTA that owns each 32-channel group (a warp's stores cover 128
    // contiguous bytes of one head's row, the form distributed shared memory
    // moves fastest; the CTA's own share is stored locally); after a cluster
    // barrier every CTA sums the C partials of its own channels and writes
    // them out.
    const int Cn = p.splits;
    constexpr int kGroups = D / 32;
    const int slmax = 32 * ((kGroups + Cn - 1) / Cn);
    float* recv = reinterpret_cast<float*>(smem);   // [C][64][slmax] (X and Q are free)
    cluster_sync();  // every CTA's mrow / lrow final; every CTA is done with X and Q
    if (tid < 64) {
      float ms[kMaxSplits], ls[kMaxSplits];
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxSplits; ++r) {
        ms[r] = -INFINITY;
        ls[r] = 0.0f;
        if (r < Cn) {
          ms[r] = peer_f32(&mrow[tid], r);
          ls[r] = peer_f32(&lrow[tid], r);
          if (ls[r] > 0.0f) M = fmaxf(M, ms[r]);
        }
      }
      float den = 0.0f;
#pragma unroll
      for (int r = 0; r < kMaxSplits; ++r)
        if (r < Cn && ls[r] > 0.0f) den += exp2f(ms[r] - M) * ls[r];
      const float lm = lrow[tid];
      fw[tid] = (lm > 0.0f && den > 0.0f) ? exp2f(mrow[tid] - M) / den : 0.0f;
    }
    __syncthreads();
    if (warp < 8) {
      const int quad = warp & 3, hf = warp >> 2;
      float f[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) f[h] = fw[32 * hf + h];
#pragma unroll 1
      for (int t = 0; t < NT; ++t) {
        const int g = 4 * t + quad;   // 32-channel group of this warp
        if (g >= kGroups) continue;   // warp-uniform
        int r = 0;
        while (r + 1 < Cn && g >= (kGroups * (r + 1)) / Cn) ++r;
        const int c0 = 32 * ((kGroups * r) / Cn);
        const int cl = 32 * g + lane - c0;
        uint32_t v[32];
        if (any) {
          tmem_ld32(tO + ((uint32_t)(32 * quad) << 16) + 64 * t + 32 * hf, v);
          tmem_ld_wait();
          reg_fence32(v);
        }
        float* dst = recv + ((size_t)split * 64 + 32 * hf) * slmax + cl;
        if (r == split) {
#pragma unroll
          for (int h = 0; h < 32; ++h)
            dst[h * slmax] = (any && f[h] != 0.0f) ? __uint_as_float(v[h]) * f[h] : 0.0f;
        } else {
          const uint32_t da = map_to_rank(dst, r);
#pragma unroll
          for (int h = 0; h < 32; ++h)
            st_cluster_f32(da + (uint32_t)(h * slmax * 4),
                           (any && f[h] != 0.0f) ? __uint_as_float(v[h]) * f[h] : 0.0f);
        }
      }
    }
    cluster_sync();  // every partial is in its owner's shared memory
    {
      const int c0 = 32 * ((kGroups * split) / Cn);
      const int w = 32 * ((kGroups * (split + 1)) / Cn) - c0;
      const int n4 = w / 4;
      const int items = p.heads * n4;
      // four items per thread and round, every load of the round in flight
      // before the sums
      constexpr int kU = 4;
      for (int it0 = tid; it0 < items; it0 += kU * kAttnThreads) {
        float4 acc[kU];
        int hh[kU], cc[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int it = it0 + u * kAttnThreads;
          hh[u] = it < items ? it / n4 : 0;
          cc[u] = it < items ? it - hh[u] * n4 : 0;
          acc[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int sp2 = 0; sp2 < kMaxSplits; ++sp2) {
          if (sp2 < Cn) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const float4 x = *reinterpret_cast<const float4*>(recv + ((size_t)sp2 * 64 + hh[u]) * slmax + 4 * cc[u]);
              acc[u].x += x.x;
              acc[u].y += x.y;
              acc[u].z += x.z;
              acc[u].w += x.w;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (it0 + u * kAttnThreads < items)
            *reinterpret_cast<float4*>(out_l + ((int64_t)row * p.heads + hh[u]) * D + c0 + 4 * cc[u]) = acc[u];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, C::kTmemCols);
  if (tid == 0 && *abort_flag) set_status(p.status, CSA2_DEV_TIMEOUT);
}

cudaError_t set_wait_limit_attention(unsigned long long ns) { return set_wait_limit_here(ns); }

template <int NSLAB>
static cudaError_t run_attention(AttnParams p, cudaStream_t s) {
  using C = AttnCfg<NSLAB>;
  auto kern = attention_kernel<NSLAB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e == cudaSuccess) e = prefer_max_shared(kern);
  if (e != cudaSuccess) return e;
  // The merge stages C x 64 x (channels of the widest share) fp32 in the X,
  // Q and P areas: fewer splits when that would not fit.
  constexpr int kGroups = C::D / 32;
  while (p.splits > 1 && p.splits * 64 * 32 * ((kGroups + p.splits - 1) / p.splits) * 4 > C::kMiscOff)
    --p.splits;
  // A CTA takes a whole SM and a cluster must fit inside one GPC, so not every
  // cluster count runs at once: take the largest split count whose clusters
  // all run in one wave (the splits of a row must also be co-resident).
  {
    static int fits[kMaxSplits + 1] = {};  // clusters of each size that run at once
    int splits = p.splits;
    while (splits > 1) {
      if (!fits[splits]) fits[splits] = max_active_clusters(kern, splits, kAttnThreads, C::kSmem) + 1;
      if (fits[splits] - 1 >= p.n_layers * p.n_rows) break;
      --splits;
    }
    p.splits = splits;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.splits, (unsigned)(p.n_layers * p.n_rows), 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the split CTAs of a row
  attr[0].val.clusterDim.x = (unsigned)p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  record_launch_begin(CSA2_KERNEL_ATTENTION, s);
  e = cudaLaunchKernelEx(&cfg, kern, p);
  record_launch_end(CSA2_KERNEL_ATTENTION, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attention(const csa2_cache& c, const AttnArgs& a, const WsLayout& L,
                             uint8_t* ws, int num_sms, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  if (a.n_layers < 1 || a.n_layers > CSA2_MAX_ATTN_LAYERS) return cudaErrorInvalidValue;
  // grid rows: one per (layer, query row)
  if ((int64_t)a.n_layers * a.n_rows > 65535) return cudaErrorInvalidConfiguration;
  // the key table holds cache rows as int32
  const int64_t rows = c.page_size ? (int64_t)c.num_pages * c.page_size : (int64_t)c.batch * c.max_len;
  if (rows > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  AttnParams p;
  p.n_layers = a.n_layers;
  for (int l = 0; l < CSA2_MAX_ATTN_LAYERS; ++l) {
    const int k = l < a.n_layers ? l : 0;
    p.q[l] = a.q[k];
    p.swa[l] = a.swa[k];
    p.out[l] = a.out[k];
  }
  p.heads = a.heads;
  p.n_rows = a.n_rows;
  p.tq = a.tq;
  p.batch = c.batch;
  p.q_pos = a.q_pos;
  p.idx = a.idx;
  p.cnt = a.cnt;
  p.kcap = a.kcap;
  p.swa_cnt = a.swa_cnt;
  p.window = a.window;
  const float scale = a.scale > 0.0f ? a.scale : 1.0f / sqrtf((float)c.dim);
  p.scale_log2 = scale * 1.4426950408889634f;
  // as many CTAs per (layer, row) as fill the SMs once
  int splits = (int)(num_sms / ((int64_t)a.n_layers * a.n_rows));
  splits = splits < 1 ? 1 : (splits > kMaxSplits ? kMaxSplits : splits);
  const int max_tiles = (a.kcap + a.window + kTile - 1) / kTile;
  if (splits > max_tiles) splits = max_tiles < 1 ? 1 : max_tiles;
  p.splits = splits;
  p.codes = c.kv_codes;
  p.scales = c.kv_scales;
  p.code_stride = c.code_stride;
  p.scale_stride = c.scale_stride;
  p.seq_len = c.seq_len;
  p.map = row_map_of(c);
  p.status = reinterpret_cast<uint32_t*>(ws + L.status);
  switch (c.dim / 64) {
    case 2: return run_attention<2>(p, s);
    case 4: return run_attention<4>(p, s);
    case 8: return run_attention<8>(p, s);
    case 9: return run_attention<9>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa2
