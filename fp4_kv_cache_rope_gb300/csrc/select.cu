// Step 3 of the path: per-query top-k selection and the block pool.
//
// Ranking (for positions and for blocks): larger score first, lower id on
// equal scores; outputs in ascending id order.  The pool keeps the
// min(2048, ceil(N/8)) blocks of 8 positions with the largest block maximum
// ("DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" knowledge
// note, section "Hierarchical Sparse Indexer: make later searches bounded";
// "Inside DeepSeek V4.1 Flash: CED, CSA2 and the 890-Byte KV Cache", section
// "Hierarchical indexing bounds later searches, not every search").
//
// The selection uses the pool itself to bound its work.  Under the ranking
// above every pool block holds its own maximum, so the P pool blocks hold P
// distinct positions ranked at least as high as the P-th block maximum; the
// k <= P best positions therefore all lie in pool blocks.  The same argument
// one level up (groups of 8 blocks ranked by their maximum) bounds the block
// selection for long sequences (and again for groups of 64 blocks when even
// the groups of 8 are too many).  Each selection then runs over at most
// 24,576 candidates held in registers by one CTA of 512 threads:
//   * keys are the order-preserving uint32 image of the fp32 scores; a radix
//     select finds the k-th largest key: the bits above the highest bit where
//     the block's largest and smallest keys differ are common, and the rest is
//     resolved 8 bits at a time with a shared-memory histogram (at most four
//     passes, stopping early once the boundary bin holds exactly the keys
//     still needed);
//   * keys above the boundary are all taken, keys on it are taken in
//     ascending id order until k are chosen; a block-wide exclusive scan
//     writes them in id order.
#include "launch.h"

namespace csa2 {

constexpr int kSelThreads = 512;
constexpr int kSelE = 48;  // candidates per thread (capacity 24,576)
constexpr int kSelCap = kSelThreads * kSelE;

struct SelectParams {
  int32_t mode;  // 0 = Full (pool + top-k from scores), 1 = top-k over pool candidates
  int32_t n_rows, tq, k, batch;
  const int32_t* batch_ids;
  const int32_t* row_len;
  const float* scores;
  int64_t score_stride;
  const float* blockmax;
  int64_t bm_stride;
  const float* cand;
  const int32_t* pool_in;
  const int32_t* pool_cnt_in;
  int32_t* out_idx;
  int32_t* out_cnt;
  int32_t* pool_out;
  int32_t* pool_cnt_out;
  uint32_t* status;
};

struct SelSmem {
  int red[32];
  int scan[32];
  uint32_t ured[2][32];
  int hist[256];
  int digit, above;
  int list[kPoolPositions];      // selected group ids of the current level
  int list2[kPoolBlocks];        // pool block ids
  int list3[kPoolBlocks];        // staging of a level's selection
};

__device__ __forceinline__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = lane < kSelThreads / 32 ? red[lane] : 0;
  t = __reduce_add_sync(0xffffffffu, t);
  __syncthreads();
  return t;
}

// Exclusive scan of one int per thread in thread order; returns the thread's
// offset, and the total through *total.
__device__ __forceinline__ int block_excl_scan(int v, int* scan, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += u;
  }
  if (lane == 31) scan[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kSelThreads / 32 ? scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    scan[lane] = t;
  }
  __syncthreads();
  const int before = (warp > 0 ? scan[warp - 1] : 0) + x - v;
  *total = scan[kSelThreads / 32 - 1];
  __syncthreads();
  return before;
}

// Select the k best of the block's candidates (key 0 = absent).  Candidate
// e of thread i has id i*kSelE + e.  Writes the selected ids, ascending, to
// out[0..k) (shared or global) and returns k.  k must not exceed the number
// of present keys.
template <typename Out>
__device__ int block_select(const uint32_t (&key)[kSelE], int k, SelSmem& sm, Out out) {
  if (k <= 0) return 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // ---- largest and smallest present key
  uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll
  for (int e = 0; e < kSelE; ++e) {
    if (key[e]) {
      mx = max(mx, key[e]);
      mn = min(mn, key[e]);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  if (lane == 0) {
    sm.ured[0][warp] = mx;
    sm.ured[1][warp] = mn;
  }
  __syncthreads();
  constexpr int kWarps = kSelThreads / 32;
  mx = __reduce_max_sync(0xffffffffu, lane < kWarps ? sm.ured[0][lane] : 0u);
  mn = __reduce_min_sync(0xffffffffu, lane < kWarps ? sm.ured[1][lane] : 0xFFFFFFFFu);
  // ---- radix passes below the common high bits
  uint32_t prefix = mx, mask = 0xFFFFFFFFu;
  int remaining = k;
  if (mx != mn) {
    int hi = 31 - __clz(mx ^ mn);
    mask = hi == 31 ? 0u : ~((2u << hi) - 1u);
    prefix = mx & mask;
    for (; hi >= 0; hi -= 8) {
      const int lo = hi >= 7 ? hi - 7 : 0;
      const int nbin = 1 << (hi - lo + 1);
      for (int i = threadIdx.x; i < 256; i += kSelThreads) sm.hist[i] = 0;
      __syncthreads();
#pragma unroll
      for (int e = 0; e < kSelE; ++e)
        if (key[e] && (key[e] & mask) == prefix)
          atomicAdd(&sm.hist[(key[e] >> lo) & (uint32_t)(nbin - 1)], 1);
      __syncthreads();
      if (warp == 0) {
        // lane holds bins 8*lane .. 8*lane+7; find the bin holding the
        // remaining-th largest key, scanning from the top
        int c[8], tot = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          c[u] = sm.hist[8 * lane + u];
          tot += c[u];
        }
        int above = tot;  // inclusive suffix over lanes >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_down_sync(0xffffffffu, above, o);
          if (lane + o < 32) above += v;
        }
        int cum = above - tot;  // keys in bins of higher lanes
#pragma unroll
        for (int u = 7; u >= 0; --u) {
          if (cum < remaining && remaining <= cum + c[u]) {
            sm.digit = 8 * lane + u;
            sm.above = cum;
          }
          cum += c[u];
        }
      }
      __syncthreads();
      const int d = sm.digit;
      remaining -= sm.above;
      prefix |= (uint32_t)d << lo;
      mask |= (uint32_t)(nbin - 1) << lo;
      const bool exact = sm.hist[d] == remaining;
      __syncthreads();
      if (exact) break;
    }
  }
  // ---- take keys above the boundary, and the first `remaining` on it
  int eq = 0;
#pragma unroll
  for (int e = 0; e < kSelE; ++e) eq += key[e] != 0u && (key[e] & mask) == prefix;
  int tot;
  const int eq_before = block_excl_scan(eq, sm.scan, &tot);
  int take = 0;
  {
    int eb = eq_before;
#pragma unroll
    for (int e = 0; e < kSelE; ++e) {
      const uint32_t km = key[e] & mask;
      const bool on = key[e] != 0u && km == prefix;
      take += (key[e] != 0u && km > prefix) || (on && eb < remaining);
      eb += on;
    }
  }
  int pos = block_excl_scan(take, sm.scan, &tot);
  {
    int eb = eq_before;
    const int base = threadIdx.x * kSelE;
#pragma unroll
    for (int e = 0; e < kSelE; ++e) {
      const uint32_t km = key[e] & mask;
      const bool on = key[e] != 0u && km == prefix;
      if ((key[e] != 0u && km > prefix) || (on && eb < remaining)) out(pos++, base + e);
      eb += on;
    }
  }
  __syncthreads();
  return k;
}

__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(SelectParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  const int row = blockIdx.x;
  const int bi = row / p.tq, tq = row % p.tq;
  const int b = p.batch_ids ? p.batch_ids[bi] : bi;
  if (b < 0 || b >= p.batch) return;
  const int64_t orow = (int64_t)b * p.tq + tq;  // output row
  const int len = p.row_len[row];
  const int base = threadIdx.x * kSelE;
  uint32_t key[kSelE];

  if (p.mode == 0) {
    const float* bm = p.blockmax + (int64_t)row * p.bm_stride;
    const float* sc = p.scores + (int64_t)row * p.score_stride;
    const int nb = (len + kBlock - 1) / kBlock;
    const int P = nb < kPoolBlocks ? nb : kPoolBlocks;
    const int kk = p.k < len ? p.k : len;
    // ---- pool: top-P blocks by block maximum.  Groups of 8^level blocks are
    // ranked by their maximum first when there are more blocks than the
    // block-wide selection holds; each level then expands the P best groups
    // into their 8 sub-groups and keeps the P best of those.
    int level = 0;
    for (int64_t ng = nb; ng > kSelCap; ng = (ng + kBlock - 1) / kBlock) ++level;
    auto group_key = [&](int64_t g, int span) -> uint32_t {
      uint32_t m = 0u;
      const int64_t first = g * span;
      for (int u = 0; u < span; ++u) {
        const int64_t i = first + u;
        if (i < nb) m = max(m, order_key(__ldg(bm + i)));
      }
      return m;
    };
    {
      int span = 1;
      for (int l = 0; l < level; ++l) span *= kBlock;
      const int64_t ng = (nb + span - 1) / span;
#pragma unroll
      for (int e = 0; e < kSelE; ++e) {
        const int64_t g = base + e;
        key[e] = g < ng ? (span == 1 ? order_key(__ldg(bm + g)) : group_key(g, span)) : 0u;
      }
      int* dst = level == 0 ? sm.list2 : sm.list;
      block_select(key, P, sm, [&](int o, int id) { dst[o] = id; });
      for (int l = level; l > 0; --l) {
        const int sub = span / kBlock;
#pragma unroll
        for (int e = 0; e < kSelE; ++e) {
          const int c = base + e;
          uint32_t v = 0u;
          if (c < P * kBlock) {
            const int64_t g = (int64_t)sm.list[c / kBlock] * kBlock + (c % kBlock);
            v = group_key(g, sub);
          }
          key[e] = v;
        }
        __syncthreads();
        int* out_list = l == 1 ? sm.list2 : sm.list;
        // expanded ids are written to a scratch copy first when overwriting list
        block_select(key, P, sm, [&](int o, int id) {
          sm.list3[o] = sm.list[id / kBlock] * kBlock + (id % kBlock);
        });
        for (int i = threadIdx.x; i < P; i += kSelThreads) out_list[i] = sm.list3[i];
        __syncthreads();
        span = sub;
      }
    }
    __syncthreads();
    if (p.pool_out) {
      int32_t* po = p.pool_out + orow * kPoolBlocks;
      for (int i = threadIdx.x; i < P; i += kSelThreads) po[i] = sm.list2[i];
    }
    if (p.pool_cnt_out && threadIdx.x == 0) p.pool_cnt_out[orow] = P;
    // ---- top-k over the pool's positions
#pragma unroll
    for (int e = 0; e < kSelE; ++e) {
      const int c = base + e;
      uint32_t v = 0;
      if (c < P * kBlock) {
        const int t = sm.list2[c / kBlock] * kBlock + (c % kBlock);
        if (t < len) v = order_key(__ldg(sc + t));
      }
      key[e] = v;
    }
    int32_t* oi = p.out_idx + orow * p.k;
    block_select(key, kk, sm, [&](int o, int id) {
      oi[o] = sm.list2[id / kBlock] * kBlock + (id % kBlock);
    });
    if (threadIdx.x == 0) p.out_cnt[orow] = kk;
  } else {
    int pc = p.pool_cnt_in[orow];
    pc = pc < 0 ? 0 : (pc > kPoolBlocks ? kPoolBlocks : pc);
    const int32_t* pool = p.pool_in + orow * kPoolBlocks;
    const float* cd = p.cand + (int64_t)row * kPoolPositions;
    for (int i = threadIdx.x; i < pc; i += kSelThreads) sm.list2[i] = pool[i];
    __syncthreads();
    int nvalid = 0;
#pragma unroll
    for (int e = 0; e < kSelE; ++e) {
      const int c = base + e;
      uint32_t v = 0;
      if (c < pc * kBlock) {
        const int blk = sm.list2[c / kBlock];
        const int64_t t = (int64_t)blk * kBlock + (c % kBlock);
        if (blk >= 0 && t < len) v = order_key(__ldg(cd + c));
      }
      key[e] = v;
      nvalid += v != 0u;
    }
    nvalid = block_sum(nvalid, sm.red);
    const int kk = p.k < nvalid ? p.k : nvalid;
    int32_t* oi = p.out_idx + orow * p.k;
    block_select(key, kk, sm, [&](int o, int id) {
      oi[o] = sm.list2[id / kBlock] * kBlock + (id % kBlock);
    });
    if (threadIdx.x == 0) p.out_cnt[orow] = kk;
  }
}

cudaError_t launch_select(const csa2_cache& c, const RowSet& rows, int mode, int32_t k,
                          const int32_t* pool_in, const int32_t* pool_cnt_in, int32_t* out_idx,
                          int32_t* out_cnt, int32_t* pool_out, int32_t* pool_cnt_out,
                          const WsLayout& L, uint8_t* ws, cudaStream_t s) {
  if (rows.n_rows <= 0) return cudaSuccess;
  SelectParams p;
  p.mode = mode;
  p.n_rows = rows.n_rows;
  p.tq = rows.tq;
  p.k = k;
  p.batch = c.batch;
  p.batch_ids = rows.batch_ids;
  p.row_len = reinterpret_cast<const int32_t*>(ws + L.row_len);
  p.scores = reinterpret_cast<const float*>(ws + L.scores);
  p.score_stride = L.score_stride;
  p.blockmax = reinterpret_cast<const float*>(ws + L.blockmax);
  p.bm_stride = L.bm_stride;
  p.cand = reinterpret_cast<const float*>(ws + L.cand);
  p.pool_in = pool_in;
  p.pool_cnt_in = pool_cnt_in;
  p.out_idx = out_idx;
  p.out_cnt = out_cnt;
  p.pool_out = pool_out;
  p.pool_cnt_out = pool_cnt_out;
  p.status = reinterpret_cast<uint32_t*>(ws + L.status);
  const int smem = (int)sizeof(SelSmem);
  cudaError_t e =
      cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  record_launch_begin(CSA2_KERNEL_SELECT, s);
  select_kernel<<<rows.n_rows, kSelThreads, smem, s>>>(p);
  record_launch_end(CSA2_KERNEL_SELECT, s);
  return cudaGetLastError();
}

}  // namespace csa2
