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
// 18,432 candidates held in registers by one CTA of 512 threads:
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
constexpr int kSelE = 36;  // candidates per thread (capacity 18,432)
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

// Candidate id i is owned by thread i / kSelE (a contiguous run of ids per
// thread, so a thread-order scan emits ids in ascending order) and stored at
// keys[i + i / kSelE]: one pad word per thread makes both the coalesced
// fills (consecutive ids) and the per-thread reads (stride kSelE + 1, an odd
// number of banks) free of bank conflicts.
constexpr int kDigitBits = 11;                 // radix digit width
constexpr int kBins = 1 << kDigitBits;         // 2,048 bins
constexpr int kRefineMax = 256;                // boundary keys ranked by counting
struct SelSmem {
  uint32_t keys[kSelThreads * (kSelE + 1)];
  int sel[kPoolBlocks];          // ids chosen by the last selection, ascending
  int list[kPoolBlocks];         // group / block ids kept by the current level
  uint32_t bkey[kRefineMax];     // boundary-bin keys and ids (ascending id)
  int bid[kRefineMax];
  uint8_t bsel[kSelCap];         // refinement verdict per id
  int red[32];
  int scan[32];
  uint32_t ured[2][32];
  // per-warp histograms, two 16-bit counters per word (a warp adds at most
  // 32 * kSelE < 65,536 to one bin)
  uint32_t whist[kSelThreads / 32][kBins / 2];
  int digit, above;
};

__device__ __forceinline__ int key_slot(int i) { return i + i / kSelE; }

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

// Exclusive scan of one int per thread in thread order.
__device__ __forceinline__ int block_excl_scan(int v, int* scan) {
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
  __syncthreads();
  return before;
}

// Selects the k best of the n first candidates (key 0 = absent) and writes
// their ids, ascending, to sm.sel[0..k).  k must not exceed the number of
// present keys.
//  1. largest / smallest present key: the bits above their highest
//     differing bit are common;
//  2. histograms of the next kDigitBits bits, restricted to the keys still
//     on the boundary, narrow the boundary bin (keys in higher bins are all
//     taken) until it holds exactly the keys still needed, or few enough to
//     rank exactly (larger key first, lower id on equal keys) by counting;
//  3. one ordered compaction writes the ids.
// Each CTA runs this code only a few times, so it is written as short loops
// (instruction lines are reused) rather than unrolled straight-line code.
__device__ __noinline__ void block_select(SelSmem& sm, int n, int k) {
  if (k <= 0) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, t = threadIdx.x;
  const int e_end = min(kSelE, max(0, n - t * kSelE));  // candidates of this thread
  const uint32_t* my = sm.keys + t * (kSelE + 1);       // this thread's keys
  constexpr int kWarps = kSelThreads / 32;
  // ---- 1. range of the present keys
  uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll 4
  for (int e = 0; e < e_end; ++e) {
    const uint32_t v = my[e];
    if (v) {
      mx = max(mx, v);
      mn = min(mn, v);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  if (lane == 0) {
    sm.ured[0][warp] = mx;
    sm.ured[1][warp] = mn;
  }
  __syncthreads();
  mx = __reduce_max_sync(0xffffffffu, lane < kWarps ? sm.ured[0][lane] : 0u);
  mn = __reduce_min_sync(0xffffffffu, lane < kWarps ? sm.ured[1][lane] : 0xFFFFFFFFu);
  // Selection state: keys with (key & mask) > prefix are taken; keys with
  // (key & mask) == prefix are on the boundary and `remaining` of them are
  // taken -- the first ones by id, or those marked in sm.bsel when refine.
  uint32_t prefix = mx, mask = 0xFFFFFFFFu;
  int remaining = k;
  bool refine = false;
  if (mx != mn) {
    int hi = 31 - __clz(mx ^ mn);
    mask = hi == 31 ? 0u : ~((2u << hi) - 1u);
    prefix = mx & mask;
    while (hi >= 0) {
      const int lo = hi >= kDigitBits - 1 ? hi - (kDigitBits - 1) : 0;
      const uint32_t bmask = (2u << (hi - lo)) - 1u;
      const int nword = (int)((bmask + 2u) >> 1);
      // ---- 2. histogram of bits [lo, hi] of the keys on the boundary
      uint32_t* wh = sm.whist[warp];
      for (int i = lane; i < nword; i += 32) wh[i] = 0u;
      __syncwarp();
#pragma unroll 4
      for (int e = 0; e < e_end; ++e) {
        const uint32_t v = my[e];
        if (v && (v & mask) == prefix) {
          const uint32_t bin = (v >> lo) & bmask;
          atomicAdd(&wh[bin >> 1], 1u << ((bin & 1u) << 4));
        }
      }
      __syncthreads();
      int c[4] = {0, 0, 0, 0};  // thread t owns bins 4t .. 4t+3
      if (2 * t < nword) {
        for (int w = 0; w < kWarps; ++w) {
          const uint32_t a = sm.whist[w][2 * t], b = (2 * t + 1 < nword) ? sm.whist[w][2 * t + 1] : 0u;
          c[0] += a & 0xFFFFu;
          c[1] += a >> 16;
          c[2] += b & 0xFFFFu;
          c[3] += b >> 16;
        }
      }
      const int mine = c[0] + c[1] + c[2] + c[3];
      const int before = block_excl_scan(mine, sm.scan);
      const int total = block_sum(mine, sm.red);
      int cum = total - before - mine;  // keys in higher bins
      for (int u = 3; u >= 0; --u) {
        if (cum < remaining && remaining <= cum + c[u]) {
          sm.digit = 4 * t + u;
          sm.above = cum;
          sm.scan[31] = c[u];  // size of the boundary bin
        }
        cum += c[u];
      }
      __syncthreads();
      const int d = sm.digit;
      remaining -= sm.above;
      const int nbd = sm.scan[31];
      prefix |= (uint32_t)d << lo;
      mask |= bmask << lo;
      __syncthreads();
      if (nbd == remaining) break;  // the whole boundary bin is taken
      if (nbd <= kRefineMax) {
        // rank the few boundary keys exactly by counting
        refine = true;
        int nb_mine = 0;
        for (int e = 0; e < e_end; ++e) nb_mine += my[e] != 0u && (my[e] & mask) == prefix;
        int o = block_excl_scan(nb_mine, sm.scan);
        for (int e = 0; e < e_end; ++e) {
          const uint32_t v = my[e];
          if (v != 0u && (v & mask) == prefix) {
            sm.bkey[o] = v;
            sm.bid[o] = t * kSelE + e;
            ++o;
          }
        }
        __syncthreads();
        // rank = keys above + equal keys with a lower id (list is in id order)
        if (t < nbd) {
          const uint32_t ki = sm.bkey[t];
          int rank = 0;
          for (int j = 0; j < nbd; ++j) {
            const uint32_t kj = sm.bkey[j];
            rank += (kj > ki) | ((kj == ki) & (j < t));
          }
          sm.bsel[sm.bid[t]] = rank < remaining ? 1 : 0;
        }
        __syncthreads();
        break;
      }
      hi = lo - 1;
    }
  }
  // ---- 3. keys above the boundary, then the boundary keys that are taken
  int eq = 0;
  if (!refine) {
    for (int e = 0; e < e_end; ++e) eq += my[e] != 0u && (my[e] & mask) == prefix;
  }
  const int eq_before = refine ? 0 : block_excl_scan(eq, sm.scan);
  int take = 0, eb = eq_before;
#pragma unroll 4
  for (int e = 0; e < e_end; ++e) {
    const uint32_t v = my[e];
    const uint32_t km = v & mask;
    const bool on = v != 0u && km == prefix;
    const bool pick = refine ? (on && sm.bsel[t * kSelE + e]) : (on && eb < remaining);
    take += (v != 0u && km > prefix) || pick;
    eb += on;
  }
  int pos = block_excl_scan(take, sm.scan);
  eb = eq_before;
#pragma unroll 4
  for (int e = 0; e < e_end; ++e) {
    const uint32_t v = my[e];
    const uint32_t km = v & mask;
    const bool on = v != 0u && km == prefix;
    const bool pick = refine ? (on && sm.bsel[t * kSelE + e]) : (on && eb < remaining);
    if ((v != 0u && km > prefix) || pick) sm.sel[pos++] = t * kSelE + e;
    eb += on;
  }
  __syncthreads();
}

// Maximum order key over blocks [g*span, g*span + span) of the row.
__device__ __forceinline__ uint32_t group_key(const float* bm, int64_t nb, int64_t g, int span) {
  uint32_t m = 0u;
  const int64_t first = g * span;
  for (int u = 0; u < span; ++u) {
    const int64_t i = first + u;
    if (i < nb) m = max(m, order_key(__ldg(bm + i)));
  }
  return m;
}

// Fills the keys of candidates 0 .. n-1 from f(i), consecutive threads on
// consecutive ids (coalesced loads), four loads in flight per thread.
template <typename F>
__device__ __forceinline__ void fill_keys(SelSmem& sm, int n, F f) {
#pragma unroll 1
  for (int r0 = 0; r0 < kSelE; r0 += 4) {
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = (r0 + u) * kSelThreads + threadIdx.x;
      v[u] = i < n ? f(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = (r0 + u) * kSelThreads + threadIdx.x;
      sm.keys[key_slot(i)] = v[u];
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(SelectParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  const int row = blockIdx.x, t = threadIdx.x;
  const int bi = row / p.tq, tq = row % p.tq;
  const int b = p.batch_ids ? p.batch_ids[bi] : bi;
  if (b < 0 || b >= p.batch) return;
  const int64_t orow = (int64_t)b * p.tq + tq;  // output row
  const int len = p.row_len[row];

  if (p.mode == 0) {
    const float* bm = p.blockmax + (int64_t)row * p.bm_stride;
    const float* sc = p.scores + (int64_t)row * p.score_stride;
    const int nb = (len + kBlock - 1) / kBlock;
    const int P = nb < kPoolBlocks ? nb : kPoolBlocks;
    const int kk = p.k < len ? p.k : len;
    // ---- pool: top-P blocks by block maximum.  When there are more blocks
    // than one selection holds, groups of 8^level blocks are ranked by their
    // maximum first; each level expands the P best groups into their 8
    // sub-groups and keeps the P best of those.
    int span = 1;
    for (int64_t ng = nb; ng > kSelCap; ng = (ng + kBlock - 1) / kBlock) span *= kBlock;
    const int ng = (int)((nb + span - 1) / span);
    fill_keys(sm, ng, [&](int g) -> uint32_t {
      return span == 1 ? order_key(__ldg(bm + g)) : group_key(bm, nb, g, span);
    });
    block_select(sm, ng, P);
    for (int i = t; i < P; i += kSelThreads) sm.list[i] = sm.sel[i];
    __syncthreads();
    for (; span > 1; span /= kBlock) {
      const int sub = span / kBlock;
      fill_keys(sm, P * kBlock, [&](int c) -> uint32_t {
        return group_key(bm, nb, (int64_t)sm.list[c / kBlock] * kBlock + c % kBlock, sub);
      });
      block_select(sm, P * kBlock, P);
      int nid[(kPoolBlocks + kSelThreads - 1) / kSelThreads];
#pragma unroll
      for (int u = 0; u < (kPoolBlocks + kSelThreads - 1) / kSelThreads; ++u) {
        const int i = t + u * kSelThreads;
        if (i < P) nid[u] = sm.list[sm.sel[i] / kBlock] * kBlock + sm.sel[i] % kBlock;
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < (kPoolBlocks + kSelThreads - 1) / kSelThreads; ++u) {
        const int i = t + u * kSelThreads;
        if (i < P) sm.list[i] = nid[u];
      }
      __syncthreads();
    }
    if (p.pool_out) {
      int32_t* po = p.pool_out + orow * kPoolBlocks;
      for (int i = t; i < P; i += kSelThreads) po[i] = sm.list[i];
    }
    if (p.pool_cnt_out && t == 0) p.pool_cnt_out[orow] = P;
    // ---- top-k over the pool's positions
    fill_keys(sm, P * kBlock, [&](int c) -> uint32_t {
      const int pos = sm.list[c / kBlock] * kBlock + (c % kBlock);
      return pos < len ? order_key(__ldg(sc + pos)) : 0u;
    });
    block_select(sm, P * kBlock, kk);
    int32_t* oi = p.out_idx + orow * p.k;
    for (int i = t; i < kk; i += kSelThreads) oi[i] = sm.list[sm.sel[i] / kBlock] * kBlock + sm.sel[i] % kBlock;
    if (t == 0) p.out_cnt[orow] = kk;
  } else {
    int pc = p.pool_cnt_in[orow];
    pc = pc < 0 ? 0 : (pc > kPoolBlocks ? kPoolBlocks : pc);
    const int32_t* pool = p.pool_in + orow * kPoolBlocks;
    const float* cd = p.cand + (int64_t)row * kPoolPositions;
    for (int i = t; i < pc; i += kSelThreads) sm.list[i] = pool[i];
    __syncthreads();
    int nvalid = 0;
    fill_keys(sm, pc * kBlock, [&](int c) -> uint32_t {
      const int blk = sm.list[c / kBlock];
      const int64_t pos = (int64_t)blk * kBlock + (c % kBlock);
      return (blk >= 0 && pos < len) ? order_key(__ldg(cd + c)) : 0u;
    });
    for (int i = t; i < pc * kBlock; i += kSelThreads) nvalid += sm.keys[key_slot(i)] != 0u;
    nvalid = block_sum(nvalid, sm.red);
    const int kk = p.k < nvalid ? p.k : nvalid;
    block_select(sm, pc * kBlock, kk);
    int32_t* oi = p.out_idx + orow * p.k;
    for (int i = t; i < kk; i += kSelThreads) oi[i] = sm.list[sm.sel[i] / kBlock] * kBlock + sm.sel[i] % kBlock;
    if (t == 0) p.out_cnt[orow] = kk;
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
