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
// the groups of 8 are too many).  Each selection therefore runs over at most
// 18,432 candidates.
//
// One query row is served by a thread-block cluster of C CTAs (C = 1, 2, 4
// or 8, as many as the SMs allow), so that a few rows still spread their
// loads and their counting over many SMs.  CTA r of the cluster holds the
// candidates with ids [r*S, r*S + S), S = E * 512, as keys (the
// order-preserving uint32 image of the fp32 scores; 0 = absent) in shared
// memory.  A selection is a radix select whose counts are exchanged through
// distributed shared memory:
//   * the cluster's largest and smallest present keys fix the common high
//     bits; histograms of the next 11 bits of the keys still on the boundary
//     (summed over the cluster) narrow the boundary bin until it holds
//     exactly the keys still needed, or at most 256 keys, which are then
//     ranked exactly (larger key first, lower id on equal keys);
//   * keys above the boundary are taken, boundary keys as ranked (or, when
//     every bit is equal, in ascending id order); each CTA writes its taken
//     ids in id order after the ones of the lower-ranked CTAs.
#include "launch.h"

namespace csa2 {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCap = 18432;      // candidates of one selection, over the cluster
constexpr int kMaxCluster = 8;
constexpr int kDigitBits = 11;      // radix digit width
constexpr int kBins = 1 << kDigitBits;
constexpr int kRefineMax = 256;     // boundary keys ranked by counting

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

// Scalars one CTA publishes to its cluster in an exchange.
struct Mail {
  uint32_t a, b;
  int32_t c, d;
};

// Local candidate id i (global id base + i) is owned by thread i / E (a
// contiguous run per thread, so a thread-order scan emits ids in ascending
// order) and stored at keys[i + i / E]: one pad word per thread makes the
// per-thread stride E + 1 odd (E = 36, 18, 10 or 6), which keeps both the
// coalesced fills and the per-thread reads free of bank conflicts.
struct SelSmem {
  uint32_t keys[kSelThreads * 37];
  alignas(16) uint32_t whist[kSelWarps][kBins / 2];  // per-warp bin counters, two 16-bit counts per word
  alignas(16) uint32_t chist[2][kBins / 2];          // this CTA's bin totals (read by the cluster)
  Mail mail[2];                          // this CTA's published scalars (read by the cluster)
  Mail pm[kMaxCluster];                  // the cluster's scalars of the last exchange
  int sel[kPoolBlocks];                  // ids this CTA selected, ascending (read by the cluster)
  int list[kPoolBlocks];                 // id behind each of this CTA's candidate slots
  uint32_t bkey[kRefineMax];             // this CTA's boundary keys and ids (read by the cluster)
  int bid[kRefineMax];
  uint32_t akey[kRefineMax];             // the cluster's boundary keys and ids
  int aid[kRefineMax];
  uint8_t bsel[kSelCap];                 // refinement verdict per local candidate
  int red[32];
  int scan[32];
  uint32_t ured[2][32];
  int peer_base[kMaxCluster], peer_cnt[kMaxCluster];
  int taken[kMaxCluster];                // refine: taken boundary keys per CTA of the cluster
  int digit, above, nbd, nloc, nb_local, n_above;
  uint32_t floor_key;                    // every key the last selection took is >= it
  uint32_t range_hi;                     // the last selection's upper key bound
};

// Publishes m, synchronises the cluster and gathers every CTA's Mail into
// sm.pm.  Each exchange flips `par`, so a buffer is rewritten only after the
// cluster has passed another barrier (every peer has read it).
__device__ __forceinline__ void exchange(SelSmem& sm, const Mail& m, int C, int& par) {
  if (threadIdx.x == 0) sm.mail[par] = m;
  cluster_sync();
  if ((int)threadIdx.x < C) {
    const Mail* src = &sm.mail[par];
    Mail r;
    r.a = peer_u32(&src->a, threadIdx.x);
    r.b = peer_u32(&src->b, threadIdx.x);
    r.c = (int32_t)peer_u32(&src->c, threadIdx.x);
    r.d = (int32_t)peer_u32(&src->d, threadIdx.x);
    sm.pm[threadIdx.x] = r;
  }
  __syncthreads();
  par ^= 1;
}

// ---------------------------------------------------------------- block scans
// Exclusive scan of one int per thread in thread order; *total gets the sum.
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
    int t = lane < kSelWarps ? scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    scan[lane] = t;
  }
  __syncthreads();
  const int before = (warp > 0 ? scan[warp - 1] : 0) + x - v;
  *total = scan[kSelWarps - 1];
  __syncthreads();
  return before;
}

// ---------------------------------------------------------------- selection
// Selects the min(k, present) best of the cluster's candidates (CTA r holds
// global ids [base, base + E*512); keys past its candidates are 0).  On
// return sm.sel holds this CTA's selected global ids in ascending order
// (sm.nloc of them), sm.peer_base / sm.peer_cnt give every CTA's share, and
// the cluster-wide number selected is returned; sm.floor_key is a key that
// every selected key reaches and sm.range_hi the largest key of the range the
// search started from.  Control flow is uniform over the cluster.  The loops over a thread's E keys are unrolled twice only: with
// 16 warps per SM the shared-memory latency is hidden across warps, and the
// smaller code keeps the function in the instruction cache.
//
// floor_key != 0 states that at least k present keys of the cluster lie in
// [floor_key, ceil_key]; the cluster-wide range exchange is then skipped and
// the search starts from that range.  Should the counts contradict it (fewer
// than k keys in range, or keys above ceil_key taken besides k), the
// selection starts again with the exchange; the counts it tests are the
// cluster's, so every CTA restarts together.
template <int E>
__device__ __noinline__ int block_select(SelSmem& sm, int base, int k, int C, int rank, int& par,
                                         uint32_t floor_key, uint32_t ceil_key) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, t = threadIdx.x;
  const uint32_t* my = sm.keys + t * (E + 1);
  if (ceil_key < floor_key) floor_key = 0u;
restart:
  // ---- 1. range and number of the present keys over the cluster
  uint32_t mx = 0u, mn = 0xFFFFFFFFu;
  int present = 0;
  if (floor_key != 0u) {
    mx = ceil_key;
    mn = floor_key;
    present = k;
  } else {
#pragma unroll 2
    for (int e = 0; e < E; ++e) {
      const uint32_t v = my[e];
      mx = max(mx, v);
      mn = min(mn, v ? v : 0xFFFFFFFFu);
      present += v != 0u;
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    present = __reduce_add_sync(0xffffffffu, present);
    if (lane == 0) {
      sm.ured[0][warp] = mx;
      sm.ured[1][warp] = mn;
      sm.red[warp] = present;
    }
    __syncthreads();
    Mail m{};
    if (warp == 0) {
      m.a = __reduce_max_sync(0xffffffffu, lane < kSelWarps ? sm.ured[0][lane] : 0u);
      m.b = __reduce_min_sync(0xffffffffu, lane < kSelWarps ? sm.ured[1][lane] : 0xFFFFFFFFu);
      m.c = __reduce_add_sync(0xffffffffu, lane < kSelWarps ? sm.red[lane] : 0);
    }
    exchange(sm, m, C, par);
    mx = 0u;
    mn = 0xFFFFFFFFu;
    present = 0;
    for (int r = 0; r < C; ++r) {
      mx = max(mx, sm.pm[r].a);
      mn = min(mn, sm.pm[r].b);
      present += sm.pm[r].c;
    }
  }
  k = min(k, present);
  if (k <= 0) {
    if (t < C) sm.peer_base[t] = sm.peer_cnt[t] = 0;
    if (t == 0) {
      sm.nloc = 0;
      sm.floor_key = 0u;
      sm.range_hi = 0u;
    }
    __syncthreads();
    return 0;
  }
  // ---- 2. narrow the boundary.  Keys with (key & mask) > prefix are taken;
  // keys with (key & mask) == prefix are on the boundary and `remaining` of
  // them are taken -- those marked in sm.bsel (refine), else the first ones
  // by id (all of them when the boundary bin holds exactly `remaining`).
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
      const int nword = (int)((bmask + 2u) >> 1);  // two 16-bit counts per word
      const int nquad = (nword + 3) >> 2;          // four words (8 bins) per owner thread
      uint32_t* wh = sm.whist[warp];
      for (int i = lane; i < nquad * 4; i += 32) wh[i] = 0u;
      __syncwarp();
#pragma unroll 2
      for (int e = 0; e < E; ++e) {
        const uint32_t v = my[e];
        if (v && (v & mask) == prefix) {
          const uint32_t bin = (v >> lo) & bmask;
          atomicAdd(&wh[bin >> 1], 1u << ((bin & 1u) << 4));
        }
      }
      __syncthreads();
      // thread t < nquad owns bins 8t .. 8t+7: this CTA's counts, then the cluster's
      const bool owns = t < nquad;
      uint4 q = make_uint4(0u, 0u, 0u, 0u);
      if (owns) {
#pragma unroll 4
        for (int w = 0; w < kSelWarps; ++w) {
          const uint4 x = *reinterpret_cast<const uint4*>(&sm.whist[w][4 * t]);
          q.x += x.x;
          q.y += x.y;
          q.z += x.z;
          q.w += x.w;
        }
      }
      int c[8];
      c[0] = (int)(q.x & 0xFFFFu); c[1] = (int)(q.x >> 16);
      c[2] = (int)(q.y & 0xFFFFu); c[3] = (int)(q.y >> 16);
      c[4] = (int)(q.z & 0xFFFFu); c[5] = (int)(q.z >> 16);
      c[6] = (int)(q.w & 0xFFFFu); c[7] = (int)(q.w >> 16);
      if (C > 1) {
        if (owns) *reinterpret_cast<uint4*>(&sm.chist[par][4 * t]) = q;
        cluster_sync();
        if (owns) {
          uint4 rq[kMaxCluster];
#pragma unroll
          for (int r = 0; r < kMaxCluster; ++r)
            rq[r] = (r < C && r != rank) ? peer_u32x4(&sm.chist[par][4 * t], r)
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int r = 0; r < kMaxCluster; ++r) {
            c[0] += (int)(rq[r].x & 0xFFFFu); c[1] += (int)(rq[r].x >> 16);
            c[2] += (int)(rq[r].y & 0xFFFFu); c[3] += (int)(rq[r].y >> 16);
            c[4] += (int)(rq[r].z & 0xFFFFu); c[5] += (int)(rq[r].z >> 16);
            c[6] += (int)(rq[r].w & 0xFFFFu); c[7] += (int)(rq[r].w >> 16);
          }
        }
        par ^= 1;
      }
      int mine = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) mine += c[u];
      int total;
      const int before = block_excl_scan(mine, sm.scan, &total);
      if (floor_key != 0u && total < remaining) {
        // only with a floor key whose promise does not hold (a NaN score
        // missing from its block maximum): redo with the range exchange.
        // total is the cluster's sum, so every CTA takes this branch.
        floor_key = 0u;
        goto restart;
      }
      int cum = total - before - mine;  // keys in higher bins
#pragma unroll
      for (int u = 7; u >= 0; --u) {
        if (cum < remaining && remaining <= cum + c[u]) {
          sm.digit = 8 * t + u;
          sm.above = cum;
          sm.nbd = c[u];
        }
        cum += c[u];
      }
      __syncthreads();
      const int d = sm.digit;
      remaining -= sm.above;
      const int nbd = sm.nbd;
      prefix |= (uint32_t)d << lo;
      mask |= bmask << lo;
      __syncthreads();
      if (nbd == remaining) break;  // the whole boundary bin is taken
      if (nbd <= kRefineMax) {
        // ---- rank the few boundary keys of the cluster exactly
        refine = true;
        if (t == 0) sm.nb_local = sm.n_above = 0;
        if (t < kMaxCluster) sm.taken[t] = 0;
        __syncthreads();
        int n_above = 0;
#pragma unroll 2
        for (int e = 0; e < E; ++e) {
          const uint32_t v = my[e];
          if (v == 0u) continue;
          if ((v & mask) == prefix) {
            const int j = atomicAdd(&sm.nb_local, 1);
            sm.bkey[j] = v;
            sm.bid[j] = base + t * E + e;
            sm.bsel[t * E + e] = 0;
          } else if ((v & mask) > prefix) {
            ++n_above;
          }
        }
        n_above = __reduce_add_sync(0xffffffffu, n_above);
        if (lane == 0 && n_above) atomicAdd(&sm.n_above, n_above);
        __syncthreads();
        Mail mb{};
        mb.c = sm.nb_local;
        mb.d = sm.n_above;
        exchange(sm, mb, C, par);
        // boundary entry t of the cluster: CTA r's entries follow those of CTAs < r
        if (t < nbd) {
          int r = 0, off = 0;
          while (r < C - 1 && t >= off + sm.pm[r].c) off += sm.pm[r++].c;
          const int i = t - off;
          if (r == rank) {
            sm.akey[t] = sm.bkey[i];
            sm.aid[t] = sm.bid[i];
          } else {
            sm.akey[t] = peer_u32(&sm.bkey[i], r);
            sm.aid[t] = (int)peer_u32(&sm.bid[i], r);
          }
        }
        __syncthreads();
        if (t < nbd) {
          const uint32_t ki = sm.akey[t];
          const int ii = sm.aid[t];
          int rk = 0;
#pragma unroll 4
          for (int j = 0; j < nbd; ++j) {
            const uint32_t kj = sm.akey[j];
            rk += (kj > ki) | ((kj == ki) & (sm.aid[j] < ii));
          }
          if (rk < remaining) {
            atomicAdd(&sm.taken[ii / (E * kSelThreads)], 1);
            if (ii >= base && ii < base + E * kSelThreads) sm.bsel[ii - base] = 1;
          }
        }
        __syncthreads();
        break;
      }
      hi = lo - 1;
    }
  }
  // ---- 3. ordered compaction.  Per thread: keys above the boundary (low
  // half) and boundary keys (high half: all of them, or the marked ones).
  int packed = 0;
#pragma unroll 2
  for (int e = 0; e < E; ++e) {
    const uint32_t v = my[e];
    const uint32_t km = v & mask;
    const bool above = v != 0u && km > prefix;
    const bool on = v != 0u && km == prefix && (!refine || sm.bsel[t * E + e]);
    packed += above ? 1 : (on ? 1 << 16 : 0);
  }
  int tot;
  const int pbefore = block_excl_scan(packed, sm.scan, &tot);
  if (!refine) {
    // (with refine, every CTA's count above the boundary came with the
    // boundary keys and its taken boundary keys were counted in sm.taken)
    Mail mc{};
    mc.c = tot & 0xFFFF;  // above the boundary
    mc.d = tot >> 16;     // on the boundary
    exchange(sm, mc, C, par);
  }
  // Boundary keys of lower-ranked CTAs come first in id order; the cluster
  // takes the first `remaining` of them (refine: exactly the marked ones).
  // Every CTA computes every CTA's share from the same exchanged counts, so
  // peer_base, peer_cnt and out_base agree across the cluster.
  int on_acc = 0, on_base = 0, out_base = 0, nloc = 0;
  for (int r = 0; r < C; ++r) {
    const int a = refine ? sm.pm[r].d : sm.pm[r].c;
    const int o = refine ? sm.taken[r] : sm.pm[r].d;
    const int taken_on = refine ? o : min(o, max(0, remaining - on_acc));
    if (r == t) {
      sm.peer_base[r] = out_base;
      sm.peer_cnt[r] = a + taken_on;
    }
    if (r == rank) {
      nloc = a + taken_on;
      on_base = on_acc;
    }
    out_base += a + taken_on;
    on_acc += o;
  }
  if (floor_key != 0u && out_base != k) {
    // keys above ceil_key were taken besides the k (NaN scores missing from
    // their block maxima): redo with the range exchange
    floor_key = 0u;
    goto restart;
  }
  const int room = refine ? 0x7FFFFFFF : max(0, remaining - on_base);  // boundary keys taken here
  int on_before = pbefore >> 16;
  int pos = (pbefore & 0xFFFF) + min(on_before, room);
#pragma unroll 2
  for (int e = 0; e < E; ++e) {
    const uint32_t v = my[e];
    const uint32_t km = v & mask;
    bool take = v != 0u && km > prefix;
    if (v != 0u && km == prefix && (!refine || sm.bsel[t * E + e])) {
      take = on_before < room;
      ++on_before;
    }
    if (take) sm.sel[pos++] = base + t * E + e;
  }
  if (t == 0) {
    sm.nloc = nloc;
    sm.floor_key = prefix;  // selected keys have (key & mask) >= prefix, low bits of prefix 0
    sm.range_hi = mx;
  }
  __syncthreads();
  return k;
}

// ---------------------------------------------------------------- fills
// Consecutive threads take consecutive ids (coalesced loads).  Every load of
// a fill is unconditional (its index is clamped into the row) and is issued
// before any value is transformed or masked, so the loads of a thread
// overlap and a fill costs about one memory round trip.
template <int E>
__device__ __forceinline__ int key_slot(int i) { return i + i / E; }

// keys of global ids [base, base + E*512): order_key(src[id]) for id < n.
template <int E>
__device__ __forceinline__ void fill_contiguous(SelSmem& sm, const float* src, int n, int base) {
  const int last = n > 0 ? n - 1 : 0;
  float v[E];
#pragma unroll
  for (int u = 0; u < E; ++u)
    v[u] = __ldg(src + min(base + u * kSelThreads + (int)threadIdx.x, last));
#pragma unroll
  for (int u = 0; u < E; ++u) {
    const int i = u * kSelThreads + threadIdx.x;
    sm.keys[key_slot<E>(i)] = base + i < n ? order_key(v[u]) : 0u;
  }
  __syncthreads();
}

// Global candidate c < 8 * P stands for position sm.list[(c - base) / 8] * 8
// + c % 8 (sm.list holds this CTA's slots); its key is order_key(src[pos])
// when pos < len, else 0; a negative or out-of-range block id gives absent
// candidates.  With by_candidate, src is indexed by c instead.
template <int E>
__device__ __forceinline__ void fill_pool_positions(SelSmem& sm, const float* src, int P, int len,
                                                    bool by_candidate, int base) {
  const int n = P * kBlock;
  const int nblk = (len + kBlock - 1) / kBlock;
  int pos[E];
  float v[E];
#pragma unroll
  for (int u = 0; u < E; ++u) {
    const int i = u * kSelThreads + threadIdx.x;
    const int blk = base + i < n ? sm.list[i / kBlock] : -1;
    pos[u] = (blk >= 0 && blk < nblk) ? blk * kBlock + (i % kBlock) : len;  // len = absent
  }
#pragma unroll
  for (int u = 0; u < E; ++u) {
    const int c = base + u * kSelThreads + threadIdx.x;
    const int at = by_candidate ? min(c, n > 0 ? n - 1 : 0) : min(pos[u], len > 0 ? len - 1 : 0);
    v[u] = __ldg(src + at);
  }
#pragma unroll
  for (int u = 0; u < E; ++u) {
    const int i = u * kSelThreads + threadIdx.x;
    sm.keys[key_slot<E>(i)] = (base + i < n && pos[u] < len) ? order_key(v[u]) : 0u;
  }
  __syncthreads();
}

// Key of a group of `span` blocks (span a power of 8 >= 8) = max order key
// over its blocks below nb.  gid(i) gives the group of local candidate i (or
// a negative id for none).  Rows of block maxima are 128-byte aligned and
// groups start at multiples of 8 blocks, so they are read as float4s.
template <int E, typename G>
__device__ __forceinline__ void fill_groups(SelSmem& sm, const float* bm, int64_t nb, int span,
                                            G gid) {
  constexpr int kBatch = E < 6 ? E : 6;
  const int64_t last4 = nb > 0 ? (nb - 1) / 4 * 4 : 0;
#pragma unroll 1
  for (int u0 = 0; u0 < E; u0 += kBatch) {
    uint32_t m[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) m[j] = 0u;
#pragma unroll 1
    for (int q = 0; q < span; q += 8) {
      float4 a[kBatch], b[kBatch];
      int64_t first[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = (u0 + j) * kSelThreads + threadIdx.x;
        const int g = u0 + j < E ? gid(i) : -1;
        first[j] = (g >= 0 ? (int64_t)g * span : nb) + q;
        a[j] = __ldg(reinterpret_cast<const float4*>(bm + min(first[j], last4)));
        b[j] = __ldg(reinterpret_cast<const float4*>(bm + min(first[j] + 4, last4)));
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float x[8] = {a[j].x, a[j].y, a[j].z, a[j].w, b[j].x, b[j].y, b[j].z, b[j].w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (first[j] + e < nb) m[j] = max(m[j], order_key(x[e]));
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (u0 + j < E) sm.keys[key_slot<E>((u0 + j) * kSelThreads + threadIdx.x)] = m[j];
  }
  __syncthreads();
}

// sm.list[s] = id selected at global rank base/8 + s (< P), read from the
// CTA that selected it; then a cluster barrier so that sm.sel may be reused.
__device__ __forceinline__ void map_slots(SelSmem& sm, int S, int base, int P, int C, int rank) {
  const int slots = S / kBlock;
  for (int s = threadIdx.x; s < slots; s += kSelThreads) {
    const int j = base / kBlock + s;
    if (j >= P) break;
    int owner = 0;
    for (int r = 0; r < C; ++r)
      if (sm.peer_base[r] <= j && j < sm.peer_base[r] + sm.peer_cnt[r]) owner = r;
    const int at = j - sm.peer_base[owner];
    sm.list[s] = owner == rank ? sm.sel[at] : (int)peer_u32(&sm.sel[at], owner);
  }
  cluster_sync();
}

// Replaces this CTA's selected candidate ids c by list[(c - base)/8]*8 + c%8
// (the sub-group or block they stand for) and publishes them to the cluster.
__device__ __forceinline__ void expand_selected(SelSmem& sm, int base) {
  for (int i = threadIdx.x; i < sm.nloc; i += kSelThreads) {
    const int c = sm.sel[i];
    sm.sel[i] = sm.list[(c - base) / kBlock] * kBlock + c % kBlock;
  }
  cluster_sync();
}

template <int E>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(SelectParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  constexpr int S = E * kSelThreads;
  griddep_wait();  // the indexer's scores, block maxima and row plan
  griddep_launch_dependents();
  const int C = cluster_size(), rank = cluster_rank();
  const int row = blockIdx.x / C, t = threadIdx.x;
  const int base = rank * S;
  const int bi = row / p.tq, tq = row % p.tq;
  const int b = p.batch_ids ? p.batch_ids[bi] : bi;
  if (b < 0 || b >= p.batch) return;  // uniform over the cluster
  const int64_t orow = (int64_t)b * p.tq + tq;  // output row
  const int len = p.row_len[row];
  int par = 0;

  if (p.mode == 0) {
    const float* bm = p.blockmax + (int64_t)row * p.bm_stride;
    const float* sc = p.scores + (int64_t)row * p.score_stride;
    const int nb = (len + kBlock - 1) / kBlock;
    int P = nb < kPoolBlocks ? nb : kPoolBlocks;
    // ---- pool: top-P blocks by block maximum.  When there are more blocks
    // than one selection holds, groups of 8^level blocks are ranked by their
    // maximum first; each level expands the P best groups into their 8
    // sub-groups and keeps the P best of those.
    int span = 1;
    for (int64_t ng = nb; ng > kSelCap; ng = (ng + kBlock - 1) / kBlock) span *= kBlock;
    const int ng = (int)((nb + span - 1) / span);
    if (span == 1)
      fill_contiguous<E>(sm, bm, ng, base);
    else
      fill_groups<E>(sm, bm, nb, span, [&](int i) { return base + i < ng ? base + i : -1; });
    // (fewer than P only if some keys are absent, i.e. NaN block maxima)
    P = block_select<E>(sm, base, P, C, rank, par, 0u, 0u);
    cluster_sync();  // every CTA's selection is final before it is read
    for (; span > 1; span /= kBlock) {
      const int sub = span / kBlock;
      map_slots(sm, S, base, P, C, rank);
      if (sub == 1)
        fill_pool_positions<E>(sm, bm, P, nb, false, base);
      else
        fill_groups<E>(sm, bm, nb, sub, [&](int i) {
          return base + i < P * kBlock ? sm.list[i / kBlock] * kBlock + i % kBlock : -1;
        });
      P = block_select<E>(sm, base, P, C, rank, par, 0u, 0u);
      expand_selected(sm, base);
    }
    if (p.pool_out) {
      int32_t* po = p.pool_out + orow * kPoolBlocks + sm.peer_base[rank];
      for (int i = t; i < sm.nloc; i += kSelThreads) po[i] = sm.sel[i];
    }
    if (p.pool_cnt_out && rank == 0 && t == 0) p.pool_cnt_out[orow] = P;
    // ---- top-k over the pool's positions.  Each of the P pool blocks holds
    // a position whose score is its block maximum, every pool block maximum
    // reaches the pool selection's floor key, and no score exceeds the
    // largest block maximum: with P >= k, at least k candidates lie in that
    // key range, which lets the selection skip its range exchange.
    const uint32_t pool_floor = P >= p.k ? sm.floor_key : 0u;
    const uint32_t pool_ceil = sm.range_hi;
    map_slots(sm, S, base, P, C, rank);
    fill_pool_positions<E>(sm, sc, P, len, false, base);
    const int kk = block_select<E>(sm, base, p.k, C, rank, par, pool_floor, pool_ceil);
    int32_t* oi = p.out_idx + orow * p.k + sm.peer_base[rank];
    for (int i = t; i < sm.nloc; i += kSelThreads) {
      const int c = sm.sel[i];
      oi[i] = sm.list[(c - base) / kBlock] * kBlock + c % kBlock;
    }
    if (rank == 0 && t == 0) p.out_cnt[orow] = kk;
  } else {
    int pc = p.pool_cnt_in[orow];
    pc = pc < 0 ? 0 : (pc > kPoolBlocks ? kPoolBlocks : pc);
    const int32_t* pool = p.pool_in + orow * kPoolBlocks;
    const float* cd = p.cand + (int64_t)row * kPoolPositions;
    for (int s = t; s < S / kBlock && base / kBlock + s < pc; s += kSelThreads)
      sm.list[s] = pool[base / kBlock + s];
    __syncthreads();
    fill_pool_positions<E>(sm, cd, pc, len, true, base);
    const int kk = block_select<E>(sm, base, p.k, C, rank, par, 0u, 0u);
    int32_t* oi = p.out_idx + orow * p.k + sm.peer_base[rank];
    for (int i = t; i < sm.nloc; i += kSelThreads) {
      const int c = sm.sel[i];
      oi[i] = sm.list[(c - base) / kBlock] * kBlock + c % kBlock;
    }
    if (rank == 0 && t == 0) p.out_cnt[orow] = kk;
  }
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

template <int E>
static cudaError_t launch_select_e(const SelectParams& p, int C, cudaStream_t s) {
  const int smem = (int)sizeof(SelSmem);
  cudaError_t e =
      cudaFuncSetAttribute(select_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = prefer_max_shared(select_kernel<E>);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.n_rows * C), 1, 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, select_kernel<E>, p);
}

cudaError_t launch_select(const csa2_cache& c, const RowSet& rows, int mode, int32_t k,
                          const int32_t* pool_in, const int32_t* pool_cnt_in, int32_t* out_idx,
                          int32_t* out_cnt, int32_t* pool_out, int32_t* pool_cnt_out,
                          const WsLayout& L, uint8_t* ws, int num_sms, cudaStream_t s) {
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
  // as many CTAs per row (one per SM) as the SMs hold, up to 8, with every
  // cluster running in one wave (a cluster must fit inside one GPC)
  int C = 1;
  while (C < kMaxCluster && (int64_t)rows.n_rows * C * 2 <= num_sms) C *= 2;
  {
    static int fits[kMaxCluster + 1] = {};  // clusters of each size that run at once
    const int smem = (int)sizeof(SelSmem);
    while (C > 1) {
      if (!fits[C]) {
        int n = 0;
        switch (C) {
          case 8: cudaFuncSetAttribute(select_kernel<6>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                  n = max_active_clusters(select_kernel<6>, 8, kSelThreads, smem); break;
          case 4: cudaFuncSetAttribute(select_kernel<10>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                  n = max_active_clusters(select_kernel<10>, 4, kSelThreads, smem); break;
          default: cudaFuncSetAttribute(select_kernel<18>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                  n = max_active_clusters(select_kernel<18>, 2, kSelThreads, smem); break;
        }
        fits[C] = n + 1;
      }
      if (fits[C] - 1 >= rows.n_rows) break;
      C /= 2;
    }
  }
  record_launch_begin(CSA2_KERNEL_SELECT, s);
  cudaError_t e;
  switch (C) {
    case 8: e = launch_select_e<6>(p, 8, s); break;
    case 4: e = launch_select_e<10>(p, 4, s); break;
    case 2: e = launch_select_e<18>(p, 2, s); break;
    default: e = launch_select_e<36>(p, 1, s); break;
  }
  record_launch_end(CSA2_KERNEL_SELECT, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace csa2
