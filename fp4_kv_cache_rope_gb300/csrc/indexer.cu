// Step 2 of the path: lightning-indexer scores on the 5th-generation tensor
// cores.
//
//   s_t = sum_h w_h * max(0, q_h . k_t)
//
// over E4M3 indexer keys k_t (di channels) and E4M3 queries q_h.  A Full layer
// scores every visible position and also emits per-8-position block maxima;
// a Reindex layer scores only the positions of the pool's blocks.  Pages:
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" knowledge
// note, section "Hierarchical Sparse Indexer: make later searches bounded"
// (the first Full indexer scans all positions; block maxima select a pool of
// at most 2,048 blocks of 8 positions; later Reindex layers score only the
// pool); "Inside DeepSeek V4.1 Flash: CED, CSA2 and the 890-Byte KV Cache",
// section "Hierarchical indexing bounds later searches, not every search".
//
// Kernel shape (two persistent CTAs per SM, 6 warps each):
//   warp 0   TMA producer: 128 key rows per stage (one 128-row box, or one box
//            per page, or one 8-row box per pool block) into a 4-deep ring,
//            plus the row's query block [Hi x di] into a double buffer;
//   warp 1   MMA issuer: D[128 positions x Hp heads] = K_tile x Q^T with
//            tcgen05.mma kind::f8f6f4 (M = 128, N = Hp, K = 32 per
//            instruction), accumulators double-buffered in tensor memory;
//            (MXFP4 keys: the warp also lays out each tile's E8M0 scales for
//            tcgen05.cp into tensor memory, ahead of block-scaled MMAs);
//   warps 2-5  epilogue: one thread per position reads its Hp accumulators
//            (tcgen05.ld 32x32b), applies ReLU and the head weights, writes
//            the fp32 score and, for Full layers, the block maximum.
// The decode indexer reads 128 bytes of key per position and does 2*Hp*di
// flops on them (128 flop/byte at Hp = 64): it is HBM bound on GB300.
#include "launch.h"

namespace csa2 {

struct IndexerParams {
  int32_t mode;  // 0 = Full, 1 = pool positions
  int32_t n_rows, tq, hi, batch;
  const int32_t* batch_ids;
  const int32_t* q_pos;
  const int32_t* seq_len;
  const int32_t* pool_blocks;
  const int32_t* pool_cnt;
  const float* w;
  RowMap map;
  int32_t rows_per_load;  // Full mode box height (128 or the page size)
  const uint8_t* idx_scales;  // MXFP4 keys: E8M0 bytes, 4 per physical row
  int64_t phys_rows;          // physical key rows (bounds of the scale copies)
  int32_t* row_len;
  int32_t* tile_prefix;
  float* scores;
  int64_t score_stride;
  float* blockmax;
  int64_t bm_stride;
  float* cand;
  uint32_t* status;
};

__device__ __forceinline__ int row_seq(const IndexerParams& p, int row) {
  const int bi = row / p.tq;
  return p.batch_ids ? p.batch_ids[bi] : bi;
}

// Visible length of query row `row` and its number of 128-wide tiles (Full:
// 128 positions per tile; Reindex: 16 pool blocks per tile).
__device__ __forceinline__ int row_tiles(const IndexerParams& p, int row, int& len_out) {
  const int b = row_seq(p, row);
  const int tq = row % p.tq;
  int len = 0;
  if (b >= 0 && b < p.batch) {
    len = p.seq_len[b];
    if (p.q_pos) {
      const int lim = p.q_pos[(int64_t)b * p.tq + tq] + 1;
      len = lim < len ? lim : len;
    }
    len = len < 0 ? 0 : (len > p.map.max_len ? p.map.max_len : len);
  }
  len_out = len;
  if (p.mode == 0) return (len + 127) / 128;
  int pc = (b >= 0 && b < p.batch) ? p.pool_cnt[(int64_t)b * p.tq + tq] : 0;
  pc = pc < 0 ? 0 : (pc > kPoolBlocks ? kPoolBlocks : pc);
  return (pc + 15) / 16;
}

// Visible length and tile count of every query row, then the prefix sum of
// tile counts (one block of 1024 threads).  Used when there are more query
// rows than the indexer computes in its own prologue.
__global__ void __launch_bounds__(1024) indexer_plan_kernel(IndexerParams p) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < p.n_rows; base += 1024) {
    const int row = base + threadIdx.x;
    int tiles = 0;
    if (row < p.n_rows) {
      int len;
      tiles = row_tiles(p, row, len);
      p.row_len[row] = len;
    }
    // block-wide inclusive scan of tiles
    int v = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += u;
      }
      warp_tot[lane] = t;
    }
    __syncthreads();
    const int incl = v + (warp > 0 ? warp_tot[warp - 1] : 0) + carry;
    if (row < p.n_rows) p.tile_prefix[row + 1] = incl;
    __syncthreads();
    if (threadIdx.x == 1023) carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) p.tile_prefix[0] = 0;
}

// Query rows up to which every indexer CTA plans the rows itself.
constexpr int kInlinePlanRows = 1024;

// Two persistent CTAs share each SM, each with its own 4-stage ring of key
// tiles: one ring keeps streaming while the other's producer or MMA thread
// is delayed (measured on the 128K decode step: 91 us against 108 us for
// one CTA per SM with an 8-stage ring, the same bytes in flight).
constexpr int kIdxCtasPerSm = 2;

// MX: MXFP4 keys (E2M1 codes + an E8M0 scale per 32 channels, di = 128).  The
// packed codes are expanded by the tensor map (CU_TENSOR_MAP_DATA_TYPE_16U4_
// ALIGN16B: 16 codes in 8 bytes, then an 8-byte gap) into the same 128-byte
// shared-memory rows the E4M3 keys use, and the MMA is the block-scaled
// kind::mxf8f6f4 with the query's scales fixed at 1.
template <int HP, int DI, bool MX = false>
struct IdxCfg {
  static constexpr int kTile = 128;
  static constexpr int kStageBytes = kTile * DI;
  static constexpr int kStages = 4;
  static constexpr int kQBytes = HP * DI;
  static constexpr int kSwizzle = DI == 128 ? 2 : (DI == 64 ? 4 : 6);
  static constexpr uint32_t kSbo = 8 * DI;
  static constexpr int kKSteps = DI / 32;
  static constexpr uint32_t kKRowBytes = MX ? DI / 2 : DI;   // global key bytes per row
  static constexpr int kSfTileBytes = MX ? kTile * 4 : 0;    // E8M0 bytes of one tile
  static constexpr int kAccCols = 2 * HP < 32 ? 32 : 2 * HP;
  // MX tensor-memory columns: A scales of accumulator a at kSfaCol + 32a (4
  // columns: row m reads column m/32), B scales at kSfbCol (N <= 64 reads 2)
  static constexpr int kSfaCol = kAccCols;
  static constexpr int kSfbCol = kAccCols + 64;
  static constexpr int kUsedCols = MX ? kSfbCol + 4 : kAccCols;
  static constexpr int kTmemCols = kUsedCols <= 32 ? 32 : (kUsedCols <= 64 ? 64 : (kUsedCols <= 128 ? 128 : 256));
  static constexpr int kSfOff = kStages * kStageBytes + 2 * kQBytes;
  // MX: the scale tiles of the two accumulators rearranged for tcgen05.cp
  // (row r holds the words of rows r, r+32, r+64, r+96), then 512 bytes of
  // E8M0 1.0 for the query scales
  static constexpr int kSfTOff = kSfOff + kStages * kSfTileBytes;
  static constexpr int kBarOff = kSfTOff + (MX ? 3 * 512 : 0);
  // mbarriers: full/empty per stage, qfull/qempty/tfull/tempty x2, drain;
  // then the abort flag and the TMEM address slot (one word each)
  static constexpr int kNumBars = 2 * kStages + 8 + 1;
  static constexpr int kBarBytes = (kNumBars * 8 + 8 + 127) / 128 * 128;
  static constexpr int kPlanOff = kBarOff + kBarBytes;  // row lengths, tile prefix
  static constexpr int kSmem = kPlanOff + 4 * (2 * kInlinePlanRows + 4);
  static_assert(kSmem <= 227 * 1024, "indexer shared memory exceeds the per-CTA limit");
};

// (d0, d1) += (w0, w1) * (max(x0, 0), max(x1, 0)) with one packed fp32 FMA
// (fma.rn per element, the same rounding as two fmaf calls).
__device__ __forceinline__ void fma2_relu(float& d0, float& d1, float w0, float w1, float x0,
                                          float x1) {
  const float a0 = fmaxf(x0, 0.0f), a1 = fmaxf(x1, 0.0f);
  asm("{\n\t.reg .b64 xa, xb, xc;\n\t"
      "mov.b64 xa, {%2, %3};\n\tmov.b64 xb, {%4, %5};\n\tmov.b64 xc, {%0, %1};\n\t"
      "fma.rn.f32x2 xc, xa, xb, xc;\n\tmov.b64 {%0, %1}, xc;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(w0), "f"(w1), "f"(a0), "f"(a1));
}

// First row whose tile range contains tile t (tile_prefix is non-decreasing).
__device__ __forceinline__ int find_row(const int32_t* prefix, int n_rows, int t) {
  int lo = 0, hi = n_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Walks the query rows of a CTA's tile range; the row's bounds and visible
// length are reloaded only when the row changes.
struct RowCursor {
  const int32_t* prefix;  // tile prefix [n_rows + 1] (shared or global memory)
  const int32_t* lens;    // visible length per row
  int row, begin, end, len;
  __device__ __forceinline__ void init(const int32_t* pre, const int32_t* ln, int n_rows, int t) {
    prefix = pre;
    lens = ln;
    row = find_row(prefix, n_rows, t);
    begin = prefix[row];
    end = prefix[row + 1];
    len = lens[row];
  }
  // Returns true when tile t starts a new row.
  __device__ __forceinline__ bool advance(const IndexerParams&, int t) {
    if (t < end) return false;
    do {
      ++row;
      begin = end;
      end = prefix[row + 1];
    } while (t >= end);
    len = lens[row];
    return true;
  }
};

template <int HP, int DI, bool MX>
__global__ void __launch_bounds__(192, kIdxCtasPerSm)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   IndexerParams p) {
  using C = IdxCfg<HP, DI, MX>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint8_t* qbuf = smem + C::kStages * C::kStageBytes;
  uint8_t* sfbuf = smem + C::kSfOff;           // MX: [kStages][128 rows][4 B]
  uint8_t* sft = smem + C::kSfTOff;            // MX: [2][32][16 B], then [32][16 B] of 1.0
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full = bars;                       // [kStages]
  uint64_t* empty = bars + C::kStages;         // [kStages]
  uint64_t* qfull = bars + 2 * C::kStages;     // [2]
  uint64_t* qempty = qfull + 2;                // [2]
  uint64_t* tfull = qempty + 2;                // [2]
  uint64_t* tempty = tfull + 2;                // [2]
  uint64_t* drain = tempty + 2;                // [1]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(drain + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();  // seq_len (the append) and, for many rows, the row plan
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1 KB alignment
    if (threadIdx.x == 0) set_status(p.status, CSA2_DEV_BAD_ALIGN);
    return;
  }
  // ---- rows: visible lengths and the tile prefix (planned here for up to
  // kInlinePlanRows rows; CTA 0 publishes them for the selection kernel)
  const int32_t* pre = p.tile_prefix;
  const int32_t* lens = p.row_len;
  if (p.n_rows <= kInlinePlanRows) {
    int32_t* s_len = reinterpret_cast<int32_t*>(smem + C::kPlanOff);
    int32_t* s_pre = s_len + kInlinePlanRows;
    for (int row = threadIdx.x; row < p.n_rows; row += blockDim.x) {
      int len;
      s_pre[row + 1] = row_tiles(p, row, len);
      s_len[row] = len;
    }
    __syncthreads();
    if (warp == 0) {
      int carry = 0;
      for (int base = 0; base < p.n_rows; base += 32) {
        const int i = base + lane;
        int v = i < p.n_rows ? s_pre[i + 1] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += u;
        }
        if (i < p.n_rows) s_pre[i + 1] = v + carry;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) s_pre[0] = 0;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
      for (int i = threadIdx.x; i < p.n_rows; i += blockDim.x) p.row_len[i] = s_len[i];
      for (int i = threadIdx.x; i <= p.n_rows; i += blockDim.x) p.tile_prefix[i] = s_pre[i];
    }
    pre = s_pre;
    lens = s_len;
  }
  const int total = pre[p.n_rows];
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(qfull + s, 1);
      mbar_init(qempty + s, 1);
      mbar_init(tfull + s, 1);
      mbar_init(tempty + s, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Zero both query buffers: rows hi..HP-1 stay zero (padded heads).
  for (int i = threadIdx.x; i < 2 * C::kQBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  if (MX)  // the query's E8M0 scales: 1.0 in every byte
    for (int i = threadIdx.x; i < 32; i += blockDim.x)
      reinterpret_cast<uint4*>(sft + 2 * 512)[i] =
          make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  fence_async_smem();
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  bool issued_mma = false;

  if (t_begin < t_end) {
    if (warp == 0) {
      // ------------------------------------------------------ TMA producer
      // The whole warp runs the loop.  Lane 0 waits on the ring and arms its
      // barriers; each lane issues the copies of the units it owns, so the
      // page-table lookups of a tile run in parallel.  On a paged cache the
      // lanes also hold a window of the row's page-table entries (pages
      // wb .. wb+63, two per lane), refilled 32 pages ahead of use: a lookup
      // that waits for memory in every tile would bound the scan, because the
      // copies of randomly placed pages keep address translation busy.
      const bool leader = lane == 0;
      auto wait_bcast = [&](uint64_t* bar, uint32_t parity) -> bool {
        int ok = 0;
        if (leader) ok = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
      };
      RowCursor rc;
      rc.init(pre, lens, p.n_rows, t_begin);
      int qn = 0, stage = 0, armed = 0;
      uint32_t phase = 0;
      int b = row_seq(p, rc.row), tq = rc.row % p.tq;
      int wseq = -1, wb = 0;          // sequence and first page of the window
      int32_t wcur = -1, wnext = -1;  // entries wb + lane and wb + 32 + lane
      const int mpp = p.map.max_pages_per_seq;
      auto pt_entry = [&](int bb, int pg) -> int32_t {
        return pg < mpp ? __ldg(p.map.page_table + (int64_t)bb * mpp + pg) : -1;
      };
      for (int t = t_begin; t < t_end; ++t) {
        const bool fresh = rc.advance(p, t) || t == t_begin;
        if (fresh) {
          b = row_seq(p, rc.row);
          tq = rc.row % p.tq;
          const int qs = qn & 1;
          if (!wait_bcast(qempty + qs, ((qn >> 1) & 1) ^ 1)) break;
          if (leader) {
            mbar_arrive_expect_tx(qfull + qs, (uint32_t)(p.hi * DI));
            tma_load_2d(qbuf + qs * C::kQBytes, &tm_q, 0, (int)(((int64_t)b * p.tq + tq) * p.hi),
                        qfull + qs);
          }
          ++qn;
        }
        if (!wait_bcast(empty + stage, phase ^ 1)) break;
        const int j = t - rc.begin;
        const int len = rc.len;
        uint8_t* dst = stages + stage * C::kStageBytes;
        // this lane's unit of the tile: its first cache row (-1: none), the
        // rows it copies and its scale bytes
        int64_t src = -1;
        int rows = 0;
        uint32_t sf_bytes = 0;
        int unit_rows = 0;
        if (p.mode == 0) {
          const int t0 = j * 128;
          if (p.map.page_size == 0) {
            if (leader) {
              src = (int64_t)b * p.map.max_len + t0;
              rows = 128;
              if (MX) {  // the tile's scale rows, cut at the end of the sequence
                const int n = p.map.max_len - t0 < 128 ? p.map.max_len - t0 : 128;
                sf_bytes = (uint32_t)(4 * n);
              }
            }
            unit_rows = 128;
          } else {
            const int rpl = p.rows_per_load;
            const int nu = 128 / rpl;  // units of the tile: pages pg0 .. pg0 + nu - 1
            const int pg0 = (int)p.map.page_of((uint32_t)t0);
            if (b != wseq || pg0 < wb || pg0 >= wb + 64) {
              wseq = b;
              wb = pg0;
              wcur = pt_entry(b, wb + lane);
              wnext = pt_entry(b, wb + 32 + lane);
            } else if (pg0 >= wb + 32) {
              wb += 32;
              wcur = wnext;
              wnext = pt_entry(b, wb + 32 + lane);
            }
            const int idx = pg0 + lane - wb;  // < 64 for the lanes that own a unit
            const int32_t e_cur = __shfl_sync(0xffffffffu, wcur, idx & 31);
            const int32_t e_next = __shfl_sync(0xffffffffu, wnext, idx & 31);
            const int32_t phys = idx < 32 ? e_cur : e_next;
            const int pos = t0 + lane * rpl;
            if (lane < nu && pos < len) {
              if (phys < 0 || phys >= p.map.num_pages) {
                set_status(p.status, CSA2_DEV_BAD_PAGE);
              } else {
                src = (int64_t)phys * p.map.page_size + p.map.in_page((uint32_t)pos);
                rows = rpl;
                sf_bytes = MX ? (uint32_t)(rpl * 4) : 0u;
              }
            }
            unit_rows = rpl;
          }
        } else {
          int pc = p.pool_cnt[(int64_t)b * p.tq + tq];
          pc = pc < 0 ? 0 : (pc > kPoolBlocks ? kPoolBlocks : pc);
          const int32_t* pool = p.pool_blocks + ((int64_t)b * p.tq + tq) * kPoolBlocks;
          // lane e < 16 owns the tile's pool block e: its id, then (paged
          // caches) its page-table entry; clamped indices keep every load
          // inside its array
          const int pi = j * 16 + lane;
          if (lane < 16 && pi < pc) {
            const int blk = __ldg(pool + (pi < kPoolBlocks ? pi : kPoolBlocks - 1));
            const int64_t t0b = (int64_t)blk * kBlock;
            if (blk < 0 || t0b >= len) {
              set_status(p.status, CSA2_DEV_BAD_POOL);
            } else if (p.map.page_size == 0) {
              src = (int64_t)b * p.map.max_len + t0b;
            } else {
              const uint32_t pg = p.map.page_of((uint32_t)t0b);
              const int32_t phys = pt_entry(b, (int)pg);
              if (phys < 0 || phys >= p.map.num_pages)
                set_status(p.status, CSA2_DEV_BAD_PAGE);
              else
                src = (int64_t)phys * p.map.page_size + p.map.in_page((uint32_t)t0b);
            }
            if (src >= 0) {
              rows = kBlock;
              // scale rows of a block, cut at the last physical row (a block
              // may run past the end of the sequence's rows; the key box is
              // clipped by the tensor map, the scale copy here)
              if (MX) {
                const int64_t n = p.phys_rows - src;
                sf_bytes = (uint32_t)(4 * (n < kBlock ? n : kBlock));
              }
            }
          }
          unit_rows = kBlock;
        }
        uint32_t bytes = (uint32_t)(rows * C::kKRowBytes) + sf_bytes;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
        if (leader) mbar_arrive_expect_tx(full + stage, bytes);
        __syncwarp();
        if (src >= 0) {
          tma_load_2d(dst + lane * unit_rows * DI, &tm_k, 0, (int)src, full + stage);
          if (MX && sf_bytes)
            bulk_load(sfbuf + stage * C::kSfTileBytes + lane * unit_rows * 4, p.idx_scales + 4 * src,
                      sf_bytes, full + stage);
        }
        ++armed;
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
      // a CTA must not exit while a copy it started still writes its shared
      // memory: after a timeout the consumers may have stopped reading the ring
      if (leader) {
        drain_armed(full, C::kStages, armed);
        drain_armed(qfull, 2, qn);
      }
    } else if (warp == 1 && (MX || lane == 0)) {
      // --------------------------------------------------------- MMA issuer
      // Lane 0 issues.  With MXFP4 keys the whole warp runs the loop: it
      // rearranges each tile's scale words for tcgen05.cp (row r of the copy
      // holds the words of tile rows r, r+32, r+64, r+96, so lane 32q + r,
      // column q receives row 32q + r's scales: where the block-scaled MMA
      // reads them), and lane 0 copies them into the accumulator's scale
      // columns ahead of its MMAs.  Waits are made warp-uniform.
      constexpr uint32_t idesc = MX ? instr_desc_mx(5, 0, 128, HP)
                                    : instr_desc(0, 0, false, false, 128, HP);
      auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        bool w = mbar_wait(bar, parity, abort_flag);
        if constexpr (MX) w = __all_sync(0xffffffffu, w);
        return w;
      };
      RowCursor rc;
      rc.init(pre, lens, p.n_rows, t_begin);
      int qn = 0, stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      const uint32_t st_base = smem_u32(stages), q_base = smem_u32(qbuf);
      if (MX && lane == 0)  // query scales (no swizzle, 16-byte rows, 8-row groups 128 B apart)
        tmem_cp_32x128b_x4(tmem + C::kSfbCol, smem_desc(smem_u32(sft + 2 * 512), 16, 128, 0));
      for (int t = t_begin; t < t_end; ++t) {
        const bool fresh = rc.advance(p, t) || t == t_begin;
        if (fresh) {
          if (qn > 0 && lane == 0) mma_commit(qempty + ((qn - 1) & 1));
          if (!wait_all(qfull + (qn & 1), (qn >> 1) & 1)) break;
          ++qn;
        }
        const int qs = (qn - 1) & 1;
        if (!wait_all(full + stage, phase)) break;
        if (!wait_all(tempty + acc, aphase ^ 1)) break;
        if (MX) {  // MMA(i-2) has finished with this accumulator's scale copy
          const uint32_t* src = reinterpret_cast<const uint32_t*>(sfbuf + stage * C::kSfTileBytes);
          reinterpret_cast<uint4*>(sft + acc * 512)[lane] =
              make_uint4(src[lane], src[32 + lane], src[64 + lane], src[96 + lane]);
          fence_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          if (MX)
            tmem_cp_32x128b_x4(tmem + C::kSfaCol + 32 * acc,
                               smem_desc(smem_u32(sft + acc * 512), 16, 128, 0));
          const uint32_t a0 = st_base + stage * C::kStageBytes;
          const uint32_t b0 = q_base + qs * C::kQBytes;
#pragma unroll
          for (int kk = 0; kk < C::kKSteps; ++kk) {
            const uint64_t ad = smem_desc(a0 + kk * 32, 16, C::kSbo, C::kSwizzle);
            const uint64_t bd = smem_desc(b0 + kk * 32, 16, C::kSbo, C::kSwizzle);
            if (MX)  // K step kk takes byte kk of each row's scale word
              mma_mx(tmem + acc * HP, ad, bd, idesc | mx_scale_ids(kk, kk),
                     tmem + C::kSfaCol + 32 * acc, tmem + C::kSfbCol, kk > 0 ? 1u : 0u);
            else
              mma_f8(tmem + acc * HP, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
          issued_mma = true;
          mma_commit(empty + stage);
          mma_commit(tfull + acc);
        }
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        if (++acc == 2) { acc = 0; aphase ^= 1; }
      }
    } else if (warp >= 2) {
      // ----------------------------------------------------------- epilogue
      const int quad = warp & 3;  // TMEM lane quadrant this warp may access
      const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
      bool ok = true;
      RowCursor rc;
      rc.init(pre, lens, p.n_rows, t_begin);
      int acc = 0;
      uint32_t aphase = 0;
      float wv[HP];
      float* out_row = nullptr;
      float* bm_row = nullptr;
      for (int t = t_begin; ok && t < t_end; ++t) {
        const bool fresh = rc.advance(p, t) || t == t_begin;
        if (fresh) {
          const int b = row_seq(p, rc.row);
          const int tq = rc.row % p.tq;
          const float* wr = p.w + ((int64_t)b * p.tq + tq) * p.hi;
#pragma unroll
          for (int h = 0; h < HP; ++h) wv[h] = h < p.hi ? __ldg(wr + h) : 0.0f;
          out_row = p.mode == 0 ? p.scores + (int64_t)rc.row * p.score_stride
                                : p.cand + (int64_t)rc.row * kPoolPositions;
          bm_row = p.blockmax + (int64_t)rc.row * p.bm_stride;
        }
        if (!mbar_wait(tfull + acc, aphase, abort_flag)) break;
        tc_fence_after();
        uint32_t r[HP];
#pragma unroll
        for (int c = 0; c < HP; c += 16) {
          uint32_t (&rr)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[c]);
          tmem_ld16(tmem + lane_base + acc * HP + c, rr);
        }
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < HP; c += 16) reg_fence(*reinterpret_cast<uint32_t(*)[16]>(&r[c]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty + acc);
        // four independent partial sums over the heads (head h into s4[h % 4]),
        // two at a time with the packed fp32 FMA, then their sum.  The
        // epilogue's instruction count is on the kernel's critical path.
        float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int h = 0; h < HP; h += 2)
          fma2_relu(s4[h & 3], s4[(h & 3) + 1], wv[h], wv[h + 1], __uint_as_float(r[h]),
                    __uint_as_float(r[h + 1]));
        const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        const int j = t - rc.begin;
        const int local = 32 * quad + lane;
        if (p.mode == 0) {
          const int pos = j * 128 + local;
          const bool valid = pos < rc.len;
          if (valid) out_row[pos] = s;
          float m = valid ? s : -INFINITY;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((lane & 7) == 0 && valid) bm_row[pos / kBlock] = m;
        } else {
          out_row[j * 128 + local] = s;
        }
        if (++acc == 2) { acc = 0; aphase ^= 1; }
      }
    }
  }
  __syncwarp();
  if (warp == 1) {
    if (lane == 0 && issued_mma) {  // let every issued MMA land before freeing TMEM
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, CSA2_DEV_TIMEOUT);
}

// ------------------------------------------------ multi-query Full indexer
// Full layers with Tq > 1 query rows per sequence (prefill chunks, multi-token
// verify): one work unit is (sequence, group of up to 128/HP consecutive query
// rows, 128-position key tile).  The MMA computes D[128 positions x
// (group x HP heads)] = K_tile x Q_group^T, so a sequence's keys are read once
// per group instead of once per query row (the per-row form re-reads them
// from L2 for every query, which bounds it on long chunks) and the tensor core
// runs N = 128.  Two accumulators of 128 columns per CTA, two CTAs per SM as
// in the per-row kernel; the four epilogue warps take the group's queries in
// turn: query g's HP accumulator columns, its head weights from shared
// memory, its own causal limit, its own score row and block maxima.
template <int HP, int DI>
struct MqCfg {
  static constexpr int kGroup = 128 / HP;           // query rows per group
  static constexpr int kN = kGroup * HP;             // 128
  static constexpr int kStageBytes = 128 * DI;
  static constexpr int kStages = 4;
  static constexpr int kQBytes = kN * DI;            // one group's query block
  static constexpr int kWBytes = kN * 4;             // one group's head weights
  static constexpr int kSwizzle = IdxCfg<HP, DI>::kSwizzle;
  static constexpr uint32_t kSbo = 8 * DI;
  static constexpr int kKSteps = DI / 32;
  static constexpr int kTmemCols = 256;
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kWOff = kQOff + 2 * kQBytes;
  static constexpr int kBarOff = kWOff + 2 * kWBytes;
  static constexpr int kNumBars = 2 * kStages + 9;
  static constexpr int kBarBytes = (kNumBars * 8 + 8 + 127) / 128 * 128;
  static constexpr int kPlanOff = kBarOff + kBarBytes;  // group tile prefix
  static constexpr int kSmem = kPlanOff + 4 * (kInlinePlanRows + 4);
  static_assert(kSmem <= 113 * 1024, "multi-query indexer: two CTAs per SM");
};

// Group gi: batch entry bi (sequence b), first query t0, gsz queries.
struct MqGroup {
  int bi, b, t0, gsz;
};
__device__ __forceinline__ MqGroup mq_group(const IndexerParams& p, int gi, int G) {
  const int gpb = (p.tq + G - 1) / G;
  MqGroup g;
  g.bi = gi / gpb;
  g.t0 = (gi - g.bi * gpb) * G;
  g.gsz = min(G, p.tq - g.t0);
  g.b = p.batch_ids ? p.batch_ids[g.bi] : g.bi;
  return g;
}

constexpr int kMqThreads = 192;  // producer, MMA issuer, 4 epilogue warps

template <int HP, int DI>
__global__ void __launch_bounds__(kMqThreads, kIdxCtasPerSm)
    indexer_mq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                      IndexerParams p, int n_groups) {
  using C = MqCfg<HP, DI>;
  constexpr int G = C::kGroup;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint8_t* qbuf = smem + C::kQOff;
  float* wbuf = reinterpret_cast<float*>(smem + C::kWOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* qfull = bars + 2 * C::kStages;
  uint64_t* qempty = qfull + 2;
  uint64_t* tfull = qempty + 2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(drain + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1) + 1;
  int32_t* s_pre = reinterpret_cast<int32_t*>(smem + C::kPlanOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();  // seq_len (the append)
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) set_status(p.status, CSA2_DEV_BAD_ALIGN);
    return;
  }
  // ---- plan: visible length of every query row (published by CTA 0 for the
  // selection kernel) and the tile prefix over groups
  if (blockIdx.x == 0) {
    for (int row = threadIdx.x; row < p.n_rows; row += blockDim.x) {
      int len;
      row_tiles(p, row, len);
      p.row_len[row] = len;
    }
  }
  for (int gi = threadIdx.x; gi < n_groups; gi += blockDim.x) {
    const MqGroup g = mq_group(p, gi, G);
    int vmax = 0;
    for (int q = 0; q < g.gsz; ++q) {
      int len;
      row_tiles(p, g.bi * p.tq + g.t0 + q, len);
      vmax = max(vmax, len);
    }
    s_pre[gi + 1] = (vmax + 127) / 128;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int i = base + lane;
      int v = i < n_groups ? s_pre[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (i < n_groups) s_pre[i + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_pre[0] = 0;
  }
  __syncthreads();
  const int total = s_pre[n_groups];
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(full + st, 1);
      mbar_init(empty + st, 1);
    }
    for (int st = 0; st < 2; ++st) {
      mbar_init(qfull + st, 1);
      mbar_init(qempty + st, 1);
      mbar_init(tfull + st, 1);
      mbar_init(tempty + st, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // zero both query blocks and weights: padded heads and queries stay zero
  for (int i = threadIdx.x; i < 2 * C::kQBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < 2 * C::kN; i += blockDim.x) wbuf[i] = 0.0f;
  fence_async_smem();
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  bool issued_mma = false;

  if (t_begin < t_end) {
    // the group of tile t and the group's first tile, walked in order
    int gcur = find_row(s_pre, n_groups, t_begin);
    auto advance = [&](int t) -> bool {  // true when tile t starts a new group
      if (t < s_pre[gcur + 1]) return false;
      while (t >= s_pre[gcur + 1]) ++gcur;
      return true;
    };
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------ TMA producer
      int qn = 0, stage = 0, armed = 0;
      uint32_t phase = 0;
      MqGroup g = mq_group(p, gcur, G);
      int vmax = 0;
      for (int t = t_begin; t < t_end; ++t) {
        const bool fresh = advance(t) || t == t_begin;
        if (fresh) {
          g = mq_group(p, gcur, G);
          vmax = 0;
          for (int q = 0; q < g.gsz; ++q) {
            int len;
            row_tiles(p, g.bi * p.tq + g.t0 + q, len);
            vmax = max(vmax, len);
          }
          const int qs = qn & 1;
          if (!mbar_wait(qempty + qs, ((qn >> 1) & 1) ^ 1, abort_flag)) break;
          const uint32_t wbytes = (uint32_t)(g.gsz * p.hi * 4);
          mbar_arrive_expect_tx(qfull + qs, (uint32_t)(g.gsz * p.hi * DI) + wbytes);
          const int64_t row0 = (int64_t)g.b * p.tq + g.t0;
          for (int q = 0; q < g.gsz; ++q)
            tma_load_2d(qbuf + qs * C::kQBytes + q * HP * DI, &tm_q, 0, (int)((row0 + q) * p.hi),
                        qfull + qs);
          bulk_load(wbuf + qs * C::kN, p.w + row0 * p.hi, wbytes, qfull + qs);
          ++qn;
        }
        if (!mbar_wait(empty + stage, phase ^ 1, abort_flag)) break;
        const int64_t t0 = (int64_t)(t - s_pre[gcur]) * 128;
        uint8_t* dst = stages + stage * C::kStageBytes;
        if (p.map.page_size == 0) {
          mbar_arrive_expect_tx(full + stage, 128 * DI);
          tma_load_2d(dst, &tm_k, 0, (int)((int64_t)g.b * p.map.max_len + t0), full + stage);
        } else {
          const int rpl = p.rows_per_load;
          const int nu = 128 / rpl;
          int nload = 0;
          int64_t src_rows[16];
          // page-table entries all requested before any is used (see above)
          const int32_t* pt = p.map.page_table + (int64_t)g.b * p.map.max_pages_per_seq;
          int32_t phys[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint32_t pg = p.map.page_of((uint32_t)(t0 + u * rpl));
            phys[u] = u < nu ? __ldg(pt + (pg < (uint32_t)p.map.max_pages_per_seq ? pg : p.map.max_pages_per_seq - 1))
                             : -1;
          }
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int64_t pos = t0 + (int64_t)u * rpl;
            src_rows[u] = -1;
            if (u < nu && pos < vmax) {
              if (phys[u] < 0 || phys[u] >= p.map.num_pages) {
                set_status(p.status, CSA2_DEV_BAD_PAGE);
              } else {
                src_rows[u] = (int64_t)phys[u] * p.map.page_size + p.map.in_page((uint32_t)pos);
                ++nload;
              }
            }
          }
          mbar_arrive_expect_tx(full + stage, (uint32_t)(nload * rpl * DI));
          for (int u = 0; u < 128 / rpl; ++u)
            if (src_rows[u] >= 0)
              tma_load_2d(dst + u * rpl * DI, &tm_k, 0, (int)src_rows[u], full + stage);
        }
        ++armed;
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
      drain_armed(full, C::kStages, armed);   // copies in flight, as above
      drain_armed(qfull, 2, qn);
    } else if (warp == 1 && lane == 0) {
      // --------------------------------------------------------- MMA issuer
      int qn = 0, stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      const uint32_t st_base = smem_u32(stages), q_base = smem_u32(qbuf);
      uint32_t idesc = 0;
      for (int t = t_begin; t < t_end; ++t) {
        const bool fresh = advance(t) || t == t_begin;
        if (fresh) {
          if (qn > 0) mma_commit(qempty + ((qn - 1) & 1));
          if (!mbar_wait(qfull + (qn & 1), (qn >> 1) & 1, abort_flag)) break;
          ++qn;
          idesc = instr_desc(0, 0, false, false, 128, mq_group(p, gcur, G).gsz * HP);
        }
        const int qs = (qn - 1) & 1;
        if (!mbar_wait(full + stage, phase, abort_flag)) break;
        if (!mbar_wait(tempty + acc, aphase ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t a0 = st_base + stage * C::kStageBytes;
        const uint32_t b0 = q_base + qs * C::kQBytes;
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_f8(tmem + acc * C::kN, smem_desc(a0 + kk * 32, 16, C::kSbo, C::kSwizzle),
                 smem_desc(b0 + kk * 32, 16, C::kSbo, C::kSwizzle), idesc, kk > 0 ? 1u : 0u);
        issued_mma = true;
        mma_commit(empty + stage);
        mma_commit(tfull + acc);
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        if (++acc == 2) { acc = 0; aphase ^= 1; }
      }
    } else if (warp >= 2) {
      // ----------------------------------------------------------- epilogue
      const int quad = warp & 3;          // tensor-memory lane quadrant
      int acc = 0, qn = 0;
      uint32_t aphase = 0;
      MqGroup g = mq_group(p, gcur, G);
      int vis[G];
      for (int t = t_begin; t < t_end; ++t) {
        const bool fresh = advance(t) || t == t_begin;
        if (fresh) {
          g = mq_group(p, gcur, G);
#pragma unroll
          for (int q = 0; q < G; ++q) {
            vis[q] = 0;
            if (q < g.gsz) row_tiles(p, g.bi * p.tq + g.t0 + q, vis[q]);
          }
          ++qn;
        }
        const float* wq = wbuf + ((qn - 1) & 1) * C::kN;
        if (!mbar_wait(tfull + acc, aphase, abort_flag)) break;
        tc_fence_after();
        const int j = t - s_pre[gcur];
        const int local = 32 * quad + lane;
        const int pos = j * 128 + local;
        for (int q = 0; q < g.gsz; ++q) {
          uint32_t r[HP];
#pragma unroll
          for (int c = 0; c < HP; c += 16) {
            uint32_t (&rr)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[c]);
            tmem_ld16(tmem + acc * C::kN + q * HP + c + ((uint32_t)(32 * quad) << 16), rr);
          }
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < HP; c += 16) reg_fence(*reinterpret_cast<uint32_t(*)[16]>(&r[c]));
          float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int h = 0; h < HP; h += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wq + q * p.hi + h);
            fma2_relu(s4[0], s4[1], w4.x, w4.y, __uint_as_float(r[h]), __uint_as_float(r[h + 1]));
            fma2_relu(s4[2], s4[3], w4.z, w4.w, __uint_as_float(r[h + 2]),
                      __uint_as_float(r[h + 3]));
          }
          const float sc = (s4[0] + s4[1]) + (s4[2] + s4[3]);
          const int64_t orow = (int64_t)g.bi * p.tq + g.t0 + q;
          const bool valid = pos < vis[q];
          if (valid) p.scores[orow * p.score_stride + pos] = sc;
          float m = valid ? sc : -INFINITY;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((lane & 7) == 0 && valid) p.blockmax[orow * p.bm_stride + pos / kBlock] = m;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty + acc);
        if (++acc == 2) { acc = 0; aphase ^= 1; }
      }
    }
  }
  __syncwarp();
  if (warp == 1) {
    if (lane == 0 && issued_mma) {
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, CSA2_DEV_TIMEOUT);
}

// Host side ---------------------------------------------------------------
cudaError_t set_wait_limit_indexer(unsigned long long ns) { return set_wait_limit_here(ns); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D byte tensor [rows, width] with a row stride, box [box_rows, width].
static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int width, int64_t stride,
                     int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)stride};
  cuuint32_t box[2] = {(cuuint32_t)width, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMapSwizzle sw = width == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : width == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                        : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Packed E2M1 rows of 128 channels (64 bytes) [rows, 128] with a row stride,
// expanded on the way into shared memory to 128-byte rows (16 codes, then 8
// bytes of gap), box [box_rows, 128 codes], 128-byte swizzle.  The mbarrier
// transaction count of one box is its global bytes: 64 per row.
static bool make_map_e2m1(CUtensorMap* m, const void* base, int64_t rows, int64_t stride,
                          int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)stride};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int HP, int DI, bool MX>
static cudaError_t run_indexer(const CUtensorMap& tk, const CUtensorMap& tq, const IndexerParams& p,
                               int num_sms, cudaStream_t s) {
  using C = IdxCfg<HP, DI, MX>;
  auto kern = indexer_kernel<HP, DI, MX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e == cudaSuccess) e = prefer_max_shared(kern);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(kIdxCtasPerSm * num_sms), 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = (size_t)C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  record_launch_begin(CSA2_KERNEL_INDEXER, s);
  e = cudaLaunchKernelEx(&cfg, kern, tk, tq, p);
  record_launch_end(CSA2_KERNEL_INDEXER, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int HP, int DI>
static cudaError_t run_indexer_mq(const CUtensorMap& tk, const CUtensorMap& tq,
                                  const IndexerParams& p, int n_groups, int num_sms,
                                  cudaStream_t s) {
  using C = MqCfg<HP, DI>;
  auto kern = indexer_mq_kernel<HP, DI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e == cudaSuccess) e = prefer_max_shared(kern);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(kIdxCtasPerSm * num_sms), 1, 1);
  cfg.blockDim = dim3(kMqThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  record_launch_begin(CSA2_KERNEL_INDEXER, s);
  e = cudaLaunchKernelEx(&cfg, kern, tk, tq, p, n_groups);
  record_launch_end(CSA2_KERNEL_INDEXER, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_indexer(const csa2_cache& c, const RowSet& rows, int mode, const uint8_t* q_idx,
                           const float* w, int32_t hi, const int32_t* pool_blocks,
                           const int32_t* pool_cnt, const WsLayout& L, uint8_t* ws, int num_sms,
                           cudaStream_t s) {
  IndexerParams p;
  p.mode = mode;
  p.n_rows = rows.n_rows;
  p.tq = rows.tq;
  p.hi = hi;
  p.batch = c.batch;
  p.batch_ids = rows.batch_ids;
  p.q_pos = rows.q_pos;
  p.seq_len = c.seq_len;
  p.pool_blocks = pool_blocks;
  p.pool_cnt = pool_cnt;
  p.w = w;
  p.map = row_map_of(c);
  p.row_len = reinterpret_cast<int32_t*>(ws + L.row_len);
  p.tile_prefix = reinterpret_cast<int32_t*>(ws + L.tile_prefix);
  p.scores = reinterpret_cast<float*>(ws + L.scores);
  p.score_stride = L.score_stride;
  p.blockmax = reinterpret_cast<float*>(ws + L.blockmax);
  p.bm_stride = L.bm_stride;
  p.cand = reinterpret_cast<float*>(ws + L.cand);
  p.status = reinterpret_cast<uint32_t*>(ws + L.status);
  if (rows.n_rows <= 0) return cudaSuccess;

  const int di = c.idx_dim;
  int64_t phys_rows;
  int box_rows;
  if (mode == 1) {
    box_rows = kBlock;
  } else if (c.page_size == 0) {
    box_rows = 128;
  } else {
    box_rows = c.page_size < 128 ? c.page_size : 128;
  }
  p.rows_per_load = box_rows;
  phys_rows = c.page_size == 0 ? (int64_t)c.batch * c.max_len : (int64_t)c.num_pages * c.page_size;
  p.phys_rows = phys_rows;
  const bool mx = c.idx_format == CSA2_IDX_MXFP4;
  p.idx_scales = mx ? c.idx_scales : nullptr;
  CUtensorMap tk, tq;
  if (mx ? !make_map_e2m1(&tk, c.idx_k, phys_rows, c.idxk_stride, box_rows)
         : !make_map(&tk, c.idx_k, phys_rows, di, c.idxk_stride, box_rows))
    return cudaErrorInvalidValue;
  const int64_t q_rows = (int64_t)c.batch * rows.tq * hi;
  if (!make_map(&tq, q_idx, q_rows, di, di, hi)) return cudaErrorInvalidValue;

  if (rows.n_rows > kInlinePlanRows) {
    prefer_max_shared(indexer_plan_kernel);
    indexer_plan_kernel<<<1, 1024, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  const int hp = hi <= 16 ? 16 : (hi <= 32 ? 32 : 64);
  if (mx) {  // MXFP4 keys: di = 128 (checked with the cache description)
    if (di != 128) return cudaErrorInvalidValue;
    if (hp == 16) return run_indexer<16, 128, true>(tk, tq, p, num_sms, s);
    if (hp == 32) return run_indexer<32, 128, true>(tk, tq, p, num_sms, s);
    return run_indexer<64, 128, true>(tk, tq, p, num_sms, s);
  }
  // several query rows per sequence in a Full layer: the multi-query kernel
  // (keys read once per group of 128/HP query rows), when its plan fits
  if (mode == 0 && rows.tq > 1 && hi % 4 == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0) {
    const int G = 128 / hp;
    const int64_t n_groups = (int64_t)(rows.n_rows / rows.tq) * ((rows.tq + G - 1) / G);
    if (n_groups <= kInlinePlanRows) {
#define CSA2_MQ_CASE(HPV, DIV) \
  if (hp == HPV && di == DIV) return run_indexer_mq<HPV, DIV>(tk, tq, p, (int)n_groups, num_sms, s);
      CSA2_MQ_CASE(16, 32) CSA2_MQ_CASE(16, 64) CSA2_MQ_CASE(16, 128)
      CSA2_MQ_CASE(32, 32) CSA2_MQ_CASE(32, 64) CSA2_MQ_CASE(32, 128)
      CSA2_MQ_CASE(64, 32) CSA2_MQ_CASE(64, 64) CSA2_MQ_CASE(64, 128)
#undef CSA2_MQ_CASE
    }
  }
#define CSA2_IDX_CASE(HPV, DIV) \
  if (hp == HPV && di == DIV) return run_indexer<HPV, DIV, false>(tk, tq, p, num_sms, s);
  CSA2_IDX_CASE(16, 32) CSA2_IDX_CASE(16, 64) CSA2_IDX_CASE(16, 128)
  CSA2_IDX_CASE(32, 32) CSA2_IDX_CASE(32, 64) CSA2_IDX_CASE(32, 128)
  CSA2_IDX_CASE(64, 32) CSA2_IDX_CASE(64, 64) CSA2_IDX_CASE(64, 128)
#undef CSA2_IDX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace csa2
