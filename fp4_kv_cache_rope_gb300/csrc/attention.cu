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
// One CTA handles a contiguous range of 64-key chunks of one query row
// (split-K over chunks).  The split CTAs of a row form one thread-block
// cluster: each stages its unnormalised output and its per-head running
// maximum and sum in shared memory, and after a cluster barrier every CTA
// merges a slice of the channels from all of them through distributed
// shared memory and writes the output.
// Nine warps, three roles:
//   data warps 4-7     gather each key's code and scale bytes (or window row)
//                      with plain vector loads one chunk ahead (index
//                      entries and page lookups two and three chunks ahead),
//                      dequantise into f16 slabs [64 keys x 64 channels]
//                      (128-byte rows, 128-byte swizzle; the X tile is double
//                      buffered), rescale the output accumulator when the
//                      running maximum jumps, and run the epilogue;
//   softmax warps 0-3  one thread per head (lanes 0-15 of each warp, the
//                      tensor-memory lanes an M=64 accumulator occupies):
//                      running maximum, rescale decision, softmax weights P
//                      (f16) for each chunk;
//   MMA warp 8         S[heads x keys] = Q . X^T (M=64, N=64, K=16), double
//                      buffered in tensor memory so that QK of chunk c+1 runs
//                      while chunk c's softmax does;  O^T[d x heads] +=
//                      X^T . P^T (M=128 channel tiles; A is the same slabs
//                      read channel-major, N = 64 heads).
#include "codec.cuh"
#include "launch.h"

namespace csa2 {

template <int NSLAB>
struct AttnCfg {
  static constexpr int D = NSLAB * 64;
  static constexpr int NT = (NSLAB + 1) / 2;     // O^T tiles of 128 channels
  static constexpr int kKeys = 64;
  static constexpr int kSlab = 64 * 128;         // one [64 x 64] f16 slab
  static constexpr int kXBytes = NSLAB * kSlab;  // one X tile (64 keys x D)
  static constexpr int kQOff = 0;
  static constexpr int kXOff = kXBytes;          // two X tiles follow Q
  static constexpr int kPOff = 3 * kXBytes;
  static constexpr int kMiscOff = kPOff + kSlab;
  static constexpr int kMiscBytes = 2048;
  static constexpr int kSmem = kMiscOff + kMiscBytes;
  static_assert(2 * kXBytes >= 64 * D * 4, "the X tiles hold the merge stage");
  static constexpr int kSCols = 2 * 64;          // two S buffers
  static constexpr int kCols = kSCols + 64 * NT;
  static constexpr int kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
  static constexpr int kPerThread = (NSLAB + 1) / 2;  // slabs per data thread
};

struct AttnParams {
  const uint16_t* q;
  int32_t heads, n_rows, tq, batch;
  const int32_t* q_pos;
  const int32_t* idx;
  const int32_t* cnt;
  int32_t kcap;
  const uint8_t* swa;
  const int32_t* swa_cnt;
  int32_t window;
  float scale_log2;  // softmax scale * log2(e)
  float* out;
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

__device__ __forceinline__ RowKeys row_keys(const AttnParams& p, int row, int D) {
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
    r.swa0 = p.swa + (int64_t)b * p.window * D;
  } else {
    // band row r holds position q_pos[b][0] - (W - 1) + r; query tq sees band
    // rows tq .. tq + W - 1 with a position >= 0
    const int p0 = p.q_pos[(int64_t)b * p.tq];
    int lo = (p.window - 1) - p0;
    lo = lo > tq ? lo : tq;
    const int hi = tq + p.window;  // exclusive
    r.n_swa = hi > lo ? hi - lo : 0;
    r.swa0 = p.swa + ((int64_t)b * (p.tq + p.window - 1) + lo) * D;
  }
  return r;
}

constexpr int kLrowOff = 128 + 2 * 64 * 4;  // lrow's byte offset in the misc area

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

// f16 copy of the query rows [heads x D] (bf16, at qs) into the swizzled Q
// slabs, by all 288 threads of the CTA (thread t of n), assuming no head needs
// scaling; returns, over the CTA, whether some |q| >= 2^14 (then the data
// warps redo the copy with a power-of-two scale per head).  Rows past `heads`
// are zero.
template <int NSLAB>
__device__ __forceinline__ bool convert_query(const uint8_t* qs, uint8_t* sq, int t, bool ok,
                                              int heads) {
  constexpr int D = NSLAB * 64;
  constexpr int kChunks = D / 8;     // 16-byte chunks per head row
  constexpr int kAll = 64 * kChunks;
  constexpr int kSlab = 64 * 128;
  constexpr int n = 288;
  bool big = false;
  for (int i0 = t; i0 < kAll; i0 += 4 * n) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + n * u;
      v[u] = (ok && i < kAll && i / kChunks < heads) ? *reinterpret_cast<const uint4*>(qs + i * 16)
                                                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
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
      *reinterpret_cast<uint4*>(sq + (c >> 3) * kSlab + h * 128 + (((c & 7) ^ (h & 7)) << 4)) =
          make_uint4(r[0], r[1], r[2], r[3]);
    }
  }
  return named_sync_or(4, 288, big);
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

// 4-byte store at byte `b` (a multiple of 4) of 16-byte column c of a
// swizzled slab row.
__device__ __forceinline__ void st_swz4(uint8_t* slab, int row, int c, int b, uint32_t v) {
  *reinterpret_cast<uint32_t*>(slab + row * 128 + ((c ^ (row & 7)) << 4) + b) = v;
}

// 16 tensor-memory lanes x 64 columns (16x256b shape, 8 repeats): thread t
// gets lanes t/4 (registers 4k, 4k+1) and t/4 + 8 (registers 4k+2, 4k+3),
// columns 8k + 2(t%4) and 8k + 2(t%4) + 1.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Where one key's bytes live: kind 0 = absent, 1 = FP4 cache row, 2 = FP8
// window row.
struct KeySrc {
  const uint8_t* a;  // codes row, or window row
  const uint8_t* s;  // scales row
  int kind;
};

// Raw bytes of one FP4 key for this thread's slabs: 32 code bytes and 4
// scale bytes per slab.  Window keys are read when they are dequantised.
template <int NP>
struct RawKey {
  uint4 c0[NP], c1[NP];
  uint32_t sc[NP];
};

// O^T *= alpha (per head column), all 128 lanes of the four data warps.
template <int NT>
__device__ __forceinline__ void rescale_output(uint32_t tO, int quad, const float* alpha) {
  tc_fence_after();
#pragma unroll 1
  for (int t = 0; t < NT; ++t) {
    const uint32_t base = tO + 64 * t + ((uint32_t)(32 * quad) << 16);
#pragma unroll
    for (int c = 0; c < 64; c += 16) {
      uint32_t v[16];
      tmem_ld16(base + c, v);
      tmem_ld_wait();
      reg_fence(v);
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) * alpha[c + u]);
      tmem_st16(base + c, v);
    }
  }
  tmem_st_wait();
  tc_fence_before();
}

// Split-K merge over the cluster of a query row:
//   o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s   per head,
// M the largest m_s with l_s > 0.  Every CTA has staged its unnormalised
// output [64][D] fp32 over its X tiles and its per-head (m, l); this CTA
// writes the channels [D*r/C, D*(r+1)/C) (in float4 columns).  Kept out of
// line so that nothing of it is live in the main loops.
template <int NSLAB>
__device__ __noinline__ void merge_splits(const AttnParams& p) {
  using C_ = AttnCfg<NSLAB>;
  constexpr int D = C_::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const float* st = reinterpret_cast<const float*>(smem + C_::kXOff);
  float* wgt = reinterpret_cast<float*>(smem + C_::kPOff);  // [kMaxSplits][64] merge weights
  float* inv_den = wgt + kMaxSplits * 64;                  // [64]
  const float* lrow = reinterpret_cast<const float*>(smem + C_::kMiscOff + kLrowOff);
  const float* mrow = lrow + 64;
  const int tid = threadIdx.x, row = blockIdx.y, r = blockIdx.x, C = p.splits;
  cluster_sync();  // every CTA's stage, mrow and lrow are written
  if (tid < 64) {
    float m[kMaxSplits], l[kMaxSplits];
    float M = -INFINITY;
#pragma unroll
    for (int u = 0; u < kMaxSplits; ++u) {
      m[u] = -INFINITY;
      l[u] = 0.0f;
      if (u < C) {
        m[u] = peer_f32(&mrow[tid], u);
        l[u] = peer_f32(&lrow[tid], u);
      }
    }
#pragma unroll
    for (int u = 0; u < kMaxSplits; ++u)
      if (l[u] > 0.0f) M = fmaxf(M, m[u]);
    float den = 0.0f;
#pragma unroll
    for (int u = 0; u < kMaxSplits; ++u) {
      const float w = l[u] > 0.0f ? exp2f(m[u] - M) : 0.0f;
      wgt[u * 64 + tid] = w;
      den += w * l[u];
    }
    inv_den[tid] = den > 0.0f ? 1.0f / den : 0.0f;
  }
  __syncthreads();
  constexpr int n4 = D / 4;
  const int q0 = n4 * r / C, q1 = n4 * (r + 1) / C, nq = q1 - q0;
  const int items = p.heads * nq;
  // four outputs per thread at a time, each reading the C stages: up to 16
  // remote float4 loads in flight
#pragma unroll 1
  for (int i0 = tid; i0 < items; i0 += 4 * blockDim.x) {
#pragma unroll 1
    for (int u0 = 0; u0 < C; u0 += 4) {
      float4 v[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = i0 + a * blockDim.x;
        const int hh = i / nq, d = 4 * (q0 + i - hh * nq);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i >= items || u0 + j >= C) continue;
          if (u0 + j == r)  // this CTA's own stage: a plain shared-memory load
            v[a][j] = *reinterpret_cast<const float4*>(st + hh * D + d);
          else
            v[a][j] = peer_f32x4(st + hh * D + d, u0 + j);
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = i0 + a * blockDim.x;
        if (i >= items) continue;
        const int hh = i / nq, d = 4 * (q0 + i - hh * nq);
        float4 num = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        float4* dst = reinterpret_cast<float4*>(p.out + ((int64_t)row * p.heads + hh) * D + d);
        if (u0 > 0) num = *dst;  // more than four splits: continue the sum
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (u0 + j < C) {
            const float w = wgt[(u0 + j) * 64 + hh];
            if (w != 0.0f) {
              num.x += w * v[a][j].x;
              num.y += w * v[a][j].y;
              num.z += w * v[a][j].z;
              num.w += w * v[a][j].w;
            }
          }
        }
        if (u0 + 4 >= C) {
          const float id = inv_den[hh];
          num = make_float4(num.x * id, num.y * id, num.z * id, num.w * id);
        }
        *dst = num;
      }
    }
  }
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

template <int NSLAB>
__global__ void __launch_bounds__(288, 1) attention_kernel(AttnParams p) {
  using C = AttnCfg<NSLAB>;
  constexpr int D = C::D;
  constexpr int NP = C::kPerThread;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sq = smem + C::kQOff;
  uint8_t* sx = smem + C::kXOff;  // X tile b at sx + b * kXBytes
  uint8_t* sp = smem + C::kPOff;
  uint8_t* misc = smem + C::kMiscOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint64_t* x_full = bars + 0;    // [2] data warps -> MMA issuer (4 arrivals)
  uint64_t* s_full = bars + 2;    // [2] QK of the chunk done
  uint64_t* pv_done = bars + 4;   // [2] PV of the chunk done (X tile and P free)
  uint64_t* dec = bars + 6;       // [2] softmax decision for the chunk (4 arrivals)
  uint64_t* resc = bars + 8;      // output rescale finished (4 arrivals)
  uint64_t* q_full = bars + 9;
  uint64_t* drain = bars + 10;
  uint64_t* p_full = bars + 11;   // softmax weights of the chunk written (4 arrivals)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 96);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 100);
  int* need_resc = reinterpret_cast<int*>(misc + 104);           // [2]
  uint32_t* vmask = reinterpret_cast<uint32_t*>(misc + 112);     // [2][2]
  float* qmul = reinterpret_cast<float*>(misc + 128);            // [64]
  float* alpha = qmul + 64;                                      // [64]
  float* lrow = alpha + 64;                                      // [64] at misc + kLrowOff
  float* mrow = lrow + 64;                                       // [64]  (ends at misc + 1152)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_status(p.status, CSA2_DEV_BAD_ALIGN);
    return;
  }
  const int row = blockIdx.y, split = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(x_full + i, 4);
      mbar_init(s_full + i, 1);
      mbar_init(pv_done + i, 1);
      mbar_init(dec + i, 4);
    }
    mbar_init(resc, 4);
    mbar_init(q_full, 1);
    mbar_init(drain, 1);
    mbar_init(p_full, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // everything read from here on may come from the previous kernels (the
  // selection, seq_len, and whatever wrote the query)
  griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) {
    // the query rows [H, D] bf16 are contiguous: one bulk copy into X tile 1,
    // which holds no slab before the second chunk
    const uint32_t qbytes = (uint32_t)(p.heads * D * 2);
    mbar_arrive_expect_tx(q_full, qbytes);
    bulk_load(sx + C::kXBytes, p.q + (int64_t)row * p.heads * D, qbytes, q_full);
  }
  const RowKeys rk = row_keys(p, row, D);
  const int nk = rk.n_global + rk.n_swa;
  const int nchunk = (nk + C::kKeys - 1) / C::kKeys;
  const int c0 = (int)((int64_t)nchunk * split / p.splits);
  const int c1 = (int)((int64_t)nchunk * (split + 1) / p.splits);
  const int nloc = c1 - c0;
  const bool direct = p.splits == 1;
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + C::kSCols;

  if (warp >= 4 && warp < 8) {
    // =============================================================== data warps
    const int dt = tid - 128;     // 0..127
    const int quad = warp & 3;    // TMEM lane quadrant of this warp
    // ---- gather / dequantise pipeline (its first index entries and rows are
    // requested before the query conversion, which hides their latency)
    const int j = dt & 63, sgrp = dt >> 6;
    auto resolve_pos = [&](int c) -> int {  // chunk-local c -> index entry (or -1)
      const int g = (c0 + c) * C::kKeys + j;
      return (c < nloc && g < rk.n_global) ? __ldg(p.idx + (int64_t)row * p.kcap + g) : -1;
    };
    auto resolve_src = [&](int c, int pos) -> KeySrc {
      KeySrc k{nullptr, nullptr, 0};
      if (c >= nloc) return k;
      const int g = (c0 + c) * C::kKeys + j;
      if (g < rk.n_global) {
        if (pos >= 0 && pos < rk.vis) {
          const int64_t r = p.map.row(rk.b, pos);
          if (r >= 0) {
            k.a = p.codes + r * p.code_stride;
            k.s = p.scales + r * p.scale_stride;
            k.kind = 1;
          } else if (sgrp == 0) {
            set_status(p.status, CSA2_DEV_BAD_PAGE);
          }
        } else if (sgrp == 0) {
          set_status(p.status, CSA2_DEV_BAD_INDEX);
        }
      } else if (g < nk) {
        k.a = rk.swa0 + (int64_t)(g - rk.n_global) * D;
        k.kind = 2;
      }
      return k;
    };
    auto load_raw = [&](const KeySrc& k, RawKey<NP>& raw) {
      if (k.kind == 1) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const int s = sgrp + 2 * i;
          if (s < NSLAB) {
            raw.c0[i] = __ldg(reinterpret_cast<const uint4*>(k.a + s * 32));
            raw.c1[i] = __ldg(reinterpret_cast<const uint4*>(k.a + s * 32 + 16));
            raw.sc[i] = __ldg(reinterpret_cast<const uint32_t*>(k.s + s * 4));
          }
        }
      }
    };
    // pipeline registers: raw bytes of chunk it+1, source of chunk it+2,
    // index entry of chunk it+3
    RawKey<NP> raw;
    KeySrc src_next = resolve_src(0, resolve_pos(0));
    load_raw(src_next, raw);
    KeySrc src_n1 = resolve_src(1, resolve_pos(1));
    int pos3 = resolve_pos(2);
    // ---- query: f16 copy of the bf16 rows, by all nine warps.  When some
    // |q| >= 2^14 the data warps redo it with each head scaled by a power of
    // two so that its f16 copy stays exact.
    bool ok = mbar_wait(q_full, 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    {
      const uint8_t* qs = sx + C::kXBytes;
      constexpr int kChunks = D / 8;  // 16-byte chunks per head row
      if (!convert_query<NSLAB>(qs, sq, tid, ok, p.heads)) {
        if (dt < 64) qmul[dt] = p.scale_log2;
      } else {
        constexpr int kPer = (kChunks + 31) / 32;
        for (int hh = 0; hh < 16; ++hh) {
          const int h = 16 * (warp - 4) + hh;
          uint4 v[kPer];
          float mx = 0.0f;
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int c = lane + 32 * i;
            v[i] = make_uint4(0, 0, 0, 0);
            if (ok && h < p.heads && c < kChunks)
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
          if (lane == 0) qmul[h] = p.scale_log2 * exp2f((float)e);
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
              st_swz(sq + (c >> 3) * C::kSlab, h, c & 7, make_uint4(o[0], o[1], o[2], o[3]));
            }
          }
        }
      }
    }
    fence_async_smem();
    named_sync(1, 288);  // Q slabs written; X tile 1 free again

    for (int it = 0; it < nloc; ++it) {
      const int buf = it & 1;
      const KeySrc src_cur = src_next;
      // X tile `buf` is free once PV of chunk it-2 has completed
      if (ok && it >= 2 && !mbar_wait(pv_done + buf, ((it - 2) >> 1) & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      uint8_t* tile = sx + buf * C::kXBytes;
      if (ok) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const int s = sgrp + 2 * i;
          if (s >= NSLAB) break;
          uint8_t* slab = tile + s * C::kSlab;
          if (src_cur.kind == 1) {
            const uint32_t cw[8] = {raw.c0[i].x, raw.c0[i].y, raw.c0[i].z, raw.c0[i].w,
                                    raw.c1[i].x, raw.c1[i].y, raw.c1[i].z, raw.c1[i].w};
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // 8 channels = 4 code bytes, group c/2
              const uint32_t sb = (raw.sc[i] >> (8 * (c >> 1))) & 0xFFu;
              const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
              const __half2 sh = *reinterpret_cast<const __half2*>(&s2);
              uint32_t o[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t v2 = e2m1x2_to_f16x2((cw[c] >> (8 * u)) & 0xFFu);
                __half2 r2 = __hmul2(*reinterpret_cast<const __half2*>(&v2), sh);
                o[u] = *reinterpret_cast<uint32_t*>(&r2);
              }
              st_swz(slab, j, c, make_uint4(o[0], o[1], o[2], o[3]));
            }
          } else if (src_cur.kind == 2) {
            const uint4* wr = reinterpret_cast<const uint4*>(src_cur.a + s * 64);
            uint4 w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) w[u] = __ldg(wr + u);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t lo = (c & 1) ? w[c >> 1].z : w[c >> 1].x;
              const uint32_t hi = (c & 1) ? w[c >> 1].w : w[c >> 1].y;
              st_swz(slab, j, c,
                     make_uint4(e4m3x2_to_f16x2(lo & 0xFFFFu), e4m3x2_to_f16x2(lo >> 16),
                                e4m3x2_to_f16x2(hi & 0xFFFFu), e4m3x2_to_f16x2(hi >> 16)));
            }
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) st_swz(slab, j, c, make_uint4(0, 0, 0, 0));
          }
        }
      }
      if (sgrp == 0) {  // warps 4 and 5 hold keys 0-31 and 32-63
        const uint32_t bal = __ballot_sync(0xffffffffu, src_cur.kind != 0);
        if (lane == 0) vmask[buf * 2 + (warp & 1)] = bal;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(x_full + buf);
      // prefetch: raw bytes of chunk it+1, source of it+2, index entry of it+3
      src_next = src_n1;
      load_raw(src_next, raw);
      src_n1 = resolve_src(it + 2, pos3);
      pos3 = resolve_pos(it + 3);
      // decision of the softmax warps for chunk it-1; PV(it-2) is complete
      if (it >= 1) {
        const int pb = (it - 1) & 1;
        if (ok && !mbar_wait(dec + pb, ((it - 1) >> 1) & 1, abort_flag)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (ok && need_resc[pb]) {
          rescale_output<C::NT>(tO, quad, alpha);
          __syncwarp();
          if (lane == 0) mbar_arrive(resc);
        }
      }
    }
    if (nloc >= 1) {
      // decision of the last chunk (needs PV of the chunk before it)
      const int last = nloc - 1, pb = last & 1;
      if (ok && last >= 1 && !mbar_wait(pv_done + (pb ^ 1), ((last - 1) >> 1) & 1, abort_flag))
        ok = false;
      if (ok && !mbar_wait(dec + pb, (last >> 1) & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      if (ok && need_resc[pb]) {
        rescale_output<C::NT>(tO, quad, alpha);
        __syncwarp();
        if (lane == 0) mbar_arrive(resc);
      }
      if (ok && !mbar_wait(pv_done + pb, (last >> 1) & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
    }
    tc_fence_after();
    named_sync(2, 288);  // lrow written by the softmax warps
    // ---- epilogue: O^T tiles, 32 channels per warp per tile; with several
    // CTAs per row the unnormalised output goes to the stage [64][D] fp32
    // (the X tiles, free now) for the cluster merge
    float* stage = reinterpret_cast<float*>(sx);
#pragma unroll 1
    for (int t = 0; t < C::NT; ++t) {
      const int s0 = (2 * t + 1 < NSLAB) ? 2 * t : NSLAB - 2;
      const int local = 32 * quad + lane;
      const int d = s0 * 64 + local;
      const bool mine = !(t == C::NT - 1 && (NSLAB & 1) && local < 64);
#pragma unroll 1
      for (int c = 0; c < 64; c += 16) {
        uint32_t v[16];
        if (nloc > 0 && ok) {
          tmem_ld16(tO + 64 * t + c + ((uint32_t)(32 * quad) << 16), v);
          tmem_ld_wait();
          reg_fence(v);
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) v[u] = 0u;
        }
        if (mine) {
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int hh = c + u;
            if (hh < p.heads) {
              const float acc = __uint_as_float(v[u]);
              if (direct) {
                const float l = lrow[hh];
                p.out[((int64_t)row * p.heads + hh) * D + d] = l > 0.0f ? acc / l : 0.0f;
              } else {
                stage[hh * D + d] = acc;
              }
            }
          }
        }
      }
    }
  } else if (warp < 4) {
    // ============================================================ softmax warps
    // Row h of an M=64 accumulator sits in tensor-memory lane
    // 32 * (h / 16) + h % 16.  A 16x256b load gives thread t of warp q the
    // rows (heads) hA = 16 q + t / 4 and hB = hA + 8, columns (keys)
    // 8 k + 2 (t % 4) + {0, 1}: each head is spread over the four threads
    // t % 4 = 0..3, each holding 16 of its 64 keys.  Running maxima agree
    // over the four threads; the sums stay per thread until the end.
    const int hA = 16 * warp + (lane >> 2), hB = hA + 8;
    const int cq = 2 * (lane & 3);  // this thread's first key in each group of 8
    {  // a share of the query conversion
      const bool okq = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag));
      convert_query<NSLAB>(sx + C::kXBytes, sq, tid, okq, p.heads);
    }
    named_sync(1, 288);  // Q slabs written
    float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
    const float qmA = qmul[hA], qmB = qmul[hB];
    bool ok = true;
    int n_resc = 0;
    for (int it = 0; it < nloc; ++it) {
      const int buf = it & 1;
      if (ok && !mbar_wait(s_full + buf, (it >> 1) & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      uint32_t sr[32];
      float mxA = -INFINITY, mxB = -INFINITY;
      if (ok) {
        tmem_ld_16x256b_x8(tmem + 64 * buf + ((uint32_t)(32 * warp) << 16), sr);
        tmem_ld_wait();
        reg_fence(*reinterpret_cast<uint32_t(*)[16]>(&sr[0]));
        reg_fence(*reinterpret_cast<uint32_t(*)[16]>(&sr[16]));
        const uint64_t mask = (uint64_t)vmask[buf * 2] | ((uint64_t)vmask[buf * 2 + 1] << 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool valid = (mask >> (8 * k + cq + e)) & 1;
            const float vA = valid ? __uint_as_float(sr[4 * k + e]) * qmA : -INFINITY;
            const float vB = valid ? __uint_as_float(sr[4 * k + 2 + e]) * qmB : -INFINITY;
            sr[4 * k + e] = __float_as_uint(vA);
            sr[4 * k + 2 + e] = __float_as_uint(vB);
            mxA = fmaxf(mxA, vA);
            mxB = fmaxf(mxB, vB);
          }
        }
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
      }
      tc_fence_before();
      // lazily raised running maximum: rescale only when it jumps by > 2^8
      bool need = false;
      float aA = 1.0f, aB = 1.0f;
      if (mxA > -INFINITY && (mA == -INFINITY || mxA > mA + 8.0f)) {
        need = true;
        aA = (mA == -INFINITY) ? 0.0f : fast_exp2(mA - mxA);
        mA = mxA;
        lA *= aA;
      }
      if (mxB > -INFINITY && (mB == -INFINITY || mxB > mB + 8.0f)) {
        need = true;
        aB = (mB == -INFINITY) ? 0.0f : fast_exp2(mB - mxB);
        mB = mxB;
        lB *= aB;
      }
      if ((lane & 3) == 0) {
        alpha[hA] = aA;
        alpha[hB] = aB;
      }
      const bool resc_needed = named_sync_or(3, 128, need) && it > 0;
      if (tid == 0) need_resc[buf] = resc_needed ? 1 : 0;
      named_sync(3, 128);
      if (lane == 0) mbar_arrive(dec + buf);
      // P and the accumulator are free once PV of chunk it-1 is done
      if (ok && it >= 1 && !mbar_wait(pv_done + (buf ^ 1), ((it - 1) >> 1) & 1, abort_flag))
        ok = false;
      if (resc_needed) {
        if (ok && !mbar_wait(resc, n_resc & 1, abort_flag)) ok = false;
        ++n_resc;
      }
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float vA0 = __uint_as_float(sr[4 * k]), vA1 = __uint_as_float(sr[4 * k + 1]);
          const float vB0 = __uint_as_float(sr[4 * k + 2]), vB1 = __uint_as_float(sr[4 * k + 3]);
          const float eA0 = vA0 == -INFINITY ? 0.0f : fast_exp2(vA0 - mA);
          const float eA1 = vA1 == -INFINITY ? 0.0f : fast_exp2(vA1 - mA);
          const float eB0 = vB0 == -INFINITY ? 0.0f : fast_exp2(vB0 - mB);
          const float eB1 = vB1 == -INFINITY ? 0.0f : fast_exp2(vB1 - mB);
          const __half2 pA = __floats2half2_rn(eA0, eA1), pB = __floats2half2_rn(eB0, eB1);
          const float2 bA = __half22float2(pA), bB = __half22float2(pB);
          lA += bA.x + bA.y;
          lB += bB.x + bB.y;
          st_swz4(sp, hA, k, 2 * cq, *reinterpret_cast<const uint32_t*>(&pA));
          st_swz4(sp, hB, k, 2 * cq, *reinterpret_cast<const uint32_t*>(&pB));
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_sync(3, 128);
      if (lane == 0) mbar_arrive(p_full);
    }
    // per-head sums over the four threads that hold the head
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    if ((lane & 3) == 0) {
      lrow[hA] = (nloc > 0 && ok) ? lA : 0.0f;
      mrow[hA] = (nloc > 0 && ok) ? mA : -INFINITY;
      lrow[hB] = (nloc > 0 && ok) ? lB : 0.0f;
      mrow[hB] = (nloc > 0 && ok) ? mB : -INFINITY;
    }
    named_sync(2, 288);
  } else {
    // ================================================================ MMA warp
    {  // a share of the query conversion
      const bool okq = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag));
      convert_query<NSLAB>(sx + C::kXBytes, sq, tid, okq, p.heads);
    }
    named_sync(1, 288);  // Q slabs written
    if (lane == 0 && nloc > 0) {
      constexpr uint32_t idesc_qk = instr_desc(0, 0, false, false, 64, 64);
      constexpr uint32_t idesc_pv = instr_desc(0, 0, true, false, 128, 64);
      const uint32_t q0 = smem_u32(sq), xb = smem_u32(sx), p0 = smem_u32(sp);
      auto issue_qk = [&](int c) {
        const uint32_t x0 = xb + (c & 1) * C::kXBytes;
        const uint32_t d = tmem + 64 * (c & 1);
#pragma unroll 1
        for (int s = 0; s < NSLAB; ++s) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(d, smem_desc(q0 + s * C::kSlab + kk * 32, 16, 1024, 2),
                    smem_desc(x0 + s * C::kSlab + kk * 32, 16, 1024, 2), idesc_qk,
                    (s | kk) != 0 ? 1u : 0u);
        }
        mma_commit(s_full + (c & 1));
      };
      bool ok = mbar_wait(x_full + 0, 0, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
      }
      auto issue_pv = [&](int c) {
        const uint32_t x0 = xb + (c & 1) * C::kXBytes;
#pragma unroll
        for (int t = 0; t < C::NT; ++t) {
          const int s0 = (2 * t + 1 < NSLAB) ? 2 * t : NSLAB - 2;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(tO + 64 * t, smem_desc(x0 + s0 * C::kSlab + kk * 2048, C::kSlab, 1024, 2),
                    smem_desc(p0 + kk * 32, 16, 1024, 2), idesc_pv, (c > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(pv_done + (c & 1));
      };
      // Whatever is ready, PV first: PV(c) once chunk c's softmax weights
      // are written, else the next QK once its X tile is dequantised.  QK can
      // run two chunks ahead of PV, which keeps the tensor pipe busy during
      // a chunk's softmax.  This is safe because X(q) is dequantised only
      // after PV(q-2) has completed, hence after the softmax has read S(q-2),
      // whose tensor-memory buffer QK(q) reuses.
      int next_qk = 1, next_pv = 0;
      const uint64_t t0 = globaltimer();
      for (uint32_t spin = 0; ok && next_pv < nloc; ++spin) {
        if (mbar_try_wait(p_full, next_pv & 1)) {
          tc_fence_after();
          issue_pv(next_pv);
          ++next_pv;
        } else if (next_qk < nloc &&
                   mbar_try_wait(x_full + (next_qk & 1), (next_qk >> 1) & 1)) {
          tc_fence_after();
          issue_qk(next_qk);
          ++next_qk;
        } else if ((spin & 63) == 63 && (*abort_flag || globaltimer() - t0 > g_wait_ns)) {
          *abort_flag = 1;
          ok = false;
        }
      }
      // let every issued MMA land before the tensor memory is freed
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
    named_sync(2, 288);
  }
  if (tid == 0) mbar_wait_drain(q_full, 0);  // the query copy, if a wait gave up early
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, C::kTmemCols);
  if (tid == 0 && *abort_flag) set_status(p.status, CSA2_DEV_TIMEOUT);
  if (p.splits > 1) merge_splits<NSLAB>(p);
}

cudaError_t set_wait_limit_attention(unsigned long long ns) { return set_wait_limit_here(ns); }

template <int NSLAB>
static cudaError_t run_attention(AttnParams p, cudaStream_t s) {
  using C = AttnCfg<NSLAB>;
  auto kern = attention_kernel<NSLAB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e == cudaSuccess) e = prefer_max_shared(kern);
  if (e != cudaSuccess) return e;
  // A CTA takes a whole SM and a cluster must fit inside one GPC, so not every
  // cluster count runs at once: take the largest split count whose clusters
  // all run in one wave (the splits of a row must also be co-resident).
  {
    static int fits[kMaxSplits + 1] = {};  // clusters of each size that run at once
    int splits = p.splits;
    while (splits > 1) {
      if (!fits[splits]) fits[splits] = max_active_clusters(kern, splits, 288, C::kSmem) + 1;
      if (fits[splits] - 1 >= p.n_rows) break;
      --splits;
    }
    p.splits = splits;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.splits, (unsigned)p.n_rows, 1);
  cfg.blockDim = dim3(288, 1, 1);
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
  AttnParams p;
  p.q = a.q;
  p.heads = a.heads;
  p.n_rows = a.n_rows;
  p.tq = a.tq;
  p.batch = c.batch;
  p.q_pos = a.q_pos;
  p.idx = a.idx;
  p.cnt = a.cnt;
  p.kcap = a.kcap;
  p.swa = a.swa;
  p.swa_cnt = a.swa_cnt;
  p.window = a.window;
  const float scale = a.scale > 0.0f ? a.scale : 1.0f / sqrtf((float)c.dim);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = a.out;
  int splits = num_sms / a.n_rows;
  splits = splits < 1 ? 1 : (splits > kMaxSplits ? kMaxSplits : splits);
  const int max_chunks = (a.kcap + a.window + 63) / 64;
  if (splits > max_chunks) splits = max_chunks < 1 ? 1 : max_chunks;
  p.splits = splits;
  p.codes = c.kv_codes;
  p.scales = c.kv_scales;
  p.code_stride = c.code_stride;
  p.scale_stride = c.scale_stride;
  p.seq_len = c.seq_len;
  p.map = RowMap{c.page_table, c.page_size, c.max_pages_per_seq, c.max_len, c.num_pages};
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
