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
// (split-K over chunks; attn_combine_kernel merges the partial results).
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
  static constexpr int kSmem = kMiscOff + 1024;
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
  float* part_o;
  float* part_ml;
  int32_t splits;
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
  float* lrow = alpha + 64;                                      // [64]  (ends at misc + 896)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_status(p.status, CSA2_DEV_BAD_ALIGN);
    return;
  }
  const int row = blockIdx.y, split = blockIdx.x;
  const RowKeys rk = row_keys(p, row, D);
  const int nk = rk.n_global + rk.n_swa;
  const int nchunk = (nk + C::kKeys - 1) / C::kKeys;
  const int c0 = (int)((int64_t)nchunk * split / p.splits);
  const int c1 = (int)((int64_t)nchunk * (split + 1) / p.splits);
  const int nloc = c1 - c0;
  const bool direct = p.splits == 1;

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
    // the query rows [H, D] bf16 are contiguous: one bulk copy into X tile 1,
    // which holds no slab before the second chunk
    const uint32_t qbytes = (uint32_t)(p.heads * D * 2);
    mbar_arrive_expect_tx(q_full, qbytes);
    bulk_load(sx + C::kXBytes, p.q + (int64_t)row * p.heads * D, qbytes, q_full);
  }
  if (warp == 8) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + C::kSCols;

  if (warp >= 4 && warp < 8) {
    // =============================================================== data warps
    const int dt = tid - 128;     // 0..127
    const int quad = warp & 3;    // TMEM lane quadrant of this warp
    // ---- query: f16 copy of the bf16 rows.  When some |q| >= 2^14 the head
    // is scaled by a power of two so that its f16 copy stays exact.
    bool ok = mbar_wait(q_full, 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    {
      const uint8_t* qs = sx + C::kXBytes;
      constexpr int kChunks = D / 8;  // 16-byte chunks per head row
      bool big = false;
      for (int i = dt; i < p.heads * kChunks && ok; i += 128) {
        const uint4 v = *reinterpret_cast<const uint4*>(qs + i * 16);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          big |= ((w4[u] & 0x7F80u) >= (141u << 7)) | (((w4[u] >> 16) & 0x7F80u) >= (141u << 7));
      }
      if (!named_sync_or(4, 128, big)) {
        constexpr int kAll = 64 * kChunks;  // multiple of 4 * 128
        static_assert(kAll % 512 == 0, "query chunks");
        for (int i0 = dt; i0 < kAll; i0 += 512) {
          uint4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + 128 * u;
            v[u] = (ok && i / kChunks < p.heads) ? *reinterpret_cast<const uint4*>(qs + i * 16)
                                                 : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + 128 * u;
            const int h = i / kChunks, c = i - h * kChunks;
            const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              __half2 h2 = __floats2half2_rn(__uint_as_float(w4[q] << 16),
                                             __uint_as_float(w4[q] & 0xFFFF0000u));
              r[q] = *reinterpret_cast<uint32_t*>(&h2);
            }
            st_swz(sq + (c >> 3) * C::kSlab, h, c & 7, make_uint4(r[0], r[1], r[2], r[3]));
          }
        }
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

    // ---- gather / dequantise pipeline
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
    // ---- epilogue: O^T tiles, 32 channels per warp per tile
    const int slot = row * p.splits + split;
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
                p.part_o[((int64_t)slot * 64 + hh) * D + d] = acc;
              }
            }
          }
        }
      }
    }
  } else if (warp < 4) {
    // ============================================================ softmax warps
    // Row h of an M=64 accumulator sits in tensor-memory lane
    // 32 * (h / 16) + h % 16: warp q, lanes 0-15, hold heads 16 q .. 16 q + 15.
    const bool act = lane < 16;
    const int h = 16 * warp + (lane & 15);
    named_sync(1, 288);  // Q slabs written
    float m_h = -INFINITY, l_h = 0.0f;
    const float qm = qmul[h];
    bool ok = true;
    int n_resc = 0;
    for (int it = 0; it < nloc; ++it) {
      const int buf = it & 1;
      if (ok && !mbar_wait(s_full + buf, (it >> 1) & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      uint32_t sr[64];
      float mx = -INFINITY;
      if (ok) {
#pragma unroll
        for (int c = 0; c < 64; c += 16)
          tmem_ld16(tmem + 64 * buf + c + ((uint32_t)(32 * warp) << 16),
                    *reinterpret_cast<uint32_t(*)[16]>(&sr[c]));
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 64; c += 16) reg_fence(*reinterpret_cast<uint32_t(*)[16]>(&sr[c]));
        const uint64_t mask = act ? ((uint64_t)vmask[buf * 2] | ((uint64_t)vmask[buf * 2 + 1] << 32)) : 0ull;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float v = ((mask >> c) & 1) ? __uint_as_float(sr[c]) * qm : -INFINITY;
          sr[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      }
      tc_fence_before();
      // lazily raised running maximum: rescale only when it jumps by > 2^8
      bool need = false;
      float a = 1.0f;
      if (mx > -INFINITY && (m_h == -INFINITY || mx > m_h + 8.0f)) {
        need = true;
        a = (m_h == -INFINITY) ? 0.0f : fast_exp2(m_h - mx);
        m_h = mx;
        l_h *= a;
      }
      if (act) alpha[h] = a;
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
      if (ok && act) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float v0 = __uint_as_float(sr[8 * c + 2 * u]);
            const float v1 = __uint_as_float(sr[8 * c + 2 * u + 1]);
            const float e0 = v0 == -INFINITY ? 0.0f : fast_exp2(v0 - m_h);
            const float e1 = v1 == -INFINITY ? 0.0f : fast_exp2(v1 - m_h);
            __half2 h2 = __floats2half2_rn(e0, e1);
            const float2 back = __half22float2(h2);
            l_h += back.x + back.y;
            o[u] = *reinterpret_cast<uint32_t*>(&h2);
          }
          st_swz(sp, h, c, make_uint4(o[0], o[1], o[2], o[3]));
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_sync(3, 128);
      if (lane == 0) mbar_arrive(p_full);
    }
    if (act) {
      lrow[h] = l_h;
      if (!direct) {
        const int slot = row * p.splits + split;
        p.part_ml[((int64_t)slot * 64 + h) * 2 + 0] = (nloc > 0 && ok) ? m_h : -INFINITY;
        p.part_ml[((int64_t)slot * 64 + h) * 2 + 1] = (nloc > 0 && ok) ? l_h : 0.0f;
      }
    }
    named_sync(2, 288);
  } else {
    // ================================================================ MMA warp
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
      // Per chunk it: PV(it) once its softmax weights are written and QK(it+1)
      // once its X tile is dequantised, whichever is ready first.
      for (int it = 0; it < nloc && ok; ++it) {
        const int buf = it & 1;
        bool qk_done = it + 1 >= nloc, pv_done_issued = false;
        const uint64_t t0 = globaltimer();
        for (uint32_t spin = 0; !(qk_done && pv_done_issued); ++spin) {
          if (!pv_done_issued && mbar_try_wait(p_full, it & 1)) {
            tc_fence_after();
            issue_pv(it);
            pv_done_issued = true;
          } else if (!qk_done && mbar_try_wait(x_full + (buf ^ 1), ((it + 1) >> 1) & 1)) {
            tc_fence_after();
            issue_qk(it + 1);
            qk_done = true;
          } else if ((spin & 63) == 63 && (*abort_flag || globaltimer() - t0 > kWaitNs)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
        }
      }
      // let every issued MMA land before the tensor memory is freed
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never);
    }
    __syncwarp();
    named_sync(2, 288);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, C::kTmemCols);
  if (tid == 0 && *abort_flag) set_status(p.status, CSA2_DEV_TIMEOUT);
}

// Merge of split-K partials: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(192) attn_combine_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml,
                                                           float* __restrict__ out, int heads,
                                                           int D, int splits) {
  __shared__ float wgt[kMaxSplits];
  __shared__ float inv_den;
  const int row = blockIdx.x, h = blockIdx.y;
  if (threadIdx.x < 32) {
    const int s = threadIdx.x;
    float m = -INFINITY, l = 0.0f;
    if (s < splits) {
      const int64_t slot = (int64_t)row * splits + s;
      m = part_ml[(slot * 64 + h) * 2 + 0];
      l = part_ml[(slot * 64 + h) * 2 + 1];
    }
    float M = l > 0.0f ? m : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = (l > 0.0f) ? exp2f(m - M) : 0.0f;
    float den = w * l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (s < splits) wgt[s] = w;
    if (s == 0) inv_den = den > 0.0f ? 1.0f / den : 0.0f;
  }
  __syncthreads();
  const float id = inv_den;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float num = 0.0f;
    for (int s = 0; s < splits; ++s) {
      const float w = wgt[s];
      if (w != 0.0f) num += w * part_o[(((int64_t)row * splits + s) * 64 + h) * D + d];
    }
    out[((int64_t)row * heads + h) * D + d] = num * id;
  }
}

template <int NSLAB>
static cudaError_t run_attention(const AttnParams& p, cudaStream_t s) {
  using C = AttnCfg<NSLAB>;
  auto kern = attention_kernel<NSLAB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, p.n_rows);
  record_launch_begin(CSA2_KERNEL_ATTENTION, s);
  kern<<<grid, 288, C::kSmem, s>>>(p);
  record_launch_end(CSA2_KERNEL_ATTENTION, s);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  dim3 g2(p.n_rows, p.heads);
  attn_combine_kernel<<<g2, 192, 0, s>>>(p.part_o, p.part_ml, p.out, p.heads, C::D, p.splits);
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
  p.part_o = reinterpret_cast<float*>(ws + L.part_o);
  p.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
  int splits = num_sms / a.n_rows;
  splits = splits < 1 ? 1 : (splits > kMaxSplits ? kMaxSplits : splits);
  const int max_chunks = (a.kcap + a.window + 63) / 64;
  if (splits > max_chunks) splits = max_chunks < 1 ? 1 : max_chunks;
  if ((int64_t)splits * a.n_rows > L.slots) splits = 1;
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
