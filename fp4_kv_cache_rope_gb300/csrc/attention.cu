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
// (split-K over chunks; partial results are merged by attn_combine_kernel).
// Warps:
//   4     producer: per chunk, cp.async.bulk gathers of each key's code row
//         (D/2 B) and scale row (D/16 B rounded up to 16), or of the window
//         row (D B), into a double-buffered raw stage;
//   0-3   dequantise the raw chunk into f16 slabs [64 keys x 64 channels]
//         (128-byte rows, 128-byte swizzle); softmax (warps 0-1, one thread
//         per head) with a lazily raised running maximum; rescale and
//         epilogue;
//   5     MMA issuer:  S[heads x keys]  = Q . X^T        (M=128, N=64, K=16,
//                      only the first 64 rows of M carry heads)
//                      O^T[d x heads] += X^T . P^T      (M=128 channel tiles,
//                      A is the same slabs read channel-major, N = 64 heads)
//         accumulators live in tensor memory: S in columns [0, 64), O^T tile
//         t in columns [64 + 64 t, 128 + 64 t).
#include "codec.cuh"
#include "launch.h"

namespace csa2 {

template <int NSLAB>
struct AttnCfg {
  static constexpr int D = NSLAB * 64;
  static constexpr int NT = (NSLAB + 1) / 2;     // O^T tiles of 128 channels
  static constexpr int kKeys = 64;
  static constexpr int kSlab = 64 * 128;         // one [64 x 64] f16 slab
  static constexpr int kQOff = 0;
  static constexpr int kXOff = NSLAB * kSlab;
  static constexpr int kPOff = 2 * NSLAB * kSlab;
  static constexpr int kRawStride = D + 16;      // bytes per key in a raw stage
  static constexpr int kRawOff = kPOff + kSlab;
  static constexpr int kRawBytes = kKeys * kRawStride;
  static constexpr int kMiscOff = kRawOff + 2 * kRawBytes;
  static constexpr int kSmem = kMiscOff + 1024;
  static constexpr int kCols = 64 + 64 * NT;
  static constexpr int kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
  static constexpr int kScaleBytes = ((D / 16) + 15) / 16 * 16;
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

// 16-byte store of f16x8 into row `row` (128-byte rows, 128-byte swizzle) of
// a slab at chunk position c (0..7).
__device__ __forceinline__ void st_swz(uint8_t* slab, int row, int c, uint4 v) {
  *reinterpret_cast<uint4*>(slab + row * 128 + ((c ^ (row & 7)) << 4)) = v;
}

template <int NSLAB>
__global__ void __launch_bounds__(192, 1) attention_kernel(AttnParams p) {
  using C = AttnCfg<NSLAB>;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sq = smem + C::kQOff;
  uint8_t* sx = smem + C::kXOff;
  uint8_t* sp = smem + C::kPOff;
  uint8_t* raw = smem + C::kRawOff;
  uint8_t* misc = smem + C::kMiscOff;
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(misc);       // [2]
  uint64_t* raw_empty = raw_full + 2;                           // [2]
  uint64_t* x_full = raw_full + 4;
  uint64_t* s_full = raw_full + 5;
  uint64_t* p_full = raw_full + 6;
  uint64_t* pv_done = raw_full + 7;
  uint64_t* drain = raw_full + 8;
  uint64_t* q_full = raw_full + 9;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 80);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 84);
  uint32_t* vmask = reinterpret_cast<uint32_t*>(misc + 88);     // [2]
  static_assert(10 * 8 <= 80, "barrier area");
  float* qmul = reinterpret_cast<float*>(misc + 128);            // [64]
  float* alpha = qmul + 64;                                      // [64]
  float* lrow = alpha + 64;                                      // [64] (ends at misc + 896)
  // key kinds (0 absent, 1 FP4 row, 2 FP8 window row) live in the 16 spare
  // bytes at offset D of each raw key slot
  auto kind_at = [&](int buf, int j) -> uint8_t& {
    return raw[buf * C::kRawBytes + j * C::kRawStride + D];
  };

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

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(raw_full + i, 1);
      mbar_init(raw_empty + i, 4);
    }
    mbar_init(x_full, 4);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    mbar_init(q_full, 1);
    *abort_flag = 0;
    fence_barrier_init();
    // the query rows [H, D] bf16 are contiguous: one bulk copy into the X
    // region, which holds no slab before the first chunk
    const uint32_t qbytes = (uint32_t)(p.heads * D * 2);
    mbar_arrive_expect_tx(q_full, qbytes);
    bulk_load(sx, p.q + (int64_t)row * p.heads * D, qbytes, q_full);
  }
  if (warp == 5) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool issued_mma = false;

  if (warp == 4) {
    // --------------------------------------------------------- producer
    for (int it = 0; it < nloc; ++it) {
      const int buf = it & 1;
      if (!mbar_wait(raw_empty + buf, ((it >> 1) & 1) ^ 1, abort_flag)) break;
      uint8_t* stage = raw + buf * C::kRawBytes;
      const uint8_t* src_a[2];
      const uint8_t* src_b[2];
      int kind[2];
      uint32_t bytes = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        const int g = (c0 + it) * C::kKeys + j;
        kind[h] = 0;
        if (g < rk.n_global) {
          const int pos = p.idx[(int64_t)row * p.kcap + g];
          if (pos >= 0 && pos < rk.vis) {
            const int64_t r = p.map.row(rk.b, pos);
            if (r >= 0) {
              kind[h] = 1;
              src_a[h] = p.codes + r * p.code_stride;
              src_b[h] = p.scales + r * p.scale_stride;
              bytes += D / 2 + C::kScaleBytes;
            } else {
              set_status(p.status, CSA2_DEV_BAD_PAGE);
            }
          } else {
            set_status(p.status, CSA2_DEV_BAD_INDEX);
          }
        } else if (g < nk) {
          kind[h] = 2;
          src_a[h] = rk.swa0 + (int64_t)(g - rk.n_global) * D;
          bytes += D;
        }
        kind_at(buf, j) = (uint8_t)kind[h];
      }
      bytes = __reduce_add_sync(0xffffffffu, bytes);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(raw_full + buf, bytes);
      __syncwarp();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint8_t* dst = stage + (lane + 32 * h) * C::kRawStride;
        if (kind[h] == 1) {
          bulk_load(dst, src_a[h], D / 2, raw_full + buf);
          bulk_load(dst + D / 2, src_b[h], C::kScaleBytes, raw_full + buf);
        } else if (kind[h] == 2) {
          bulk_load(dst, src_a[h], D, raw_full + buf);
        }
      }
    }
    // wind down: let copies still in flight land before the CTA exits
    if (*abort_flag && lane == 0) {
      volatile int never = 0;
      for (int i = 0; i < 2; ++i) mbar_wait(raw_full + i, 0, &never);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = instr_desc(0, 0, false, false, 128, 64);
      constexpr uint32_t idesc_pv = instr_desc(0, 0, true, false, 128, 64);
      const uint32_t q0 = smem_u32(sq), x0 = smem_u32(sx), p0 = smem_u32(sp);
      for (int it = 0; it < nloc; ++it) {
        if (!mbar_wait(x_full, it & 1, abort_flag)) break;
        tc_fence_after();
#pragma unroll 1
        for (int s = 0; s < NSLAB; ++s) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_f16(tmem, smem_desc(q0 + s * C::kSlab + kk * 32, 16, 1024, 2),
                    smem_desc(x0 + s * C::kSlab + kk * 32, 16, 1024, 2), idesc_qk,
                    (s | kk) != 0 ? 1u : 0u);
          }
        }
        issued_mma = true;
        mma_commit(s_full);
        if (!mbar_wait(p_full, it & 1, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < C::NT; ++t) {
          const int s0 = (2 * t + 1 < NSLAB) ? 2 * t : NSLAB - 2;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_f16(tmem + 64 + 64 * t,
                    smem_desc(x0 + s0 * C::kSlab + kk * 2048, C::kSlab, 1024, 2),
                    smem_desc(p0 + kk * 32, 16, 1024, 2), idesc_pv,
                    (it > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(pv_done);
      }
      if (issued_mma) {
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------- warps 0-3: compute threads
    // Query: per-head power-of-two scale so that the f16 copy is exact.
    // Warp w converts heads 16w .. 16w+15 from the bf16 rows staged in sx.
    bool ok = mbar_wait(q_full, 0, abort_flag);
    constexpr int kChunks = D / 8;                 // 16-byte chunks per head row
    constexpr int kPer = (kChunks + 31) / 32;
    for (int hh = 0; hh < 16; ++hh) {
      const int h = 16 * warp + hh;
      uint4 v[kPer];
      float mx = 0.0f;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int c = lane + 32 * i;
        v[i] = make_uint4(0, 0, 0, 0);
        if (ok && h < p.heads && c < kChunks)
          v[i] = *reinterpret_cast<const uint4*>(sx + (h * D + c * 8) * 2);
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
    fence_async_smem();
    named_sync(1, 128);

    const int h = tid;  // softmax head of warps 0-1
    float m_h = -INFINITY, l_h = 0.0f;
    const float qm = tid < 64 ? qmul[tid] : 0.0f;
    const int j = tid & 63;         // dequant key of this thread
    const int sgrp = tid >> 6;      // slabs sgrp, sgrp+2, ...
    // Every compute thread runs all nloc iterations and the same sequence of
    // named barriers; after a wait gives up (ok == false) the work is skipped.
    ok = __all_sync(0xffffffffu, ok);
    for (int it = 0; it < nloc; ++it) {
      const int buf = it & 1;
      if (ok && !mbar_wait(raw_full + buf, (it >> 1) & 1, abort_flag)) ok = false;
      if (ok && it > 0 && !mbar_wait(pv_done, (it - 1) & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      // ---- dequantise key j into slabs sgrp, sgrp + 2, ...
      const uint8_t* kr = raw + buf * C::kRawBytes + j * C::kRawStride;
      const int kind = ok ? kind_at(buf, j) : 0;
      for (int s = sgrp; s < NSLAB; s += 2) {
        uint8_t* slab = sx + s * C::kSlab;
        if (kind == 1) {
          const uint4 cw0 = *reinterpret_cast<const uint4*>(kr + s * 32);
          const uint4 cw1 = *reinterpret_cast<const uint4*>(kr + s * 32 + 16);
          const uint32_t scw = *reinterpret_cast<const uint32_t*>(kr + D / 2 + s * 4);
          const uint32_t cw[8] = {cw0.x, cw0.y, cw0.z, cw0.w, cw1.x, cw1.y, cw1.z, cw1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 8 channels = 4 code bytes, group c/2
            const uint32_t sb = (scw >> (8 * (c >> 1))) & 0xFFu;
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
        } else if (kind == 2) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint2 bw = *reinterpret_cast<const uint2*>(kr + s * 64 + c * 8);
            const uint32_t o0 = e4m3x2_to_f16x2(bw.x & 0xFFFFu);
            const uint32_t o1 = e4m3x2_to_f16x2(bw.x >> 16);
            const uint32_t o2 = e4m3x2_to_f16x2(bw.y & 0xFFFFu);
            const uint32_t o3 = e4m3x2_to_f16x2(bw.y >> 16);
            st_swz(slab, j, c, make_uint4(o0, o1, o2, o3));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) st_swz(slab, j, c, make_uint4(0, 0, 0, 0));
        }
      }
      if (tid < 64) {
        const uint32_t bal = __ballot_sync(0xffffffffu, kind != 0);
        if (lane == 0) vmask[warp] = bal;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(raw_empty + buf);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(x_full);

      // ---- softmax over this chunk (warps 0-1: thread = head)
      if (ok && !mbar_wait(s_full, it & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      named_sync(1, 128);  // vmask written by warps 0-1 is visible to all
      uint32_t sr[64];
      float mx = -INFINITY;
      uint64_t mask = 0;
      if (warp < 2 && ok) {
#pragma unroll
        for (int c = 0; c < 64; c += 16)
          tmem_ld16(tmem + c + ((uint32_t)(32 * warp) << 16), *reinterpret_cast<uint32_t(*)[16]>(&sr[c]));
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 64; c += 16) reg_fence(*reinterpret_cast<uint32_t(*)[16]>(&sr[c]));
        mask = (uint64_t)vmask[0] | ((uint64_t)vmask[1] << 32);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float v = ((mask >> c) & 1) ? __uint_as_float(sr[c]) * qm : -INFINITY;
          sr[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      }
      bool need = false;
      float a = 1.0f;
      if (warp < 2 && mx > -INFINITY && (m_h == -INFINITY || mx > m_h + 8.0f)) {
        need = true;
        a = (m_h == -INFINITY) ? 0.0f : exp2f(m_h - mx);
        m_h = mx;
        l_h *= a;
      }
      if (warp < 2) alpha[h] = a;
      const bool any = named_sync_or(1, 128, need);
      if (any && it > 0 && ok) {
        // rescale the running output O^T (all 128 lanes, 64 head columns per tile)
        float av[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) av[c] = alpha[c];
#pragma unroll 1
        for (int t = 0; t < C::NT; ++t) {
          const uint32_t base = tmem + 64 + 64 * t + ((uint32_t)(32 * warp) << 16);
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            uint32_t v[16];
            tmem_ld16(base + c, v);
            tmem_ld_wait();
            reg_fence(v);
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) * av[c + u]);
            tmem_st16(base + c, v);
          }
        }
        tmem_st_wait();
      }
      if (warp < 2 && ok) {
        uint8_t* prow = sp;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float v0 = __uint_as_float(sr[8 * c + 2 * u]);
            const float v1 = __uint_as_float(sr[8 * c + 2 * u + 1]);
            const float e0 = v0 == -INFINITY ? 0.0f : exp2f(v0 - m_h);
            const float e1 = v1 == -INFINITY ? 0.0f : exp2f(v1 - m_h);
            __half2 h2 = __floats2half2_rn(e0, e1);
            l_h += __low2float(h2) + __high2float(h2);
            o[u] = *reinterpret_cast<uint32_t*>(&h2);
          }
          st_swz(prow, h, c, make_uint4(o[0], o[1], o[2], o[3]));
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ---- epilogue
    if (ok && nloc > 0) ok = mbar_wait(pv_done, (nloc - 1) & 1, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (warp < 2) lrow[h] = l_h;
    named_sync(1, 128);
    const bool direct = p.splits == 1;
    const int slot = row * p.splits + split;
    if (warp < 2 && !direct) {
      p.part_ml[((int64_t)slot * 64 + h) * 2 + 0] = (nloc > 0 && ok) ? m_h : -INFINITY;
      p.part_ml[((int64_t)slot * 64 + h) * 2 + 1] = (nloc > 0 && ok) ? l_h : 0.0f;
    }
#pragma unroll 1
    for (int t = 0; t < C::NT; ++t) {
      const int s0 = (2 * t + 1 < NSLAB) ? 2 * t : NSLAB - 2;
      const int local = 32 * warp + lane;
      const int d = s0 * 64 + local;
      const bool mine = !(t == C::NT - 1 && (NSLAB & 1) && local < 64);
      uint32_t v[64];
      if (nloc > 0 && ok) {
#pragma unroll
        for (int c = 0; c < 64; c += 16)
          tmem_ld16(tmem + 64 + 64 * t + c + ((uint32_t)(32 * warp) << 16),
                    *reinterpret_cast<uint32_t(*)[16]>(&v[c]));
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 64; c += 16) reg_fence(*reinterpret_cast<uint32_t(*)[16]>(&v[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) v[c] = 0u;
      }
      if (mine) {
#pragma unroll
        for (int hh = 0; hh < 64; ++hh) {
          if (hh >= p.heads) break;
          const float acc = __uint_as_float(v[hh]);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, C::kTmemCols);
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
  kern<<<grid, 192, C::kSmem, s>>>(p);
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
