// Step 1 of the path: RoPE + FP4 (E2M1 x E4M3-per-16) quantisation + append,
// the indexer key (E4M3 per channel, or MXFP4: E2M1 with an E8M0 scale per 32
// channels), and the plain FP8 (E4M3) cast used for the SWA window and the
// indexer queries.
//
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" knowledge
// note, section "FP4 main KV: trade precision for bytes, not for a new GEMM":
// the main cache is quantised after RoPE to E2M1 values with one E4M3 scale
// per 16 channels and no second global scale; the SWA cache stays FP8.
// "Inside DeepSeek V4.1 Flash: CED, CSA2 and the 890-Byte KV Cache", section
// "Reconstructing the 890-byte cache budget": D/2 code bytes + D/16 scale
// bytes per entry.
//
// The unit of work is one group of 16 channels of one row: rotate the pairs
// that fall in the RoPE slice, take the group maximum, encode the scale and
// the 16 codes, store 8 code bytes and one scale byte.  Large appends stream
// their rows through shared memory with bulk copies issued several chunks
// ahead (quant_stream_kernel); small ones (decode) give each thread one group
// read straight from global memory.  The work is HBM bound: 3.5 KB read and
// 452 B written per D = 576 row with its indexer key.
#include "codec.cuh"
#include "launch.h"

namespace csa2 {

// Appends of at most this many 16-channel groups run as one cluster of up to
// 8 CTAs that also advances seq_len (decode steps: B x (D + di) / 16 groups).
constexpr int64_t kSmallAppendGroups = 8 * 512;

struct QuantParams {
  const float* kv;
  const float* z;       // pair compression: logits [B, 2T, D], else null
  const float* idx_in;
  uint8_t* codes;
  uint8_t* scales;
  uint8_t* idx_k;
  uint8_t* idx_scales;  // MXFP4 keys: 4 E8M0 bytes per row
  int32_t idx_mx;       // 1: MXFP4 indexer keys, 0: E4M3
  int64_t code_stride, scale_stride, idxk_stride;
  int32_t* seq_len;
  const float* rope_cos;
  const float* rope_sin;
  RowMap map;
  int32_t B, T, D, R, di;
  int32_t groups_main, groups_total;  // per row
  int32_t row0;                         // first row (b * T + i) of this launch
  uint32_t n_groups;                    // groups of this launch (< 2^31)
  uint32_t* status;
  // streaming kernel: rows of the launch and the shared-memory stage layout
  // (one slot per row: fp32 input row(s), indexer key row, cos row, sin row)
  int32_t n_rows;
  int32_t s_rows, s_stage_bytes, s_slot_bytes, s_slot_used, s_kv_bytes, s_idx_bytes;
  int32_t s_plain_groups;              // main groups before the first RoPE channel
  uint32_t s_inv_plain, s_inv_rope, s_inv_idx;  // ceil(2^20 / n): item -> row mapping
};

// ------------------------------------------------------ m = 2 compression
// An encoder entry combines two source positions with per-channel weights:
// the softmax of the two compression logits ("DeepSeek-V4.1-Flash" knowledge
// note, symbol table and "Causal Encoder-Decoder": Z_l is the weight used when
// forming a compressed global KV entry; "Inside DeepSeek V4.1 Flash", "CSA2:
// reuse memory and reuse selection independently": non-overlapping groups, no
// positional embedding).  Every step is one fp32 rounding, written out (no
// library exponential, no contraction), so the rows -- and the FP4 codes they
// decide -- are reproducible exactly: e^x for x <= 0 by Cody-Waite reduction
// with ln 2 split as 2839/4096 + remainder, then the degree-7 Taylor series.
constexpr float kInvLn2 = (float)(1.0 / 0.6931471805599453);
constexpr float kLn2Hi = (float)(2839.0 / 4096.0);
constexpr float kLn2Lo = (float)(0.6931471805599453 - 2839.0 / 4096.0);

__device__ __forceinline__ float exp_nonpos(float x) {
  if (x < -80.0f) return 0.0f;
  const float k = rintf(__fmul_rn(x, kInvLn2));
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(k, kLn2Hi)), __fmul_rn(k, kLn2Lo));
  float p = (float)(1.0 / 5040.0);
  p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 720.0));
  p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 120.0));
  p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 24.0));
  p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 6.0));
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  // times 2^k, exact: k >= -116 here, so the result stays a normal float
  return __fmul_rn(p, __int_as_float((127 + (int)k) << 23));
}

// c = w0 x0 + w1 x1 with (w0, w1) the softmax of (z0, z1).
__device__ __forceinline__ float combine_pair(float x0, float x1, float z0, float z1) {
  const float d = __fsub_rn(z1, z0);
  const float t = exp_nonpos(-fabsf(d));
  const float s = __fadd_rn(1.0f, t);
  const float big = __fdiv_rn(1.0f, s), small = __fdiv_rn(t, s);
  const float w0 = d >= 0.0f ? small : big;
  const float w1 = d >= 0.0f ? big : small;
  return __fadd_rn(__fmul_rn(w0, x0), __fmul_rn(w1, x1));
}

// ------------------------------------------------------------ group encoders
// Shared by both kernels below.  Source pointers are generic: rows in global
// memory (the per-thread kernel) or their staged copy in shared memory (the
// streaming kernel).

// MXFP4 indexer key, one 32-channel block: the E8M0 scale code is the OCP
// Microscaling shared exponent floor(log2 amax) - 2 (E2M1's top binade is
// 2^2), read off the fp32 exponent field of amax and clamped at code 0;
// codes = E2M1(x * 2^(127 - code)), an exact power-of-two scaling.
__device__ __noinline__ void encode_idx_mx(const QuantParams& p, const float* src, int gi,
                                           int64_t r) {
  float y[32];
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 f = s4[v];
    y[4 * v + 0] = f.x;
    y[4 * v + 1] = f.y;
    y[4 * v + 2] = f.z;
    y[4 * v + 3] = f.w;
  }
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(y[e]));
  const int bexp = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  const uint32_t code = bexp > 2 ? (uint32_t)(bexp - 2) : 0u;
  const float inv = __uint_as_float((254u - code) << 23);  // 2^(127 - code), a normal float
  uint32_t w[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint32_t x = 0;
#pragma unroll
    for (int e = 0; e < 8; e += 2)
      x |= e2m1x2_from_f32(__fmul_rn(y[8 * v + e], inv), __fmul_rn(y[8 * v + e + 1], inv))
           << (4 * e);
    w[v] = x;
  }
  *reinterpret_cast<uint4*>(p.idx_k + r * p.idxk_stride + 16 * gi) = make_uint4(w[0], w[1], w[2], w[3]);
  p.idx_scales[r * 4 + gi] = (uint8_t)code;
}

// Indexer key group gi (16 channels): plain E4M3 per element.
__device__ __forceinline__ void encode_idx_e4m3(const QuantParams& p, const float (&y)[16], int gi,
                                                int64_t r) {
  uint32_t w[4];
#pragma unroll
  for (int v = 0; v < 4; ++v)
    w[v] = e4m3x2_from_f32(y[4 * v], y[4 * v + 1]) |
           (e4m3x2_from_f32(y[4 * v + 2], y[4 * v + 3]) << 16);
  *reinterpret_cast<uint4*>(p.idx_k + r * p.idxk_stride + 16 * gi) =
      make_uint4(w[0], w[1], w[2], w[3]);
}

// Main-KV group g (16 channels, after the pair combination): RoPE on the
// interleaved pairs of the last R channels, with cs / sn the cos / sin row of
// the entry's position (R / 2 values each); then the E4M3 scale and the 16
// E2M1 codes.
__device__ __forceinline__ void encode_main(const QuantParams& p, float (&y)[16], int g,
                                            const float* cs, const float* sn, int64_t r) {
  // two fp32 products and one add/sub per rotated output, each rounded once
  // (no contraction into an FMA)
  const int c0 = 16 * g;
  const int rope0 = p.D - p.R;
  if (c0 + 16 > rope0) {
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int c = c0 + e;
      if (c >= rope0) {
        const int j = (c - rope0) >> 1;
        const float co = cs[j], si = sn[j];
        const float x0 = y[e], x1 = y[e + 1];
        y[e] = __fsub_rn(__fmul_rn(x0, co), __fmul_rn(x1, si));
        y[e + 1] = __fadd_rn(__fmul_rn(x0, si), __fmul_rn(x1, co));
      }
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(y[e]));
  // scale byte E4M3(fl(amax / 6)) and its exact value (through f16, which
  // holds every E4M3 value)
  const uint32_t sc = e4m3x2_from_f32(__fdiv_rn(amax, 6.0f), 0.0f) & 0xFFu;
  const float s = __half2float(__ushort_as_half((unsigned short)(e4m3x2_to_f16x2(sc) & 0xFFFFu)));
  uint32_t lo = 0, hi = 0;
  if (s != 0.0f) {
    // The code of each value is E2M1(fl(y / s)).  y * fl(1 / s), rounded,
    // is within 2.5 ulp of fl(y / s) (two roundings of 2^-24 relative each,
    // against half an ulp), so both give the same code unless an E2M1
    // rounding boundary (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5: at most three
    // significant bits, so their low 21 mantissa bits are zero) lies within
    // a few ulps of the product.  Such groups take the quotients themselves.
    // (The test also flags other values with few significant bits, zero
    // among them; those groups just take the slower exact path.  The sign
    // bit does not reach the low 21 bits, so it needs no masking.)
    const float inv = __frcp_rn(s);
    float q[16];
    uint32_t dist = 0xFFFFFFFFu;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      q[e] = __fmul_rn(y[e], inv);
      dist = min(dist, (__float_as_uint(q[e]) + 8u) & 0x1FFFFFu);
    }
    if (dist <= 16u) {
#pragma unroll
      for (int e = 0; e < 16; ++e) q[e] = __fdiv_rn(y[e], s);
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      lo |= e2m1x2_from_f32(q[e], q[e + 1]) << (4 * e);
      hi |= e2m1x2_from_f32(q[8 + e], q[9 + e]) << (4 * e);
    }
  }
  *reinterpret_cast<uint2*>(p.codes + r * p.code_stride + 8 * g) = make_uint2(lo, hi);
  p.scales[r * p.scale_stride + g] = (uint8_t)sc;
}

// 16 consecutive fp32 values.
__device__ __forceinline__ void load16(const float* src, float (&y)[16]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const float4 f = s4[v];
    y[4 * v + 0] = f.x;
    y[4 * v + 1] = f.y;
    y[4 * v + 2] = f.z;
    y[4 * v + 3] = f.w;
  }
}

// 16 channels of a compressed entry from the source rows x0, x1 and their
// logits z0, z1.
__device__ __forceinline__ void load16_pair(const float* x0, const float* x1, const float* z0,
                                            const float* z1, float (&y)[16]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const float4 a = reinterpret_cast<const float4*>(x0)[v];
    const float4 c = reinterpret_cast<const float4*>(x1)[v];
    const float4 u = reinterpret_cast<const float4*>(z0)[v];
    const float4 w = reinterpret_cast<const float4*>(z1)[v];
    y[4 * v + 0] = combine_pair(a.x, c.x, u.x, w.x);
    y[4 * v + 1] = combine_pair(a.y, c.y, u.y, w.y);
    y[4 * v + 2] = combine_pair(a.z, c.z, u.z, w.z);
    y[4 * v + 3] = combine_pair(a.w, c.w, u.w, w.w);
  }
}

// Destination row of launch row lrow (row row0 + lrow = b * T + i, entry i of
// sequence b, at position seq_len[b] + i), or -1 after recording why not.
__device__ __forceinline__ int64_t dest_row(const QuantParams& p, int32_t row32, int64_t* pos_out) {
  const int b = row32 / p.T;
  const int i = row32 - b * p.T;
  const int64_t pos = (int64_t)p.seq_len[b] + i;
  *pos_out = pos;
  if (pos >= p.map.max_len || pos < 0) {
    set_status(p.status, CSA2_DEV_OVERFLOW);
    return -1;
  }
  const int64_t r = p.map.row(b, pos);
  if (r < 0) set_status(p.status, CSA2_DEV_BAD_PAGE);
  return r;
}

// ------------------------------------------------------ per-thread kernel
// Quantises group gid of the launch (row row0 + gid / groups_total, group
// gid % groups_total) straight from global memory.  Rows (B * T) and a
// launch's groups fit in 31 bits, so the index arithmetic is 32-bit (a 64-bit
// division is a long software sequence on the GPU).  Used for the small
// appends and for inputs the streaming kernel cannot copy in bulk.
__device__ __forceinline__ void quant_group(const QuantParams& p, uint32_t gid) {
  const uint32_t lrow = gid / (uint32_t)p.groups_total;
  const int g = (int)(gid - lrow * (uint32_t)p.groups_total);
  const int32_t row32 = p.row0 + (int32_t)lrow;
  const int64_t row = row32;
  const bool is_idx = g >= p.groups_main;
  if (is_idx && p.idx_mx) {
    int64_t pos;
    const int64_t r = dest_row(p, row32, &pos);
    if (r >= 0) encode_idx_mx(p, p.idx_in + row * p.di + 32 * (g - p.groups_main),
                              g - p.groups_main, r);
    return;
  }
  // the input rows do not depend on the position: request them first
  float y[16];
  if (p.z && !is_idx) {  // entry i of sequence b from source rows 2i, 2i+1
    const int64_t r0 = row * 2 * p.D + 16 * g;
    load16_pair(p.kv + r0, p.kv + r0 + p.D, p.z + r0, p.z + r0 + p.D, y);
  } else {
    load16(is_idx ? p.idx_in + row * p.di + 16 * (g - p.groups_main) : p.kv + row * p.D + 16 * g,
           y);
  }
  int64_t pos;
  const int64_t r = dest_row(p, row32, &pos);
  if (r < 0) return;
  if (is_idx) {
    encode_idx_e4m3(p, y, g - p.groups_main, r);
    return;
  }
  const int half = p.R >> 1;
  encode_main(p, y, g, p.rope_cos + pos * half, p.rope_sin + pos * half, r);
}

__global__ void __launch_bounds__(256) quant_append_kernel(QuantParams p) {
  const uint32_t gid = blockIdx.x * blockDim.x + threadIdx.x;
  if (gid < p.n_groups) quant_group(p, gid);
}

// ------------------------------------------------------- streaming kernel
// Large appends.  A persistent CTA walks chunks of rps rows (chunk c,
// c + grid, ...) through a ring of kStreamStages shared-memory stages:
//
// * warp 16 (producer): per chunk, lane l bulk-copies row l's inputs (the
//   fp32 row -- or the two source rows and their logits -- and the indexer
//   key row) into slot l of the stage, resolves the row's destination
//   (seq_len, page table), records it, and copies the cos / sin rows of its
//   position; each lane arrives once on the stage's `full` barrier.
// * warps 0-15: wait for the stage, quantise its rows' groups from shared
//   memory with the encoders above (thread = group), and release the stage.
//
// The copies run up to kStreamStages - 1 chunks ahead of the arithmetic, so
// the HBM reads stay in flight while groups are encoded, and the dependent
// seq_len -> page-table lookups sit off the arithmetic's path.
constexpr int kStreamStages = 3;
constexpr int kStreamWarps = 16;
constexpr int kStreamThreads = 32 * (kStreamWarps + 1);
constexpr int kStreamStageBytes = 34 * 1024;   // 11 rows of D = 576 with their keys

__device__ __forceinline__ void stream_group(const QuantParams& p, const uint8_t* slot, int g,
                                             int64_t r) {
  const float* in = reinterpret_cast<const float*>(slot);
  const float* idx = reinterpret_cast<const float*>(slot + p.s_kv_bytes);
  if (g >= p.groups_main) {
    const int gi = g - p.groups_main;
    if (p.idx_mx) {
      encode_idx_mx(p, idx + 32 * gi, gi, r);
    } else {
      float y[16];
      load16(idx + 16 * gi, y);
      encode_idx_e4m3(p, y, gi, r);
    }
    return;
  }
  float y[16];
  if (p.z) {
    const int D = p.D;
    load16_pair(in + 16 * g, in + D + 16 * g, in + 2 * D + 16 * g, in + 3 * D + 16 * g, y);
  } else {
    load16(in + 16 * g, y);
  }
  const float* cs = reinterpret_cast<const float*>(slot + p.s_kv_bytes + p.s_idx_bytes);
  encode_main(p, y, g, cs, cs + (p.R >> 1), r);
}

__global__ void __launch_bounds__(kStreamThreads, 2) quant_stream_kernel(QuantParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rps = p.s_rows, stage_bytes = p.s_stage_bytes;
  int64_t* meta = reinterpret_cast<int64_t*>(smem + kStreamStages * stage_bytes);  // [S][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + kStreamStages * 32);
  uint64_t* empty = full + kStreamStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStreamStages);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreamStages; ++s) {
      mbar_init(full + s, 32);
      mbar_init(empty + s, kStreamWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  griddep_launch_dependents();   // the seq_len update may launch; it waits for this grid
  const int64_t nrows = p.n_rows;
  const int64_t nchunks = (nrows + rps - 1) / rps;

  if (warp == kStreamWarps) {
    int armed = 0;
    for (int j = 0;; ++j) {
      const int64_t c = blockIdx.x + (int64_t)j * gridDim.x;
      if (c >= nchunks) break;
      const int s = j % kStreamStages;
      bool ok = true;
      if (j >= kStreamStages)
        ok = mbar_wait(empty + s, (uint32_t)((j / kStreamStages - 1) & 1), abort_flag);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;   // all lanes arrive on `full`, or none
      // the input rows do not depend on the position: their copies go out
      // first, then the destination lookup and the cos / sin rows
      const int64_t lr = c * rps + lane;
      const bool have = lane < rps && lr < nrows;
      const int64_t row = p.row0 + lr;
      uint8_t* slot = smem + s * stage_bytes + lane * p.s_slot_bytes;
      const uint32_t kvb = (uint32_t)p.s_kv_bytes;
      if (have) {
        mbar_expect_tx(full + s, kvb + (uint32_t)p.s_idx_bytes);
        if (p.z) {
          bulk_load(slot, p.kv + row * 2 * p.D, kvb / 2, full + s);
          bulk_load(slot + kvb / 2, p.z + row * 2 * p.D, kvb / 2, full + s);
        } else {
          bulk_load(slot, p.kv + row * p.D, kvb, full + s);
        }
        if (p.s_idx_bytes)
          bulk_load(slot + kvb, p.idx_in + row * p.di, (uint32_t)p.s_idx_bytes, full + s);
      }
      // seq_len and the page table may still be written by the previous
      // kernel (an earlier append's seq_len update): wait for it once
      if (j == 0) griddep_wait();
      int64_t r = -1, pos = 0;
      if (have) r = dest_row(p, (int32_t)row, &pos);
      const int half = p.R >> 1;
      const uint32_t hb = (uint32_t)half * 4u;
      const uint32_t rope_bytes = r >= 0 && half > 0 ? 2u * hb : 0u;
      if (lane < rps) meta[s * 32 + lane] = r;
      mbar_arrive_expect_tx(full + s, rope_bytes);   // this lane's one arrival
      if (rope_bytes) {
        uint8_t* rs = slot + kvb + p.s_idx_bytes;
        bulk_load(rs, p.rope_cos + pos * half, hb, full + s);
        bulk_load(rs + hb, p.rope_sin + pos * half, hb, full + s);
      }
      ++armed;
    }
    // every armed stage has landed before the CTA may exit
    drain_armed(full, kStreamStages, armed);
    return;
  }

  const int gm = p.groups_main, gx = p.groups_total - p.groups_main;
  const int gp = p.s_plain_groups, gr = gm - gp;   // groups without / with RoPE channels
  for (int j = 0;; ++j) {
    const int64_t c = blockIdx.x + (int64_t)j * gridDim.x;
    if (c >= nchunks) break;
    const int s = j % kStreamStages;
    if (!mbar_wait(full + s, (uint32_t)((j / kStreamStages) & 1), abort_flag)) break;
    const int rows_here = (int)(nrows - c * rps < rps ? nrows - c * rps : rps);
    // the plain main groups of every row, then the groups that hold RoPE
    // channels, then the indexer-key groups, so that a warp's lanes mostly
    // run the same code
    const int plain_items = rows_here * gp;
    const int main_items = plain_items + rows_here * gr;
    const int items = main_items + rows_here * gx;
    const uint8_t* stage = smem + s * stage_bytes;
    for (int it = threadIdx.x; it < items; it += kStreamWarps * 32) {
      // k / n (n = gp, gr or gx) as a product: the launcher keeps items * n
      // below 2^20, so floor(k * ceil(2^20 / n) / 2^20) = floor(k / n) (the
      // rounding-up error, below k / 2^20, stays below 1 / n)
      int l, g;
      if (it < plain_items) {
        l = (int)(((uint32_t)it * p.s_inv_plain) >> 20);
        g = it - l * gp;
      } else if (it < main_items) {
        const int k = it - plain_items;
        l = (int)(((uint32_t)k * p.s_inv_rope) >> 20);
        g = gp + k - l * gr;
      } else {
        const int k = it - main_items;
        l = (int)(((uint32_t)k * p.s_inv_idx) >> 20);
        g = gm + k - l * gx;
      }
      const int64_t r = meta[s * 32 + l];
      if (r >= 0) stream_group(p, stage + l * p.s_slot_bytes, g, r);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, CSA2_DEV_TIMEOUT);
}

// Small appends (decode): one thread-block cluster of up to 8 CTAs does every
// group; after a cluster barrier (every read of seq_len precedes it) CTA 0
// advances seq_len, so no second launch is needed.
//
// The groups are quantised and stored before the dependency wait, so that
// they overlap the previous kernel's tail (on the SMs it leaves free): the
// new rows go to positions >= seq_len, which no kernel of the path reads
// before they are appended, and seq_len itself is written only by appends.
// Only the seq_len update waits, because the previous kernel may still read
// seq_len.  The inputs are the caller's (see csa2_quant_append).
__global__ void __launch_bounds__(512) quant_append_cluster_kernel(QuantParams p) {
  const uint32_t gid = blockIdx.x * blockDim.x + threadIdx.x;
  if (gid < p.n_groups) quant_group(p, gid);
  griddep_wait();
  griddep_launch_dependents();
  cluster_sync();
  if (blockIdx.x == 0) {
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      const int64_t n = (int64_t)p.seq_len[b] + p.T;
      p.seq_len[b] = (int32_t)(n > p.map.max_len ? p.map.max_len : n);
    }
  }
}

__global__ void advance_len_kernel(int32_t* seq_len, int32_t B, int32_t T, int32_t max_len) {
  griddep_wait();   // every read of seq_len by the append grid is done
  griddep_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int64_t n = (int64_t)seq_len[b] + T;
    seq_len[b] = (int32_t)(n > max_len ? max_len : n);
  }
}

__global__ void __launch_bounds__(256) fp8_quant_kernel(const float* __restrict__ x, int64_t n,
                                                        uint8_t* __restrict__ out) {
  const int64_t i4 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i4 + 3 < n && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
      ((reinterpret_cast<uintptr_t>(out) & 3) == 0)) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(x + i4));
    *reinterpret_cast<uint32_t*>(out + i4) = e4m3_encode(f.x) | (e4m3_encode(f.y) << 8) |
                                              (e4m3_encode(f.z) << 16) |
                                              (e4m3_encode(f.w) << 24);
  } else {
    for (int64_t i = i4; i < n && i < i4 + 4; ++i) out[i] = (uint8_t)e4m3_encode(x[i]);
  }
}

cudaError_t launch_fp8_quant(const float* x, int64_t n, uint8_t* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t threads = (n + 3) / 4;
  const int64_t blocks = (threads + 255) / 256;
  fp8_quant_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, n, out);
  return cudaGetLastError();
}

cudaError_t launch_quant_append(const csa2_cache& c, const float* kv, const float* z,
                                const float* idx_in, int32_t T, uint32_t* status, int num_sms,
                                cudaStream_t s) {
  QuantParams p;
  p.kv = kv;
  p.z = z;
  p.idx_in = idx_in;
  p.codes = c.kv_codes;
  p.scales = c.kv_scales;
  p.idx_k = c.idx_k;
  p.idx_scales = c.idx_scales;
  p.idx_mx = c.idx_format == CSA2_IDX_MXFP4 ? 1 : 0;
  p.code_stride = c.code_stride;
  p.scale_stride = c.scale_stride;
  p.idxk_stride = c.idxk_stride;
  p.seq_len = c.seq_len;
  p.rope_cos = c.rope_cos;
  p.rope_sin = c.rope_sin;
  p.map = row_map_of(c);
  p.B = c.batch;
  p.T = T;
  p.D = c.dim;
  p.R = c.rope_dim;
  p.di = c.idx_dim;
  p.groups_main = c.dim / kGroup;
  p.groups_total = p.groups_main + (idx_in ? c.idx_dim / (p.idx_mx ? 32 : 16) : 0);
  p.status = status;
  p.row0 = 0;
  const int64_t total = (int64_t)c.batch * T * p.groups_total;
  if ((int64_t)c.batch * T > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  if (total <= kSmallAppendGroups) {
    p.n_groups = (uint32_t)total;
    const int ctas = (int)((total + 511) / 512);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(512, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = prefer_max_shared(quant_append_cluster_kernel);
    if (e != cudaSuccess) return e;
    record_launch_begin(CSA2_KERNEL_QUANT, s);
    e = cudaLaunchKernelEx(&cfg, quant_append_cluster_kernel, p);
    record_launch_end(CSA2_KERNEL_QUANT, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  prefer_max_shared(advance_len_kernel);
  const int64_t rows = (int64_t)c.batch * T;
  // the streaming kernel bulk-copies whole rows: every source row and the
  // cos / sin rows must start on 16 bytes and span a multiple of 16 bytes
  // (kv, z and the indexer rows are 16-byte aligned, D and di multiples of 16)
  const int half = p.R >> 1;
  bool stream = p.R == 0 || ((half % 4) == 0 && (reinterpret_cast<uintptr_t>(p.rope_cos) & 15) == 0 &&
                             (reinterpret_cast<uintptr_t>(p.rope_sin) & 15) == 0);
  if (stream) {
    p.s_kv_bytes = (z ? 4 : 1) * p.D * 4;
    p.s_idx_bytes = idx_in ? p.di * 4 : 0;
    p.s_slot_used = p.s_kv_bytes + p.s_idx_bytes + 2 * half * 4;
    p.s_slot_bytes = (p.s_slot_used + 15) & ~15;
    // rows per chunk: as many as a stage holds, but few enough that every
    // CTA of a full wave gets about three chunks (so short appends pipeline)
    const int64_t wave = (int64_t)num_sms * 2;
    int64_t rps = kStreamStageBytes / p.s_slot_bytes;
    const int64_t spread = (rows + 3 * wave - 1) / (3 * wave);
    if (spread < rps) rps = spread;
    rps = rps < 1 ? 1 : (rps > 32 ? 32 : rps);
    auto inv20 = [](uint32_t n) { return n ? ((1u << 20) + n - 1) / n : 0u; };
    p.s_plain_groups = (p.D - p.R) / kGroup;
    const uint32_t gx = (uint32_t)(p.groups_total - p.groups_main);
    p.s_inv_plain = inv20((uint32_t)p.s_plain_groups);
    p.s_inv_rope = inv20((uint32_t)(p.groups_main - p.s_plain_groups));
    p.s_inv_idx = inv20(gx);
    p.s_rows = (int32_t)rps;
    p.s_stage_bytes = (int32_t)rps * p.s_slot_bytes;
    const int64_t gmax = p.groups_main > (int64_t)gx ? p.groups_main : (int64_t)gx;  // >= gp, gr
    if (rps * p.groups_total * gmax >= ((int64_t)1 << 20)) stream = false;
    const int smem = kStreamStages * p.s_stage_bytes + kStreamStages * 32 * 8 +
                     2 * kStreamStages * 8 + 16;
    stream = stream && smem <= 227 * 1024 &&
             cudaFuncSetAttribute(quant_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem) == cudaSuccess;
    int occ = 0;
    if (stream)
      stream = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, quant_stream_kernel,
                                                             kStreamThreads, smem) == cudaSuccess &&
               occ > 0;
    if (stream) {
      p.row0 = 0;
      p.n_rows = (int32_t)rows;
      const int64_t chunks = (rows + rps - 1) / rps;
      const int64_t cap = (int64_t)num_sms * occ;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(chunks < cap ? chunks : cap), 1, 1);
      cfg.blockDim = dim3(kStreamThreads, 1, 1);
      cfg.dynamicSmemBytes = (size_t)smem;
      cfg.stream = s;
      cudaLaunchAttribute attr[1] = {pdl_attribute()};
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      record_launch_begin(CSA2_KERNEL_QUANT, s);
      const cudaError_t el = cudaLaunchKernelEx(&cfg, quant_stream_kernel, p);
      record_launch_end(CSA2_KERNEL_QUANT, s);
      if (el != cudaSuccess) return el;
    }
  }
  if (!stream) {
    prefer_max_shared(quant_append_kernel);
    // launches of at most 2^30 groups (whole rows), each indexed in 32 bits
    const int64_t rows_per = ((int64_t)1 << 30) / p.groups_total;
    record_launch_begin(CSA2_KERNEL_QUANT, s);
    for (int64_t r0 = 0; r0 < rows; r0 += rows_per) {
      const int64_t nr = rows - r0 < rows_per ? rows - r0 : rows_per;
      p.row0 = (int32_t)r0;
      p.n_groups = (uint32_t)(nr * p.groups_total);
      quant_append_kernel<<<(unsigned)((p.n_groups + 255) / 256), 256, 0, s>>>(p);
    }
    record_launch_end(CSA2_KERNEL_QUANT, s);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // launched early too: it waits for the append grid before touching seq_len
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((c.batch + 127) / 128), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, advance_len_kernel, c.seq_len, c.batch, T, c.max_len);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t set_wait_limit_quant(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace csa2
