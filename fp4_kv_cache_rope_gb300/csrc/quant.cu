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
// One thread owns one group of 16 channels of one row: it loads 64 bytes of
// fp32, rotates the pairs that fall in the RoPE slice, takes the group
// maximum, encodes the scale and the 16 codes, and stores 8 code bytes and
// one scale byte.  Consecutive threads own consecutive groups, so loads and
// stores are coalesced.  The kernel is HBM bound (2.3 KB read, 324 B written
// per D = 576 row).
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

// MXFP4 indexer key, one 32-channel block per thread: the E8M0 scale code is
// the OCP Microscaling shared exponent floor(log2 amax) - 2 (E2M1's top
// binade is 2^2), read off the fp32 exponent field of amax and clamped at
// code 0; codes = E2M1(x * 2^(127 - code)), an exact power-of-two scaling.
__device__ __noinline__ void quant_idx_mx(const QuantParams& p, int64_t row, int b, int i,
                                          int gi) {
  float y[32];
  const float4* src = reinterpret_cast<const float4*>(p.idx_in + row * p.di + 32 * gi);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 f = __ldg(src + v);
    y[4 * v + 0] = f.x;
    y[4 * v + 1] = f.y;
    y[4 * v + 2] = f.z;
    y[4 * v + 3] = f.w;
  }
  const int64_t pos = (int64_t)p.seq_len[b] + i;
  if (pos >= p.map.max_len || pos < 0) {
    set_status(p.status, CSA2_DEV_OVERFLOW);
    return;
  }
  const int64_t r = p.map.row(b, pos);
  if (r < 0) {
    set_status(p.status, CSA2_DEV_BAD_PAGE);
    return;
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
    for (int e = 0; e < 8; ++e) x |= e2m1_encode(__fmul_rn(y[8 * v + e], inv)) << (4 * e);
    w[v] = x;
  }
  *reinterpret_cast<uint4*>(p.idx_k + r * p.idxk_stride + 16 * gi) = make_uint4(w[0], w[1], w[2], w[3]);
  p.idx_scales[r * 4 + gi] = (uint8_t)code;
}

// Quantises group gid of the launch (row row0 + gid / groups_total, group
// gid % groups_total).  Rows (B * T) and a launch's groups fit in 31 bits, so
// the index arithmetic is 32-bit (a 64-bit division is a long software
// sequence on the GPU).
__device__ __forceinline__ void quant_group(const QuantParams& p, uint32_t gid) {
  const uint32_t lrow = gid / (uint32_t)p.groups_total;
  const int g = (int)(gid - lrow * (uint32_t)p.groups_total);
  const int32_t row32 = p.row0 + (int32_t)lrow;
  const int b = row32 / p.T;
  const int i = row32 - b * p.T;
  const int64_t row = row32;
  const bool is_idx = g >= p.groups_main;
  if (is_idx && p.idx_mx) {
    quant_idx_mx(p, row, b, i, g - p.groups_main);
    return;
  }
  // the input rows do not depend on the position: request them first
  float y[16];
  {
    if (p.z && !is_idx) {  // entry i of sequence b from source rows 2i, 2i+1
      const int64_t r0 = ((int64_t)b * p.T + i) * 2 * p.D + 16 * g;
      const float4* x0 = reinterpret_cast<const float4*>(p.kv + r0);
      const float4* x1 = reinterpret_cast<const float4*>(p.kv + r0 + p.D);
      const float4* z0 = reinterpret_cast<const float4*>(p.z + r0);
      const float4* z1 = reinterpret_cast<const float4*>(p.z + r0 + p.D);
      float4 a[4], c[4], u[4], v4[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        a[v] = __ldg(x0 + v);
        c[v] = __ldg(x1 + v);
        u[v] = __ldg(z0 + v);
        v4[v] = __ldg(z1 + v);
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        y[4 * v + 0] = combine_pair(a[v].x, c[v].x, u[v].x, v4[v].x);
        y[4 * v + 1] = combine_pair(a[v].y, c[v].y, u[v].y, v4[v].y);
        y[4 * v + 2] = combine_pair(a[v].z, c[v].z, u[v].z, v4[v].z);
        y[4 * v + 3] = combine_pair(a[v].w, c[v].w, u[v].w, v4[v].w);
      }
    } else {
      const float4* src =
          is_idx ? reinterpret_cast<const float4*>(p.idx_in + row * p.di + 16 * (g - p.groups_main))
                 : reinterpret_cast<const float4*>(p.kv + row * p.D + 16 * g);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float4 f = __ldg(src + v);
        y[4 * v + 0] = f.x;
        y[4 * v + 1] = f.y;
        y[4 * v + 2] = f.z;
        y[4 * v + 3] = f.w;
      }
    }
  }
  const int64_t pos = (int64_t)p.seq_len[b] + i;
  if (pos >= p.map.max_len || pos < 0) {
    set_status(p.status, CSA2_DEV_OVERFLOW);
    return;
  }
  const int64_t r = p.map.row(b, pos);
  if (r < 0) {
    set_status(p.status, CSA2_DEV_BAD_PAGE);
    return;
  }

  if (is_idx) {  // indexer key: plain E4M3 per element
    const int gi = g - p.groups_main;
    uint32_t w[4];
#pragma unroll
    for (int v = 0; v < 4; ++v)
      w[v] = e4m3_encode(y[4 * v]) | (e4m3_encode(y[4 * v + 1]) << 8) |
             (e4m3_encode(y[4 * v + 2]) << 16) | (e4m3_encode(y[4 * v + 3]) << 24);
    *reinterpret_cast<uint4*>(p.idx_k + r * p.idxk_stride + 16 * gi) =
        make_uint4(w[0], w[1], w[2], w[3]);
    return;
  }

  // RoPE on interleaved pairs of the last R channels: two fp32 products and one
  // add/sub per output, each rounded once (no contraction into an FMA).
  const int c0 = 16 * g;
  const int rope0 = p.D - p.R;
  if (c0 + 16 > rope0) {
    const int half = p.R >> 1;
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int c = c0 + e;
      if (c >= rope0) {
        const int j = (c - rope0) >> 1;
        const float cs = __ldg(p.rope_cos + pos * half + j);
        const float sn = __ldg(p.rope_sin + pos * half + j);
        const float x0 = y[e], x1 = y[e + 1];
        y[e] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
        y[e + 1] = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
      }
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(y[e]));
  const uint32_t sc = e4m3_encode_mag(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_decode(sc);
  uint32_t lo = 0, hi = 0;
  if (s != 0.0f) {
#pragma unroll
    for (int e = 0; e < 8; ++e) lo |= e2m1_encode(__fdiv_rn(y[e], s)) << (4 * e);
#pragma unroll
    for (int e = 0; e < 8; ++e) hi |= e2m1_encode(__fdiv_rn(y[8 + e], s)) << (4 * e);
  }
  *reinterpret_cast<uint2*>(p.codes + r * p.code_stride + 8 * g) = make_uint2(lo, hi);
  p.scales[r * p.scale_stride + g] = (uint8_t)sc;
}

__global__ void __launch_bounds__(256) quant_append_kernel(QuantParams p) {
  const uint32_t gid = blockIdx.x * blockDim.x + threadIdx.x;
  if (gid < p.n_groups) quant_group(p, gid);
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
                                const float* idx_in, int32_t T, uint32_t* status,
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
  prefer_max_shared(quant_append_kernel);
  prefer_max_shared(advance_len_kernel);
  // launches of at most 2^30 groups (whole rows), each indexed in 32 bits
  const int64_t rows = (int64_t)c.batch * T;
  const int64_t rows_per = ((int64_t)1 << 30) / p.groups_total;
  record_launch_begin(CSA2_KERNEL_QUANT, s);
  for (int64_t r0 = 0; r0 < rows; r0 += rows_per) {
    const int64_t nr = rows - r0 < rows_per ? rows - r0 : rows_per;
    p.row0 = (int32_t)r0;
    p.n_groups = (uint32_t)(nr * p.groups_total);
    quant_append_kernel<<<(unsigned)((p.n_groups + 255) / 256), 256, 0, s>>>(p);
  }
  record_launch_end(CSA2_KERNEL_QUANT, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  advance_len_kernel<<<(c.batch + 127) / 128, 128, 0, s>>>(c.seq_len, c.batch, T, c.max_len);
  return cudaGetLastError();
}

}  // namespace csa2
