// The CSA2 hot path as plain C++ on the host cores: test infrastructure and
// the timed CPU baseline, never the product path.  It shares no code, header
// or table with the CUDA library; the format tables below are built from the
// formats' definitions.  Compiled with -ffp-contract=off, so every float
// operation is one IEEE rounding, as written.
//
// Pages followed (titles and sections):
//   "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
//   (knowledge note): "FP4 main KV: trade precision for bytes, not for a new
//   GEMM" (E2M1 codes, one E4M3 scale per 16 channels, quantised after
//   RoPE), "Hierarchical Sparse Indexer: make later searches bounded" (the
//   indexer score, top-k, the block pool), "Putting It Together" steps 5-8
//   (score, select, dequantise, sparse attention with the local window).
//
// Each function restates the same definition as the numpy oracle
// (oracle/csa2.py), in loops: one std::thread per core takes a contiguous
// share of the positions (scores) or heads (attention).
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <thread>
#include <vector>

namespace {

// ------------------------------------------------------------------ formats
// E4M3 "FN": sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
// subnormal (m / 8 * 2^-6); 0x7F / 0xFF are NaN and never produced.
double e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xF, m = c & 7;
  double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, (int)e - 10);
  if ((c & 0x7F) == 0x7F) v = NAN;
  return (c & 0x80) ? -v : v;
}

// E2M1: sign in bit 3, magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
const double kE2m1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
double e2m1_value(uint32_t c) { return (c & 8) ? -kE2m1Mag[c & 7] : kE2m1Mag[c & 7]; }

struct Tables {
  double e4m3[256];
  double e4m3_finite[127];  // magnitudes of codes 0..126, increasing
  Tables() {
    for (int c = 0; c < 256; ++c) e4m3[c] = e4m3_value((uint32_t)c);
    for (int c = 0; c < 127; ++c) e4m3_finite[c] = e4m3_value((uint32_t)c);
  }
};
const Tables& tables() {
  static const Tables t;
  return t;
}

// Index of the nearest entry of the increasing table t[0..n) to mag >= 0;
// a tie goes to the even index; at or above the last entry, the last index.
int nearest_code(double mag, const double* t, int n) {
  if (mag >= t[n - 1]) return n - 1;
  int hi = (int)(std::lower_bound(t, t + n, mag) - t);  // first t >= mag
  if (hi == 0) return 0;
  const int lo = hi - 1;
  const double dl = mag - t[lo], dh = t[hi] - mag;
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return (lo % 2 == 0) ? lo : hi;
}

uint32_t e4m3_encode(float x) {
  const double mag = fabs((double)x);
  const uint32_t code = (uint32_t)nearest_code(mag, tables().e4m3_finite, 127);
  return code | (signbit(x) ? 0x80u : 0u);
}

uint32_t e2m1_encode(float x) {
  const double mag = fabs((double)x);
  const uint32_t code = (uint32_t)nearest_code(mag, kE2m1Mag, 8);
  return code | (signbit(x) ? 8u : 0u);
}

// Runs f(lo, hi) over [0, n) cut into `threads` contiguous shares.
template <typename F>
void parallel_for(int64_t n, int threads, F f) {
  if (threads <= 1 || n < 2 * threads) {
    f((int64_t)0, n);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t) {
    const int64_t lo = n * t / threads, hi = n * (t + 1) / threads;
    pool.emplace_back([=] { f(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

int cref_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? (int)n : 1;
}

// ---------------------------------------------------- step 1: RoPE + FP4
// Pre-RoPE fp32 rows kv [n, D] at positions pos[n] -> codes [n, D/2] (element
// 2j in the low nibble of byte j) and scales [n, D/16].  RoPE on pairs
// (D-R+2i, D-R+2i+1) with (c, s) = (cos_tab, sin_tab)[pos][i]:
// y0 = x0*c - x1*s, y1 = x0*s + x1*c, each operation one fp32 rounding.  Per
// group of 16: scale code = E4M3(amax / 6) (fp32 division), s its value,
// codes = E2M1(y / s) (fp32 division), all zero when s == 0.
void cref_quant_append_rows(const float* kv, const int64_t* pos, int64_t n, int32_t D,
                            const float* cos_tab, const float* sin_tab, int32_t R,
                            uint8_t* codes, uint8_t* scales) {
  std::vector<float> y((size_t)D);
  const int half = R / 2;
  for (int64_t r = 0; r < n; ++r) {
    const float* x = kv + r * D;
    memcpy(y.data(), x, sizeof(float) * (size_t)D);
    for (int i = 0; i < half; ++i) {
      const float c = cos_tab[pos[r] * half + i], s = sin_tab[pos[r] * half + i];
      const float x0 = x[D - R + 2 * i], x1 = x[D - R + 2 * i + 1];
      const float a = x0 * c, b = x1 * s, e = x0 * s, f = x1 * c;
      y[D - R + 2 * i] = a - b;
      y[D - R + 2 * i + 1] = e + f;
    }
    for (int g = 0; g < D / 16; ++g) {
      float amax = 0.0f;
      for (int e = 0; e < 16; ++e) amax = std::max(amax, fabsf(y[16 * g + e]));
      const float sixth = amax / 6.0f;
      const uint32_t sc = e4m3_encode(sixth);
      const float s = (float)tables().e4m3[sc];
      scales[r * (D / 16) + g] = (uint8_t)sc;
      for (int e = 0; e < 16; e += 2) {
        uint32_t lo = 0, hi = 0;
        if (s != 0.0f) {
          const float q0 = y[16 * g + e] / s, q1 = y[16 * g + e + 1] / s;
          lo = e2m1_encode(q0);
          hi = e2m1_encode(q1);
        }
        codes[r * (D / 2) + 8 * g + e / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

// ----------------------------------------- step 1b: m = 2 pair compression
// e^x for fp32 x <= 0, one fp32 rounding per operation, 0 below -80:
// k = rint(x / ln 2), r = (x - k ln2_hi) - k ln2_lo (ln2_hi = 2839/4096 has 12
// significant bits, so k ln2_hi is exact), e^r by Horner on the degree-7
// Taylor polynomial, times 2^k (k >= -116 keeps the result normal).
float exp_neg_f32(float x) {
  const float inv_ln2 = (float)(1.0 / 0.6931471805599453);
  const float ln2_hi = (float)(2839.0 / 4096.0);
  const float ln2_lo = (float)(0.6931471805599453 - 2839.0 / 4096.0);
  if (x < -80.0f) return 0.0f;
  const float k = rintf(x * inv_ln2);
  const float r = (x - k * ln2_hi) - k * ln2_lo;
  static const double fact[8] = {1.0, 1.0, 2.0, 6.0, 24.0, 120.0, 720.0, 5040.0};
  float p = (float)(1.0 / fact[7]);
  for (int i = 6; i >= 0; --i) p = p * r + (float)(1.0 / fact[i]);
  return ldexpf(p, (int)k);
}

// Source rows kv [2T, D] and their logits z [2T, D] -> T compressed rows:
// per channel, with d = z1 - z0 and t = e^-|d|, the larger logit's row gets
// 1 / (1 + t) and the other t / (1 + t) (a softmax over the pair);
// c = w0 x0 + w1 x1, each operation one fp32 rounding.
void cref_compress_pairs(const float* kv, const float* z, int64_t T, int32_t D, float* out) {
  for (int64_t j = 0; j < T; ++j)
    for (int c = 0; c < D; ++c) {
      const float z0 = z[(2 * j) * D + c], z1 = z[(2 * j + 1) * D + c];
      const float d = z1 - z0;
      const float t = exp_neg_f32(-fabsf(d));
      const float s = 1.0f + t;
      const float big = 1.0f / s, small = t / s;
      const float w0 = d >= 0.0f ? small : big;
      const float w1 = d >= 0.0f ? big : small;
      const float a = w0 * kv[(2 * j) * D + c], b = w1 * kv[(2 * j + 1) * D + c];
      out[j * D + c] = a + b;
    }
}

// The codecs over a range of fp32 bit patterns: for i in [first, first + n)
// the value with bit pattern i, its E2M1 code and its E4M3 code (0xFF for
// NaN patterns, which the encoders never receive).
void cref_encode_range(uint64_t first, int64_t n, uint8_t* e2m1, uint8_t* e4m3,
                       int32_t threads) {
  parallel_for(n, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) {
      const uint32_t bits = (uint32_t)(first + (uint64_t)i);
      float x;
      memcpy(&x, &bits, sizeof x);
      if (isnan(x)) {
        e2m1[i] = 0xFF;
        e4m3[i] = 0xFF;
        continue;
      }
      e2m1[i] = (uint8_t)e2m1_encode(x);
      e4m3[i] = (uint8_t)e4m3_encode(x);
    }
  });
}

// ------------------------------------------------ step 2: indexer scores
// s_t = sum_h w_h * max(0, sum_d q[h, d] k[t, d]) in fp64, q and k decoded
// from E4M3 (k rows k_stride bytes apart).  Every product of two E4M3 values
// and every partial sum of one row's di products is exact in fp64.
void cref_index_scores(const uint8_t* q_codes, const float* w, int32_t Hi, int32_t di,
                       const uint8_t* k_codes, int64_t k_stride, int64_t n, double* out,
                       int32_t threads) {
  const Tables& T = tables();
  std::vector<double> q((size_t)Hi * di);
  for (int64_t i = 0; i < (int64_t)Hi * di; ++i) q[i] = T.e4m3[q_codes[i]];
  parallel_for(n, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> k((size_t)di);
    for (int64_t t = lo; t < hi; ++t) {
      const uint8_t* kc = k_codes + t * k_stride;
      for (int d = 0; d < di; ++d) k[d] = T.e4m3[kc[d]];
      double s = 0.0;
      for (int h = 0; h < Hi; ++h) {
        double dot = 0.0;
        for (int d = 0; d < di; ++d) dot += q[(size_t)h * di + d] * k[d];
        s += (double)w[h] * (dot > 0.0 ? dot : 0.0);
      }
      out[t] = s;
    }
  });
}

// The same score with MXFP4 keys: E2M1 codes (element 2j in the low nibble
// of byte j) times one E8M0 scale 2^(code - 127) per 32 channels.
void cref_index_scores_mx(const uint8_t* q_codes, const float* w, int32_t Hi, int32_t di,
                          const uint8_t* k_codes, int64_t k_stride, const uint8_t* k_scales,
                          int64_t s_stride, int64_t n, double* out, int32_t threads) {
  const Tables& T = tables();
  std::vector<double> q((size_t)Hi * di);
  for (int64_t i = 0; i < (int64_t)Hi * di; ++i) q[i] = T.e4m3[q_codes[i]];
  parallel_for(n, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> k((size_t)di);
    for (int64_t t = lo; t < hi; ++t) {
      const uint8_t* kc = k_codes + t * k_stride;
      const uint8_t* ks = k_scales + t * s_stride;
      for (int d = 0; d < di; ++d) {
        const uint32_t c = (kc[d / 2] >> (4 * (d & 1))) & 0xF;
        k[d] = e2m1_value(c) * ldexp(1.0, (int)ks[d / 32] - 127);
      }
      double s = 0.0;
      for (int h = 0; h < Hi; ++h) {
        double dot = 0.0;
        for (int d = 0; d < di; ++d) dot += q[(size_t)h * di + d] * k[d];
        s += (double)w[h] * (dot > 0.0 ? dot : 0.0);
      }
      out[t] = s;
    }
  });
}

// ------------------------------------------------------- step 3: selection
// Per block of 8 positions, the largest score among the positions that exist.
void cref_block_maxima(const double* scores, int64_t n, double* out) {
  for (int64_t b = 0; b * 8 < n; ++b) {
    double m = -INFINITY;
    for (int64_t t = 8 * b; t < n && t < 8 * b + 8; ++t) m = std::max(m, scores[t]);
    out[b] = m;
  }
}

// The k best of n (score descending, id ascending on equal scores), written
// to out in ascending id order; ids == NULL means ids 0..n-1.  Returns the
// count, min(k, n).
int64_t cref_topk(const double* scores, const int64_t* ids, int64_t n, int64_t k, int64_t* out) {
  if (k > n) k = n;
  if (k <= 0) return 0;
  std::vector<int64_t> ord((size_t)n);
  for (int64_t i = 0; i < n; ++i) ord[i] = i;
  auto id = [&](int64_t i) { return ids ? ids[i] : i; };
  auto better = [&](int64_t a, int64_t b) {
    if (scores[a] != scores[b]) return scores[a] > scores[b];
    return id(a) < id(b);
  };
  std::nth_element(ord.begin(), ord.begin() + (k - 1), ord.end(), better);
  for (int64_t i = 0; i < k; ++i) out[i] = id(ord[i]);
  std::sort(out, out + k);
  return k;
}

// ------------------------------------------- step 4: FP4 dequantisation
// (codes [rows, D/2] at code_stride, scales [rows, D/16] at scale_stride) ->
// fp64 rows [rows, D]: E2M1(code) * E4M3(scale of the channel's group).
void cref_dequant_fp4(const uint8_t* codes, int64_t code_stride, const uint8_t* scales,
                      int64_t scale_stride, int64_t rows, int32_t D, double* out) {
  const Tables& T = tables();
  for (int64_t r = 0; r < rows; ++r)
    for (int c = 0; c < D; ++c) {
      const uint32_t code = (codes[r * code_stride + c / 2] >> (4 * (c & 1))) & 0xF;
      out[r * D + c] = e2m1_value(code) * T.e4m3[scales[r * scale_stride + c / 16]];
    }
}

// Plain E4M3 codes -> fp64 (the FP8 window rows).
void cref_decode_e4m3(const uint8_t* codes, int64_t n, double* out) {
  const Tables& T = tables();
  for (int64_t i = 0; i < n; ++i) out[i] = T.e4m3[codes[i]];
}

// ----------------------------------------------------- step 5: attention
// One softmax per head over the n rows (selected rows, then window rows),
// K = V = the row: o_h = sum_j p_j x_j / sum_j p_j with
// p_j = exp(scale * q_h . x_j - max_j(...)); all in fp64; n == 0 gives zeros.
void cref_attention(const double* q, int32_t H, int32_t D, const double* rows, int64_t n,
                    double scale, double* out, int32_t threads) {
  parallel_for(H, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> p((size_t)(n > 0 ? n : 1));
    for (int64_t h = lo; h < hi; ++h) {
      double* o = out + h * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (n == 0) continue;
      const double* qh = q + h * D;
      double m = -INFINITY;
      for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qh[d] * rows[j * D + d];
        p[j] = scale * dot;
        m = std::max(m, p[j]);
      }
      double den = 0.0;
      for (int64_t j = 0; j < n; ++j) {
        p[j] = exp(p[j] - m);
        den += p[j];
      }
      for (int64_t j = 0; j < n; ++j)
        for (int d = 0; d < D; ++d) o[d] += p[j] * rows[j * D + d];
      for (int d = 0; d < D; ++d) o[d] /= den;
    }
  });
}

}  // extern "C"
