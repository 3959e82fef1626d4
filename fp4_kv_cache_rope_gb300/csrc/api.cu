// C-ABI entry points of libcsa2: host-side validation, workspace carving and
// kernel launches.  Every entry point returns a csa2_status and never throws.
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "launch.h"

using namespace csa2;

namespace {

bool mult16(int64_t x) { return x % 16 == 0; }

// Structural checks of the cache description.
bool cache_ok(const csa2_cache* c) {
  if (!c) return false;
  if (c->batch <= 0 || c->dim <= 0 || c->dim % 64 != 0 || c->dim > 576) return false;
  if (c->rope_dim < 0 || c->rope_dim % 2 != 0 || c->rope_dim > c->dim) return false;
  if (c->idx_dim != 32 && c->idx_dim != 64 && c->idx_dim != 128) return false;
  if (c->max_len <= 0 || c->max_len > CSA2_MAX_LEN) return false;
  if (c->page_size < 0) return false;
  if (c->page_size > 0) {
    if (c->page_size % 8 != 0) return false;
    if (!(128 % c->page_size == 0 || c->page_size % 128 == 0)) return false;
    if (!c->page_table || c->max_pages_per_seq <= 0 || c->num_pages <= 0) return false;
    if ((int64_t)c->max_pages_per_seq * c->page_size < c->max_len) return false;
  }
  if (!c->kv_codes || !c->kv_scales || !c->idx_k || !c->seq_len) return false;
  if (c->code_stride < c->dim / 2 || !mult16(c->code_stride)) return false;
  const int64_t scb = ((c->dim / 16) + 15) / 16 * 16;
  if (c->scale_stride < scb || !mult16(c->scale_stride)) return false;
  if (c->idx_format == CSA2_IDX_E4M3) {
    if (c->idxk_stride < c->idx_dim || !mult16(c->idxk_stride)) return false;
  } else if (c->idx_format == CSA2_IDX_MXFP4) {
    // the packed-E2M1 tensor map wants 32-byte aligned rows of 128 channels;
    // a tile's scale rows are copied in 16-byte aligned runs
    if (c->idx_dim != 128 || c->idxk_stride < 64 || c->idxk_stride % 32 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(c->idx_k) & 31) != 0) return false;
    if (!c->idx_scales || c->idx_scale_stride != 4) return false;
    if ((reinterpret_cast<uintptr_t>(c->idx_scales) & 15) != 0) return false;
    if (c->page_size == 0 && c->max_len % 4 != 0) return false;
  } else {
    return false;
  }
  if (c->rope_dim > 0 && (!c->rope_cos || !c->rope_sin)) return false;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

csa2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

WsLayout layout_for(const csa2_cache* c, int64_t rows) {
  return ws_layout(c->max_len, rows);
}

cudaEvent_t g_events[4][2] = {};

}  // namespace

namespace csa2 {
// Under stream capture the records are external, so that they become event
// nodes timing every replay instead of capture-internal dependencies; the
// external flag is only valid while the stream is capturing.
static void record_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}
void record_launch_begin(int family, cudaStream_t s) {
  if (g_events[family][0]) record_event(g_events[family][0], s);
}
void record_launch_end(int family, cudaStream_t s) {
  if (g_events[family][1]) record_event(g_events[family][1], s);
}
}  // namespace csa2

extern "C" {

csa2_status csa2_set_launch_events(int32_t family, void* begin, void* end) {
  if (family < 0 || family > 3 || ((begin == nullptr) != (end == nullptr))) return CSA2_ERR_INVALID;
  g_events[family][0] = static_cast<cudaEvent_t>(begin);
  g_events[family][1] = static_cast<cudaEvent_t>(end);
  return CSA2_OK;
}

csa2_status csa2_set_wait_limit(uint64_t ns) {
  const unsigned long long v = ns == 0 ? (unsigned long long)kWaitNs : (unsigned long long)ns;
  cudaError_t e = set_wait_limit_indexer(v);
  if (e == cudaSuccess) e = set_wait_limit_attention(v);
  if (e == cudaSuccess) e = set_wait_limit_quant(v);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return from_cuda(e);
}

size_t csa2_workspace_size(const csa2_cache* cache, int32_t max_rows, int32_t heads) {
  if (!cache_ok(cache) || max_rows <= 0 || heads <= 0 || heads > 64) return 0;
  return layout_for(cache, max_rows).total;
}

int64_t csa2_entry_bytes(int32_t dim) { return dim <= 0 ? 0 : (int64_t)dim / 2 + dim / 16; }

csa2_status csa2_fp8_quant(const float* x, int64_t n, uint8_t* out, void* stream) {
  if (n < 0 || (n > 0 && (!x || !out))) return CSA2_ERR_INVALID;
  return from_cuda(launch_fp8_quant(x, n, out, (cudaStream_t)stream));
}

csa2_status csa2_quant_append(const csa2_cache* cache, const float* kv, const float* idx_k_in,
                              int32_t T, void* ws, void* stream) {
  if (!cache_ok(cache) || !kv || !ws || T < 0 || !aligned16(kv) || !aligned16(ws))
    return CSA2_ERR_INVALID;
  if (idx_k_in && !aligned16(idx_k_in)) return CSA2_ERR_INVALID;
  if (T == 0) return CSA2_OK;
  if (T > cache->max_len) return CSA2_ERR_INVALID;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const WsLayout L = layout_for(cache, 1);
  return from_cuda(launch_quant_append(*cache, kv, nullptr, idx_k_in, T,
                                       reinterpret_cast<uint32_t*>(w + L.status), num_sms(),
                                       (cudaStream_t)stream));
}

csa2_status csa2_quant_append_pairs(const csa2_cache* cache, const float* kv, const float* z,
                                    const float* idx_k_in, int32_t T, void* ws, void* stream) {
  if (!cache_ok(cache) || !kv || !z || !ws || T < 0 || !aligned16(kv) || !aligned16(z) ||
      !aligned16(ws))
    return CSA2_ERR_INVALID;
  if (idx_k_in && !aligned16(idx_k_in)) return CSA2_ERR_INVALID;
  if (T == 0) return CSA2_OK;
  if (T > cache->max_len) return CSA2_ERR_INVALID;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const WsLayout L = layout_for(cache, 1);
  return from_cuda(launch_quant_append(*cache, kv, z, idx_k_in, T,
                                       reinterpret_cast<uint32_t*>(w + L.status), num_sms(),
                                       (cudaStream_t)stream));
}

static csa2_status index_common(const csa2_cache* cache, int mode, const uint8_t* q_idx,
                                const float* w, int32_t Hi, int32_t Tq, const int32_t* q_pos,
                                const int32_t* pool_in, const int32_t* pool_cnt_in,
                                const int32_t* batch_ids, int32_t n_batch, int32_t k,
                                int32_t* out_idx, int32_t* out_cnt, int32_t* pool_out,
                                int32_t* pool_cnt_out, void* ws, void* stream) {
  if (!cache_ok(cache) || !q_idx || !w || !out_idx || !out_cnt || !ws) return CSA2_ERR_INVALID;
  if (Hi < 1 || Hi > 64 || Tq < 1 || k < 1 || k > CSA2_MAX_TOPK) return CSA2_ERR_INVALID;
  if (n_batch < 0 || n_batch > cache->batch || (!batch_ids && n_batch != cache->batch))
    return CSA2_ERR_INVALID;
  if (Tq > 1 && !q_pos) return CSA2_ERR_INVALID;
  if (mode == 1 && (!pool_in || !pool_cnt_in)) return CSA2_ERR_INVALID;
  if ((pool_out == nullptr) != (pool_cnt_out == nullptr)) return CSA2_ERR_INVALID;
  if (!aligned16(q_idx) || !aligned16(ws)) return CSA2_ERR_INVALID;
  if (n_batch == 0) return CSA2_OK;
  const int64_t rows = (int64_t)n_batch * Tq;
  if (rows > (1 << 24)) return CSA2_ERR_INVALID;
  RowSet rs{(int32_t)rows, Tq, batch_ids, q_pos};
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const WsLayout L = layout_for(cache, rows);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_indexer(*cache, rs, mode, q_idx, w, Hi, pool_in, pool_cnt_in, L, wsb,
                                 num_sms(), s);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  e = launch_select(*cache, rs, mode, k, pool_in, pool_cnt_in, out_idx, out_cnt, pool_out,
                    pool_cnt_out, L, wsb, num_sms(), s);
  return from_cuda(e);
}

csa2_status csa2_index_full(const csa2_cache* cache, const uint8_t* q_idx, const float* w,
                            int32_t Hi, int32_t Tq, const int32_t* q_pos,
                            const int32_t* batch_ids, int32_t n_batch, int32_t k,
                            int32_t* out_idx, int32_t* out_cnt, int32_t* pool_blocks,
                            int32_t* pool_cnt, void* ws, void* stream) {
  return index_common(cache, 0, q_idx, w, Hi, Tq, q_pos, nullptr, nullptr, batch_ids, n_batch, k,
                      out_idx, out_cnt, pool_blocks, pool_cnt, ws, stream);
}

csa2_status csa2_index_reindex(const csa2_cache* cache, const uint8_t* q_idx, const float* w,
                               int32_t Hi, int32_t Tq, const int32_t* q_pos,
                               const int32_t* pool_blocks, const int32_t* pool_cnt,
                               const int32_t* batch_ids, int32_t n_batch, int32_t k,
                               int32_t* out_idx, int32_t* out_cnt, void* ws, void* stream) {
  return index_common(cache, 1, q_idx, w, Hi, Tq, q_pos, pool_blocks, pool_cnt, batch_ids,
                      n_batch, k, out_idx, out_cnt, nullptr, nullptr, ws, stream);
}

static csa2_status attn_common(const csa2_cache* cache, int32_t L, const uint16_t* const* q,
                               int32_t H, int32_t Tq, const int32_t* q_pos, const int32_t* idx,
                               const int32_t* cnt, int32_t kcap, const uint8_t* const* swa,
                               const int32_t* swa_cnt, int32_t W, float scale, float* const* out,
                               void* ws, void* stream) {
  if (!cache_ok(cache) || !q || !idx || !cnt || !out || !ws) return CSA2_ERR_INVALID;
  if (L < 1 || L > CSA2_MAX_ATTN_LAYERS) return CSA2_ERR_INVALID;
  if (H < 1 || H > 64 || kcap < 0 || W < 0 || Tq < 1) return CSA2_ERR_INVALID;
  if (W > 0 && !swa) return CSA2_ERR_INVALID;
  for (int l = 0; l < L; ++l) {
    if (!q[l] || !out[l] || !aligned16(q[l]) || !aligned16(out[l])) return CSA2_ERR_INVALID;
    if (W > 0 && (!swa[l] || !aligned16(swa[l]))) return CSA2_ERR_INVALID;
  }
  if (!aligned16(ws)) return CSA2_ERR_INVALID;
  if (isnan(scale)) return CSA2_ERR_INVALID;
  const int64_t rows = (int64_t)cache->batch * Tq;
  if ((int64_t)L * rows > 65535) return CSA2_ERR_INVALID;
  AttnArgs a;
  a.n_layers = L;
  for (int l = 0; l < CSA2_MAX_ATTN_LAYERS; ++l) {
    const int k = l < L ? l : 0;
    a.q[l] = q[k];
    a.swa[l] = W > 0 ? swa[k] : nullptr;
    a.out[l] = out[k];
  }
  a.heads = H;
  a.n_rows = (int32_t)rows;
  a.tq = Tq;
  a.q_pos = q_pos;
  a.idx = idx;
  a.cnt = cnt;
  a.kcap = kcap;
  a.swa_cnt = swa_cnt;
  a.window = W;
  a.scale = scale;
  const WsLayout Lw = layout_for(cache, rows);
  return from_cuda(launch_attention(*cache, a, Lw, static_cast<uint8_t*>(ws), num_sms(),
                                    (cudaStream_t)stream));
}

csa2_status csa2_attn_decode(const csa2_cache* cache, const uint16_t* q, int32_t H,
                             const int32_t* idx, const int32_t* cnt, int32_t kcap,
                             const uint8_t* swa, const int32_t* swa_cnt, int32_t W,
                             float softmax_scale, float* out, void* ws, void* stream) {
  return attn_common(cache, 1, &q, H, 1, nullptr, idx, cnt, kcap, &swa, swa_cnt, W,
                     softmax_scale, &out, ws, stream);
}

csa2_status csa2_attn_decode_layers(const csa2_cache* cache, int32_t L, const uint16_t* const* q,
                                    int32_t H, const int32_t* idx, const int32_t* cnt,
                                    int32_t kcap, const uint8_t* const* swa,
                                    const int32_t* swa_cnt, int32_t W, float softmax_scale,
                                    float* const* out, void* ws, void* stream) {
  if (!q || !out || (W > 0 && !swa)) return CSA2_ERR_INVALID;
  return attn_common(cache, L, q, H, 1, nullptr, idx, cnt, kcap, swa, swa_cnt, W, softmax_scale,
                     out, ws, stream);
}

csa2_status csa2_attn_prefill(const csa2_cache* cache, const uint16_t* q, int32_t H, int32_t Tq,
                              const int32_t* q_pos, const int32_t* idx, const int32_t* cnt,
                              int32_t kcap, const uint8_t* swa, int32_t W, float softmax_scale,
                              float* out, void* ws, void* stream) {
  if (!q_pos) return CSA2_ERR_INVALID;
  if (W < 1) return CSA2_ERR_INVALID;
  return attn_common(cache, 1, &q, H, Tq, q_pos, idx, cnt, kcap, &swa, nullptr, W, softmax_scale,
                     &out, ws, stream);
}

csa2_status csa2_get_status(void* ws, uint32_t* host_status, void* stream) {
  if (!ws || !host_status) return CSA2_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(host_status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
  return *host_status ? CSA2_ERR_DEVICE : CSA2_OK;
}

csa2_status csa2_reset_status(void* ws, void* stream) {
  if (!ws) return CSA2_ERR_INVALID;
  return from_cuda(cudaMemsetAsync(ws, 0, sizeof(uint32_t), (cudaStream_t)stream));
}

const char* csa2_status_string(csa2_status status) {
  switch (status) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID: return "invalid argument";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_UNSUPPORTED: return "unsupported";
    case CSA2_ERR_TIMEOUT: return "timeout";
    case CSA2_ERR_DEVICE: return "device status set";
  }
  return "unknown status";
}

}  // extern "C"

// ------------------------------------------------- index_full without a workspace
//
// csa2_index_full_noalloc serves callers that are handed their device buffers
// and may not create more: a host engine that reserves the GPU's memory for
// its own pools at start-up and forbids side allocations, or a hot loop that
// cannot take the implicit device synchronisation and unbounded latency of a
// cudaMalloc.  Its scratch (status word, per-row lengths, scores, block
// maxima) lives in one fixed array of CSA2_NOALLOC_SCRATCH_BYTES bytes that
// every GPU loading this library's device code holds until the process exits.
// All calls on a device share that array and it keeps the previous call's
// contents; only the status word must start at zero and each call clears it.
// Two calls whose work overlaps on the GPU (different streams, or threads that
// do not order their streams) race on the array.
namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[CSA2_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoallocMaxDevices] = {};

// Device address of the scratch array on the current device.  Looked up once
// per device (with that device current); the first lookup may load this
// library's device code onto the device.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    // The host-side name of the array only identifies it; the device address
    // comes from the runtime.
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if ((reinterpret_cast<uintptr_t>(p) & 255) != 0) return cudaErrorMisalignedAddress;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" csa2_status csa2_index_full_noalloc(
    const csa2_cache* cache, const uint8_t* q_idx, const float* w, int32_t Hi, int32_t Tq,
    const int32_t* q_pos, const int32_t* batch_ids, int32_t n_batch, int32_t k, int32_t* out_idx,
    int32_t* out_cnt, int32_t* pool_blocks, int32_t* pool_cnt, uint32_t* status, void* stream) {
  if (!cache_ok(cache) || Tq < 1 || n_batch < 0 || n_batch > cache->batch) return CSA2_ERR_INVALID;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3) != 0) return CSA2_ERR_INVALID;
  const int64_t rows = (int64_t)n_batch * Tq;
  if (rows > (1 << 24)) return CSA2_ERR_INVALID;
  if (rows > 0 && layout_for(cache, rows).total > (size_t)CSA2_NOALLOC_SCRATCH_BYTES)
    return CSA2_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s) != cudaSuccess) return CSA2_ERR_CUDA;
  const csa2_status r = csa2_index_full(cache, q_idx, w, Hi, Tq, q_pos, batch_ids, n_batch, k,
                                        out_idx, out_cnt, pool_blocks, pool_cnt, scratch, stream);
  if (r != CSA2_OK) return r;
  if (status && cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDefault, s) !=
                    cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}
