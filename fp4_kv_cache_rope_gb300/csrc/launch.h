// Host-side launch functions shared between the C-ABI layer (api.cu) and the
// kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"
#include "common.cuh"

namespace csa2 {

// Every kernel of the path asks for the largest shared-memory carveout, so
// that consecutive kernels of a step never make an SM change its L1/shared
// split between launches.
// Launch attribute that lets a kernel overlap the tail of the previous kernel
// of its stream (it must call griddep_wait() before using that kernel's work).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

template <typename Kernel>
inline cudaError_t prefer_max_shared(Kernel kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

// How many clusters of `cluster` CTAs (each `threads` threads and `smem`
// dynamic shared-memory bytes) the GPU runs at once; 0 when unknown.
template <typename Kernel>
inline int max_active_clusters(Kernel kern, int cluster, int threads, int smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear the error; the caller falls back
    return 0;
  }
  return n;
}

// Limit of the bounded on-chip waits of each kernel file (0 = the default).
cudaError_t set_wait_limit_indexer(unsigned long long ns);
cudaError_t set_wait_limit_attention(unsigned long long ns);
cudaError_t set_wait_limit_quant(unsigned long long ns);

// Benchmark instrumentation (api.cu): records the family's begin/end events
// on stream s when they are set.
void record_launch_begin(int family, cudaStream_t s);
void record_launch_end(int family, cudaStream_t s);

// quant.cu
cudaError_t launch_fp8_quant(const float* x, int64_t n, uint8_t* out, cudaStream_t s);
cudaError_t launch_quant_append(const csa2_cache& c, const float* kv, const float* z,
                                const float* idx_in, int32_t T, uint32_t* status, int num_sms,
                                cudaStream_t s);

// Description of the query rows of one indexer call.
struct RowSet {
  int32_t n_rows;           // n_batch * Tq
  int32_t tq;               // queries per sequence
  const int32_t* batch_ids; // [n_batch] or null (identity)
  const int32_t* q_pos;     // [B, Tq] or null (decode)
};

// indexer.cu: mode 0 = Full (all visible positions), 1 = pool positions.
cudaError_t launch_indexer(const csa2_cache& c, const RowSet& rows, int mode,
                           const uint8_t* q_idx, const float* w, int32_t hi,
                           const int32_t* pool_blocks, const int32_t* pool_cnt,
                           const WsLayout& L, uint8_t* ws, int num_sms, cudaStream_t s);

// select.cu
cudaError_t launch_select(const csa2_cache& c, const RowSet& rows, int mode, int32_t k,
                          const int32_t* pool_in, const int32_t* pool_cnt_in, int32_t* out_idx,
                          int32_t* out_cnt, int32_t* pool_out, int32_t* pool_cnt_out,
                          const WsLayout& L, uint8_t* ws, int num_sms, cudaStream_t s);

// attention.cu
struct AttnArgs {
  // per layer (n_layers of them; the layers share idx, cnt and swa_cnt)
  const uint16_t* q[CSA2_MAX_ATTN_LAYERS];    // bf16 [rows, H, D]
  const uint8_t* swa[CSA2_MAX_ATTN_LAYERS];   // decode [B, W, D]; prefill band [B, Tq+W-1, D]
  float* out[CSA2_MAX_ATTN_LAYERS];           // [rows, H, D]
  int32_t n_layers;
  int32_t heads;
  int32_t n_rows;           // B * Tq
  int32_t tq;               // 1 for decode
  const int32_t* q_pos;     // prefill positions [B, Tq] or null
  const int32_t* idx;       // [rows, kcap]
  const int32_t* cnt;       // [rows]
  int32_t kcap;
  const int32_t* swa_cnt;   // decode only, or null
  int32_t window;
  float scale;
};
cudaError_t launch_attention(const csa2_cache& c, const AttnArgs& a, const WsLayout& L,
                             uint8_t* ws, int num_sms, cudaStream_t s);

}  // namespace csa2
