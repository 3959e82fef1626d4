/*
 * csa2.h -- C ABI of the CSA2 sparse-attention path over an FP4 global KV cache
 * (GB300 / sm_103a).
 *
 * The path, as the pages describe it:
 *   1. main-KV rows are rotated (RoPE) and then quantised to E2M1 values with
 *      one E4M3 scale per 16 channels, no second global scale, and appended to
 *      the cache ("DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
 *      Compression" knowledge note, section "FP4 main KV: trade precision for
 *      bytes, not for a new GEMM"; "Inside DeepSeek V4.1 Flash: CED, CSA2 and
 *      the 890-Byte KV Cache", section "Reconstructing the 890-byte cache
 *      budget");
 *   2. a lightning indexer scores cached positions against FP8 indexer keys;
 *   3. a top-k is selected per query; a Full layer also keeps a pool of at most
 *      2,048 blocks of 8 positions ranked by block-maximum score, which Reindex
 *      layers search; Reuse layers take the previous selection unchanged
 *      (knowledge note, sections "CSA2: share cache, refresh selection only
 *      when needed" and "Hierarchical Sparse Indexer: make later searches
 *      bounded");
 *   4. the selected FP4 rows are gathered and dequantised;
 *   5. one softmax runs over those rows together with an FP8 sliding window
 *      (SWA) of the most recent rows (knowledge note, "Putting It Together",
 *      steps 5-8).
 *
 * Layer modes are chosen by which calls the caller makes: Full =
 * csa2_index_full then csa2_attn_*; Reindex = csa2_index_reindex with the pool
 * of the last Full call, then csa2_attn_*; Reuse = csa2_attn_* with the
 * previous index set.
 *
 * Conventions for every call
 *  - All array arguments are DEVICE pointers to caller-owned memory unless a
 *    comment says "host".  The library allocates no device memory.
 *  - `stream` is a cudaStream_t passed as void*.  Calls enqueue kernels on it
 *    and return without synchronising (except csa2_get_status).
 *  - `ws` is a caller-owned device workspace of at least csa2_workspace_size()
 *    bytes, 256-byte aligned.  It holds scratch and a 32-bit device status word.
 *    Calls that share one workspace must be ordered on one stream.
 *  - Return value: CSA2_OK, or CSA2_ERR_INVALID for an argument rejected on
 *    the host (nothing is launched), or CSA2_ERR_CUDA when a launch failed.
 *  - Faults found on the device (an index past the visible length, a page id
 *    out of range, an append past max_len, a bounded wait that gave up) are
 *    never trapped: the kernel skips the offending row or element and ORs a
 *    CSA2_DEV_* bit into the status word, read with csa2_get_status.
 *  - No C++ exception crosses this boundary.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID = 1,      /* argument rejected on the host; nothing launched */
  CSA2_ERR_CUDA = 2,         /* a CUDA runtime or driver call failed */
  CSA2_ERR_UNSUPPORTED = 3,  /* valid request outside the shapes the library runs */
  CSA2_ERR_TIMEOUT = 4,      /* reserved for host-side waits */
  CSA2_ERR_DEVICE = 5        /* csa2_get_status found device status bits set */
} csa2_status;

/* Bits of the device status word. */
#define CSA2_DEV_BAD_INDEX 0x1u   /* selected position < 0 or >= visible length */
#define CSA2_DEV_BAD_PAGE 0x2u    /* page-table entry outside [0, num_pages) */
#define CSA2_DEV_OVERFLOW 0x4u    /* append past max_len */
#define CSA2_DEV_TIMEOUT 0x8u     /* a bounded on-chip wait gave up */
#define CSA2_DEV_BAD_POOL 0x10u   /* pool block id outside the visible blocks */
#define CSA2_DEV_BAD_ALIGN 0x20u  /* on-chip buffer misaligned (kernel skipped work) */

/* Largest k and the pool capacity (blocks of 8 positions). */
#define CSA2_MAX_TOPK 2048
#define CSA2_MAX_ATTN_LAYERS 8   /* layers of one csa2_attn_decode_layers call */
#define CSA2_POOL_BLOCKS 2048
#define CSA2_BLOCK 8
/* Longest sequence (positions) the selection kernels accept. */
#define CSA2_MAX_LEN (1 << 21)

/*
 * One shared global cache (one CSA2 group).  Row layout of the cache:
 *   kv_codes  [rows, code_stride]  E2M1 codes, two per byte, channel 2j in the
 *                                  low nibble of byte j (D/2 bytes used)
 *   kv_scales [rows, scale_stride] one E4M3 scale byte per 16 channels, in
 *                                  channel order (D/16 bytes used)
 *   idx_k     [rows, idxk_stride]  indexer key in one of two formats (idx_format):
 *     CSA2_IDX_E4M3  one E4M3 byte per channel (di bytes used)
 *     CSA2_IDX_MXFP4 E2M1 codes, two per byte, channel 2j in the low nibble
 *                    of byte j (di/2 bytes used), with
 *   idx_scales [rows, idx_scale_stride] one E8M0 byte 2^(code-127) per 32
 *                    channels, in channel order (MXFP4 only: di/32 bytes).
 *     The MXFP4 form is the released implementation's indexer key: 128 x 4/8
 *     + 128/32 = 68 bytes per entry ("Inside DeepSeek V4.1 Flash: CED, CSA2
 *     and the 890-Byte KV Cache", sections "Reconstructing the 890-byte cache
 *     budget" and "How the derived numbers were built").
 * The physical row of position t of sequence b is
 *   page_size == 0 : b * max_len + t
 *   page_size  > 0 : page_table[b * max_pages_per_seq + t / page_size]
 *                    * page_size + t % page_size
 */
typedef struct csa2_cache {
  int32_t batch;              /* B sequences */
  int32_t dim;                /* D channels per main-KV row; multiple of 64, <= 576 */
  int32_t rope_dim;           /* R: the last R channels are rotated; even, <= D */
  int32_t idx_dim;            /* di: 32, 64 or 128 */
  int32_t page_size;          /* 0 = contiguous; else a multiple of 8 that divides 128
                                 or a multiple of 128 */
  int32_t max_pages_per_seq;  /* columns of page_table (paged only) */
  int32_t max_len;            /* capacity in positions per sequence; <= CSA2_MAX_LEN */
  int32_t num_pages;          /* physical pages (paged), used for bounds checks */
  uint8_t *kv_codes;
  int64_t code_stride;        /* bytes per row, >= D/2, multiple of 16 */
  uint8_t *kv_scales;
  int64_t scale_stride;       /* bytes per row, >= round_up(D/16, 16), multiple of 16 */
  uint8_t *idx_k;
  int64_t idxk_stride;        /* bytes per row, >= di, multiple of 16 */
  const int32_t *page_table;  /* [B, max_pages_per_seq] or NULL when page_size == 0 */
  int32_t *seq_len;           /* [B] visible positions; advanced by csa2_quant_append */
  const float *rope_cos;      /* [max_len, R/2] fp32: cos(p * theta^(-2i/R)) */
  const float *rope_sin;      /* [max_len, R/2] fp32: sin(p * theta^(-2i/R)) */
  /* Indexer-key format.  Zero-initialised descriptions get CSA2_IDX_E4M3.
   * CSA2_IDX_MXFP4 requires di = 128, idx_k 32-byte aligned with
   * idxk_stride >= 64 and a multiple of 32, idx_scales 16-byte aligned with
   * idx_scale_stride == 4, and max_len a multiple of 4 when page_size == 0. */
  int32_t idx_format;
  uint8_t *idx_scales;        /* MXFP4 only; NULL for E4M3 */
  int64_t idx_scale_stride;   /* MXFP4 only: 4 */
} csa2_cache;

#define CSA2_IDX_E4M3 0
#define CSA2_IDX_MXFP4 1

/*
 * Workspace bytes for calls on `cache` that process at most `max_rows` query
 * rows (B * Tq of one call) with `heads` attention heads.  Returns 0 when the
 * cache description is invalid.
 */
size_t csa2_workspace_size(const csa2_cache *cache, int32_t max_rows, int32_t heads);

/*
 * Bytes of one FP4 main-KV entry as stored algorithmically: D/2 code bytes +
 * D/16 scale bytes (288 for D = 512, 324 for D = 576).
 */
int64_t csa2_entry_bytes(int32_t dim);

/*
 * FP8 cast used for the SWA window rows and the indexer operands: every fp32
 * x[i] becomes the E4M3 code of the nearest representable value, ties to the
 * even code, saturating at +-448, sign bit copied from x (so -0.0 -> 0x80).
 * x: device fp32 [n]; out: device uint8 [n].  Non-finite inputs: unspecified.
 */
csa2_status csa2_fp8_quant(const float *x, int64_t n, uint8_t *out, void *stream);

/*
 * Step 1: RoPE + FP4 quantisation + append.
 * kv:       device fp32 [B, T, D], rows BEFORE rotation.
 * idx_k_in: device fp32 [B, T, di] or NULL; when given it is written to the
 *           same rows' indexer key: E4M3 as csa2_fp8_quant casts, or MXFP4:
 *           per 32 channels the E8M0 scale code is max(E - 2, 0) where E is
 *           the biased exponent field of the block's fp32 amax (the OCP
 *           Microscaling rule 2^(floor(log2 amax) - 2)), and each code is
 *           E2M1(x / scale) (RNE, saturating at 6, sign copied).
 * Row i of sequence b lands at position p = seq_len[b] + i: channels D-R+2j
 * and D-R+2j+1 are rotated by (c, s) = (rope_cos, rope_sin)[p][j] as
 * y0 = x0*c - x1*s, y1 = x0*s + x1*c in fp32 with one rounding per operation;
 * per group of 16 channels the scale byte is E4M3(amax/6) (correctly rounded
 * fp32 division, RNE, saturating) and each code is E2M1(y/scale) (RNE,
 * saturating, sign copied), all codes 0 when the scale decodes to 0.
 * Afterwards seq_len[b] += T.  A row with p >= max_len is skipped and sets
 * CSA2_DEV_OVERFLOW.
 * Ordering: appends are launched so that they may start while the previous
 * kernel on the stream finishes, when that kernel allows its dependents to
 * launch early (the library's own kernels do).  They read kv / idx_k_in
 * before waiting for it; small appends (decode sizes) also write the new rows
 * before the wait, large ones write them after reading seq_len behind the
 * wait; seq_len is updated only after the previous kernel completes.  The
 * kernel just before this call must therefore not write kv or idx_k_in after
 * allowing early launch (kernels that do not use programmatic launch never
 * overlap it).
 */
csa2_status csa2_quant_append(const csa2_cache *cache, const float *kv, const float *idx_k_in,
                              int32_t T, void *ws, void *stream);

/*
 * Step 1 for an encoder cache (compression ratio m = 2): entry i of sequence
 * b combines source rows 2i and 2i+1 and is appended at entry position
 * p = seq_len[b] + i ("DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
 * Compression" knowledge note, symbol table (m = 2 in the encoder; Z_l the
 * weight used when forming a compressed entry) and "Causal Encoder-Decoder";
 * "Inside DeepSeek V4.1 Flash: CED, CSA2 and the 890-Byte KV Cache", "CSA2:
 * reuse memory and reuse selection independently": non-overlapping groups,
 * no positional embedding).  The pages do not print the combination; this
 * library takes a per-channel softmax of the two logits:
 *   d = z1 - z0, t = e^-|d| (0 when |d| > 80), s = 1 + t,
 *   the larger logit's row gets 1/s, the other t/s, c = w0 x0 + w1 x1,
 * every operation one fp32 rounding (e^x by Cody-Waite reduction with ln 2 =
 * 2839/4096 + (ln 2 - 2839/4096), then Horner on the degree-7 Taylor
 * polynomial, times 2^k).  The entry is then rotated at p and quantised
 * exactly as csa2_quant_append does.
 * kv, z:    device fp32 [B, 2T, D] source rows before rotation and their
 *           compression logits, 16-byte aligned.
 * idx_k_in: device fp32 [B, T, di] (one indexer key per entry) or NULL.
 * Afterwards seq_len[b] += T (entries).  Errors and ordering (kv, z and
 * idx_k_in read before the previous kernel completes) as csa2_quant_append.
 */
csa2_status csa2_quant_append_pairs(const csa2_cache *cache, const float *kv, const float *z,
                                    const float *idx_k_in, int32_t T, void *ws, void *stream);

/*
 * Steps 2-3, Full layer: score every visible position and select.
 * q_idx:    device E4M3 [B, Tq, Hi, di] indexer queries.
 * w:        device fp32 [B, Tq, Hi] head weights.
 * Hi:       indexer heads, 1..64.
 * q_pos:    device int32 [B, Tq] inclusive causal limit per query, or NULL for
 *           decode (visible = [0, seq_len[b])).
 * batch_ids, n_batch: device int32 subset of sequences to process, or NULL
 *           with n_batch = B.
 * k:        1..CSA2_MAX_TOPK.
 * Score of position t: s_t = sum_h w_h * max(0, q_h . k_t) (fp32 accumulate);
 * with MXFP4 keys k_t is the E2M1 code times its block's E8M0 scale (the
 * tensor cores apply the scale per 32 channels).
 * Outputs (only rows of the processed sequences are written):
 *   out_idx     [B, Tq, k]  int32 positions of the top min(k, visible) scores
 *                           ranked by (score desc, position asc), written in
 *                           ascending position order; cnt entries used
 *   out_cnt     [B, Tq]     int32
 *   pool_blocks [B, Tq, CSA2_POOL_BLOCKS] int32 or NULL: block ids b (positions
 *                           8b..8b+7) of the min(2048, ceil(visible/8)) blocks
 *                           with the largest block maximum (ties: lower id),
 *                           ascending
 *   pool_cnt    [B, Tq]     int32 or NULL
 */
csa2_status csa2_index_full(const csa2_cache *cache, const uint8_t *q_idx, const float *w,
                            int32_t Hi, int32_t Tq, const int32_t *q_pos,
                            const int32_t *batch_ids, int32_t n_batch, int32_t k,
                            int32_t *out_idx, int32_t *out_cnt, int32_t *pool_blocks,
                            int32_t *pool_cnt, void *ws, void *stream);

/*
 * csa2_index_full without a caller workspace.  The paper has no counterpart:
 * this entry point exists for callers that may not allocate device memory --
 * an engine that hands this library only the buffers it reserved for it at
 * start-up, or a latency-critical loop that cannot afford cudaMalloc's
 * implicit synchronisation.  Arguments and results are those of
 * csa2_index_full, with `ws` replaced by:
 *   status: device (or pinned host) uint32, 4-byte aligned, or NULL; receives
 *           this call's device status word (CSA2_DEV_* bits), stream ordered.
 * The scratch is one fixed array of CSA2_NOALLOC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads the library's device code until the
 * process exits; the call allocates no memory (no cudaMalloc, no library
 * allocator).  With S = max_len rounded up to 128 and M = S/8 rounded up to
 * 32, a call on rows = n_batch*Tq query rows needs about
 * rows*(4*S + 4*M + 65536) + 1024 bytes (each part rounded up to 256 B),
 * e.g. 32 rows at max_len 131,136 need 21 MB and one row at CSA2_MAX_LEN
 * needs 9.5 MB; larger requests return CSA2_ERR_UNSUPPORTED with nothing
 * launched.
 * The first call on a device looks up the array's device address (and may
 * load the library's device code there); make that first call before any
 * stream capture.  Every call on a device shares the array and finds the
 * previous call's contents in it; each call clears the status word it needs
 * at zero.  Calls whose GPU work overlaps (other streams, unordered threads)
 * race on the array: order them on one stream.
 */
#define CSA2_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
csa2_status csa2_index_full_noalloc(const csa2_cache *cache, const uint8_t *q_idx,
                                    const float *w, int32_t Hi, int32_t Tq, const int32_t *q_pos,
                                    const int32_t *batch_ids, int32_t n_batch, int32_t k,
                                    int32_t *out_idx, int32_t *out_cnt, int32_t *pool_blocks,
                                    int32_t *pool_cnt, uint32_t *status, void *stream);

/*
 * Steps 2-3, Reindex layer: score only the pool's visible positions with this
 * layer's own indexer query and select its top-k (same ranking and output
 * order as csa2_index_full).  pool_blocks [B, Tq, CSA2_POOL_BLOCKS] must be
 * ascending block ids (as csa2_index_full writes them); pool_cnt [B, Tq].
 * A block id past the visible blocks sets CSA2_DEV_BAD_POOL and is skipped.
 */
csa2_status csa2_index_reindex(const csa2_cache *cache, const uint8_t *q_idx, const float *w,
                               int32_t Hi, int32_t Tq, const int32_t *q_pos,
                               const int32_t *pool_blocks, const int32_t *pool_cnt,
                               const int32_t *batch_ids, int32_t n_batch, int32_t k,
                               int32_t *out_idx, int32_t *out_cnt, void *ws, void *stream);

/*
 * Steps 4-5, decode: for each sequence b and head h,
 *   o = sum_j softmax_j(scale * q_h . x_j) * x_j
 * over j = the cnt[b] selected global rows idx[b][0..cnt) (dequantised
 * E2M1 x E4M3) followed by the swa_cnt[b] window rows swa[b][0..swa_cnt)
 * (E4M3 per element, no scale).  K = V = the dequantised row (value width D).
 * q:    device bf16 bits [B, H, D], already rotated; H <= 64.
 * idx:  device int32 [B, kcap]; cnt: device int32 [B] (clamped to kcap).
 * swa:  device E4M3 [B, W, D]; swa_cnt: device int32 [B] or NULL (= W).
 * softmax_scale <= 0 selects 1/sqrt(D).  out: device fp32 [B, H, D],
 * 16-byte aligned.
 * A row with no keys gives zeros.  An index outside [0, seq_len[b]) sets
 * CSA2_DEV_BAD_INDEX and is left out of the softmax.
 * When the SMs outnumber the query rows, the keys of a row are split over a
 * thread-block cluster of up to 8 CTAs whose partial results are merged in
 * distributed shared memory; the workspace holds no partial outputs.
 * Ordering: the kernel may start while the previous kernel on the stream
 * finishes, when that kernel allows its dependents to launch early (the
 * library's own kernels do), and copies q before waiting for it; idx, cnt,
 * seq_len and the cache rows are read only after it completes.  The kernel
 * just before this call must therefore not write q after allowing early
 * launch.
 */
csa2_status csa2_attn_decode(const csa2_cache *cache, const uint16_t *q, int32_t H,
                             const int32_t *idx, const int32_t *cnt, int32_t kcap,
                             const uint8_t *swa, const int32_t *swa_cnt, int32_t W,
                             float softmax_scale, float *out, void *ws, void *stream);

/*
 * Steps 4-5, decode, for L layers that attend over the same selection of the
 * same cache: the CSA2 groups of "DeepSeek-V4.1-Flash: Pushing the Limits of
 * KV Cache Compression" (knowledge note, section "CSA2: share cache, refresh
 * selection only when needed"), where the Reuse layers that follow a Full or
 * Reindex layer take its top-k unchanged.  Layer l gives exactly what
 * csa2_attn_decode(cache, q[l], H, idx, cnt, kcap, swa[l], swa_cnt, W,
 * softmax_scale, out[l], ws, stream) gives; one launch serves all L layers, so
 * each (layer, sequence) row gets fewer split-K CTAs (none, when L * B rows
 * fill the SMs) and the launch's fixed costs are paid once.
 * L: 1..CSA2_MAX_ATTN_LAYERS.  q, swa, out: HOST arrays of L device pointers
 * with the layouts of csa2_attn_decode; idx, cnt, swa_cnt shared.  L * B must
 * not exceed 65,535.  Errors and ordering as csa2_attn_decode.
 */
csa2_status csa2_attn_decode_layers(const csa2_cache *cache, int32_t L, const uint16_t *const *q,
                                    int32_t H, const int32_t *idx, const int32_t *cnt,
                                    int32_t kcap, const uint8_t *const *swa,
                                    const int32_t *swa_cnt, int32_t W, float softmax_scale,
                                    float *const *out, void *ws, void *stream);

/*
 * Steps 4-5, prefill chunk: as csa2_attn_decode for Tq query rows per
 * sequence.  q: bf16 [B, Tq, H, D]; q_pos [B, Tq] positions (visible global
 * positions are <= q_pos); idx [B, Tq, kcap]; cnt [B, Tq].
 * swa: E4M3 band [B, Tq + W - 1, D]; band row r holds position
 * q_pos[b][0] - (W - 1) + r, and query tq attends to band rows tq .. tq+W-1
 * whose positions are >= 0 (the W most recent positions up to itself).
 * out: fp32 [B, Tq, H, D], 16-byte aligned.  Ordering as csa2_attn_decode.
 */
csa2_status csa2_attn_prefill(const csa2_cache *cache, const uint16_t *q, int32_t H, int32_t Tq,
                              const int32_t *q_pos, const int32_t *idx, const int32_t *cnt,
                              int32_t kcap, const uint8_t *swa, int32_t W, float softmax_scale,
                              float *out, void *ws, void *stream);

/* Copies the device status word to *host_status after the stream drains.
 * Returns CSA2_ERR_DEVICE when any bit is set. */
csa2_status csa2_get_status(void *ws, uint32_t *host_status, void *stream);

/* Clears the device status word (stream ordered). */
csa2_status csa2_reset_status(void *ws, void *stream);

/*
 * Optional instrumentation for benchmarks: while set, the main kernel of the
 * given family is bracketed by cudaEventRecord(begin) / cudaEventRecord(end)
 * on the stream of the call that launches it.  Families:
 *   CSA2_KERNEL_QUANT (step 1), CSA2_KERNEL_INDEXER (step 2),
 *   CSA2_KERNEL_SELECT (step 3), CSA2_KERNEL_ATTENTION (steps 4-5).
 * begin/end are cudaEvent_t passed as void*; NULL/NULL turns it off.  While
 * the stream is being captured the records are external
 * (cudaEventRecordExternal): event nodes that time every replay of the graph.
 * Process-wide setting, not thread safe; it does not change any result.
 */
#define CSA2_KERNEL_QUANT 0
#define CSA2_KERNEL_INDEXER 1
#define CSA2_KERNEL_SELECT 2
#define CSA2_KERNEL_ATTENTION 3
csa2_status csa2_set_launch_events(int32_t family, void *begin, void *end);

/* Time after which a bounded on-chip wait of the kernels gives up, in
 * nanoseconds (default 2e9: two seconds); 0 restores the default.
 * The indexer and attention kernels keep their pipeline stages in step with
 * mbarriers.  Each wait on one is bounded by the GPU's global timer.  When a
 * wait runs out the kernel stops its pipeline, sets CSA2_DEV_TIMEOUT in the
 * workspace status word, waits for the copies and MMAs it has already
 * started, frees its tensor memory and returns.  No data computed by that
 * launch may be used.  This call exists so that tests can make a wait run out
 * on an ordinary launch.  It sets the limit for the current device and
 * affects kernels launched after it returns.  It synchronises with the
 * device, and it is not thread safe.  Errors: CSA2_ERR_CUDA when the device
 * copy fails.  No counterpart on the pages (an implementation safety limit). */
csa2_status csa2_set_wait_limit(uint64_t ns);

/* Static string for a status code. */
const char *csa2_status_string(csa2_status status);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */
