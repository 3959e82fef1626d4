"""The CSA2 hot path, step by step, as plain numpy (oracle side).

Pages followed (titles and sections):

[KN]  "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
      (knowledge note): "CSA2: share cache, refresh selection only when
      needed" (mode table), "Hierarchical Sparse Indexer: make later searches
      bounded", "FP4 main KV: trade precision for bytes, not for a new GEMM",
      "Putting It Together" (steps 5-8 of the request trace).
[ID]  "Inside DeepSeek V4.1 Flash: CED, CSA2 and the 890-Byte KV Cache":
      "CSA2: reuse memory and reuse selection independently", "Hierarchical
      indexing bounds later searches, not every search", "Reconstructing the
      890-byte cache budget".
[MT]  "DeepSeek-V4.1-Flash：把 KV 缓存压缩从“算法点”推进为“部署系统”":
      section "3. FP4 主 KV" (quantised after RoPE, dequantised before
      attention, SWA kept in FP8).
[EB]  "The 890-Byte Token - DeepSeek-V4.1 Flash's Elegant KV Cache
      Optimizations": "FP4 main KV cache" (range after normalisation),
      "Hierarchical Sparse Indexer".

Readings of points the pages leave open:

* RoPE rotates the last ``rope_dim`` channels in interleaved pairs
  (2i, 2i+1) with angle p * theta**(-2i/rope_dim); the cos/sin table is an
  fp32 input; each output takes two fp32 products and one fp32 add/sub, each
  rounded once (no fused multiply-add).
* FP4 scale = E4M3(RNE(amax / 6)) with a correctly rounded fp32 division; a
  zero scale gives all-zero codes; codes = E2M1(RNE(y / scale)); element 2j
  in the low nibble of byte j.
* Indexer score s_t = sum_h w_h * max(0, q_h . k_t) over E4M3 operands, no
  extra constant factor.
* MXFP4 indexer key (the alternative key format): per block of 32 channels
  the E8M0 scale is 2^(floor(log2 amax) - 2), the OCP Microscaling rule
  (E2M1's largest binade has exponent 2), clamped below at 2^-127 (code 0,
  also used for an all-zero block); codes = E2M1(RNE(x / scale)), saturating
  at 6, sign copied, packed like the main-KV codes.  The query stays E4M3.
* Ranking order for top-k and for the pool: larger score first, lower index
  on equal scores.  The pool keeps min(2048, ceil(N/8)) blocks of 8
  positions ranked by block maximum.  Outputs are sorted ascending.
* Attention: one softmax over the selected global rows followed by the SWA
  rows (no de-duplication), K = V = the dequantised row, logit scale
  1/sqrt(D) unless given.
"""
from __future__ import annotations

import math

import numpy as np

from .formats import (E8M0_BIAS, e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode,
                      e8m0_decode)

GROUP = 16          # channels per E4M3 scale of the main-KV format
MX_BLOCK = 32       # channels per E8M0 scale of the MXFP4 indexer key
E2M1_EMAX = 2       # exponent of E2M1's largest binade (4 <= |v| <= 6)
BLOCK = 8           # positions per pool block
POOL_BLOCKS = 2048  # pool capacity in blocks


# ---------------------------------------------------------------- step 1: RoPE
def rope_rotate(x, pos, cos_tab, sin_tab, rope_dim):
    """Rotate the last ``rope_dim`` channels of fp32 rows ``x`` [n, D] at positions ``pos``.

    [KN] "FP4 main KV": the cache is quantised after RoPE; [MT] "3. FP4 主 KV".
    Pair i is (D-R+2i, D-R+2i+1); with (c, s) = table[pos, i]:
    y0 = x0*c - x1*s,  y1 = x0*s + x1*c  (fp32, one rounding per operation).
    Pinned: identity at position 0, exact rotation of unit vectors, norm kept
    within fp32 rounding, agreement with complex multiplication in fp64.
    """
    x = np.asarray(x, dtype=np.float32)
    y = x.copy()
    if rope_dim == 0:
        return y
    d = x.shape[-1]
    pos = np.asarray(pos, dtype=np.int64)
    c = np.asarray(cos_tab, dtype=np.float32)[pos]
    s = np.asarray(sin_tab, dtype=np.float32)[pos]
    x0 = x[:, d - rope_dim::2]
    x1 = x[:, d - rope_dim + 1::2]
    y[:, d - rope_dim::2] = (x0 * c) - (x1 * s)
    y[:, d - rope_dim + 1::2] = (x0 * s) + (x1 * c)
    return y


# ------------------------------------------------------- step 1: FP4 quantise
def quantize_fp4(y):
    """Post-RoPE fp32 rows [n, D] -> (codes uint8 [n, D/2], scales uint8 [n, D/16]).

    [KN] "FP4 main KV": E2M1 values, one E4M3 scale per 16 channels, no second
    global scale; [ID] "Reconstructing the 890-byte cache budget": 512 x 4/8 +
    512/16 bytes per entry.
    For each group of 16 channels: amax = max|y|; scale code = E4M3(amax/6);
    s = value of that code; codes = E2M1(y/s), or all zero when s == 0.
    Pinned: zero groups, exact power-of-two groups, saturation, the per-element
    error bound of the E2M1 grid, byte counts of the pages.
    """
    y = np.asarray(y, dtype=np.float32)
    n, d = y.shape
    g = y.reshape(n, d // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1)
    scale_code = e4m3_encode(amax / np.float32(6.0))
    s = e4m3_decode(scale_code).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = g / s[..., None]
    codes = e2m1_encode(np.where(s[..., None] == 0, np.float32(0.0), q))
    codes = np.where(s[..., None] == 0, np.uint8(0), codes).reshape(n, d)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scale_code.astype(np.uint8)


def dequantize_fp4(codes, scales, dim):
    """(codes [n, D/2], scales [n, >= D/16]) -> float64 rows [n, D].

    [KN] "Putting It Together", step 8: FP4 blocks are dequantised when
    attention needs them.  x = E2M1(code) * E4M3(scale of the channel's group).
    """
    codes = np.asarray(codes, dtype=np.uint8)[:, : dim // 2]
    lo = e2m1_decode(codes & 0xF)
    hi = e2m1_decode(codes >> 4)
    v = np.empty((codes.shape[0], dim), dtype=np.float64)
    v[:, 0::2] = lo
    v[:, 1::2] = hi
    s = e4m3_decode(np.asarray(scales, dtype=np.uint8)[:, : dim // GROUP])
    return v * np.repeat(s, GROUP, axis=1)


def quant_append_rows(kv, pos, cos_tab, sin_tab, rope_dim):
    """Pre-RoPE fp32 rows and their positions -> the bytes appended to the cache."""
    return quantize_fp4(rope_rotate(kv, pos, cos_tab, sin_tab, rope_dim))


# ------------------------------------------ step 1b: m = 2 pair compression
# The exponential of the pair weights, written out so that every operation is
# one fp32 rounding (Cody-Waite range reduction, then the Taylor series of
# e^r to degree 7): the kernels evaluate the same sequence, so the compressed
# rows -- and the FP4 codes they decide -- agree bit for bit.
INV_LN2 = np.float32(1.0 / math.log(2.0))
LN2_HI = np.float32(2839.0 / 4096.0)                 # 12 significant bits: k * LN2_HI is exact
LN2_LO = np.float32(math.log(2.0) - 2839.0 / 4096.0)
EXP_TAYLOR = [np.float32(1.0 / math.factorial(i)) for i in range(8)]
EXP_MIN = np.float32(-80.0)                          # below: e^x is taken as 0


def exp_neg_f32(x):
    """e^x for fp32 x <= 0, one fp32 rounding per operation; 0 below -80.

    k = rint(x / ln 2); r = (x - k ln2_hi) - k ln2_lo; e^r by Horner on the
    degree-7 Taylor polynomial; times 2^k (exact: k >= -116 keeps it normal).
    Pinned: within 4 ulp of e^x across [-80, 0], exactly 1 at 0.
    """
    x = np.asarray(x, dtype=np.float32)
    xc = np.maximum(x, EXP_MIN)          # below the cut the result is 0 anyway
    k = np.rint(xc * INV_LN2).astype(np.float32)
    r = (xc - k * LN2_HI) - k * LN2_LO
    p = EXP_TAYLOR[7]
    for c in EXP_TAYLOR[6::-1]:
        p = p * r + c
    t = np.ldexp(p, k.astype(np.int32)).astype(np.float32)
    return np.where(x < EXP_MIN, np.float32(0.0), t).astype(np.float32)


def pair_weights(z0, z1):
    """Per-channel softmax of the two compression logits of a pair (fp32).

    [KN] "Causal Encoder-Decoder" and the symbol table: Z_l is the weight used
    when forming a compressed global KV entry; [ID] "CSA2: reuse memory and
    reuse selection independently": CSA2 groups non-overlapping source
    positions and drops the compressor's positional embedding.  The pages do
    not print the combination; the reading is a softmax of Z over the group's
    positions, channel by channel.  With d = z1 - z0 and t = e^-|d|:
    the larger logit gets 1 / (1 + t), the other t / (1 + t).
    Pinned: equal logits give exactly (1/2, 1/2); the weights sum to 1 within
    1 ulp; swapping the pair swaps them; far-apart logits select one row.
    """
    z0 = np.asarray(z0, dtype=np.float32)
    z1 = np.asarray(z1, dtype=np.float32)
    d = z1 - z0
    t = exp_neg_f32(-np.abs(d))
    s = np.float32(1.0) + t
    big = np.float32(1.0) / s
    small = t / s
    w1 = np.where(d >= 0, big, small).astype(np.float32)
    w0 = np.where(d >= 0, small, big).astype(np.float32)
    return w0, w1


def compress_pairs(kv, z):
    """Source rows [2T, D] and their logits [2T, D] -> T compressed rows (fp32).

    Entry j combines source positions 2j and 2j+1 (m = 2, the encoder's
    ratio, [KN] symbol table): c = w0 * x0 + w1 * x1 per channel, two fp32
    products and one fp32 sum.  The entry is then rotated at its compressed
    position j and quantised like any main-KV row.
    """
    kv = np.asarray(kv, dtype=np.float32)
    z = np.asarray(z, dtype=np.float32)
    w0, w1 = pair_weights(z[0::2], z[1::2])
    return (w0 * kv[0::2] + w1 * kv[1::2]).astype(np.float32)


def fp8_cast(x):
    """fp32 -> E4M3 codes (SWA rows, indexer keys and queries)."""
    return e4m3_encode(x)


def quantize_mxfp4(x):
    """fp32 indexer-key rows [n, d] -> (codes uint8 [n, d/2], E8M0 scales uint8 [n, d/32]).

    [ID] "Reconstructing the 890-byte cache budget": the indexer key keeps
    32-channel groups with E8M0 scales, 128 x 4/8 + 128/32 = 68 bytes;
    "How the derived numbers were built": MXFP4, one scale per 32.
    Per block: amax = max|x|; e = floor(log2 amax) - 2 (the OCP Microscaling
    shared-exponent rule for E2M1), at least -127; scale = 2^e (code e + 127);
    codes = E2M1(x / scale) (RNE, saturating, sign copied).  An all-zero block
    takes code 0.  x / scale is exact (a power-of-two division of an fp32
    value, computed in fp64).
    Pinned: the exponent against the fp32 bit pattern, saturation between 6
    and 8 times the scale, grid values reproduced exactly, the per-element
    error bound, zero and tiny blocks, the pages' byte count.
    """
    x = np.asarray(x, dtype=np.float32)
    n, d = x.shape
    g = x.reshape(n, d // MX_BLOCK, MX_BLOCK).astype(np.float64)
    amax = np.max(np.abs(g), axis=-1)
    _, ex = np.frexp(amax)                  # amax = m * 2^ex, 0.5 <= m < 1
    e = np.where(amax > 0, ex - 1 - E2M1_EMAX, -E8M0_BIAS)
    e = np.maximum(e, -E8M0_BIAS)
    scale = np.ldexp(1.0, e)
    codes = e2m1_encode(g / scale[..., None]).reshape(n, d)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, (e + E8M0_BIAS).astype(np.uint8)


def dequantize_mxfp4(codes, scales, dim):
    """(codes [n, d/2], E8M0 scales [n, d/32]) -> float64 rows [n, d]."""
    codes = np.asarray(codes, dtype=np.uint8)[:, : dim // 2]
    v = np.empty((codes.shape[0], dim), dtype=np.float64)
    v[:, 0::2] = e2m1_decode(codes & 0xF)
    v[:, 1::2] = e2m1_decode(codes >> 4)
    s = e8m0_decode(np.asarray(scales, dtype=np.uint8)[:, : dim // MX_BLOCK])
    return v * np.repeat(s, MX_BLOCK, axis=1)


# -------------------------------------------------------- step 2: indexer score
def indexer_scores(q_codes, w, k_codes):
    """Lightning-indexer scores of one query against key rows (fp64).

    [KN] "Hierarchical Sparse Indexer"; [ID] "Hierarchical indexing bounds
    later searches".  s_t = sum_h w_h * max(0, sum_d q[h,d] k[t,d]) with
    q, k decoded from E4M3.  The inner products are exact in fp64 (products
    of two E4M3 values have at most 8 significant bits and 128 of them sum
    well inside 53 bits).
    Pinned: with one head and w = 1 it equals ReLU(q.k) computed in exact
    rational arithmetic.
    """
    q = e4m3_decode(q_codes).reshape(len(w), -1)
    k = e4m3_decode(k_codes).reshape(-1, q.shape[1])
    return indexer_scores_values(q, w, k)


def indexer_scores_values(q, w, k):
    """s_t = sum_h w_h * max(0, q_h . k_t) for decoded q [Hi, di] and keys k [n, di] (fp64).

    Shared by both key formats: the E4M3 keys above and the MXFP4 keys
    (decoded by dequantize_mxfp4).  Every product is exact in fp64 (at most
    6 significant bits times a power of two); with MXFP4 keys whose blocks sit
    at very different scales the fp64 sum itself may round.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64).reshape(-1, q.shape[1])
    dots = k @ q.T
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)


def block_maxima(scores):
    """Per 8-position block: max score over the positions that exist."""
    scores = np.asarray(scores, dtype=np.float64)
    n = len(scores)
    nb = -(-n // BLOCK)
    pad = np.full(nb * BLOCK, -np.inf)
    pad[:n] = scores
    return pad.reshape(nb, BLOCK).max(axis=1)


# ------------------------------------------------------------ step 3: selection
def topk(scores, k, ids=None):
    """The k best ids by (score descending, id ascending), returned ascending."""
    scores = np.asarray(scores, dtype=np.float64)
    ids = np.arange(len(scores)) if ids is None else np.asarray(ids)
    k = min(k, len(scores))
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    order = np.lexsort((ids, -scores))
    return np.sort(ids[order[:k]]).astype(np.int64)


def full_select(scores, k, pool_blocks=POOL_BLOCKS):
    """Full layer: top-k positions and the block pool.

    [KN] "Hierarchical Sparse Indexer": the first Full indexer scores all
    positions and block maxima select a shared pool; [ID] "Hierarchical
    indexing": up to 2,048 blocks of eight positions, at most 16,384
    candidates.  Returns (idx ascending, pool block ids ascending).
    """
    n = len(scores)
    idx = topk(scores, k)
    bm = block_maxima(scores)
    pool = topk(bm, min(pool_blocks, len(bm)))
    return idx, pool


def pool_positions(pool, n):
    """Positions covered by the pool blocks that are < n, ascending."""
    pool = np.asarray(pool, dtype=np.int64)
    pos = (pool[:, None] * BLOCK + np.arange(BLOCK)[None, :]).reshape(-1)
    return pos[pos < n]


def reindex_select(q_codes, w, k_codes_of, pool, n, k):
    """Reindex layer: own indexer query over the pool's positions only.

    [KN] "CSA2" mode table (Reindex reuses main KV and indexer K, computes a
    new indexer Q and a fresh top-k) and "Hierarchical Sparse Indexer" (later
    Reindex layers score only the pool).  ``k_codes_of(positions)`` returns
    the E4M3 indexer-key rows of those positions.
    """
    pos = pool_positions(pool, n)
    s = indexer_scores(q_codes, w, k_codes_of(pos))
    return topk(s, k, ids=pos)


# --------------------------------------------------- steps 4-5: attention
def sparse_attention(q, rows, scale=None):
    """One softmax over ``rows`` (selected global rows then SWA rows), K = V = rows.

    [KN] "CSA2" (every mode computes its own Q and SWA path) and "Putting It
    Together" step 7 (sparse attention with local SWA); [ID] "CSA2: reuse
    memory and reuse selection independently" (the query attends to the
    selected entries together with the local window).
    q: float64 [H, D]; rows: float64 [n, D].  Output float64 [H, D]; n == 0
    gives zeros.  Pinned: equals dense attention when every row is selected;
    one row gives that row; equal logits give the mean; invariant to adding a
    constant to every logit.
    """
    q = np.asarray(q, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(q.shape[1])
    if rows.shape[0] == 0:
        return np.zeros_like(q)
    logits = scale * (q @ rows.T)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    return (p @ rows) / p.sum(axis=1, keepdims=True)


def swa_rows_decode(swa_codes):
    """FP8 SWA rows -> float64 (plain per-element E4M3, no scale)."""
    return e4m3_decode(swa_codes)


def swa_band_rows(p0, tq, window):
    """Rows of a prefill chunk's SWA band that query ``tq`` attends.

    [KN] "Putting It Together": every query also attends its local sliding
    window of the most recent positions.  The chunk's queries sit at
    positions p0 .. p0+T-1 and share one band of T+W-1 FP8 rows, row r
    holding position p0-(W-1)+r.  Query tq at position p = p0+tq sees the
    window positions max(0, p-W+1) .. p, i.e. band rows
    max(tq, W-1-p0) .. tq+W-1 (rows of negative positions are skipped).
    Pinned against a brute-force walk over the positions each query sees.
    """
    lo = max(tq, (window - 1) - p0)
    return np.arange(lo, tq + window, dtype=np.int64)
