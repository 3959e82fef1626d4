"""Bit-exact GPU check of the main-KV FP4 append on the format's edges.

"DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", section
"FP4 main KV: trade precision for bytes, not for a new GEMM": each post-RoPE
row is stored as E2M1 values with one E4M3 scale per 16 channels and no
global scale.  The seeded workload rows never reach the corners of that
format, so these rows are built by hand:

* an all-zero group, an all -0.0 group, tiny negatives next to a unit amax
  (sign-kept zero code 0x8);
* groups whose amax is 6 * 2^e for every e in [-9, 8] (exact scales);
* amax 2,688, 2,689 and 1e6 (scale saturation at 448, codes clamped at 6);
* amax / 6 in the E4M3 subnormal range, including the tie that rounds to a
  zero scale;
* elements whose quotient y / s is exactly an E2M1 midpoint (0.25, 0.75,
  1.25, 1.75, 2.5, 3.5, 5) or one fp32 ulp either side, at several scales;
* rows appended at position 0 and at position max_len - 1, with edge values
  in the rotated channels too.

The append kernels are covered: one large append (the streaming kernel),
then decode appends of one row per sequence (the cluster kernel), on a
contiguous and on a paged cache; and a large append whose cos / sin rows
cannot be bulk-copied (the per-thread kernel).  Codes and scale
bytes are compared with the oracle's quantiser bit for bit; the indexer-key
bytes written by the same calls are compared with the oracle's E4M3 cast.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle import formats as F  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import Workload  # noqa: E402

D, R, DI = 576, 64, 128
MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)


def _group_mids(scale, nudge):
    """16 values at one scale: +-6*scale (the amax, so the scale code is exact)
    and the seven midpoints times the scale, each moved by `nudge` ulps."""
    v = MIDS * np.float32(scale)
    if nudge > 0:
        v = np.nextafter(v, np.float32(np.inf))
    elif nudge < 0:
        v = np.nextafter(v, np.float32(0.0))
    g = np.concatenate([[6.0 * scale], v, -v, [-6.0 * scale]]).astype(np.float32)
    return g


def edge_groups(rng):
    """A list of 16-channel groups (fp32) that reach the format's corners."""
    groups = [np.zeros(16, np.float32), np.full(16, -0.0, np.float32)]
    tiny = np.full(16, -1e-30, np.float32)
    tiny[0] = 1.0
    tiny[1] = 1e-30
    groups.append(tiny)
    for e in range(-9, 9):                       # exact scales 2^e
        g = rng.uniform(-1.0, 1.0, 16).astype(np.float32) * np.float32(6.0 * 2.0 ** e)
        g[rng.integers(16)] = np.float32(6.0 * 2.0 ** e) * (1 if e % 2 else -1)
        groups.append(g)
    for amax in (2688.0, 2689.0, 1e6, 1e30):    # saturation
        g = rng.uniform(-1.0, 1.0, 16).astype(np.float32) * np.float32(amax)
        g[3] = np.float32(-amax)
        groups.append(g)
    for m in (7.0, 5.0, 3.0, 2.0, 1.5, 1.0, 0.75, 0.5, 0.49, 0.25):   # amax / 6 = m * 2^-9
        g = rng.uniform(-1.0, 1.0, 16).astype(np.float32) * np.float32(6.0 * m * 2.0 ** -9)
        g[5] = np.float32(6.0 * m * 2.0 ** -9)
        groups.append(g)
    for scale in (1.0, 0.5, 1.125, 2.0 ** -9, 3.0 * 2.0 ** -9, 448.0, 0.875 * 2.0 ** -6):
        for nudge in (0, 1, -1):
            groups.append(_group_mids(scale, nudge))
    return groups


def edge_rows(rng, n):
    """n rows of D channels: the edge groups laid over the first D - R
    channels (which RoPE leaves as they are), normal values elsewhere; every
    fourth row and the last row also carry edge groups in the rotated
    channels (unchanged at position 0, rotated elsewhere)."""
    groups = edge_groups(rng)
    rows = rng.standard_normal((n, D)).astype(np.float32)
    gi = 0
    for r in range(n):
        for g in range((D - R) // 16):
            rows[r, 16 * g: 16 * g + 16] = groups[gi % len(groups)]
            gi += 1
        if r % 4 == 0 or r == n - 1:
            for g in range((D - R) // 16, D // 16):
                rows[r, 16 * g: 16 * g + 16] = groups[gi % len(groups)]
                gi += 1
    return rows


def idx_edge_rows(rng, n):
    """Indexer-key rows around the E4M3 grid: midpoints, saturation, tiny."""
    fin = F.e4m3_decode(np.arange(0x7F)).astype(np.float32)
    mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)
    pool = np.concatenate([mids, np.nextafter(mids, np.float32(0)), fin,
                           [0.0, -0.0, 448.0, 464.0, 1e6, 1e-12]]).astype(np.float32)
    x = rng.choice(pool, size=(n, DI)).astype(np.float32)
    return x * rng.choice(np.array([1.0, -1.0], np.float32), size=(n, DI))


def read_rows(cache, b, positions):
    ix = torch.tensor([cache.physical_row(b, int(t)) for t in positions], dtype=torch.long,
                      device="cuda")
    return (cache.codes.index_select(0, ix).cpu().numpy()[:, : D // 2],
            cache.scales.index_select(0, ix).cpu().numpy()[:, : D // 16],
            cache.idx_k.index_select(0, ix).cpu().numpy()[:, :DI])


@pytest.mark.parametrize("page", [0, 64], ids=["contiguous", "paged64"])
def test_main_kv_quantiser_edges_bit_exact(page):
    n_big = 256
    wl = Workload(f"quant-edges-p{page}", 2, [n_big, n_big], D, R, 64, DI, 64, 64, 128,
                  seed=71, page_size=page)
    dw = DeviceWorkload(wl, build_cache=False)
    L = wl.max_len
    rng = np.random.default_rng(71 + page)
    kv = [edge_rows(rng, L) for _ in range(wl.batch)]
    ik = [idx_edge_rows(rng, L) for _ in range(wl.batch)]
    # one large append per sequence (the grid kernel): positions 0 .. n_big-1
    for b in range(wl.batch):
        K.quant_append(dw.seq_view(b), torch.from_numpy(kv[b][:n_big]).cuda(),
                       torch.from_numpy(ik[b][:n_big]).cuda(), n_big, dw.ws)
    # decode appends, one row of every sequence per call (the cluster kernel),
    # up to the last position max_len - 1
    for t in range(n_big, L):
        K.quant_append(dw.cache, torch.from_numpy(np.stack([kv[b][t] for b in range(wl.batch)])).cuda(),
                       torch.from_numpy(np.stack([ik[b][t] for b in range(wl.batch)])).cuda(), 1, dw.ws)
    torch.cuda.synchronize()
    assert K.get_status(dw.ws) == 0
    for b in range(wl.batch):
        assert int(dw.cache.seq_len[b]) == L
        pos = np.arange(L)
        codes, scales, idxk = read_rows(dw.cache, b, pos)
        rc, rs = O.quant_append_rows(kv[b], pos, dw.rope_cos, dw.rope_sin, R)
        bad = np.nonzero(np.any(codes != rc, axis=1) | np.any(scales != rs, axis=1))[0]
        assert len(bad) == 0, f"b={b}: {len(bad)} rows differ, first at position {bad[:4]}"
        assert np.array_equal(idxk, O.fp8_cast(ik[b])), b
    # the edges were actually reached
    _, rs = O.quant_append_rows(kv[0], np.arange(L), dw.rope_cos, dw.rope_sin, R)
    assert (rs == 0x7E).any() and (rs == 0).any() and ((rs > 0) & (rs < 8)).any()


def test_large_append_per_thread_kernel():
    """A RoPE slice of 12 channels: cos / sin rows of 24 bytes are no multiple
    of 16, so a large append takes the per-thread kernel instead of the
    streaming one.  Codes, scales and indexer keys bit-exact."""
    r12, n = 12, 300
    wl = Workload("quant-rope12", 1, [n], D, r12, 64, DI, 64, 64, 128, seed=73)
    dw = DeviceWorkload(wl, build_cache=False)
    rng = np.random.default_rng(73)
    kv = edge_rows(rng, n)
    ik = idx_edge_rows(rng, n)
    K.quant_append(dw.seq_view(0), torch.from_numpy(kv).cuda(), torch.from_numpy(ik).cuda(), n,
                   dw.ws)
    torch.cuda.synchronize()
    assert K.get_status(dw.ws) == 0
    assert int(dw.cache.seq_len[0]) == n
    pos = np.arange(n)
    codes, scales, idxk = read_rows(dw.cache, 0, pos)
    rc, rs = O.quant_append_rows(kv, pos, dw.rope_cos, dw.rope_sin, r12)
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs)
    assert np.array_equal(idxk, O.fp8_cast(ik))
