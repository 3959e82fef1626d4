"""The README's example runs as printed, and its selection and attention
agree with the oracle on the same inputs."""
import os
import re

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from checks import attended_set, check_attention, check_select  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle import formats as F  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs_and_matches_the_oracle():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert len(blocks) == 1
    torch.manual_seed(0)
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    B, k, N, D, R, di = env["B"], env["k"], env["N"], env["D"], env["R"], env["di"]
    cache = env["cache"]
    assert cache.seq_len.cpu().tolist() == [N] * B
    q_idx, w = env["q_idx"].cpu().numpy(), env["w"].cpu().numpy()
    cos_tab, sin_tab = cache.rope_cos.cpu().numpy(), cache.rope_sin.cpu().numpy()
    rows = np.arange(N)
    for b in range(B):
        r0 = b * cache.max_len
        codes = cache.codes[r0: r0 + N, : D // 2].cpu().numpy()
        scales = cache.scales[r0: r0 + N, : D // 16].cpu().numpy()
        idxk = cache.idx_k[r0: r0 + N, :di].cpu().numpy()
        rc, rs = O.quant_append_rows(env["kv"][b].cpu().numpy(), rows, cos_tab, sin_tab, R)
        assert np.array_equal(codes, rc) and np.array_equal(scales, rs), b
        assert np.array_equal(idxk, F.e4m3_encode(env["idx_keys"][b].cpu().numpy())), b
        s = O.indexer_scores(q_idx[b, 0], w[b, 0], idxk)
        gi = env["idx"][b, 0, : int(env["cnt"][b, 0])].cpu().numpy()
        check_select(gi, s, rows, k, f"README top-k b={b}")
        ridx, _ = O.full_select(s, k)
        use = attended_set(gi, ridx)
        sel = O.dequantize_fp4(codes[use], scales[use], D)
        win = O.swa_rows_decode(env["swa"][b].cpu().numpy())
        q = env["q"][b].float().cpu().numpy().astype(np.float64)
        ref = O.sparse_attention(q, np.concatenate([sel, win]))
        check_attention(env["out"][b].cpu().numpy(), ref, f"README attention b={b}")
