"""Standalone top-k select (fm_topk_select) vs the oracle / brute force."""
import numpy as np
import pytest

import pins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch, torch.device("cuda:0")


def run(torch, dev, scores, k, n_valid=None):
    import sparse_attention_kv_c4_gb300 as fm
    rows = scores.shape[0]
    sd = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).to(dev)
    nv = None if n_valid is None else torch.from_numpy(np.asarray(n_valid, np.int32)).to(dev)
    idx = torch.full((rows, k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((rows, k), 7.0, dtype=torch.float32, device=dev)
    fm.fm_topk_select(sd, k, idx, sc, n_valid=nv)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("rows,n,k", [(3, 4096, 512), (2, 65536, 512), (4, 12288, 512), (5, 700, 512),
                                      (3, 513, 512), (2, 3000, 1), (2, 5000, 1024), (1, 0, 16), (2, 1, 512)])
def test_topk_random(torch_dev, orc, rows, n, k):
    torch, dev = torch_dev
    rng = np.random.default_rng(n + k)
    s = rng.standard_normal((rows, n)).astype(np.float32) * 3
    idx, sc = run(torch, dev, s, k)
    for r in range(rows):
        ref, _, m = orc.topk(np.arange(n), s[r].astype(np.float64), k)
        assert (idx[r] == ref).all()
        sel = ref[:m]
        assert (sc[r][:m] == s[r][sel]).all() and np.isneginf(sc[r][m:]).all()


def test_topk_heavy_ties_and_specials(torch_dev, orc):
    torch, dev = torch_dev
    rng = np.random.default_rng(3)
    n, k = 20000, 512
    s = rng.integers(-4, 5, (3, n)).astype(np.float32)
    s[0, ::7] = -0.0
    s[1, ::11] = np.nan
    s[1, ::13] = -np.inf
    s[2, :] = 1.5  # all equal: lowest ids win
    idx, sc = run(torch, dev, s, k)
    for r in range(3):
        want = pins.expected_topk(list(range(n)), [float(v) for v in s[r]], k)
        assert list(idx[r]) == want


def test_topk_n_valid(torch_dev, orc):
    torch, dev = torch_dev
    rng = np.random.default_rng(5)
    s = rng.standard_normal((4, 3000)).astype(np.float32)
    nv = [3000, 0, 100, 1200]
    idx, sc = run(torch, dev, s, 512, n_valid=nv)
    for r in range(4):
        ref, _, _ = orc.topk(np.arange(nv[r]), s[r, : nv[r]].astype(np.float64), 512)
        assert (idx[r] == ref).all()
