"""Standalone top-k select (fm_topk_select) vs the oracle / brute force.

Rows span the one-CTA select's regimes: short rows taken whole (<= 4096),
sampled rows with the bitmap emit (<= 131072) and longer rows with the
sorting emit; rows whose sample misleads the threshold take the exact radix
path.  Every case must give the oracle's exact answer.
"""
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


def run(torch, dev, scores, k, n_valid=None, ld=None):
    import sparse_attention_kv_c4_gb300 as fm
    rows, n = scores.shape
    ld = n if ld is None else ld
    buf = np.full((rows, ld), 1e30, dtype=np.float32)  # padding past n must never be read as a score
    buf[:, :n] = scores
    sd = torch.from_numpy(buf).to(dev)[:, :n]
    nv = None if n_valid is None else torch.from_numpy(np.asarray(n_valid, np.int32)).to(dev)
    idx = torch.full((rows, k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((rows, k), 7.0, dtype=torch.float32, device=dev)
    fm.fm_topk_select(sd, k, idx, sc, n_valid=nv)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), sc.cpu().numpy()


def check_rows(orc, s, k, idx, sc, n_valid=None):
    for r in range(s.shape[0]):
        nr = s.shape[1] if n_valid is None else n_valid[r]
        ref, _, m = orc.topk(np.arange(nr), s[r, :nr].astype(np.float64), k)
        assert (idx[r] == ref).all(), r
        sel = ref[:m]
        assert (sc[r][:m] == s[r][sel]).all() and np.isneginf(sc[r][m:]).all(), r


@pytest.mark.parametrize("rows,n,k", [(3, 4096, 512), (2, 65536, 512), (4, 12288, 512), (5, 700, 512),
                                      (3, 513, 512), (2, 3000, 1), (2, 5000, 1024), (1, 0, 16), (2, 1, 512),
                                      (3, 4097, 512), (2, 131072, 512), (3, 24577, 1), (2, 40000, 1024),
                                      (2, 9000, 16), (2, 65537, 512), (400, 12288, 512), (3, 3073, 512),
                                      (2, 8191, 1024), (2, 200000, 512)])
def test_topk_random(torch_dev, orc, rows, n, k):
    torch, dev = torch_dev
    rng = np.random.default_rng(n + k)
    s = rng.standard_normal((rows, n)).astype(np.float32) * 3
    idx, sc = run(torch, dev, s, k)
    check_rows(orc, s, k, idx, sc)


@pytest.mark.parametrize("n", [20000, 65536, 262144])
def test_topk_heavy_ties_and_specials(torch_dev, orc, n):
    torch, dev = torch_dev
    rng = np.random.default_rng(3)
    k = 512
    s = rng.integers(-4, 5, (6, n)).astype(np.float32)
    s[0, ::7] = -0.0
    s[1, ::11] = np.nan
    s[1, ::13] = -np.inf
    s[2, :] = 1.5  # all equal: lowest ids win
    s[3, :] = -np.inf  # threshold at -inf: every score is compared by composite
    s[4, :] = np.nan  # NaN ranks as -inf
    s[5, : n // 2] = -np.inf
    idx, sc = run(torch, dev, s, k)
    for r in range(s.shape[0]):
        want = pins.expected_topk(list(range(n)), [float(v) for v in s[r]], k)
        assert list(idx[r]) == want, r


def test_topk_adversarial_order(torch_dev, orc):
    """Rows whose sample misleads the threshold (sorted, one hot block at the
    end, values hidden between the sample runs) must still come out exact:
    the select then redoes the row with the exact radix path."""
    torch, dev = torch_dev
    n, k = 65536, 512
    rng = np.random.default_rng(11)
    s = np.empty((5, n), np.float32)
    s[0] = np.arange(n, dtype=np.float32)  # ascending
    s[1] = -np.arange(n, dtype=np.float32)  # descending
    s[2] = rng.standard_normal(n).astype(np.float32)
    s[2, -600:] += 50.0  # hot block at the end
    s[3] = rng.standard_normal(n).astype(np.float32)
    # large values only between the sample runs (runs of 64 at multiples of (n-64)/31)
    for run_i in range(31):
        a = run_i * (n - 64) // 31 + 64
        s[3, a:a + 40] += 30.0
    s[4] = rng.standard_normal(n).astype(np.float32) * 1e-30  # tiny magnitudes, subnormal keys
    idx, sc = run(torch, dev, s, k)
    check_rows(orc, s, k, idx, sc)


def test_topk_n_valid(torch_dev, orc):
    torch, dev = torch_dev
    rng = np.random.default_rng(5)
    s = rng.standard_normal((6, 30000)).astype(np.float32)
    nv = [30000, 0, 100, 1200, 4096, 4097]
    idx, sc = run(torch, dev, s, 512, n_valid=nv)
    check_rows(orc, s, 512, idx, sc, n_valid=nv)


@pytest.mark.parametrize("ld", [12289, 12290, 12291])
def test_topk_unaligned_rows(torch_dev, orc, ld):
    """Row strides that are not a multiple of 4 floats: rows lose 16-byte
    alignment and take the scalar-load path."""
    torch, dev = torch_dev
    rng = np.random.default_rng(ld)
    n = 12288
    s = rng.standard_normal((4, n)).astype(np.float32)
    idx, sc = run(torch, dev, s, 512, ld=ld)
    check_rows(orc, s, 512, idx, sc)

