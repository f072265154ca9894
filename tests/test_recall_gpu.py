"""Page recall (fm_page_recall) vs the oracle: bit-exact page ids, densities
and counts, at small ragged sizes, at the three serving configurations
(256K / 512K / 1M context with KMAX 96 / 192 / 384) and on edge cases."""
import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch, torch.device("cuda:0")


def run(torch, dev, mask, S, kmax, sink=0, recent=0, with_density=True):
    import sparse_attention_kv_c4_gb300 as fm
    B = mask.shape[0]
    md = torch.from_numpy(np.ascontiguousarray(mask).view(np.int32)).to(dev)
    pages = torch.full((B, kmax), -7, dtype=torch.int32, device=dev)
    dens = torch.full((B, kmax), -7, dtype=torch.int32, device=dev) if with_density else None
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    fm.fm_page_recall(md, S, kmax, pages, dens, n, sink=sink, recent=recent)
    torch.cuda.synchronize()
    return pages.cpu().numpy(), (dens.cpu().numpy() if with_density else None), n.cpu().numpy()


def check(orc, torch, dev, mask, S, kmax, sink=0, recent=0):
    pages, dens, n = run(torch, dev, mask, S, kmax, sink, recent)
    wp, wd, wn = orc.page_recall(mask, S, kmax, sink=sink, recent=recent)
    assert (n == wn).all(), (n, wn)
    assert (pages == wp).all()
    assert (dens == wd).all()


@pytest.mark.parametrize("S", [1, 63, 64, 65, 1000, 4097, 20000])
@pytest.mark.parametrize("kmax", [1, 7, 96])
def test_recall_small(torch_dev, orc, S, kmax):
    torch, dev = torch_dev
    cfg = gen.RecallCfg("t", B=5, S=S, kmax=kmax, seed=S * 131 + kmax)
    mask = gen.recall_mask(cfg)
    check(orc, torch, dev, mask, S, kmax)
    rng = np.random.default_rng(S + kmax)
    check(orc, torch, dev, mask, S, kmax, sink=int(rng.integers(0, 200)), recent=int(rng.integers(0, 300)))


@pytest.mark.parametrize("cfg", [gen.RECALL_256K, gen.RECALL_512K, gen.RECALL_1M], ids=lambda c: c.name)
def test_recall_serving_configs(torch_dev, orc, cfg):
    torch, dev = torch_dev
    mask = gen.recall_mask(cfg)
    check(orc, torch, dev, mask, cfg.S, cfg.kmax)
    check(orc, torch, dev, mask, cfg.S, cfg.kmax, sink=4, recent=256)


def test_recall_edges(torch_dev, orc):
    torch, dev = torch_dev
    S = 64 * 40 + 9
    words = (S + 31) // 32
    zero = np.zeros((2, words), np.uint32)
    pages, dens, n = run(torch, dev, zero, S, 16)
    assert (n == 0).all() and (pages == -1).all() and (dens == -1).all()
    # every chunk resident, more pages requested than exist
    ones = np.full((2, words), 0xFFFFFFFF, np.uint32)
    check(orc, torch, dev, ones, S, 64)
    # bits past S are ignored (garbage in the last word)
    ragged = gen.recall_mask(gen.RecallCfg("t", B=3, S=S, kmax=8, seed=5))
    ragged[:, -1] |= np.uint32(0xFFFFFFFF) << np.uint32(S % 32)
    check(orc, torch, dev, ragged, S, 8)
    # the sink / recency tail cover the whole history, and all densities tie
    check(orc, torch, dev, zero, S, 5, sink=S)
    check(orc, torch, dev, zero, S, 5, recent=10 * S)
    # S = 0: nothing to recall; density_out and n_out are optional
    pages, dens, n = run(torch, dev, np.zeros((2, 1), np.uint32), 0, 4)
    assert (n == 0).all() and (pages == -1).all()
    pages, dens, n = run(torch, dev, ones, S, 8, with_density=False)
    wp, _, wn = orc.page_recall(ones, S, 8)
    assert (pages == wp).all() and (n == wn).all()


def test_recall_feeds_the_paged_scorer(torch_dev, orc):
    """The recalled page ids are a valid page table: distinct, in range and
    exactly n per request (the paged scorer rejects repeats)."""
    torch, dev = torch_dev
    cfg = gen.RECALL_1M
    pages, dens, n = run(torch, dev, gen.recall_mask(cfg), cfg.S, cfg.kmax)
    n_pages = (cfg.S + 63) // 64
    for b in range(cfg.B):
        got = pages[b, : n[b]]
        assert (np.diff(got) > 0).all() and got[0] >= 0 and got[-1] < n_pages
        assert (pages[b, n[b]:] == -1).all()
