"""Memory Indexer kernel (fm_memindex_score_mask) vs the oracle, on the GPU."""
import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch, torch.device("cuda:0")


def _run(torch, dev, q, w, K, threshold=0.5, want_maxsig=True, want_logits=True, keys_dev=None):
    import sparse_attention_kv_c4_gb300 as fm
    B, L, _, _ = q.shape
    S = K.shape[2] if keys_dev is None else keys_dev.shape[2]
    qd = torch.from_numpy(q.view(np.int16)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    Kd = torch.from_numpy(K.view(np.int16)).to(dev) if keys_dev is None else keys_dev
    mask = torch.full((B, (S + 31) // 32), -1, dtype=torch.int32, device=dev)
    maxsig = torch.full((B, S), np.nan, dtype=torch.float32, device=dev) if want_maxsig else None
    logits = torch.full((B, L, S), np.nan, dtype=torch.float32, device=dev) if want_logits else None
    fm.fm_memindex_score_mask(qd, wd, Kd, mask, maxsig, logits, threshold=threshold)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    return (mask.cpu().numpy().view(np.uint32), None if maxsig is None else maxsig.cpu().numpy(),
            None if logits is None else logits.cpu().numpy())


@pytest.mark.parametrize("B,L,S,frac", [(1, 1, 4096, 0.12), (2, 3, 1000, 0.12), (3, 3, 129, 0.25),
                                        (1, 2, 31, 0.05), (2, 4, 640, 0.12), (1, 3, 1, 0.5), (5, 3, 300, 0.0)])
def test_memindex_matches_oracle(torch_dev, orc, B, L, S, frac):
    torch, dev = torch_dev
    cfg = gen.MemIndexCfg("t", B=B, L=L, S=S, hot_frac=frac, seed=gen.BASE_SEED + 1000 + S)
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    mask, maxsig, logits = _run(torch, dev, q, w, K)
    x = orc.memindex_logits(q, w, K)
    parity.assert_logits_close(logits, x)
    m = x.max(axis=1)
    parity.assert_mask_parity(mask, m, S)
    _, ref_sig = orc.memindex_select(x, 0.5)
    assert np.all(np.abs(maxsig - ref_sig) <= 0.25 * parity.tol(m) + 2e-6)


def test_memindex_tiny_config(torch_dev, orc):
    """The tiny workload: 1 query, 1 layer, S=4096, 12% planted."""
    torch, dev = torch_dev
    cfg = gen.TINY
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    mask, maxsig, logits = _run(torch, dev, q, w, K)
    x = orc.memindex_logits(q, w, K)
    parity.assert_logits_close(logits, x)
    parity.assert_mask_parity(mask, x.max(axis=1), cfg.S)
    bits, _ = parity.mask_bits(mask, cfg.S)
    assert bits[0, gen.planted(cfg, 0, 0)].all()


def test_memindex_threshold_other_than_half(torch_dev, orc):
    torch, dev = torch_dev
    cfg = gen.MemIndexCfg("t", B=2, L=3, S=777, seed=77)
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    for thr in (0.25, 0.75, 0.9):
        mask, _, _ = _run(torch, dev, q, w, K, threshold=thr, want_maxsig=False, want_logits=False)
        x = orc.memindex_logits(q, w, K)
        ref_mask, ref_sig = orc.memindex_select(x, thr)
        lg = float(np.log(thr / (1 - thr)))
        parity.assert_mask_parity(mask, x.max(axis=1), cfg.S, thr_logit=lg)


def test_memindex_strided_keys(torch_dev, orc):
    """Keys inside a larger buffer (padded layer and request strides)."""
    torch, dev = torch_dev
    cfg = gen.MemIndexCfg("t", B=2, L=3, S=500, seed=91)
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    big = np.zeros((cfg.B, cfg.L + 1, cfg.S + 24, cfg.d), dtype=np.uint16)
    big[:, : cfg.L, : cfg.S] = K
    Kd = torch.from_numpy(big.view(np.int16)).to(dev)[:, : cfg.L, : cfg.S]
    mask, _, logits = _run(torch, dev, q, w, K, keys_dev=Kd, want_maxsig=False)
    x = orc.memindex_logits(q, w, K)
    parity.assert_logits_close(logits, x)
    parity.assert_mask_parity(mask, x.max(axis=1), cfg.S)


def test_generator_device_matches_host(torch_dev):
    """gen's CUDA fill kernels reproduce the host generator bit for bit."""
    torch, dev = torch_dev
    cfg = gen.MemIndexCfg("t", B=3, L=3, S=3000, seed=5)
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    hot_d = torch.from_numpy(hot).to(dev)
    Kd = torch.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=torch.int16, device=dev)
    gen.memindex_keys_device(cfg, hot_d.data_ptr(), Kd.data_ptr(), cfg.L * cfg.S * cfg.d, cfg.S * cfg.d)
    torch.cuda.synchronize()
    assert (Kd.cpu().numpy().view(np.uint16) == K).all()
    pc = gen.PagedCfg("t", requests=2, layers=3, n_pages=40, R=5, seed=6)
    logical, phys, owner = gen.paged_tables(pc)
    k8, sc = gen.paged_pool_host(pc, owner)
    own_d = torch.from_numpy(owner).to(dev)
    k8d = torch.empty((pc.P, pc.page, pc.d), dtype=torch.uint8, device=dev)
    scd = torch.empty((pc.P, pc.page), dtype=torch.float32, device=dev)
    gen.paged_pool_device(pc, own_d.data_ptr(), k8d.data_ptr(), scd.data_ptr())
    torch.cuda.synchronize()
    assert (k8d.cpu().numpy() == k8).all() and (scd.cpu().numpy().view(np.uint32) == sc.view(np.uint32)).all()


def _sampled_full_size(torch, dev, orc, cfg, n_samples, want_maxsig):
    """Full-size workload filled on the device; oracle on sampled chunks."""
    import sparse_attention_kv_c4_gb300 as fm
    q, w, hot = gen.memindex_qw(cfg)
    hot_d = torch.from_numpy(hot).to(dev)
    Kd = torch.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=torch.int16, device=dev)
    gen.memindex_keys_device(cfg, hot_d.data_ptr(), Kd.data_ptr(), cfg.L * cfg.S * cfg.d, cfg.S * cfg.d)
    qd = torch.from_numpy(q.view(np.int16)).to(dev)
    wd = torch.from_numpy(w).to(dev)
    mask = torch.empty((cfg.B, (cfg.S + 31) // 32), dtype=torch.int32, device=dev)
    maxsig = torch.empty((cfg.B, cfg.S), dtype=torch.float32, device=dev) if want_maxsig else None
    fm.fm_memindex_score_mask(qd, wd, Kd, mask, maxsig)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    del Kd
    mask = mask.cpu().numpy().view(np.uint32)
    bits, tail = parity.mask_bits(mask, cfg.S)
    assert not tail.any()
    rng = np.random.default_rng(cfg.seed)
    for b in rng.choice(cfg.B, size=min(cfg.B, 4), replace=False):
        s = np.sort(rng.choice(cfg.S, size=n_samples, replace=False))
        xs = np.empty((cfg.L, len(s)))
        for l in range(cfg.L):
            rows = gen.memindex_key_rows(cfg, int(b), l, s, hot)
            for i in range(len(s)):
                xs[l, i] = orc.score_bf16(q[b, l], w[b, l], rows[i])
        m = xs.max(axis=0)
        exempt = np.abs(m) <= parity.tol(m)
        assert not ((bits[b, s] != (m >= 0)) & ~exempt).any()
        if want_maxsig:
            sig = 1 / (1 + np.exp(-m))
            got = maxsig[b].cpu().numpy()[s] if hasattr(maxsig, "cpu") else maxsig[b, s]
            assert np.all(np.abs(got - sig) <= 0.25 * parity.tol(m) + 2e-6)
        for l in range(cfg.L):  # every planted chunk is resident
            pl = gen.planted(cfg, int(b), l)
            assert bits[b, pl].all()
    frac = bits.mean()
    assert cfg.hot_frac * 0.8 < frac < cfg.hot_frac + 0.9, frac


# The 256K workload and the 1M workload at 12% planted are compared in full
# in test_full_configs_gpu.py; the 1M workload's other planted fractions are
# sampled here.
@pytest.mark.parametrize("frac", [0.05, 0.25])
def test_memindex_1m_full_size_sampled(torch_dev, orc, frac):
    torch, dev = torch_dev
    cfg = gen.replace(gen.MEMINDEX_1M, hot_frac=frac)
    _sampled_full_size(torch, dev, orc, cfg, 300, want_maxsig=True)
