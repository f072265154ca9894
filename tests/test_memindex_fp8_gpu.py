"""Memory Indexer over compressed E4M3 keys (fm_memindex_score_mask_fp8) vs
the oracle on the GPU: logits within the fp8 tolerance, the resident mask
bit-exact outside the tolerance band, max-sigmoid, strided inputs, the
device generator, and the 1M workload sampled at full size."""
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


def _run(torch, dev, q, w, k8d, scd, S, threshold=0.5, want_logits=True):
    import sparse_attention_kv_c4_gb300 as fm
    B, L = q.shape[:2]
    qd = torch.from_numpy(q.view(np.int16)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    mask = torch.full((B, (S + 31) // 32), -1, dtype=torch.int32, device=dev)
    maxsig = torch.full((B, S), np.nan, dtype=torch.float32, device=dev)
    logits = torch.full((B, L, S), np.nan, dtype=torch.float32, device=dev) if want_logits else None
    ws = torch.empty(fm.fm_memindex_fp8_workspace(B, L), dtype=torch.uint8, device=dev)
    fm.fm_memindex_score_mask_fp8(qd, wd, k8d, scd, mask, maxsig, logits, threshold=threshold, workspace=ws)
    torch.cuda.synchronize()
    st = fm.fm_device_status(reset=True)
    assert st == 0, f"device status {st:#x}"
    return (mask.cpu().numpy().view(np.uint32), maxsig.cpu().numpy(),
            None if logits is None else logits.cpu().numpy())


def _check(orc, q, w, k8, sc, mask, maxsig, logits, S, thr=0.5):
    x = orc.memindex_logits_fp8(q, w, k8, sc)
    if logits is not None:
        parity.assert_logits_close(logits, x, fp8=True)
    m = x.max(axis=1)
    t = float(np.log(thr / (1 - thr)))
    parity.assert_mask_parity(mask, m, S, thr_logit=t, fp8=True)
    _, ref_sig = orc.memindex_select(x, thr)
    assert np.all(np.abs(maxsig - ref_sig) <= 0.25 * parity.tol(m, fp8=True) + 2e-6)


@pytest.mark.parametrize("B,L,S,frac", [(1, 1, 4096, 0.12), (2, 3, 1000, 0.12), (3, 3, 129, 0.25),
                                        (1, 2, 31, 0.05), (2, 4, 640, 0.12), (1, 3, 1, 0.5), (5, 3, 300, 0.0),
                                        (1, 4, 2000, 0.3)])
def test_memindex_fp8_matches_oracle(torch_dev, orc, B, L, S, frac):
    torch, dev = torch_dev
    cfg = gen.MemIndexCfg("t", B=B, L=L, S=S, hot_frac=frac, seed=gen.BASE_SEED + 2000 + S)
    q, w, hot = gen.memindex_qw(cfg)
    k8, sc = gen.memindex_fp8_keys_host(cfg, hot)
    mask, maxsig, logits = _run(torch, dev, q, w, torch.from_numpy(k8).to(dev), torch.from_numpy(sc).to(dev), S)
    _check(orc, q, w, k8, sc, mask, maxsig, logits, S)


def test_memindex_fp8_threshold_and_strides(torch_dev, orc):
    """A threshold other than 0.5, keys and scales living inside larger
    buffers (layer / request strides beyond the dense ones), and zero and
    negative scales."""
    torch, dev = torch_dev
    B, L, S = 2, 3, 700
    cfg = gen.MemIndexCfg("t", B=B, L=L, S=S, seed=gen.BASE_SEED + 2100)
    q, w, hot = gen.memindex_qw(cfg)
    k8, sc = gen.memindex_fp8_keys_host(cfg, hot)
    sc[0, 1, ::7] = 0.0
    sc[1, 2, ::5] *= -1.0
    big_k = torch.zeros((B, L + 1, S + 16, 128), dtype=torch.uint8, device=dev)
    big_k[:, :L, :S] = torch.from_numpy(k8).to(dev)
    big_s = torch.zeros((B, L + 2, S + 5), dtype=torch.float32, device=dev)
    big_s[:, :L, :S] = torch.from_numpy(sc).to(dev)
    mask, maxsig, logits = _run(torch, dev, q, w, big_k[:, :L, :S], big_s[:, :L, :S], S, threshold=0.75)
    _check(orc, q, w, k8, sc, mask, maxsig, logits, S, thr=0.75)


def test_memindex_fp8_device_generator_matches_host(torch_dev):
    torch, dev = torch_dev
    cfg = gen.MemIndexCfg("t", B=2, L=3, S=640, seed=gen.BASE_SEED + 2200)
    q, w, hot = gen.memindex_qw(cfg)
    k8, sc = gen.memindex_fp8_keys_host(cfg, hot)
    hot_d = torch.from_numpy(hot).to(dev)
    own_d = torch.from_numpy(gen.memindex_fp8_owner(cfg)).to(dev)
    k8d = torch.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=torch.uint8, device=dev)
    scd = torch.empty((cfg.B, cfg.L, cfg.S), dtype=torch.float32, device=dev)
    gen.memindex_fp8_keys_device(cfg, hot_d.data_ptr(), own_d.data_ptr(), k8d.data_ptr(), scd.data_ptr())
    torch.cuda.synchronize()
    assert (k8d.cpu().numpy() == k8).all()
    assert (scd.cpu().numpy().view(np.uint32) == sc.view(np.uint32)).all()


@pytest.mark.parametrize("frac", [0.05, 0.12])
def test_memindex_fp8_1m_full_size_sampled(torch_dev, orc, frac):
    """30 requests x 3 layers x 262144 chunks of compressed keys (3.1 GB),
    filled on the device; the oracle on sampled chunks."""
    torch, dev = torch_dev
    cfg = gen.replace(gen.MEMINDEX_1M, hot_frac=frac)
    q, w, hot = gen.memindex_qw(cfg)
    hot_d = torch.from_numpy(hot).to(dev)
    own_d = torch.from_numpy(gen.memindex_fp8_owner(cfg)).to(dev)
    k8d = torch.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=torch.uint8, device=dev)
    scd = torch.empty((cfg.B, cfg.L, cfg.S), dtype=torch.float32, device=dev)
    gen.memindex_fp8_keys_device(cfg, hot_d.data_ptr(), own_d.data_ptr(), k8d.data_ptr(), scd.data_ptr())
    mask, maxsig, _ = _run(torch, dev, q, w, k8d, scd, cfg.S, want_logits=False)
    del k8d, scd
    bits, tail = parity.mask_bits(mask, cfg.S)
    assert not tail.any()
    rng = np.random.default_rng(cfg.seed + 1)
    for b in rng.choice(cfg.B, size=3, replace=False):
        s = np.sort(rng.choice(cfg.S, size=300, replace=False))
        xs = np.empty((cfg.L, len(s)))
        for l in range(cfg.L):
            rows, scs = gen.memindex_fp8_key_rows(cfg, int(b), l, s, hot)
            for i in range(len(s)):
                xs[l, i] = orc.score_fp8(q[b, l], w[b, l], rows[i], scs[i])
        m = xs.max(axis=0)
        exempt = np.abs(m) <= parity.tol(m, fp8=True)
        assert not ((bits[b, s] != (m >= 0)) & ~exempt).any()
        sig = 1 / (1 + np.exp(-m))
        assert np.all(np.abs(maxsig[b, s] - sig) <= 0.25 * parity.tol(m, fp8=True) + 2e-6)
        for l in range(cfg.L):  # every planted chunk is resident
            assert bits[b, gen.planted(cfg, int(b), l)].all()
