"""The trained retriever's Memory Indexer (fm_retriever_score_mask) vs the
oracle on the GPU: 128 or 64 heads over packed compressed_k rows, the max
(union) and mean ensembles, strided inputs, and the 1M workload at full size
on sampled chunks."""
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


def _run(torch, dev, q, w, ck_dev, S, mode, threshold=0.5, want_logits=True):
    import sparse_attention_kv_c4_gb300 as fm
    B, L, n_h = q.shape[:3]
    qd = torch.from_numpy(q.view(np.int16)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    mask = torch.full((B, (S + 31) // 32), -1, dtype=torch.int32, device=dev)
    ens = torch.full((B, S), np.nan, dtype=torch.float32, device=dev)
    logits = torch.full((B, L, S), np.nan, dtype=torch.float32, device=dev) if want_logits else None
    ws = torch.empty(fm.fm_retriever_workspace(B, L, n_h), dtype=torch.uint8, device=dev)
    fm.fm_retriever_score_mask(qd, wd, ck_dev, mask, ens, logits, ensemble=mode, threshold=threshold, workspace=ws)
    torch.cuda.synchronize()
    st = fm.fm_device_status(reset=True)
    assert st == 0, f"device status {st:#x}"
    return (mask.cpu().numpy().view(np.uint32), ens.cpu().numpy(),
            None if logits is None else logits.cpu().numpy())


def _check_ensemble(orc, x, mask, ens, S, mode, thr):
    """x [B,L,S] oracle logits (fp64)."""
    ref_mask, ref_e = orc.memindex_ensemble(x, mode, thr)
    band = 0.25 * parity.tol(np.abs(x).max(axis=1), fp8=True)  # sigma' <= 1/4
    assert np.all(np.abs(ens - ref_e) <= band + 2e-6), np.abs(ens - ref_e).max()
    bits, tail = parity.mask_bits(mask, S)
    assert not tail.any()
    ref_bits, _ = parity.mask_bits(ref_mask, S)
    bad = (bits != ref_bits) & (np.abs(ref_e - thr) > band)
    assert not bad.any(), f"{int(bad.sum())} mask bits differ outside the band, e.g. {np.argwhere(bad)[:3]}"


@pytest.mark.parametrize("B,L,S,n_h,mode,frac", [
    (1, 3, 4096, 128, 0, 0.12), (1, 3, 4096, 128, 1, 0.12), (2, 4, 1000, 128, 1, 0.25), (3, 1, 132, 128, 0, 0.05),
    (2, 2, 640, 64, 0, 0.12), (2, 3, 644, 64, 1, 0.3), (1, 3, 4, 128, 1, 0.5), (5, 3, 300, 128, 0, 0.0)])
def test_retriever_matches_oracle(torch_dev, orc, B, L, S, n_h, mode, frac):
    torch, dev = torch_dev
    cfg = gen.MemIndexCfg("t", B=B, L=L, S=S, n_h=n_h, hot_frac=frac, seed=gen.BASE_SEED + 3000 + S + n_h)
    q, w, hot = gen.memindex_qw(cfg)
    k8, sc = gen.memindex_fp8_keys_host(cfg, hot)
    ck = gen.pack_compressed_k(k8, sc)
    mask, ens, logits = _run(torch, dev, q, w, torch.from_numpy(ck).to(dev), S, mode)
    k8o, sco = orc.unpack_compressed_k(ck)
    x = orc.memindex_logits_fp8(q, w, k8o, sco)
    parity.assert_logits_close(logits, x, fp8=True)
    # the exact query split (and, at 128 heads and up to 3 layers, q_w in four
    # E4M3 terms for the ReLU's linear half) leaves only fp32 rounding
    err = float(np.max(np.abs(logits - x) / (np.abs(x) + 1.0)))
    assert err < 2e-3, f"retriever logit relative error {err} (expected ~1e-5)"
    _check_ensemble(orc, x, mask, ens, S, mode, 0.5)


def test_retriever_threshold_strides_and_scales(torch_dev, orc):
    """Threshold 0.7 (mean) and 0.3 (max); packed rows inside a larger buffer
    (request and layer strides beyond the dense ones); zero and negative
    scales."""
    torch, dev = torch_dev
    B, L, S = 2, 3, 520
    cfg = gen.MemIndexCfg("t", B=B, L=L, S=S, n_h=128, seed=gen.BASE_SEED + 3100)
    q, w, hot = gen.memindex_qw(cfg)
    k8, sc = gen.memindex_fp8_keys_host(cfg, hot)
    sc[0, 1, ::7] = 0.0
    sc[1, 2, ::5] *= -1.0
    ck = gen.pack_compressed_k(k8, sc)
    big = torch.zeros((B, L + 1, S + 12, 132), dtype=torch.uint8, device=dev)
    big[:, :L, :S] = torch.from_numpy(ck).to(dev)
    k8o, sco = orc.unpack_compressed_k(ck)
    x = orc.memindex_logits_fp8(q, w, k8o, sco)
    for mode, thr in ((1, 0.7), (0, 0.3)):
        mask, ens, logits = _run(torch, dev, q, w, big[:, :L, :S], S, mode, threshold=thr)
        parity.assert_logits_close(logits, x, fp8=True)
        _check_ensemble(orc, x, mask, ens, S, mode, thr)


def test_retriever_rejects_bad_args(torch_dev):
    torch, dev = torch_dev
    import sparse_attention_kv_c4_gb300 as fm
    q = torch.zeros((1, 3, 128, 128), dtype=torch.int16, device=dev)
    w = torch.zeros((1, 3, 128), dtype=torch.float32, device=dev)
    mask = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    ws = torch.empty(fm.fm_retriever_workspace(1, 3, 128), dtype=torch.uint8, device=dev)
    ck = torch.zeros((1, 3, 30, 132), dtype=torch.uint8, device=dev)  # S % 4 != 0
    with pytest.raises(fm.FmError):
        fm.fm_retriever_score_mask(q, w, ck, mask, workspace=ws)
    ck = torch.zeros((1, 3, 32, 132), dtype=torch.uint8, device=dev)
    with pytest.raises(fm.FmError):
        fm.fm_retriever_score_mask(q, w, ck, mask, ensemble=2, workspace=ws)
    with pytest.raises(fm.FmError):
        fm.fm_retriever_score_mask(q, w, ck, mask, threshold=1.0, workspace=ws)
    with pytest.raises(fm.FmError):
        fm.fm_retriever_score_mask(q, w, ck, mask, workspace=ws[:100])
    assert fm.fm_device_status(reset=True) == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_retriever_1m_full_size_sampled(torch_dev, orc, mode):
    """30 requests x 3 layers x 262144 packed rows (3.1 GB) at 128 heads,
    filled on the device; the oracle on sampled chunks."""
    torch, dev = torch_dev
    cfg = gen.RETRIEVER_1M
    q, w, hot = gen.memindex_qw(cfg)
    hot_d = torch.from_numpy(hot).to(dev)
    own_d = torch.from_numpy(gen.memindex_fp8_owner(cfg)).to(dev)
    k8d = torch.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=torch.uint8, device=dev)
    scd = torch.empty((cfg.B, cfg.L, cfg.S), dtype=torch.float32, device=dev)
    gen.memindex_fp8_keys_device(cfg, hot_d.data_ptr(), own_d.data_ptr(), k8d.data_ptr(), scd.data_ptr())
    ck = torch.cat([k8d, scd.view(torch.uint8).view(cfg.B, cfg.L, cfg.S, 4)], dim=-1)
    del k8d, scd
    mask, ens, _ = _run(torch, dev, q, w, ck, cfg.S, mode, want_logits=False)
    del ck
    bits, tail = parity.mask_bits(mask, cfg.S)
    assert not tail.any()
    rng = np.random.default_rng(cfg.seed + mode)
    for b in rng.choice(cfg.B, size=3, replace=False):
        s = np.sort(rng.choice(cfg.S, size=200, replace=False))
        x = np.empty((1, cfg.L, len(s)))
        for l in range(cfg.L):
            rows, scs = gen.memindex_fp8_key_rows(cfg, int(b), l, s, hot)
            for i in range(len(s)):
                x[0, l, i] = orc.score_fp8(q[b, l], w[b, l], rows[i], scs[i])
        ref_mask, ref_e = orc.memindex_ensemble(x, mode, 0.5)
        band = 0.25 * parity.tol(np.abs(x).max(axis=1), fp8=True)[0]
        assert np.all(np.abs(ens[b, s] - ref_e[0]) <= band + 2e-6)
        ref_bits, _ = parity.mask_bits(ref_mask, len(s))
        bad = (bits[b, s] != ref_bits[0]) & (np.abs(ref_e[0] - 0.5) > band)
        assert not bad.any()
        if mode == 0:  # the union keeps every planted chunk
            for l in range(cfg.L):
                assert bits[b, gen.planted(cfg, int(b), l)].all()
