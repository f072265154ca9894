"""Prefill top-k (fm_index_prefill_topk) vs the oracle, on the GPU."""
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


def run_prefill(torch, dev, q, w, pos, K, k, ratio=4):
    import sparse_attention_kv_c4_gb300 as fm
    T = q.shape[0]
    S = K.shape[0]
    qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    pd = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int64)).to(dev)
    kd = torch.from_numpy(np.ascontiguousarray(K).view(np.int16)).to(dev)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((T, k), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_index_prefill_workspace(T, S), dtype=torch.uint8, device=dev)
    fm.fm_index_prefill_topk(qd, wd, pd, kd, k, idx, sc, ratio=ratio, workspace=ws)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    return idx.cpu().numpy(), sc.cpu().numpy()


def check(orc, q, w, pos, K, idx, sc, k, ratio=4, rows=None):
    rows = range(q.shape[0]) if rows is None else rows
    rows = list(rows)
    ref_idx, _ = orc.prefill_topk(q[rows], w[rows], np.asarray(pos)[rows], K, ratio=ratio, k=k)
    exempt = 0
    for n, t in enumerate(rows):
        cache = {}

        def score(s, t=t):
            if s not in cache:
                cache[s] = orc.score_bf16(q[t], w[t], K[s])
            return cache[s]
        exempt += parity.assert_topk_parity(idx[t], ref_idx[n], score, k, got_scores=sc[t])
    return exempt


def small(T, S, seed, pos=None):
    cfg = gen.PrefillCfg("t", T=T, S=S, pos0=4 * S + 17, seed=seed)
    return gen.prefill_host(cfg, pos=pos)


@pytest.mark.parametrize("T,S,k", [(37, 1000, 512), (4, 128, 64), (9, 4097, 512), (64, 3000, 1024), (5, 700, 1)])
def test_prefill_matches_oracle(torch_dev, orc, T, S, k):
    torch, dev = torch_dev
    q, w, pos, K = small(T, S, seed=T * 7 + S)
    idx, sc = run_prefill(torch, dev, q, w, pos, K, k)
    check(orc, q, w, pos, K, idx, sc, k)


def test_prefill_causal_limit_bites(torch_dev, orc):
    torch, dev = torch_dev
    T, S = 41, 2000
    pos = np.array([0, 1, 3, 4, 5, 8, 100, 511, 2047, 2048, 2052, 4000, 7999, 8000, 8004, 100000] +
                   list(range(5000, 5000 + 25 * 97, 97)), dtype=np.int64)
    q, w, _, K = small(T, S, seed=3, pos=pos)
    idx, sc = run_prefill(torch, dev, q, w, pos, K, 512)
    check(orc, q, w, pos, K, idx, sc, 512)
    for t in range(T):
        lim = min(S, max(0, int(pos[t])) // 4)
        sel = idx[t][idx[t] >= 0]
        assert len(sel) == min(512, lim) and (sel < lim).all()


def test_prefill_other_ratio(torch_dev, orc):
    torch, dev = torch_dev
    q, w, _, K = small(12, 900, seed=4)
    pos = np.arange(12, dtype=np.int64) * 300
    idx, sc = run_prefill(torch, dev, q, w, pos, K, 128, ratio=3)
    check(orc, q, w, pos, K, idx, sc, 128, ratio=3)


@pytest.mark.parametrize("variant", ["positions_262144", "positions_0", "positions_near_end"])
def test_prefill_full_size_sampled(torch_dev, orc, variant):
    """T=4096 queries x S=65536 chunks; sampled rows recomputed by the oracle."""
    torch, dev = torch_dev
    cfg = gen.PREFILL
    pos = {"positions_262144": cfg.pos0 + np.arange(cfg.T),
           "positions_0": np.arange(cfg.T),
           "positions_near_end": 4 * cfg.S - 4096 + np.arange(cfg.T)}[variant].astype(np.int64)
    q, w, pos, K = gen.prefill_host(cfg, pos=pos)
    idx, sc = run_prefill(torch, dev, q, w, pos, K, cfg.k)
    rng = np.random.default_rng(11)
    rows = sorted(set(rng.choice(cfg.T, size=6, replace=False).tolist()) | {0, cfg.T - 1})
    check(orc, q, w, pos, K, idx, sc, cfg.k, rows=rows)


@pytest.mark.parametrize("T,S,start,ratio", [(37, 1000, None, 4), (9, 4097, 0, 4), (6, 300, -3, 4), (11, 900, 0, 3)])
def test_prefill_scores_match_oracle(torch_dev, orc, T, S, start, ratio):
    """fm_index_prefill_scores: every element against the oracle's scores,
    -inf exactly where s >= the token's causal limit.  start=None puts every
    position past 4S (nothing masked); 0 makes the limit bite inside the row
    and skip whole 128-chunk tiles; negative positions mask the whole row."""
    torch, dev = torch_dev
    import sparse_attention_kv_c4_gb300 as fm
    pos = None if start is None else np.arange(start, start + T, dtype=np.int64) * 97
    q, w, pos, K = small(T, S, seed=T * 11 + S, pos=pos)
    ref = orc.prefill_logits(q, w, pos, K, ratio=ratio)
    out = torch.full((T, S), 7.0, dtype=torch.float32, device=dev)
    fm.fm_index_prefill_scores(torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).to(dev),
                               torch.from_numpy(np.ascontiguousarray(w)).to(dev),
                               torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int64)).to(dev),
                               torch.from_numpy(np.ascontiguousarray(K).view(np.int16)).to(dev), out, ratio=ratio)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    got = out.cpu().numpy().astype(np.float64)
    masked = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), masked)
    parity.assert_logits_close(got[~masked], ref[~masked])


def test_prefill_scores_full_size_sampled(torch_dev, orc):
    """The bench's launch (4096 tokens x 65536 chunks): sampled rows against
    the oracle."""
    torch, dev = torch_dev
    import sparse_attention_kv_c4_gb300 as fm
    cfg = gen.PREFILL
    q, w, pos, K = gen.prefill_host(cfg)
    out = torch.empty((cfg.T, cfg.S), dtype=torch.float32, device=dev)
    fm.fm_index_prefill_scores(torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).to(dev),
                               torch.from_numpy(np.ascontiguousarray(w)).to(dev),
                               torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int64)).to(dev),
                               torch.from_numpy(np.ascontiguousarray(K).view(np.int16)).to(dev), out)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    rows = [0, 1, 2, 3, 1021, 2050, 4095]
    ref = orc.prefill_logits(q[rows], w[rows], pos[rows], K)
    parity.assert_logits_close(out[rows].cpu().numpy(), ref)
