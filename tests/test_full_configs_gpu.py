"""The benchmark workloads compared with the oracle in full, on the GPU.

Every output of these workloads is checked, not a sample:
  - the tiny workload (1 query, 1 layer, S = 4096, 12% planted): its resident
    mask and its top-512 over all chunks, through two CUDA paths (the dense
    prefill call at a position that sees every chunk, and the Memory
    Indexer's logits followed by the standalone top-k);
  - the Memory Indexer at 256K context (76 requests x 3 layers x 65536
    chunks) and at 1M context (30 x 3 x 262144, 12% planted): every logit,
    every mask bit and every max-sigmoid;
  - the native paged top-512 at 512K context (1260 queries x 192 pages) and
    at 1M context (630 queries x 384 pages): every query's id set and scores.
The keys are filled on the device by the generator's CUDA kernels and
regenerated bit for bit on the host for the oracle, one request at a time.
"""
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


def test_tiny_config_mask_and_top512(torch_dev, orc):
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    cfg = gen.TINY
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    x = orc.memindex_logits(q, w, K)[0, 0]
    ids = np.arange(cfg.S, dtype=np.int64)
    ref_idx, _, n = orc.topk(ids, x, 512)
    assert n == 512
    planted = np.flatnonzero(gen.planted(cfg, 0, 0))
    assert 0 < len(planted) <= 512

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    qd, wd, Kd = t(q.view(np.int16)), t(w), t(K.view(np.int16))
    mask = torch.empty((1, cfg.S // 32), dtype=torch.int32, device=dev)
    logits = torch.empty((1, 1, cfg.S), dtype=torch.float32, device=dev)
    fm.fm_memindex_score_mask(qd, wd, Kd, mask, None, logits)
    # path 1: the Memory Indexer's logits, then the standalone top-512
    idx1 = torch.empty((1, 512), dtype=torch.int32, device=dev)
    sc1 = torch.empty((1, 512), dtype=torch.float32, device=dev)
    fm.fm_topk_select(logits[0], 512, idx1, sc1)
    # path 2: the dense prefill call, one token whose causal limit is S
    pos = torch.tensor([4 * cfg.S], dtype=torch.int64, device=dev)
    idx2 = torch.empty((1, 512), dtype=torch.int32, device=dev)
    sc2 = torch.empty((1, 512), dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_index_prefill_workspace(1, cfg.S), dtype=torch.uint8, device=dev)
    fm.fm_index_prefill_topk(qd[0], wd[0], pos, Kd[0, 0], 512, idx2, sc2, workspace=ws)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0

    parity.assert_logits_close(logits.cpu().numpy()[0, 0], x)
    parity.assert_mask_parity(mask.cpu().numpy().view(np.uint32), x[None], cfg.S)
    for idx, sc in ((idx1, sc1), (idx2, sc2)):
        got = idx.cpu().numpy()
        parity.assert_topk_rows_parity(got, sc.cpu().numpy(), ref_idx[None], ids[None], x[None])
        assert set(planted.tolist()) <= set(got[0].tolist()), "a planted chunk is missing from the top-512"


def _memindex_full(torch, dev, orc, cfg):
    import sparse_attention_kv_c4_gb300 as fm
    q, w, hot = gen.memindex_qw(cfg)
    hot_d = torch.from_numpy(hot).to(dev)
    Kd = torch.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=torch.int16, device=dev)
    gen.memindex_keys_device(cfg, hot_d.data_ptr(), Kd.data_ptr(), cfg.L * cfg.S * cfg.d, cfg.S * cfg.d)
    mask = torch.empty((cfg.B, (cfg.S + 31) // 32), dtype=torch.int32, device=dev)
    maxsig = torch.empty((cfg.B, cfg.S), dtype=torch.float32, device=dev)
    logits = torch.empty((cfg.B, cfg.L, cfg.S), dtype=torch.float32, device=dev)
    fm.fm_memindex_score_mask(torch.from_numpy(q.view(np.int16)).to(dev), torch.from_numpy(w).to(dev), Kd, mask,
                              maxsig, logits)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    del Kd
    mask = mask.cpu().numpy().view(np.uint32)
    maxsig = maxsig.cpu().numpy()
    logits = logits.cpu().numpy()
    torch.cuda.empty_cache()
    s_all = np.arange(cfg.S, dtype=np.int64)
    exempt = 0
    for b in range(cfg.B):
        Kb = np.stack([gen.memindex_key_rows(cfg, b, l, s_all, hot) for l in range(cfg.L)])[None]
        x = orc.memindex_logits(q[b:b + 1], w[b:b + 1], Kb)[0]
        parity.assert_logits_close(logits[b], x, what=f"request {b} logits")
        m = x.max(axis=0)
        exempt += parity.assert_mask_parity(mask[b:b + 1], m[None], cfg.S)
        sig = 1.0 / (1.0 + np.exp(-m))
        assert np.all(np.abs(maxsig[b] - sig) <= 0.25 * parity.tol(m) + 2e-6), f"request {b} max-sigmoid"
        bits, _ = parity.mask_bits(mask[b:b + 1], cfg.S)
        for l in range(cfg.L):
            assert bits[0, gen.planted(cfg, b, l)].all(), f"request {b} layer {l}: planted chunk not resident"
    return exempt


def test_memindex_256k_full(torch_dev, orc):
    torch, dev = torch_dev
    _memindex_full(torch, dev, orc, gen.MEMINDEX_256K)


def test_memindex_1m_full(torch_dev, orc):
    torch, dev = torch_dev
    _memindex_full(torch, dev, orc, gen.MEMINDEX_1M)


@pytest.mark.parametrize("cfg", [gen.PAGED_512K, gen.PAGED_1M], ids=lambda c: c.name)
def test_paged_full(torch_dev, orc, cfg):
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    logical, phys, owner = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    own_d = torch.from_numpy(owner).to(dev)
    k8d = torch.empty((cfg.P, cfg.page, cfg.d), dtype=torch.uint8, device=dev)
    scd = torch.empty((cfg.P, cfg.page), dtype=torch.float32, device=dev)
    gen.paged_pool_device(cfg, own_d.data_ptr(), k8d.data_ptr(), scd.data_ptr())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    idx = torch.full((cfg.Q, cfg.k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((cfg.Q, cfg.k), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(cfg.Q, cfg.R), dtype=torch.uint8, device=dev)
    fm.fm_native_topk_paged(t(q.view(np.int16)), t(w), k8d, scd, t(phys), t(logical), cfg.k, idx, sc, workspace=ws)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    del k8d, scd, own_d, ws
    torch.cuda.empty_cache()
    # the oracle per group of requests, over a local pool of the group's pages
    group = 3 * cfg.layers
    for q0 in range(0, cfg.Q, group):
        qs = np.arange(q0, min(cfg.Q, q0 + group))
        local = np.arange(len(qs) * cfg.R, dtype=np.int32).reshape(len(qs), cfg.R)
        table = np.zeros_like(phys)
        table[qs] = local
        k8l, scl = gen.paged_pool_rows(cfg, logical, table, queries=qs, n_pool=len(qs) * cfg.R)
        ref_idx, _, ref_lg = orc.paged_topk(q[qs], w[qs], k8l, scl, local, logical[qs], k=cfg.k, want_logits=True)
        cand = (logical[qs].astype(np.int64)[:, :, None] * cfg.page + np.arange(cfg.page)).reshape(len(qs), -1)
        parity.assert_topk_rows_parity(idx[qs], sc[qs], ref_idx, cand, ref_lg, fp8=True)
