"""Level-2 resident mask and fused remap (fm_native_topk_paged_ex) vs the
oracle: only resident chunks are candidates (one mask row per request,
shared by its layers), and the remap emits reserve cells for the same
selection in the same order."""
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


def case(seed, requests=2, layers=3, n_pages=40, R=7, resident=0.35):
    cfg = gen.PagedCfg("t", requests=requests, layers=layers, n_pages=n_pages, R=R, seed=seed)
    logical, phys, owner = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    k8, scale = gen.paged_pool_host(cfg, owner)
    mask = gen.recall_mask(gen.RecallCfg("t", B=requests, S=n_pages * 64, kmax=1, cold=resident, hot_frac=0.05,
                                         seed=seed + 1))
    return cfg, q, w, k8, scale, phys, logical, mask


def run(torch, dev, q, w, k8, scale, phys, logical, k, mask, mask_group, id_mode, n_res=None):
    import sparse_attention_kv_c4_gb300 as fm
    Q, R = phys.shape
    t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).to(dev)
    idx = torch.full((Q, k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((Q, k), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(Q, R), dtype=torch.uint8, device=dev)
    fm.fm_native_topk_paged_ex(t(q, np.int16), t(w), t(k8), t(scale), t(phys.astype(np.int32)),
                               t(logical.astype(np.int32)), k, idx, sc,
                               n_res=None if n_res is None else t(np.asarray(n_res, np.int32)),
                               res_mask=None if mask is None else t(mask, np.int32), mask_group=mask_group,
                               id_mode=id_mode, workspace=ws)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    return idx.cpu().numpy(), sc.cpu().numpy()


def check_logical(orc, cfg, q, w, k8, scale, phys, logical, mask, k, idx, sc, n_res=None):
    ref_idx, _, ref_lg = orc.paged_topk(q, w, k8, scale, phys, logical, n_res=n_res, k=k, want_logits=True,
                                        res_mask=mask, mask_group=cfg.layers)
    Q, R = phys.shape
    for qi in range(Q):
        nr = R if n_res is None else max(0, min(R, int(n_res[qi])))
        score = {int(logical[qi, j]) * 64 + o: ref_lg[qi, j * 64 + o] for j in range(nr) for o in range(64)}
        parity.assert_topk_parity(idx[qi], ref_idx[qi], score.__getitem__, k, fp8=True, got_scores=sc[qi])
        # every selected chunk is resident
        row = mask[qi // cfg.layers]
        for c in (int(v) for v in idx[qi] if v >= 0):
            assert (int(row[c >> 5]) >> (c & 31)) & 1, (qi, c)


@pytest.mark.parametrize("k,R,resident", [(64, 7, 0.35), (512, 7, 0.35), (512, 12, 0.9), (1024, 30, 0.5),
                                          (512, 30, 0.02)])
def test_mask_matches_oracle(torch_dev, orc, k, R, resident):
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical, mask = case(300 + R, R=R, n_pages=max(40, 2 * R), resident=resident)
    idx, sc = run(torch, dev, q, w, k8, scale, phys, logical, k, mask, cfg.layers, 0)
    check_logical(orc, cfg, q, w, k8, scale, phys, logical, mask, k, idx, sc)


def test_remap_is_the_same_selection_in_reserve_cells(torch_dev, orc):
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical, mask = case(401, R=9)
    for m in (None, mask):
        a, sa = run(torch, dev, q, w, k8, scale, phys, logical, 200, m, cfg.layers, 0)
        b, sb = run(torch, dev, q, w, k8, scale, phys, logical, 200, m, cfg.layers, 1)
        for qi in range(cfg.Q):
            cell = {int(logical[qi, j]) * 64 + o: int(phys[qi, j]) * 64 + o for j in range(cfg.R) for o in range(64)}
            assert [cell[c] if c >= 0 else -1 for c in a[qi]] == list(b[qi]), qi
        assert (sa == sb).all()
        # and the oracle's remapped selection agrees outside the tolerance band
        ref, _ = orc.paged_topk(q, w, k8, scale, phys, logical, k=200, res_mask=m, mask_group=cfg.layers, id_mode=1)
        for qi in range(cfg.Q):
            assert len(set(b[qi]) ^ set(ref[qi])) <= 4, qi


def test_mask_edges(torch_dev, orc):
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical, mask = case(402, R=6)
    # empty resident set: nothing selected
    zero = np.zeros_like(mask)
    idx, sc = run(torch, dev, q, w, k8, scale, phys, logical, 64, zero, cfg.layers, 0)
    assert (idx == -1).all() and np.isneginf(sc).all()
    # all resident: the same as no mask
    ones = np.full_like(mask, 0xFFFFFFFF)
    a, _ = run(torch, dev, q, w, k8, scale, phys, logical, 300, ones, cfg.layers, 0)
    b, _ = run(torch, dev, q, w, k8, scale, phys, logical, 300, None, cfg.layers, 0)
    assert (a == b).all()
    # a short mask row: words past it count as non-resident; one row per query; n_res
    short = mask[:, :20].copy()
    per_query = np.repeat(short, cfg.layers, axis=0)
    n_res = [6, 0, 3, 6, 1, 5]
    idx, sc = run(torch, dev, q, w, k8, scale, phys, logical, 128, per_query, 1, 0, n_res=n_res)
    check_logical(orc, gen.replace(cfg, layers=1), q, w, k8, scale, phys, logical, per_query, 128, idx, sc,
                  n_res=n_res)


def test_mask_full_size_sampled(torch_dev, orc):
    """The 1M paged workload (630 queries x 384 pages) with a Memory-Indexer
    style mask per request: sampled queries against the oracle."""
    torch, dev = torch_dev
    import sparse_attention_kv_c4_gb300 as fm
    cfg = gen.PAGED_1M
    logical, phys, owner = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    own_d = torch.from_numpy(owner).to(dev)
    k8 = torch.empty((cfg.P, cfg.page, cfg.d), dtype=torch.uint8, device=dev)
    sc8 = torch.empty((cfg.P, cfg.page), dtype=torch.float32, device=dev)
    gen.paged_pool_device(cfg, own_d.data_ptr(), k8.data_ptr(), sc8.data_ptr())
    mask = gen.recall_mask(gen.RecallCfg("t", B=cfg.requests, S=cfg.n_pages * 64, kmax=1, seed=77))
    t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).to(dev)
    idx = torch.empty((cfg.Q, cfg.k), dtype=torch.int32, device=dev)
    sc = torch.empty((cfg.Q, cfg.k), dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(cfg.Q, cfg.R), dtype=torch.uint8, device=dev)
    fm.fm_native_topk_paged_ex(t(q, np.int16), t(w), k8, sc8, t(phys), t(logical), cfg.k, idx, sc,
                               res_mask=t(mask, np.int32), mask_group=cfg.layers, workspace=ws)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    for qi in (0, 21 * 7 + 3, cfg.Q - 1):
        a, b = divmod(qi, cfg.layers)
        k8s = np.empty((cfg.R, 64, cfg.d), np.uint8)
        scs = np.empty((cfg.R, 64), np.float32)
        for j in range(cfg.R):
            lp = int(logical[qi, j])
            k8s[j], scs[j] = gen.paged_chunk_rows(cfg, a, b, np.arange(lp * 64, lp * 64 + 64))
        sub_phys = np.arange(cfg.R, dtype=np.int32)[None, :]
        ref, _, lg = orc.paged_topk(q[qi:qi + 1], w[qi:qi + 1], k8s, scs, sub_phys, logical[qi:qi + 1], k=cfg.k,
                                    want_logits=True, res_mask=mask[a:a + 1])
        score = {int(logical[qi, j]) * 64 + o: lg[0, j * 64 + o] for j in range(cfg.R) for o in range(64)}
        parity.assert_topk_parity(idx[qi], ref[0], score.__getitem__, cfg.k, fp8=True, got_scores=sc[qi])
