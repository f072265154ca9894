"""Native paged top-k (fm_native_topk_paged) vs the oracle, on the GPU."""
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


def run_paged(torch, dev, q, w, k8, scale, phys, logical, k, n_res=None, pool_dev=None):
    import sparse_attention_kv_c4_gb300 as fm
    Q, R = phys.shape
    qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    if pool_dev is None:
        kd = torch.from_numpy(np.ascontiguousarray(k8)).to(dev)
        sd = torch.from_numpy(np.ascontiguousarray(scale)).to(dev)
    else:
        kd, sd = pool_dev
    pd = torch.from_numpy(np.ascontiguousarray(phys, dtype=np.int32)).to(dev)
    ld = torch.from_numpy(np.ascontiguousarray(logical, dtype=np.int32)).to(dev)
    nd = None if n_res is None else torch.from_numpy(np.asarray(n_res, dtype=np.int32)).to(dev)
    idx = torch.full((Q, k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((Q, k), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(Q, R), dtype=torch.uint8, device=dev)
    fm.fm_native_topk_paged(qd, wd, kd, sd, pd, ld, k, idx, sc, n_res=nd, workspace=ws)
    torch.cuda.synchronize()
    status = fm.fm_device_status(reset=True)
    return idx.cpu().numpy(), sc.cpu().numpy(), status


def check_rows(orc, q, w, k8, scale, phys, logical, idx, sc, k, n_res=None):
    ref_idx, ref_sc, ref_lg = orc.paged_topk(q, w, k8, scale, phys, logical, n_res=n_res, k=k, want_logits=True)
    Q, R = phys.shape
    exempt = 0
    for qi in range(Q):
        nr = R if n_res is None else max(0, min(R, int(n_res[qi])))
        score = {int(logical[qi, j]) * 64 + o: ref_lg[qi, j * 64 + o] for j in range(nr) for o in range(64)}
        exempt += parity.assert_topk_parity(idx[qi], ref_idx[qi], score.__getitem__, k, fp8=True,
                                            got_scores=sc[qi])
    return exempt


def small_case(seed, requests=2, layers=3, n_pages=40, R=7):
    cfg = gen.PagedCfg("t", requests=requests, layers=layers, n_pages=n_pages, R=R, seed=seed)
    logical, phys, owner = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    k8, scale = gen.paged_pool_host(cfg, owner)
    return cfg, q, w, k8, scale, phys, logical


@pytest.mark.parametrize("k,R", [(64, 7), (512, 7), (100, 1), (512, 12), (1024, 30)])
def test_paged_matches_oracle(torch_dev, orc, k, R):
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(100 + R, R=R, n_pages=max(40, 2 * R))
    idx, sc, status = run_paged(torch, dev, q, w, k8, scale, phys, logical, k)
    assert status == 0
    check_rows(orc, q, w, k8, scale, phys, logical, idx, sc, k)


def test_paged_scores_close_to_oracle_everywhere(torch_dev, orc):
    """With k >= candidates every resident chunk is returned with its score."""
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(5, R=5)
    idx, sc, status = run_paged(torch, dev, q, w, k8, scale, phys, logical, 1024)
    _, _, ref_lg = orc.paged_topk(q, w, k8, scale, phys, logical, k=1024, want_logits=True)
    for qi in range(cfg.Q):
        sel = idx[qi][idx[qi] >= 0]
        assert len(sel) == 5 * 64
        score = {int(logical[qi, j]) * 64 + o: ref_lg[qi, j * 64 + o] for j in range(5) for o in range(64)}
        ref = np.array([score[int(i)] for i in sel])
        err = parity.assert_logits_close(sc[qi][: len(sel)], ref, fp8=True)
        assert err < 2e-3, f"paged score relative error {err} (expected ~1e-5)"


def test_paged_nres_and_row_order(torch_dev, orc):
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(9, requests=3, layers=2, R=9)
    n_res = np.array([9, 0, 3, 4, 1, 12], dtype=np.int32)
    idx, sc, status = run_paged(torch, dev, q, w, k8, scale, phys, logical, 128, n_res=n_res)
    assert status == 0
    check_rows(orc, q, w, k8, scale, phys, logical, idx, sc, 128, n_res=n_res)
    assert (idx[1] == -1).all()
    perm = np.random.default_rng(1).permutation(9)
    idx2, sc2, _ = run_paged(torch, dev, q, w, k8, scale, phys[:, perm].copy(), logical[:, perm].copy(), 128)
    idx3, sc3, _ = run_paged(torch, dev, q, w, k8, scale, phys, logical, 128)
    assert (idx2 == idx3).all() and np.array_equal(sc2, sc3)


def test_paged_ties_choose_lower_ids(torch_dev):
    """q = 0 gives every chunk the score 0: the k lowest chunk ids win."""
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(11, R=6)
    q = np.zeros_like(q)
    idx, sc, status = run_paged(torch, dev, q, w, k8, scale, phys, logical, 100)
    for qi in range(cfg.Q):
        ids = sorted(int(lp) * 64 + o for lp in logical[qi] for o in range(64))
        assert list(idx[qi]) == ids[:100]
        assert (sc[qi] == 0).all()


def test_paged_bad_pages_are_flagged_and_skipped(torch_dev, orc):
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(13, R=6)
    phys = phys.copy()
    logical = logical.copy()
    phys[0, 2] = cfg.P + 5          # out of range
    logical[1, 4] = logical[1, 1]   # repeated logical page
    idx, sc, status = run_paged(torch, dev, q, w, k8, scale, phys, logical, 512)
    assert status & 0x1 and status & 0x4
    row0 = set(int(i) for i in idx[0] if i >= 0)
    assert len(row0) == 5 * 64 and not any(i // 64 == logical[0, 2] for i in row0)
    row1 = [int(i) for i in idx[1] if i >= 0]
    assert len(row1) == 5 * 64 and len(set(row1)) == len(row1)
    # the surviving rows equal the oracle's on the tables with the flagged
    # entries removed: the out-of-range entry of row 0, and the later of the
    # two entries of row 1 that repeat a logical page (the first one listed is
    # kept); removed entries go last and n_res leaves them out
    keep = {0: [0, 1, 3, 4, 5], 1: [0, 1, 2, 3, 5]}
    n_res = np.full(cfg.Q, 6, dtype=np.int32)
    for r, cols in keep.items():
        order = cols + [c for c in range(6) if c not in cols]
        phys[r], logical[r] = phys[r, order], logical[r, order]
        n_res[r] = len(cols)
    phys[0, 5] = 0  # the removed entry is past n_res; any in-range value
    check_rows(orc, q, w, k8, scale, phys, logical, idx, sc, 512, n_res=n_res)


def test_paged_scale_signs(torch_dev, orc):
    """Negative and zero chunk scales take the general ReLU(scale * dot) path."""
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(17, R=4)
    scale = scale.copy()
    scale[::3, ::5] *= -1.0
    scale[1::4, 3::7] = 0.0
    idx, sc, status = run_paged(torch, dev, q, w, k8, scale, phys, logical, 200)
    assert status == 0
    check_rows(orc, q, w, k8, scale, phys, logical, idx, sc, 200)


# The 512K and 1M paged workloads are compared in full in test_full_configs_gpu.py.


def test_paged_full_history_whole_rows(torch_dev, orc):
    """Full-history scoring: every page of a 4096-page (1M-token) history is
    listed, in a shuffled table order; each query's 262144 chunks are all
    candidates and the whole rows are compared with the oracle."""
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(gen.BASE_SEED + 910, requests=1, layers=2, n_pages=4096,
                                                     R=4096)
    assert sorted(logical[0].tolist()) == list(range(4096))
    idx, sc, status = run_paged(torch, dev, q, w, k8, scale, phys, logical, 512)
    assert status == 0
    check_rows(orc, q, w, k8, scale, phys, logical, idx, sc, 512)


def test_paged_full_history_1m_sampled(torch_dev, orc):
    """The full-history configuration at full size (630 queries x 4096 pages,
    21.8 GB pool filled on the device); sampled queries recomputed by the
    oracle over all 262144 of their chunks."""
    torch, dev = torch_dev
    cfg = gen.PAGED_FULL_1M
    logical, phys, owner = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    own_d = torch.from_numpy(owner).to(dev)
    k8d = torch.empty((cfg.P, cfg.page, cfg.d), dtype=torch.uint8, device=dev)
    scd = torch.empty((cfg.P, cfg.page), dtype=torch.float32, device=dev)
    gen.paged_pool_device(cfg, own_d.data_ptr(), k8d.data_ptr(), scd.data_ptr())
    idx, sc, status = run_paged(torch, dev, q, w, None, None, phys, logical, cfg.k, pool_dev=(k8d, scd))
    assert status == 0
    del k8d, scd, own_d
    torch.cuda.empty_cache()
    rng = np.random.default_rng(cfg.seed)
    for qi in rng.choice(cfg.Q, size=2, replace=False):
        a, b = qi // cfg.layers, qi % cfg.layers
        k8s, scs = gen.paged_chunk_rows(cfg, a, b, np.arange(cfg.n_pages * cfg.page))
        k8s = k8s.reshape(cfg.n_pages, cfg.page, cfg.d)
        scs = scs.reshape(cfg.n_pages, cfg.page)
        # logical page j sits in local pool page j
        check_rows(orc, q[qi:qi + 1], w[qi:qi + 1], k8s, scs, logical[qi:qi + 1], logical[qi:qi + 1],
                   idx[qi:qi + 1], sc[qi:qi + 1], cfg.k)


def test_check_device_status_reports_bounds(torch_dev, orc):
    """fm_check_device_status turns the flagged status word into
    FM_ERR_DEVICE_BOUNDS once, and clears it."""
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    cfg, q, w, k8, scale, phys, logical = small_case(19, R=4)
    fm.fm_check_device_status()  # a clean word to start from
    phys = phys.copy()
    phys[2, 1] = -3
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    idx = torch.empty((cfg.Q, 64), dtype=torch.int32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(cfg.Q, cfg.R), dtype=torch.uint8, device=dev)
    fm.fm_native_topk_paged(t(q.view(np.int16)), t(w), t(k8), t(scale), t(phys), t(logical), 64, idx, workspace=ws)
    with pytest.raises(fm.FmError) as e:
        fm.fm_check_device_status()
    assert e.value.status == fm.FM_ERR_DEVICE_BOUNDS and "out of range" in str(e.value)
    fm.fm_check_device_status()  # cleared
