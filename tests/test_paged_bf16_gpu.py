"""Native paged top-k over a pool of bf16 keys (fm_native_topk_paged with
key_dtype FM_DTYPE_BF16, no scale) vs the oracle, on the GPU."""
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


def case(seed, requests=2, layers=3, n_pages=40, R=7):
    cfg = gen.PagedCfg("t", requests=requests, layers=layers, n_pages=n_pages, R=R, seed=seed)
    logical, phys, _ = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    kbf = gen.paged_pool_rows_bf16(cfg, logical, phys)
    return cfg, q, w, kbf, phys, logical


def run(torch, dev, q, w, kbf, phys, logical, k, n_res=None, res_mask=None, mask_group=1, id_mode=0):
    import sparse_attention_kv_c4_gb300 as fm
    Q, R = phys.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    idx = torch.full((Q, k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((Q, k), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(Q, R), dtype=torch.uint8, device=dev)
    args = (t(q.view(np.int16)), t(w), t(kbf.view(np.int16)), None, t(phys.astype(np.int32)),
            t(logical.astype(np.int32)), k, idx, sc)
    nr = None if n_res is None else t(np.asarray(n_res, np.int32))
    if res_mask is None and id_mode == 0:
        fm.fm_native_topk_paged(*args, n_res=nr, workspace=ws)
    else:
        fm.fm_native_topk_paged_ex(*args, n_res=nr, res_mask=None if res_mask is None else t(res_mask),
                                   mask_group=mask_group, id_mode=id_mode, workspace=ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), sc.cpu().numpy(), fm.fm_device_status(reset=True)


def check(orc, q, w, kbf, phys, logical, idx, sc, k, n_res=None):
    ref_idx, _, ref_lg = orc.paged_topk_bf16(q, w, kbf, phys, logical, n_res=n_res, k=k, want_logits=True)
    Q, R = phys.shape
    cand = (logical.astype(np.int64)[:, :, None] * 64 + np.arange(64)).reshape(Q, -1).copy()
    if n_res is not None:
        for qi in range(Q):
            cand[qi, max(0, min(R, int(n_res[qi]))) * 64:] = -1
    return parity.assert_topk_rows_parity(idx, sc, ref_idx, cand, ref_lg)


@pytest.mark.parametrize("k,R", [(64, 7), (512, 7), (100, 1), (512, 12), (1024, 30)])
def test_bf16_pool_matches_oracle(torch_dev, orc, k, R):
    torch, dev = torch_dev
    cfg, q, w, kbf, phys, logical = case(300 + R, R=R, n_pages=max(40, 2 * R))
    idx, sc, status = run(torch, dev, q, w, kbf, phys, logical, k)
    assert status == 0
    check(orc, q, w, kbf, phys, logical, idx, sc, k)


def test_bf16_pool_many_tiles_per_cta(torch_dev, orc):
    """Enough tiles that every CTA of the persistent scorer runs its stage
    ring around many times and crosses query boundaries (4 x 21 queries x
    384 pages)."""
    torch, dev = torch_dev
    cfg, q, w, kbf, phys, logical = case(333, requests=4, layers=21, n_pages=4096, R=384)
    idx, sc, status = run(torch, dev, q, w, kbf, phys, logical, 512)
    assert status == 0
    check(orc, q, w, kbf, phys, logical, idx, sc, 512)


def test_bf16_pool_nres_row_order_and_bad_pages(torch_dev, orc):
    torch, dev = torch_dev
    cfg, q, w, kbf, phys, logical = case(341, requests=3, layers=2, R=9)
    n_res = np.array([9, 0, 3, 4, 1, 12], dtype=np.int32)
    idx, sc, status = run(torch, dev, q, w, kbf, phys, logical, 128, n_res=n_res)
    assert status == 0
    check(orc, q, w, kbf, phys, logical, idx, sc, 128, n_res=n_res)
    perm = np.random.default_rng(2).permutation(9)
    idx2, sc2, _ = run(torch, dev, q, w, kbf, phys[:, perm], logical[:, perm], 128, n_res=None)
    idx3, sc3, _ = run(torch, dev, q, w, kbf, phys, logical, 128)
    assert (idx2 == idx3).all() and np.array_equal(sc2, sc3)
    bad = phys.copy()
    bad[0, 2] = cfg.P + 1
    idx4, sc4, status = run(torch, dev, q, w, kbf, bad, logical, 128)
    assert status & 0x1
    keep = [0, 1, 3, 4, 5, 6, 7, 8, 2]
    nr = np.full(cfg.Q, 9, np.int32)
    nr[0] = 8
    p2, l2 = phys.copy(), logical.copy()
    p2[0], l2[0] = phys[0, keep], logical[0, keep]
    check(orc, q, w, kbf, p2, l2, idx4, sc4, 128, n_res=nr)


def test_bf16_pool_resident_mask_and_remap(torch_dev, orc):
    torch, dev = torch_dev
    cfg, q, w, kbf, phys, logical = case(353, requests=2, layers=3, n_pages=30, R=6)
    rng = np.random.default_rng(4)
    mask = np.packbits(rng.random((cfg.requests, 30 * 64)) < 0.3, axis=-1, bitorder="little").view("<u4")
    mask = mask.reshape(cfg.requests, -1)
    idx0, sc0, status = run(torch, dev, q, w, kbf, phys, logical, 100, res_mask=mask, mask_group=cfg.layers)
    assert status == 0
    ref0, _, ref_lg = orc.paged_topk_bf16(q, w, kbf, phys, logical, k=100, res_mask=mask, mask_group=cfg.layers,
                                          want_logits=True)
    bits = np.unpackbits(mask.view(np.uint8), axis=-1, bitorder="little")
    cand = (logical.astype(np.int64)[:, :, None] * 64 + np.arange(64)).reshape(cfg.Q, -1).copy()
    for qi in range(cfg.Q):
        cand[qi, ~bits[qi // cfg.layers][cand[qi]].astype(bool)] = -1  # non-resident: not a candidate
    parity.assert_topk_rows_parity(idx0, sc0, ref0, cand, ref_lg)
    # the fused remap emits the same selection as reserve cells, in the order
    # of the logical ids: exact wherever the selection equals the oracle's
    idx1, sc1, status = run(torch, dev, q, w, kbf, phys, logical, 100, res_mask=mask, mask_group=cfg.layers,
                            id_mode=1)
    assert status == 0
    ref1, _ = orc.paged_topk_bf16(q, w, kbf, phys, logical, k=100, res_mask=mask, mask_group=cfg.layers, id_mode=1)
    same = (idx0 == ref0).all(axis=1)
    assert same.sum() >= cfg.Q - 1
    assert (idx1[same] == ref1[same]).all()
    assert np.array_equal(sc1, sc0)


def test_bf16_pool_takes_no_scale(torch_dev):
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    q = torch.zeros((2, 64, 128), dtype=torch.int16, device=dev)
    w = torch.zeros((2, 64), dtype=torch.float32, device=dev)
    pool = torch.zeros((3, 64, 128), dtype=torch.int16, device=dev)
    scale = torch.ones((3, 64), dtype=torch.float32, device=dev)
    table = torch.zeros((2, 1), dtype=torch.int32, device=dev)
    idx = torch.empty((2, 8), dtype=torch.int32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(2, 1), dtype=torch.uint8, device=dev)
    with pytest.raises(fm.FmError) as e:
        fm.fm_native_topk_paged(q, w, pool, scale, table, table, 8, idx, workspace=ws)
    assert e.value.status == fm.FM_ERR_INVALID_ARG


def test_bf16_pool_device_fill_matches_host(torch_dev):
    """The generator's device fill of a bf16 pool (used by the benchmark row)
    gives the host builder's values bit for bit."""
    torch, dev = torch_dev
    cfg = gen.PagedCfg("t", requests=2, layers=3, n_pages=50, R=6, seed=361)
    logical, phys, owner = gen.paged_tables(cfg)
    host = gen.paged_pool_rows_bf16(cfg, logical, phys)
    own_d = torch.from_numpy(owner).to(dev)
    kd = torch.empty((cfg.P, cfg.page, cfg.d), dtype=torch.int16, device=dev)
    gen.paged_pool_bf16_device(cfg, own_d.data_ptr(), kd.data_ptr())
    torch.cuda.synchronize()
    assert (kd.cpu().numpy().view(np.uint16) == host).all()
