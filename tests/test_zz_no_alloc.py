"""The scratch-free paged top-k (fm_native_topk_paged_noalloc).

Callers that cannot allocate device memory -- an engine whose KV-cache pool
owns nearly all of HBM, a decode loop that must not stall on cudaMalloc's
implicit synchronisation, a plugin host with no allocator -- use this entry
point instead of fm_native_topk_paged.  It must give the same top-k ids and
scores as the workspace entry point, on every call, even though all calls
share one scratch array that keeps the previous call's contents.  This file
is collected last so that a run stopping at its first failure has already run
every other test.  Its cases check the no-allocation call against the oracle
as well as against the workspace entry point, at the scratch array's size
limit and on the long-table (R > 1024) path.
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


def _case(torch, dev, seed, requests, layers, R):
    cfg = gen.PagedCfg("t", requests=requests, layers=layers, n_pages=4 * R + 5, R=R, seed=seed)
    logical, phys, owner = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    k8, scale = gen.paged_pool_host(cfg, owner)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return cfg, (t(q.view(np.int16)), t(w), t(k8), t(scale), t(phys), t(logical))


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(torch_dev, orc):
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    # two different problems back to back: the second call reuses a scratch
    # array that still holds the first call's data
    for seed, requests, layers, R, k in [(41, 2, 3, 9, 256), (42, 3, 2, 5, 512)]:
        cfg, args = _case(torch, dev, seed, requests, layers, R)
        Q = cfg.Q
        idx_ws = torch.full((Q, k), -7, dtype=torch.int32, device=dev)
        sc_ws = torch.full((Q, k), 7.0, dtype=torch.float32, device=dev)
        ws = torch.empty(fm.fm_native_topk_paged_workspace(Q, R), dtype=torch.uint8, device=dev)
        fm.fm_native_topk_paged(*args, k, idx_ws, sc_ws, workspace=ws)
        idx_na = torch.full((Q, k), -9, dtype=torch.int32, device=dev)
        sc_na = torch.full((Q, k), 9.0, dtype=torch.float32, device=dev)
        fm.fm_native_topk_paged_noalloc(*args, k, idx_na, sc_na)
        torch.cuda.synchronize()
        assert fm.fm_device_status(reset=True) == 0
        a, b = idx_ws.cpu().numpy(), idx_na.cpu().numpy()
        assert (a == b).all(), "top-k ids differ from the workspace entry point"
        sa, sb = sc_ws.cpu().numpy(), sc_na.cpu().numpy()
        n = a >= 0
        parity.assert_logits_close(sb[n], sa[n], fp8=True, what="noalloc scores")
        assert np.isneginf(sb[~n]).all()
        q, w = gen.paged_qw(cfg)
        logical, phys, _ = gen.paged_tables(cfg)
        k8, scale = gen.paged_pool_rows(cfg, logical, phys)
        ref_idx, cand, ref_lg = _oracle_rows(orc, cfg, q, w, k8, scale, phys, logical, k)
        parity.assert_topk_rows_parity(b, sb, ref_idx, cand, ref_lg, fp8=True)


def _oracle_rows(orc, cfg, q, w, k8, scale, phys, logical, k):
    ref_idx, _, ref_lg = orc.paged_topk(q, w, k8, scale, phys, logical, k=k, want_logits=True)
    cand = (logical.astype(np.int64)[:, :, None] * 64 + np.arange(64)).reshape(cfg.Q, -1)
    return ref_idx, cand, ref_lg


@pytest.mark.parametrize("requests,layers,R,k", [
    (8, 17, 384, 512),   # 136 queries: the largest batch whose workspace fits the 16 MiB scratch
    (1, 3, 1500, 512),   # a table longer than 1024 entries (the 1024-thread prep kernel)
])
def test_noalloc_at_its_size_limits_matches_oracle(torch_dev, orc, requests, layers, R, k):
    """The scratch filled to its limit, and the long-table prep path, against
    the workspace entry point (bit for bit) and the oracle (parity rules)."""
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    cfg = gen.PagedCfg("t", requests=requests, layers=layers, n_pages=max(2048, 2 * R), R=R,
                       seed=gen.BASE_SEED + 700 + R)
    Q = cfg.Q
    assert fm.fm_native_topk_paged_workspace(Q, R) <= fm.FM_NOALLOC_SCRATCH_BYTES
    if R == 384:
        assert fm.fm_native_topk_paged_workspace(Q + 1, R) > fm.FM_NOALLOC_SCRATCH_BYTES
    logical, phys, _ = gen.paged_tables(cfg)
    q, w = gen.paged_qw(cfg)
    k8, scale = gen.paged_pool_rows(cfg, logical, phys)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    args = (t(q.view(np.int16)), t(w), t(k8), t(scale), t(phys), t(logical))
    idx_na = torch.full((Q, k), -9, dtype=torch.int32, device=dev)
    sc_na = torch.full((Q, k), 9.0, dtype=torch.float32, device=dev)
    fm.fm_native_topk_paged_noalloc(*args, k, idx_na, sc_na)
    idx_ws = torch.full((Q, k), -7, dtype=torch.int32, device=dev)
    sc_ws = torch.full((Q, k), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_native_topk_paged_workspace(Q, R), dtype=torch.uint8, device=dev)
    fm.fm_native_topk_paged(*args, k, idx_ws, sc_ws, workspace=ws)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    a, b = idx_na.cpu().numpy(), idx_ws.cpu().numpy()
    assert (a == b).all(), "top-k ids differ from the workspace entry point"
    sa = sc_na.cpu().numpy()
    assert np.array_equal(sa.view(np.uint32), sc_ws.cpu().numpy().view(np.uint32))
    ref_idx, cand, ref_lg = _oracle_rows(orc, cfg, q, w, k8, scale, phys, logical, k)
    parity.assert_topk_rows_parity(a, sa, ref_idx, cand, ref_lg, fp8=True)


def test_noalloc_rejects_sizes_beyond_its_scratch(torch_dev):
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    Q, R = 137, 384  # one query more than the built-in scratch holds
    assert fm.fm_native_topk_paged_workspace(Q, R) > fm.FM_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((Q, 64, 128), dtype=torch.int16, device=dev)
    w = torch.zeros((Q, 64), dtype=torch.float32, device=dev)
    pool = torch.zeros((1, 64, 128), dtype=torch.uint8, device=dev)
    scale = torch.ones((1, 64), dtype=torch.float32, device=dev)
    table = torch.zeros((Q, R), dtype=torch.int32, device=dev)
    idx = torch.empty((Q, 512), dtype=torch.int32, device=dev)
    with pytest.raises(fm.FmError) as e:
        fm.fm_native_topk_paged_noalloc(q, w, pool, scale, table, table, 512, idx)
    assert e.value.status == fm.FM_ERR_INVALID_ARG and "scratch" in str(e.value)
