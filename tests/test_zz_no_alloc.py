"""The scratch-free paged top-k (fm_native_topk_paged_noalloc).

Callers that cannot allocate device memory -- an engine whose KV-cache pool
owns nearly all of HBM, a decode loop that must not stall on cudaMalloc's
implicit synchronisation, a plugin host with no allocator -- use this entry
point instead of fm_native_topk_paged.  It must give the same top-k ids and
scores as the workspace entry point, on every call, even though all calls
share one scratch array that keeps the previous call's contents.  This file
is collected last so that a run stopping at its first failure has already run
every other test.
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


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(torch_dev):
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


def test_noalloc_rejects_sizes_beyond_its_scratch(torch_dev):
    import sparse_attention_kv_c4_gb300 as fm
    torch, dev = torch_dev
    Q, R = 1024, 2048  # needs far more than the built-in scratch
    assert fm.fm_native_topk_paged_workspace(Q, R) > 16 << 20
    q = torch.zeros((Q, 64, 128), dtype=torch.int16, device=dev)
    w = torch.zeros((Q, 64), dtype=torch.float32, device=dev)
    pool = torch.zeros((1, 64, 128), dtype=torch.uint8, device=dev)
    scale = torch.ones((1, 64), dtype=torch.float32, device=dev)
    table = torch.zeros((Q, R), dtype=torch.int32, device=dev)
    idx = torch.empty((Q, 512), dtype=torch.int32, device=dev)
    with pytest.raises(fm.FmError) as e:
        fm.fm_native_topk_paged_noalloc(q, w, pool, scale, table, table, 512, idx)
    assert e.value.status == fm.FM_ERR_INVALID_ARG and "scratch" in str(e.value)
