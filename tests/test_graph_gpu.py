"""The whole indexer path captured in one CUDA graph ([RM] key optimisations:
"Two-level recall inside cuda-graph").  Every entry point is asynchronous on
the caller's stream and allocates nothing, so a decode cycle (Memory Indexer
-> page recall -> masked paged top-k with remap) and a prefill call can be
captured once and replayed; replays must reproduce the eager results bit for
bit (the kernels are deterministic: fixed MMA order, exact top-k with ids in
order)."""
import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch, torch.device("cuda:0")


def test_decode_and_prefill_in_one_graph(torch_dev):
    torch, dev = torch_dev
    import sparse_attention_kv_c4_gb300 as fm
    t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).to(dev)

    # Memory Indexer over 2 requests x 3 layers x 40 pages of chunks
    layers, n_pages = 3, 40
    mi = gen.MemIndexCfg("g", B=2, L=layers, S=n_pages * 64, seed=gen.BASE_SEED + 200)
    q, w, hot = gen.memindex_qw(mi)
    K = gen.memindex_keys_host(mi, hot)
    mq, mw, mK = t(q, np.int16), t(w), t(K, np.int16)
    mask = torch.empty((mi.B, (mi.S + 31) // 32), dtype=torch.int32, device=dev)
    maxsig = torch.empty((mi.B, mi.S), dtype=torch.float32, device=dev)
    # page recall of that mask
    kmax = 9
    pages = torch.empty((mi.B, kmax), dtype=torch.int32, device=dev)
    n_rec = torch.empty((mi.B,), dtype=torch.int32, device=dev)
    # native paged top-k of 2 x 3 queries over a seeded pool, confined to the
    # Memory Indexer's mask, ids remapped to reserve cells
    pc = gen.PagedCfg("g", requests=mi.B, layers=layers, n_pages=n_pages, R=9, seed=gen.BASE_SEED + 201)
    logical, phys, owner = gen.paged_tables(pc)
    pq, pw = gen.paged_qw(pc)
    k8, scale = gen.paged_pool_host(pc, owner)
    pq_d, pw_d, k8_d, sc_d, ph_d, lg_d = t(pq, np.int16), t(pw), t(k8), t(scale), t(phys), t(logical)
    pidx = torch.empty((pc.Q, 256), dtype=torch.int32, device=dev)
    pscore = torch.empty((pc.Q, 256), dtype=torch.float32, device=dev)
    pws = torch.empty(fm.fm_native_topk_paged_workspace(pc.Q, pc.R), dtype=torch.uint8, device=dev)
    # prefill: 64 tokens against 4096 chunks
    pf = gen.PrefillCfg("g", T=64, S=4096, pos0=4 * 4000, seed=gen.BASE_SEED + 202)
    fq, fw, fpos, fK = gen.prefill_host(pf)
    fq_d, fw_d, fpos_d, fK_d = t(fq, np.int16), t(fw), t(fpos), t(fK, np.int16)
    fidx = torch.empty((pf.T, pf.k), dtype=torch.int32, device=dev)
    fscore = torch.empty((pf.T, pf.k), dtype=torch.float32, device=dev)
    fws = torch.empty(fm.fm_index_prefill_workspace(pf.T, pf.S), dtype=torch.uint8, device=dev)

    outs = [mask, maxsig, pages, n_rec, pidx, pscore, fidx, fscore]

    def step():
        fm.fm_memindex_score_mask(mq, mw, mK, mask, maxsig)
        fm.fm_page_recall(mask, mi.S, kmax, pages, None, n_rec, recent=64)
        fm.fm_native_topk_paged_ex(pq_d, pw_d, k8_d, sc_d, ph_d, lg_d, 256, pidx, pscore, res_mask=mask,
                                   mask_group=layers, id_mode=1, workspace=pws)
        fm.fm_index_prefill_topk(fq_d, fw_d, fpos_d, fK_d, pf.k, fidx, fscore, workspace=fws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager, outside capture: loads every kernel and sets its attributes
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    assert fm.fm_device_status(reset=True) == 0

    for o in outs:
        o.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        for o in outs:
            o.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, eager):
            assert torch.equal(a, b)
    assert fm.fm_device_status(reset=True) == 0
    # the graph is live: the recalled pages and the masked selection are non-trivial
    assert int(n_rec.min()) > 0 and int((pidx >= 0).sum()) > 0


def test_query_chain_layers_in_one_graph(torch_dev):
    """Three layers of the query chain (its second to fourth kernels use
    programmatic dependent launch) captured in one CUDA graph, followed by
    the retriever over the chain's output: replays reproduce the eager
    results bit for bit (the K-split partials are summed in a fixed order)."""
    torch, dev = torch_dev
    import sparse_attention_kv_c4_gb300 as fm
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).to(dev)
    T, L, n_h, dim, r = 6, 3, 128, 1024, 512
    sets = [[t(a) for a in gen.query_chain_inputs(T, dim=dim, r=r, n_h=n_h, seed=gen.BASE_SEED + 700 + l)]
            for l in range(L)]
    q = torch.empty((T, L, n_h, 128), dtype=torch.int16, device=dev)
    w = torch.empty((T, L, n_h), dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_query_chain_workspace(T, r, n_h), dtype=torch.uint8, device=dev)
    S = 1024
    cfg = gen.MemIndexCfg("gq", B=T, L=L, S=S, n_h=n_h, seed=gen.BASE_SEED + 710)
    k8, sc = gen.memindex_fp8_keys_host(cfg, np.zeros((T, L, n_h), np.float32))
    ck = torch.from_numpy(gen.pack_compressed_k(k8, sc)).to(dev)
    mask = torch.empty((T, S // 32), dtype=torch.int32, device=dev)
    ens = torch.empty((T, S), dtype=torch.float32, device=dev)
    rws = torch.empty(fm.fm_retriever_workspace(T, L, n_h), dtype=torch.uint8, device=dev)
    # the chain's per-layer outputs are strided views of q / w ([T, L, ...])
    q_l = [torch.empty((T, n_h, 128), dtype=torch.int16, device=dev) for _ in range(L)]
    w_l = [torch.empty((T, n_h), dtype=torch.float32, device=dev) for _ in range(L)]

    def run():
        for l, (hidden, wq_a, q_norm, wq_b, w_proj, pos) in enumerate(sets):
            fm.fm_query_chain(hidden, wq_a, q_norm, wq_b, w_proj, pos, q_l[l], w_l[l], workspace=ws)
        for l in range(L):
            q[:, l].copy_(q_l[l])
            w[:, l].copy_(w_l[l])
        fm.fm_retriever_score_mask(q, w, ck, mask, ens, workspace=rws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    ref = [x.clone() for x in (q, w, mask, ens)]
    for x in (q, w, mask, ens):
        x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    for _ in range(3):
        for x in (q, w, mask, ens):
            x.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip((q, w, mask, ens), ref):
            assert torch.equal(a, b)
    assert fm.fm_device_status(reset=True) == 0
