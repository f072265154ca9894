"""The query side of a CSA layer (fm_query_chain: wq_a -> RMSNorm -> wq_b ->
YaRN rotary -> Walsh-Hadamard, and the head weights) vs the oracle, on the
GPU, at the retriever's sizes (dim 4096, rank 2048, 128 heads of 128).

Tolerance: the only rounding beyond fp32 accumulation is the bf16 RMSNorm
output fed to wq_b (relative 2^-9 per element); wq_b, the rotation and the
orthonormal Hadamard carry that to at most a few 2^-9 of a head's rms, so q
(fp32) must agree within 2^-6 of the head's rms; the bf16 q within that plus
half a bf16 ulp; w (fp32 GEMM, no rounding) within 1e-5 of its rms."""
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


def _run(torch, dev, inputs, n_h):
    import sparse_attention_kv_c4_gb300 as fm
    hidden, wq_a, q_norm, wq_b, w_proj, pos = inputs
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).to(dev)
    T = hidden.shape[0]
    q = torch.zeros((T, n_h, 128), dtype=torch.int16, device=dev)
    q32 = torch.zeros((T, n_h, 128), dtype=torch.float32, device=dev)
    w = torch.zeros((T, n_h), dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_query_chain_workspace(T, wq_a.shape[0], n_h), dtype=torch.uint8, device=dev)
    fm.fm_query_chain(t(hidden), t(wq_a), t(q_norm), t(wq_b), t(w_proj), t(pos), q, w, q_out_f32=q32, workspace=ws)
    torch.cuda.synchronize()
    qb = (q.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return qb, q32.cpu().numpy().astype(np.float64), w.cpu().numpy().astype(np.float64)


def _check(q_ref, w_ref, qb, q32, w):
    rms = np.sqrt((q_ref ** 2).mean(axis=-1, keepdims=True))
    tol = 2.0 ** -6 * rms + 1e-6
    assert np.all(np.abs(q32 - q_ref) <= tol), float((np.abs(q32 - q_ref) / rms).max())
    assert np.all(np.abs(qb - q_ref) <= tol + 2.0 ** -8 * np.abs(q_ref))
    wr = np.sqrt((w_ref ** 2).mean(axis=-1, keepdims=True))
    assert np.all(np.abs(w - w_ref) <= 1e-5 * wr + 1e-8), float((np.abs(w - w_ref) / wr).max())


@pytest.mark.parametrize("T,n_h", [(3, 128), (5, 64), (1, 128)])
def test_query_chain_matches_oracle(torch_dev, orc, T, n_h):
    torch, dev = torch_dev
    inputs = gen.query_chain_inputs(T, n_h=n_h, seed=gen.BASE_SEED + 500 + T + n_h)
    q_ref, w_ref = orc.query_chain(*inputs, n_h=n_h)
    _check(q_ref, w_ref, *_run(torch, dev, inputs, n_h))


def test_query_chain_decode_batch(torch_dev, orc):
    """A decode batch of 30 tokens (one per request of the 1M-context
    workload) at the retriever's sizes: the projections' token operand spans
    two 16-row groups and the K splits of both GEMMs are summed."""
    torch, dev = torch_dev
    inputs = gen.query_chain_inputs(30, seed=gen.BASE_SEED + 560)
    q_ref, w_ref = orc.query_chain(*inputs, n_h=128)
    _check(q_ref, w_ref, *_run(torch, dev, inputs, 128))


@pytest.mark.parametrize("T", [40, 256, 300])
def test_query_chain_many_tokens(torch_dev, orc, T):
    """More tokens than one projection launch takes (256): 300 tokens run as
    blocks of 256 and 44; dims not multiples of 64 leave ragged K chunks."""
    torch, dev = torch_dev
    inputs = gen.query_chain_inputs(T, dim=520, r=264, n_h=8, seed=gen.BASE_SEED + 570 + T)
    q_ref, w_ref = orc.query_chain(*inputs, n_h=8)
    _check(q_ref, w_ref, *_run(torch, dev, inputs, 8))


def test_query_chain_small_dims_and_positions(torch_dev, orc):
    """Other widths (dim 512, rank 256) and positions across the whole range,
    including ones where fp32 angles would be off by whole radians."""
    torch, dev = torch_dev
    pos = np.array([0, 1, 4095, 65536, 300000, (1 << 20) - 1, (1 << 31) - 1], dtype=np.int64)
    inputs = gen.query_chain_inputs(len(pos), dim=512, r=256, n_h=8, seed=gen.BASE_SEED + 520, pos=pos)
    q_ref, w_ref = orc.query_chain(*inputs, n_h=8)
    _check(q_ref, w_ref, *_run(torch, dev, inputs, 8))


def test_query_chain_feeds_the_retriever(torch_dev, orc):
    """End to end: the chain's q and w drive the retriever over packed keys;
    its logits match the oracle's logits computed from the oracle's own chain
    output (within the fp8 tolerance widened by the chain's bf16 rounding)."""
    torch, dev = torch_dev
    import parity
    import sparse_attention_kv_c4_gb300 as fm
    L, S = 3, 512
    chains = [gen.query_chain_inputs(2, seed=gen.BASE_SEED + 530 + l) for l in range(L)]
    refs = [orc.query_chain(*c, n_h=128) for c in chains]
    outs = [_run(torch, dev, c, 128) for c in chains]
    # q [B=2, L, 128, 128] bf16 from the GPU chain; the oracle's q rounded the same way
    q_gpu = np.stack([o[0] for o in outs], axis=1)
    w_gpu = np.stack([o[2] for o in outs], axis=1).astype(np.float32)
    qbits = (q_gpu.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    cfg = gen.MemIndexCfg("chain", B=2, L=L, S=S, n_h=128, seed=gen.BASE_SEED + 540)
    hot = np.zeros((2, L, 128), np.float32)
    k8, sc = gen.memindex_fp8_keys_host(cfg, hot)
    ck = gen.pack_compressed_k(k8, sc)
    mask = torch.empty((2, S // 32), dtype=torch.int32, device=dev)
    logits = torch.empty((2, L, S), dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_retriever_workspace(2, L, 128), dtype=torch.uint8, device=dev)
    fm.fm_retriever_score_mask(torch.from_numpy(qbits.view(np.int16)).to(dev), torch.from_numpy(w_gpu).to(dev),
                               torch.from_numpy(ck).to(dev), mask, None, logits, workspace=ws)
    torch.cuda.synchronize()
    x_gpu = logits.cpu().numpy()
    x_same_q = orc.memindex_logits_fp8(qbits, w_gpu, k8, sc)  # the retriever is exact on its own inputs
    parity.assert_logits_close(x_gpu, x_same_q, fp8=True)
    q_ref = np.stack([r[0] for r in refs], axis=1)
    w_ref = np.stack([r[1] for r in refs], axis=1).astype(np.float32)
    u = q_ref.astype(np.float32).view(np.uint32).astype(np.uint64)
    q_ref_bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    x_ref = orc.memindex_logits_fp8(q_ref_bits, w_ref, k8, sc)
    assert np.all(np.abs(x_gpu - x_ref) <= 2.0 ** -5 * (np.abs(x_ref) + np.abs(x_ref).mean()) + 1e-3)


@pytest.mark.parametrize("L,T,n_h,dim,r", [(3, 30, 128, 4096, 2048), (2, 5, 64, 1024, 512), (4, 300, 8, 520, 264)])
def test_query_chain_layers_match_oracle(torch_dev, orc, L, T, n_h, dim, r):
    """fm_query_chain_layers: every layer against the oracle's chain for that
    layer (its own weights, the shared positions), outputs in [T, L, ...]."""
    torch, dev = torch_dev
    import sparse_attention_kv_c4_gb300 as fm
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).to(dev)
    ins = [gen.query_chain_inputs(T, dim=dim, r=r, n_h=n_h, seed=gen.BASE_SEED + 800 + 10 * L + l) for l in range(L)]
    pos = ins[0][5]
    dev_in = [[t(a) for a in x[:5]] for x in ins]
    q = torch.zeros((T, L, n_h, 128), dtype=torch.int16, device=dev)
    q32 = torch.zeros((T, L, n_h, 128), dtype=torch.float32, device=dev)
    w = torch.zeros((T, L, n_h), dtype=torch.float32, device=dev)
    ws = torch.empty(fm.fm_query_chain_layers_workspace(L, T, r, n_h), dtype=torch.uint8, device=dev)
    fm.fm_query_chain_layers([x[0] for x in dev_in], [x[1] for x in dev_in], [x[2] for x in dev_in],
                             [x[3] for x in dev_in], [x[4] for x in dev_in], t(pos), q, w, q_out_f32=q32,
                             workspace=ws)
    torch.cuda.synchronize()
    assert fm.fm_device_status(reset=True) == 0
    qb_all = (q.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for l in range(L):
        hidden, wq_a, q_norm, wq_b, w_proj, _ = ins[l]
        q_ref, w_ref = orc.query_chain(hidden, wq_a, q_norm, wq_b, w_proj, pos, n_h=n_h)
        _check(q_ref, w_ref, qb_all[:, l], q32[:, l].cpu().numpy().astype(np.float64),
               w[:, l].cpu().numpy().astype(np.float64))
