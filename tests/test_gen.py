"""The synthetic input generator: determinism, distributions, encoders."""
import numpy as np
import pytest

import gen


def test_q_deterministic_and_normalish():
    cfg = gen.MemIndexCfg("t", B=2, L=3, S=64, seed=123)
    q1, w1, hot1 = gen.memindex_qw(cfg)
    q2, w2, hot2 = gen.memindex_qw(cfg)
    assert (q1 == q2).all() and (hot1 == hot2).all()
    qf = (q1.astype(np.uint32) << 16).view(np.float32)
    assert abs(qf.mean()) < 0.02 and abs(qf.std() - 1.0) < 0.02
    assert np.allclose(np.linalg.norm(hot1, axis=-1), 1.0, atol=1e-6)
    assert (w1[..., :8] == 1.0).all() and (w1[..., 8:] == np.float32(-0.2)).all()


def test_keys_rows_match_dense_and_variance():
    cfg = gen.MemIndexCfg("t", B=1, L=2, S=300, seed=5)
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    s = np.array([0, 17, 299, 5])
    assert (gen.memindex_key_rows(cfg, 0, 1, s, hot) == K[0, 1, s]).all()
    pl = gen.planted(cfg, 0, 1)
    kf = (K[0, 1].astype(np.uint32) << 16).view(np.float32)
    cold = kf[~pl]
    assert abs(cold.std() * np.sqrt(128) - 1.0) < 0.03
    # planted rows point along the hot direction with norm ~3
    hotp = kf[pl] @ hot[0, 1]
    assert (hotp > 2.5).all()


def test_e4m3_encoder_matches_torch_rne():
    """gen's fp32 -> E4M3 encoder (RNE, in range) equals PyTorch's cast."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01,
                        np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -9])])
    x = x[np.abs(x) <= 448].astype(np.float32)
    enc = np.array([gen_codec(float(v)) for v in x], dtype=np.uint8)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (enc == want).all(), np.nonzero(enc != want)[0][:5]


def gen_codec(v):
    """Call gen.h's element encoders through a two-line C shim."""
    import ctypes
    if not hasattr(gen_codec, "fn"):
        import os, subprocess, tempfile
        d = tempfile.mkdtemp()
        src = os.path.join(d, "c.c")
        with open(src, "w") as f:
            f.write('#include "gen.h"\nuint8_t enc(float f){return gen_e4m3_rne_sat(f);}\n'
                    'uint16_t bf(float f){return gen_bf16_rne(f);}\n')
        so = os.path.join(d, "c.so")
        subprocess.run(["gcc", "-O2", "-shared", "-fPIC", "-ffp-contract=off", "-I", gen.HERE, "-o", so, src,
                        "-lm"], check=True)
        lib = ctypes.CDLL(so)
        lib.enc.argtypes = [ctypes.c_float]
        lib.enc.restype = ctypes.c_uint8
        lib.bf.argtypes = [ctypes.c_float]
        lib.bf.restype = ctypes.c_uint16
        gen_codec.fn = lib
    return gen_codec.fn.enc(v)


def test_bf16_rne_matches_torch():
    torch = pytest.importorskip("torch")
    gen_codec(0.0)
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * 10).astype(np.float32)
    got = np.array([gen_codec.fn.bf(float(v)) for v in x], dtype=np.uint16)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (got == want).all()


def test_paged_tables_shapes_and_distinct():
    cfg = gen.PagedCfg("t", requests=3, layers=4, n_pages=50, R=7, seed=9)
    logical, phys, owner = gen.paged_tables(cfg)
    assert logical.shape == (12, 7) and phys.shape == (12, 7)
    for r in range(3):
        rows = logical[r * 4:(r + 1) * 4]
        assert (rows == rows[0]).all() and len(set(rows[0].tolist())) == 7
    assert sorted(phys.reshape(-1).tolist()) == list(range(cfg.P))
    for qi in range(12):
        for j in range(7):
            p = phys[qi, j]
            assert tuple(owner[p]) == (qi // 4, qi % 4, logical[qi, j])


def test_pool_host_rows_consistent():
    cfg = gen.PagedCfg("t", requests=2, layers=2, n_pages=10, R=3, page=8, seed=4)
    logical, phys, owner = gen.paged_tables(cfg)
    k8, scale = gen.paged_pool_host(cfg, owner)
    a, b, lp = owner[5]
    k8r, scr = gen.paged_chunk_rows(cfg, a, b, np.arange(lp * 8, lp * 8 + 8))
    assert (k8r == k8[5]).all() and (scr == scale[5]).all()
    assert ((k8 & 0x7F) != 0x7F).all()


def test_pool_rows_match_pool_host():
    """The batched pool builder gives paged_pool_host's pages, also when the
    tables are renumbered to a local pool."""
    cfg = gen.PagedCfg("t", requests=2, layers=3, n_pages=30, R=4, seed=8)
    logical, phys, owner = gen.paged_tables(cfg)
    k8, scale = gen.paged_pool_host(cfg, owner)
    k8b, scb = gen.paged_pool_rows(cfg, logical, phys)
    assert (k8b == k8).all() and (scb.view(np.uint32) == scale.view(np.uint32)).all()
    qs = [3, 4]
    local = np.arange(len(qs) * cfg.R, dtype=np.int32).reshape(len(qs), cfg.R)
    table = np.zeros_like(phys)
    table[qs] = local
    k8l, scl = gen.paged_pool_rows(cfg, logical, table, queries=qs, n_pool=len(qs) * cfg.R)
    assert (k8l == k8[phys[qs].reshape(-1)]).all() and (scl == scale[phys[qs].reshape(-1)]).all()
