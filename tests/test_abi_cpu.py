"""The C ABI library loads, exports every declared entry point and rejects bad
arguments on the host before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fm_index.h")


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fm_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import sparse_attention_kv_c4_gb300 as fm
    if not os.path.exists(fm.LIB_PATH):
        from sparse_attention_kv_c4_gb300 import _build
        _build.build()
    return fm.lib()


def test_header_declares_the_boundary():
    names = declared()
    for n in ("fm_memindex_score_mask", "fm_native_topk_paged", "fm_index_prefill_topk", "fm_index_prefill_scores",
              "fm_topk_select",
              "fm_native_topk_paged_workspace", "fm_index_prefill_workspace", "fm_topk_workspace",
              "fm_retriever_score_mask", "fm_retriever_workspace",
              "fm_query_chain", "fm_query_chain_workspace", "fm_query_chain_layers", "fm_query_chain_layers_workspace",
              "fm_last_error", "fm_device_status", "fm_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_version(lib):
    assert lib.fm_version() >= 10000


def test_memindex_rejects_bad_args_on_host(lib):
    import sparse_attention_kv_c4_gb300 as fm
    f = lib.fm_memindex_score_mask
    fake = 4096  # never dereferenced: validation fails first
    # n_h != 64
    assert f(fake, fake, fake, 3 * 128 * 128, 128 * 128, 1, 3, 128, 32, 128, 0.5, fake, None, None, None) == 1
    assert "n_h" in fm.fm_last_error()
    # L > 4
    assert f(fake, fake, fake, 5 * 128 * 128, 128 * 128, 1, 5, 128, 64, 128, 0.5, fake, None, None, None) == 1
    # threshold outside (0, 1)
    assert f(fake, fake, fake, 3 * 128 * 128, 128 * 128, 1, 3, 128, 64, 128, 1.0, fake, None, None, None) == 1
    # NULL mask
    assert f(fake, fake, fake, 3 * 128 * 128, 128 * 128, 1, 3, 128, 64, 128, 0.5, None, None, None, None) == 1
    # misaligned keys
    assert f(fake, fake, fake + 2, 3 * 128 * 128, 128 * 128, 1, 3, 128, 64, 128, 0.5, fake, None, None, None) == 1
    # overlapping strides
    assert f(fake, fake, fake, 128 * 128, 128 * 128, 2, 3, 128, 64, 128, 0.5, fake, None, None, None) == 1
    # empty work is OK without a device
    assert f(None, None, None, 0, 0, 0, 3, 128, 64, 128, 0.5, None, None, None, None) == 0


def test_page_recall_rejects_bad_args_on_host(lib):
    import sparse_attention_kv_c4_gb300 as fm
    fm.lib()  # sets argtypes
    f = lib.fm_page_recall
    fake = 4096  # never dereferenced: validation fails first
    assert f(fake, 2, 1024, 0, 0, 0, fake, None, None, None) == 1  # kmax < 1
    assert "kmax" in fm.fm_last_error()
    assert f(fake, 2, 1024, 0, 0, 65537, fake, None, None, None) == 1  # kmax too large
    assert f(fake, 2, 1024, -1, 0, 8, fake, None, None, None) == 1  # negative sink
    assert f(fake, 2, 1024, 0, -3, 8, fake, None, None, None) == 1  # negative recent
    assert f(fake, 2, 1 << 31, 0, 0, 8, fake, None, None, None) == 1  # S too large
    assert f(None, 2, 1024, 0, 0, 8, fake, None, None, None) == 1  # NULL mask
    assert f(fake, 2, 1024, 0, 0, 8, None, None, None, None) == 1  # NULL pages_out
    assert f(fake + 2, 2, 1024, 0, 0, 8, fake, None, None, None) == 1  # misaligned mask
    assert f(None, 0, 1024, 0, 0, 8, None, None, None, None) == 0  # empty work is OK without a device


def test_prefill_scores_rejects_bad_args_on_host(lib):
    import sparse_attention_kv_c4_gb300 as fm
    fm.lib()  # sets argtypes
    f = lib.fm_index_prefill_scores
    fake = 4096  # never dereferenced: validation fails first
    assert f(fake, fake, fake, fake, 8, 100, 32, 128, 4, fake, None) == 1  # n_h != 64
    assert "n_h" in fm.fm_last_error()
    assert f(fake, fake, fake, fake, 8, 100, 64, 128, 0, fake, None) == 1  # ratio < 1
    assert f(fake, fake, fake, fake, 8, 1 << 31, 64, 128, 4, fake, None) == 1  # S too large
    assert f(fake, fake, fake, fake, 8, 100, 64, 128, 4, None, None) == 1  # NULL logits_out
    assert f(fake + 8, fake, fake, fake, 8, 100, 64, 128, 4, fake, None) == 1  # misaligned q
    assert f(fake, fake, fake, fake, 8, 100, 64, 128, 4, fake + 2, None) == 1  # misaligned logits_out
    assert f(None, None, None, None, 0, 100, 64, 128, 4, None, None) == 0  # T = 0: nothing to do


def test_query_chain_layers_rejects_bad_args_on_host(lib):
    import ctypes
    import sparse_attention_kv_c4_gb300 as fm
    fm.lib()  # sets argtypes
    f = lib.fm_query_chain_layers
    fake = 4096  # never dereferenced: validation fails first
    ptrs = (ctypes.c_void_p * 4)(fake, fake, fake, fake)
    rope = (160000.0, 16.0, 65536.0, 32.0, 1.0, 1e-6)

    def call(L, T=4, dim=512, r=256, n_h=8, hd=128, rd=64, arrs=ptrs, q=fake, w=fake, ws=None, wsb=0):
        return f(L, arrs, arrs, arrs, arrs, arrs, fake, T, dim, r, n_h, hd, rd, *rope, q, None, w, ws, wsb, None)
    assert call(0) == 1 and "L=0" in fm.fm_last_error()          # no layers
    assert call(5) == 1                                          # more than four layers
    assert call(2, hd=64) == 1                                   # head_dim must be 128
    assert call(2, dim=516) == 1                                 # dim not a multiple of 8
    assert call(2, q=None) == 1                                  # NULL q_out
    null_layer = (ctypes.c_void_p * 4)(fake, None, fake, fake)
    assert call(2, arrs=null_layer) == 1 and "layer 1" in fm.fm_last_error()
    misaligned = (ctypes.c_void_p * 4)(fake, fake + 8, fake, fake)
    assert call(2, arrs=misaligned) == 1
    assert call(2) == 5                                          # no workspace: FM_ERR_WORKSPACE
    assert call(2, T=0) == 0                                     # nothing to do
    assert fm.fm_query_chain_layers_workspace(3, 30, 2048, 128) > fm.fm_query_chain_workspace(30, 2048, 128)
    assert fm.fm_query_chain_layers_workspace(1, 30, 2048, 128) == fm.fm_query_chain_workspace(30, 2048, 128)
    assert fm.fm_query_chain_layers_workspace(5, 30, 2048, 128) == 0


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import sparse_attention_kv_c4_gb300 as fm
    monkeypatch.setattr(fm, "_lib", None)
    monkeypatch.setattr(fm, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        fm.lib()


def test_topk_workspace_size_contract(lib):
    """fm_topk_workspace is host-only arithmetic; the select needs no scratch."""
    lib.fm_topk_workspace.argtypes = [ctypes.c_int, ctypes.c_int64]
    lib.fm_topk_workspace.restype = ctypes.c_size_t
    for rows, n in ((8, 4096), (8, 65536), (0, 65536), (4096, 131073)):
        assert lib.fm_topk_workspace(rows, n) == 0


def test_paged_workspace_accepts_a_whole_1m_history(lib):
    """Page tables of up to 4096 entries (a 1M-token request's every page) are
    accepted; one more is rejected (size 0)."""
    lib.fm_native_topk_paged_workspace.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.fm_native_topk_paged_workspace.restype = ctypes.c_size_t
    ws = lib.fm_native_topk_paged_workspace(630, 4096)
    assert ws >= 630 * 4096 * 64 * 4  # the score rows alone
    assert lib.fm_native_topk_paged_workspace(630, 4097) == 0
    assert lib.fm_native_topk_paged_workspace(1, 0) == 0


def test_memindex_fp8_workspace_contract(lib):
    """The fp8 Memory Indexer's workspace holds, per (request, layer), the
    split query's two 80-row E4M3 term blocks (64 heads, then the weighted
    query sum's four terms and zeros) and 68 floats of weights: at least
    20,752 bytes each; L outside 1..4 or a negative B sizes nothing."""
    lib.fm_memindex_fp8_workspace.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.fm_memindex_fp8_workspace.restype = ctypes.c_size_t
    per = 2 * 80 * 128 + 68 * 4
    for B, L in ((1, 1), (4, 3), (30, 3), (2, 4)):
        ws = lib.fm_memindex_fp8_workspace(B, L)
        assert ws >= B * L * per and ws % 256 == 0, (B, L, ws)
    assert lib.fm_memindex_fp8_workspace(1, 0) == 0 and lib.fm_memindex_fp8_workspace(1, 5) == 0
    assert lib.fm_memindex_fp8_workspace(-1, 3) == 0
    assert lib.fm_memindex_fp8_workspace(0, 3) == 0


def test_retriever_workspace_and_host_checks(lib):
    """Workspace sizing is host arithmetic; bad arguments are rejected before
    any device work (no GPU needed)."""
    lib.fm_retriever_workspace.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.fm_retriever_workspace.restype = ctypes.c_size_t
    assert lib.fm_retriever_workspace(30, 3, 128) >= 30 * 3 * (2 * 128 * 128 + 128 * 4)
    assert lib.fm_retriever_workspace(30, 3, 64) >= 30 * 3 * (2 * 64 * 128 + 64 * 4)
    assert lib.fm_retriever_workspace(1, 3, 96) == 0 and lib.fm_retriever_workspace(1, 5, 128) == 0
    f = lib.fm_retriever_score_mask
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 2 + [ctypes.c_int] * 2 + [ctypes.c_int64] + \
        [ctypes.c_int] * 3 + [ctypes.c_float] + [ctypes.c_void_p] * 4 + [ctypes.c_size_t, ctypes.c_void_p]
    INVALID = 1
    base = dict(B=1, L=3, S=64, n_h=128, d=128, ens=0, thr=0.5)

    def call(**kw):
        a = dict(base, **kw)
        return f(8, 8, 8, 0, 0, a["B"], a["L"], a["S"], a["n_h"], a["d"], a["ens"], a["thr"], 8, None, None, 256, 1 << 20,
                 None)
    assert call(n_h=96) == INVALID
    assert call(d=64) == INVALID
    assert call(S=30) == INVALID        # packed rows need S % 4 == 0
    assert call(L=5) == INVALID
    assert call(ens=2) == INVALID
    assert call(thr=0.0) == INVALID


def test_python_constants_match_header():
    """The binding's status codes, device-status bits and the no-allocation
    scratch size are the header's."""
    import sparse_attention_kv_c4_gb300 as fm
    src = open(HEADER).read()
    enum = dict((k, int(v)) for k, v in re.findall(r"\b(FM_(?:OK|ERR_[A-Z_]+))\s*=\s*(\d+)", src))
    assert enum, "no status codes found"
    for k, v in enum.items():
        assert getattr(fm, k) == v, k
    for k, v in re.findall(r"#define (FM_DEVERR_[A-Z_]+) (0x[0-9a-f]+)u", src):
        assert getattr(fm, k) == int(v, 16), k
    m = re.search(r"#define FM_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", src)
    assert m and fm.FM_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_check_device_status_is_exported(lib):
    assert hasattr(lib, "fm_check_device_status")


def test_paged_rejects_bad_key_dtype_on_host(lib):
    import sparse_attention_kv_c4_gb300 as fm
    fm.lib()  # sets argtypes
    f = lib.fm_native_topk_paged
    fake = 4096  # never dereferenced: validation fails first

    def call(dtype, scale, ws=fake, wsb=1 << 30):
        return f(fake, fake, fake, dtype, scale, 8, fake, fake, None, 2, 3, 64, 128, 512, fake, None, ws, wsb, None)
    assert call(0, fake) == fm.FM_ERR_INVALID_ARG and "key_dtype" in fm.fm_last_error()
    assert call(3, fake) == fm.FM_ERR_INVALID_ARG
    assert call(fm.FM_DTYPE_BF16, fake) == fm.FM_ERR_INVALID_ARG and "k_scale" in fm.fm_last_error()
    assert call(fm.FM_DTYPE_FP8_E4M3, None) == fm.FM_ERR_INVALID_ARG  # an E4M3 pool needs its scales
    assert call(fm.FM_DTYPE_BF16, None, ws=None) == fm.FM_ERR_WORKSPACE
