"""GB300-native Lookahead-Sparse-Attention c4 indexer.

Thin Python binding of ``libfm_index.so`` (C ABI in ``include/fm_index.h``):
the functions below carry the C names and only marshal torch tensors into
pointers, sizes and the current CUDA stream.  Every step of the indexer runs
in the library's sm_103a kernels; there is no Python or CPU fallback, and
importing a function whose library is missing raises.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "FmError", "lib", "fm_version", "fm_last_error", "fm_device_status", "fm_check_device_status", "fm_memindex_score_mask",
    "fm_topk_workspace", "fm_topk_select", "fm_native_topk_paged_workspace", "fm_native_topk_paged",
    "fm_index_prefill_workspace", "fm_index_prefill_topk", "fm_native_topk_paged_noalloc", "fm_page_recall",
    "fm_native_topk_paged_ex", "fm_memindex_fp8_workspace", "fm_memindex_score_mask_fp8",
    "fm_index_prefill_scores", "fm_retriever_workspace", "fm_retriever_score_mask", "fm_query_chain_workspace",
    "fm_query_chain", "fm_query_chain_layers_workspace", "fm_query_chain_layers", "LIB_PATH",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfm_index.so")

FM_OK, FM_ERR_INVALID_ARG, FM_ERR_UNSUPPORTED, FM_ERR_CUDA = 0, 1, 2, 3
FM_ERR_DEVICE_BOUNDS, FM_ERR_WORKSPACE, FM_ERR_DEVICE_TIMEOUT = 4, 5, 6
FM_DEVERR_PAGE_RANGE, FM_DEVERR_TIMEOUT, FM_DEVERR_DUP_PAGE = 0x1, 0x2, 0x4
FM_DTYPE_BF16, FM_DTYPE_FP8_E4M3 = 1, 2  # key element types of a paged pool
FM_NOALLOC_SCRATCH_BYTES = 16 << 20  # the no-allocation paged top-k's built-in scratch (fm_index.h)

_VP, _I64, _I32, _F, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class FmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"fm status {status}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libfm_index.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.fm_version.restype = ctypes.c_int
        L.fm_last_error.restype = ctypes.c_char_p
        L.fm_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), _I32, _VP]
        L.fm_check_device_status.argtypes = [_VP]
        L.fm_check_device_status.restype = ctypes.c_int
        L.fm_memindex_score_mask.argtypes = [_VP, _VP, _VP, _I64, _I64, _I32, _I32, _I64, _I32, _I32, _F, _VP,
                                             _VP, _VP, _VP]
        for name in ("fm_topk_workspace",):
            if hasattr(L, name):
                getattr(L, name).argtypes = [_I32, _I64]
                getattr(L, name).restype = _SZ
        if hasattr(L, "fm_topk_select"):
            L.fm_topk_select.argtypes = [_VP, _I64, _VP, _I32, _I64, _I32, _VP, _VP, _VP, _SZ, _VP]
        if hasattr(L, "fm_native_topk_paged_workspace"):
            L.fm_native_topk_paged_workspace.argtypes = [_I32, _I32]
            L.fm_native_topk_paged_workspace.restype = _SZ
            L.fm_native_topk_paged.argtypes = [_VP, _VP, _VP, _I32, _VP, _I64, _VP, _VP, _VP, _I32, _I32, _I32,
                                               _I32, _I32, _VP, _VP, _VP, _SZ, _VP]
        if hasattr(L, "fm_native_topk_paged_ex"):
            L.fm_native_topk_paged_ex.argtypes = [_VP, _VP, _VP, _I32, _VP, _I64, _VP, _VP, _VP, _I32, _I32, _I32,
                                                  _I32, _I32, _VP, _I64, _I32, _I32, _VP, _VP, _VP, _SZ, _VP]
        if hasattr(L, "fm_native_topk_paged_noalloc"):
            L.fm_native_topk_paged_noalloc.argtypes = [_VP, _VP, _VP, _VP, _I64, _VP, _VP, _VP, _I32, _I32, _I32,
                                                       _I32, _I32, _VP, _VP, _VP]
            L.fm_native_topk_paged_noalloc.restype = ctypes.c_int
        if hasattr(L, "fm_index_prefill_workspace"):
            L.fm_index_prefill_workspace.argtypes = [_I32, _I64]
            L.fm_index_prefill_workspace.restype = _SZ
            L.fm_index_prefill_topk.argtypes = [_VP, _VP, _VP, _VP, _I32, _I64, _I32, _I32, _I32, _I32, _VP, _VP,
                                                _VP, _SZ, _VP]
        if hasattr(L, "fm_index_prefill_scores"):
            L.fm_index_prefill_scores.argtypes = [_VP, _VP, _VP, _VP, _I32, _I64, _I32, _I32, _I32, _VP, _VP]
            L.fm_index_prefill_scores.restype = ctypes.c_int
        if hasattr(L, "fm_memindex_score_mask_fp8"):
            L.fm_memindex_fp8_workspace.argtypes = [_I32, _I32]
            L.fm_memindex_fp8_workspace.restype = _SZ
            L.fm_memindex_score_mask_fp8.argtypes = [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _I32, _I32, _I64,
                                                     _I32, _I32, _F, _VP, _VP, _VP, _VP, _SZ, _VP]
        if hasattr(L, "fm_retriever_score_mask"):
            L.fm_retriever_workspace.argtypes = [_I32, _I32, _I32]
            L.fm_retriever_workspace.restype = _SZ
            L.fm_retriever_score_mask.argtypes = [_VP, _VP, _VP, _I64, _I64, _I32, _I32, _I64, _I32, _I32, _I32, _F,
                                                  _VP, _VP, _VP, _VP, _SZ, _VP]
        if hasattr(L, "fm_query_chain"):
            L.fm_query_chain_workspace.argtypes = [_I32, _I32, _I32]
            L.fm_query_chain_workspace.restype = _SZ
            _D = ctypes.c_double
            L.fm_query_chain.argtypes = [_VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32, _I32, _I32, _D, _D, _D,
                                         _D, _D, _F, _VP, _VP, _VP, _VP, _SZ, _VP]
        if hasattr(L, "fm_query_chain_layers"):
            _D = ctypes.c_double
            L.fm_query_chain_layers_workspace.argtypes = [_I32, _I32, _I32, _I32]
            L.fm_query_chain_layers_workspace.restype = _SZ
            L.fm_query_chain_layers.argtypes = [_I32, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32, _I32,
                                                _I32, _D, _D, _D, _D, _D, _F, _VP, _VP, _VP, _VP, _SZ, _VP]
            L.fm_query_chain_layers.restype = ctypes.c_int
        if hasattr(L, "fm_page_recall"):
            L.fm_page_recall.argtypes = [_VP, _I32, _I64, _I64, _I64, _I32, _VP, _VP, _VP, _VP]
        for name in ("fm_memindex_score_mask", "fm_topk_select", "fm_native_topk_paged", "fm_index_prefill_topk",
                     "fm_device_status", "fm_page_recall", "fm_native_topk_paged_ex", "fm_memindex_score_mask_fp8"):
            if hasattr(L, name):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != FM_OK:
        raise FmError(status, fm_last_error())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def fm_version() -> int:
    return lib().fm_version()


def fm_last_error() -> str:
    return lib().fm_last_error().decode()


def fm_device_status(reset: bool = True, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().fm_device_status(ctypes.byref(v), int(reset), _stream(stream)))
    return v.value


def fm_check_device_status(stream=None) -> None:
    """Raise FmError (FM_ERR_DEVICE_BOUNDS or FM_ERR_DEVICE_TIMEOUT) when a
    kernel flagged the device status word since its last reset; clears it."""
    _check(lib().fm_check_device_status(_stream(stream)))


def fm_memindex_score_mask(q, w, keys, mask_out, maxsig_out=None, logits_out=None, threshold: float = 0.5,
                           stream=None) -> None:
    """q [B,L,64,128] bf16, w [B,L,64] fp32, keys [B,L,S,128] bf16 (any b/l
    strides, rows dense), mask_out [B, ceil(S/32)] int32/uint32,
    maxsig_out [B,S] fp32 or None, logits_out [B,L,S] fp32 or None."""
    B, L, n_h, d = q.shape
    S = keys.shape[2]
    if keys.stride(3) != 1 or keys.stride(2) != d:
        raise ValueError("keys rows must be dense [.., S, d]")
    _check(lib().fm_memindex_score_mask(_ptr(q), _ptr(w), _ptr(keys), keys.stride(0), keys.stride(1), B, L, S, n_h,
                                        d, float(threshold), _ptr(mask_out), _ptr(maxsig_out), _ptr(logits_out),
                                        _stream(stream)))


def fm_memindex_fp8_workspace(B: int, L: int) -> int:
    return lib().fm_memindex_fp8_workspace(B, L)


def fm_memindex_score_mask_fp8(q, w, k8, k_scale, mask_out, maxsig_out=None, logits_out=None, threshold: float = 0.5,
                               workspace=None, stream=None) -> None:
    """q [B,L,64,128] bf16, w [B,L,64] fp32, k8 [B,L,S,128] uint8 E4M3 codes
    (any b/l strides, rows dense), k_scale [B,L,S] fp32 (any b/l strides,
    unit s stride), mask_out [B, ceil(S/32)], maxsig_out [B,S] or None,
    logits_out [B,L,S] or None, workspace >= fm_memindex_fp8_workspace(B, L)."""
    B, L, n_h, d = q.shape
    S = k8.shape[2]
    if k8.stride(3) != 1 or k8.stride(2) != d or k_scale.stride(2) != 1:
        raise ValueError("k8 rows must be dense [.., S, d] and k_scale rows dense [.., S]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_memindex_score_mask_fp8(_ptr(q), _ptr(w), _ptr(k8), _ptr(k_scale), k8.stride(0), k8.stride(1),
                                            k_scale.stride(0), k_scale.stride(1), B, L, S, n_h, d, float(threshold),
                                            _ptr(mask_out), _ptr(maxsig_out), _ptr(logits_out), _ptr(workspace),
                                            ws_bytes, _stream(stream)))


# The retriever's rotary hyperparameters ("FlashMemory-DeepSeek-V4" README, "Hyperparameters").
RETRIEVER_ROPE = dict(rope_base=160000.0, rope_factor=16.0, rope_orig_len=65536.0, rope_beta_fast=32.0,
                      rope_beta_slow=1.0)


def fm_query_chain_workspace(T: int, r: int, n_h: int) -> int:
    return lib().fm_query_chain_workspace(T, r, n_h)


def fm_query_chain(hidden, wq_a, q_norm, wq_b, w_proj, pos, q_out, w_out, q_out_f32=None, eps: float = 1e-6,
                   workspace=None, stream=None, **rope) -> None:
    """hidden [T,dim] bf16, wq_a [r,dim], q_norm [r], wq_b [n_h*128, r], w_proj [n_h,dim] bf16,
    pos [T] int64 -> q_out [T,n_h,128] bf16, w_out [T,n_h] fp32 (q_out_f32 optional)."""
    cfg = dict(RETRIEVER_ROPE, **rope)
    T, dim = hidden.shape
    r = wq_a.shape[0]
    n_h = w_proj.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_query_chain(_ptr(hidden), _ptr(wq_a), _ptr(q_norm), _ptr(wq_b), _ptr(w_proj), _ptr(pos), T, dim,
                                r, n_h, 128, 64, cfg["rope_base"], cfg["rope_factor"], cfg["rope_orig_len"],
                                cfg["rope_beta_fast"], cfg["rope_beta_slow"], float(eps), _ptr(q_out),
                                _ptr(q_out_f32), _ptr(w_out), _ptr(workspace), ws_bytes, _stream(stream)))


def fm_query_chain_layers_workspace(L: int, T: int, r: int, n_h: int) -> int:
    return lib().fm_query_chain_layers_workspace(L, T, r, n_h)


def fm_query_chain_layers(hidden, wq_a, q_norm, wq_b, w_proj, pos, q_out, w_out, q_out_f32=None, eps: float = 1e-6,
                          workspace=None, stream=None, **rope) -> None:
    """hidden, wq_a, q_norm, wq_b, w_proj: sequences of L device tensors (one
    per layer, shapes as fm_query_chain); pos [T] int64 -> q_out [T,L,n_h,128]
    bf16, w_out [T,L,n_h] fp32 (q_out_f32 optional)."""
    cfg = dict(RETRIEVER_ROPE, **rope)
    L = len(hidden)
    T, dim = hidden[0].shape
    r = wq_a[0].shape[0]
    n_h = w_proj[0].shape[0]
    arr = lambda ts: (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_query_chain_layers(L, arr(hidden), arr(wq_a), arr(q_norm), arr(wq_b), arr(w_proj), _ptr(pos), T,
                                       dim, r, n_h, 128, 64, cfg["rope_base"], cfg["rope_factor"],
                                       cfg["rope_orig_len"], cfg["rope_beta_fast"], cfg["rope_beta_slow"], float(eps),
                                       _ptr(q_out), _ptr(q_out_f32), _ptr(w_out), _ptr(workspace), ws_bytes,
                                       _stream(stream)))


ENSEMBLE_MAX, ENSEMBLE_MEAN = 0, 1


def fm_retriever_workspace(B: int, L: int, n_h: int = 128) -> int:
    return lib().fm_retriever_workspace(B, L, n_h)


def fm_retriever_score_mask(q, w, compressed_k, mask_out, ens_out=None, logits_out=None, ensemble: int = ENSEMBLE_MAX,
                            threshold: float = 0.5, workspace=None, stream=None) -> None:
    """q [B,L,n_h,128] bf16 (n_h 64 or 128), w [B,L,n_h] fp32, compressed_k
    [B,L,S,132] uint8 packed rows (any b/l strides, rows dense), mask_out
    [B, ceil(S/32)], ens_out [B,S] or None, logits_out [B,L,S] or None,
    ensemble ENSEMBLE_MAX or ENSEMBLE_MEAN, workspace >=
    fm_retriever_workspace(B, L, n_h)."""
    B, L, n_h, d = q.shape
    S = compressed_k.shape[2]
    if compressed_k.stride(3) != 1 or compressed_k.stride(2) != d + 4:
        raise ValueError("compressed_k rows must be dense [.., S, 132]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_retriever_score_mask(_ptr(q), _ptr(w), _ptr(compressed_k), compressed_k.stride(0),
                                         compressed_k.stride(1), B, L, S, n_h, d, int(ensemble), float(threshold),
                                         _ptr(mask_out), _ptr(ens_out), _ptr(logits_out), _ptr(workspace), ws_bytes,
                                         _stream(stream)))


def fm_topk_workspace(rows: int, n: int) -> int:
    return lib().fm_topk_workspace(rows, n)


def fm_topk_select(scores, k: int, idx_out, score_out=None, n_valid=None, n=None, workspace=None,
                   stream=None) -> None:
    """scores [rows, ld] fp32 (row stride ld, unit column stride); n_valid [rows]
    int32 or None; idx_out [rows, k] int32; score_out [rows, k] fp32 or None."""
    rows, ld = scores.shape[0], scores.stride(0)
    n = scores.shape[1] if n is None else n
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_topk_select(_ptr(scores), ld, _ptr(n_valid), rows, n, k, _ptr(idx_out), _ptr(score_out),
                                _ptr(workspace), ws_bytes, _stream(stream)))


def fm_native_topk_paged_workspace(Q: int, R: int) -> int:
    return lib().fm_native_topk_paged_workspace(Q, R)


def _key_dtype(k_pool) -> int:
    """The pool's key type from its tensor dtype: uint8 holds E4M3 codes;
    int16 / bfloat16 hold bf16 keys."""
    import torch
    if k_pool.dtype == torch.uint8:
        return FM_DTYPE_FP8_E4M3
    if k_pool.dtype in (torch.int16, torch.bfloat16):
        return FM_DTYPE_BF16
    raise ValueError(f"k_pool dtype {k_pool.dtype}: uint8 (E4M3 codes) or int16/bfloat16 (bf16 keys)")


def fm_native_topk_paged(q, w, k_pool, k_scale, page_phys, page_logical, k: int, idx_out, score_out=None,
                         n_res=None, workspace=None, stream=None) -> None:
    """q [Q,64,128] bf16, w [Q,64] fp32, k_pool [P,64,128]: uint8 E4M3 codes
    with k_scale [P,64] fp32, or int16/bfloat16 bf16 keys with k_scale None;
    page_phys/page_logical [Q,R] int32, n_res [Q] int32 or None, idx_out
    [Q,k] int32, score_out [Q,k] fp32 or None."""
    Q, n_h, d = q.shape
    R = page_phys.shape[1]
    P = k_pool.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_native_topk_paged(_ptr(q), _ptr(w), _ptr(k_pool), _key_dtype(k_pool), _ptr(k_scale), P,
                                      _ptr(page_phys),
                                      _ptr(page_logical), _ptr(n_res), Q, R, n_h, d, k, _ptr(idx_out),
                                      _ptr(score_out), _ptr(workspace), ws_bytes, _stream(stream)))


def fm_native_topk_paged_ex(q, w, k_pool, k_scale, page_phys, page_logical, k: int, idx_out, score_out=None,
                            n_res=None, res_mask=None, mask_group: int = 1, id_mode: int = 0, workspace=None,
                            stream=None) -> None:
    """fm_native_topk_paged plus the Level-2 resident mask res_mask
    [rows, mask_ld] int32/uint32 (row qi // mask_group per query, or None) and
    id_mode (0 = logical chunk ids, 1 = reserve cells phys * 64 + o)."""
    Q, n_h, d = q.shape
    R = page_phys.shape[1]
    P = k_pool.shape[0]
    mask_ld = 0 if res_mask is None else res_mask.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_native_topk_paged_ex(_ptr(q), _ptr(w), _ptr(k_pool), _key_dtype(k_pool), _ptr(k_scale), P,
                                         _ptr(page_phys),
                                         _ptr(page_logical), _ptr(n_res), Q, R, n_h, d, k, _ptr(res_mask), mask_ld,
                                         mask_group, id_mode, _ptr(idx_out), _ptr(score_out), _ptr(workspace),
                                         ws_bytes, _stream(stream)))


def fm_native_topk_paged_noalloc(q, w, k_pool, k_scale, page_phys, page_logical, k: int, idx_out, score_out=None,
                                 n_res=None, stream=None) -> None:
    """fm_native_topk_paged without a workspace, for callers that cannot
    allocate device memory: the scratch is a fixed 16 MiB array inside the
    library (shared by all calls; serialise calls that could overlap)."""
    Q, n_h, d = q.shape
    R = page_phys.shape[1]
    P = k_pool.shape[0]
    _check(lib().fm_native_topk_paged_noalloc(_ptr(q), _ptr(w), _ptr(k_pool), _ptr(k_scale), P, _ptr(page_phys),
                                              _ptr(page_logical), _ptr(n_res), Q, R, n_h, d, k, _ptr(idx_out),
                                              _ptr(score_out), _stream(stream)))


def fm_index_prefill_workspace(T: int, S: int) -> int:
    return lib().fm_index_prefill_workspace(T, S)


def fm_index_prefill_topk(q, w, pos, keys, k: int, idx_out, score_out=None, ratio: int = 4, workspace=None,
                          stream=None) -> None:
    """q [T,64,128] bf16, w [T,64] fp32, pos [T] int64, keys [S,128] bf16,
    idx_out [T,k] int32, score_out [T,k] fp32 or None."""
    T, n_h, d = q.shape
    S = keys.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fm_index_prefill_topk(_ptr(q), _ptr(w), _ptr(pos), _ptr(keys), T, S, n_h, d, ratio, k,
                                       _ptr(idx_out), _ptr(score_out), _ptr(workspace), ws_bytes, _stream(stream)))


def fm_index_prefill_scores(q, w, pos, keys, logits_out, ratio: int = 4, stream=None) -> None:
    """q [T,64,128] bf16, w [T,64] fp32, pos [T] int64, keys [S,128] bf16,
    logits_out [T,S] fp32 (contiguous): the dense scores, -inf past each
    token's causal limit."""
    T, n_h, d = q.shape
    S = keys.shape[0]
    _check(lib().fm_index_prefill_scores(_ptr(q), _ptr(w), _ptr(pos), _ptr(keys), T, S, n_h, d, ratio,
                                         _ptr(logits_out), _stream(stream)))


def fm_page_recall(mask, S: int, kmax: int, pages_out, density_out=None, n_out=None, sink: int = 0, recent: int = 0,
                   stream=None) -> None:
    """mask [B, ceil(S/32)] int32/uint32 (fm_memindex_score_mask's output),
    pages_out [B, kmax] int32, density_out [B, kmax] int32 or None, n_out [B]
    int32 or None."""
    B = mask.shape[0]
    _check(lib().fm_page_recall(_ptr(mask), B, S, sink, recent, kmax, _ptr(pages_out), _ptr(density_out),
                                _ptr(n_out), _stream(stream)))
