"""CPU oracle for the LSA c4 indexer hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (sparse_attention_kv_c4_gb300)
never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation, one OpenMP
split over independent outputs).  This module only compiles it, loads it with
ctypes and marshals numpy arrays.  Every function cites, in ``oracle.c``, the
passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
SO = os.path.join(HERE, "liborc.so")

u16p = ctypes.POINTER(ctypes.c_uint16)
u8p = ctypes.POINTER(ctypes.c_uint8)
u32p = ctypes.POINTER(ctypes.c_uint32)
f32p = ctypes.POINTER(ctypes.c_float)
f64p = ctypes.POINTER(ctypes.c_double)
i32p = ctypes.POINTER(ctypes.c_int32)
i64p = ctypes.POINTER(ctypes.c_int64)
I64, I32, D, F = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_float


def compile_oracle(src: str = SRC, so: str = SO, extra=()) -> str:
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11",
           *extra, "-o", so, src, "-lm"]
    subprocess.run(cmd, check=True)
    return so


def build() -> str:
    return compile_oracle()


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a, t):
    return a.ctypes.data_as(t) if a is not None else None


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, so: str = SO):
        lib = ctypes.CDLL(so)
        lib.orc_bf16.argtypes = [ctypes.c_uint16]
        lib.orc_bf16.restype = D
        lib.orc_e4m3.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3.restype = D
        lib.orc_sigmoid.argtypes = [D]
        lib.orc_sigmoid.restype = D
        lib.orc_score_bf16.argtypes = [u16p, f32p, u16p, I32, I32]
        lib.orc_score_bf16.restype = D
        lib.orc_score_fp8.argtypes = [u16p, f32p, u8p, F, I32, I32]
        lib.orc_score_fp8.restype = D
        lib.orc_memindex_logits.argtypes = [u16p, f32p, u16p, I64, I64, I64, I64, I64, I32, I32, f64p]
        lib.orc_memindex_logits_fp8.argtypes = [u16p, f32p, u8p, f32p, I64, I64, I64, I64, I64, I64, I64, I32, I32,
                                                f64p]
        lib.orc_memindex_select.argtypes = [f64p, I64, I64, I64, D, u32p, f64p]
        lib.orc_unpack_compressed_k.argtypes = [u8p, I64, I32, u8p, f32p]
        lib.orc_rmsnorm.argtypes = [f64p, u16p, I32, D, f64p]
        lib.orc_yarn_freq.argtypes = [I32, I32, D, D, D, D, D]
        lib.orc_yarn_freq.restype = D
        lib.orc_rope_yarn.argtypes = [f64p, I32, I32, I64, D, D, D, D, D]
        lib.orc_hadamard.argtypes = [f64p, I32, f64p]
        lib.orc_query_chain.argtypes = [u16p, u16p, u16p, u16p, u16p, i64p, I64, I32, I32, I32, I32, I32, D, D, D, D,
                                        D, D, f64p, f64p]
        lib.orc_memindex_ensemble.argtypes = [f64p, I64, I64, I64, I32, D, u32p, f64p]
        lib.orc_topk.argtypes = [i64p, f64p, I64, I32, i32p, f64p]
        lib.orc_topk.restype = ctypes.c_int
        lib.orc_paged_topk.argtypes = [u16p, f32p, u8p, f32p, i32p, i32p, i32p, I64, I64, I32, I32, I32,
                                       I32, i32p, f64p, f64p]
        lib.orc_paged_topk_ex.argtypes = [u16p, f32p, u8p, f32p, i32p, i32p, i32p, I64, I64, I32, I32, I32, I32,
                                          u32p, I64, I32, I32, i32p, f64p, f64p]
        lib.orc_paged_topk_bf16_ex.argtypes = [u16p, f32p, u16p, i32p, i32p, i32p, I64, I64, I32, I32, I32, I32,
                                               u32p, I64, I32, I32, i32p, f64p, f64p]
        lib.orc_causal_limit.argtypes = [I64, I64, I32]
        lib.orc_causal_limit.restype = I64
        lib.orc_prefill_topk.argtypes = [u16p, f32p, i64p, u16p, I64, I64, I32, I32, I32, I32, i32p, f64p]
        lib.orc_page_recall.argtypes = [u32p, I64, I64, I64, I64, I32, I32, i32p, i32p, i32p]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        self.lib = lib
        self.path = so

    # -- element decoding ----------------------------------------------------
    def bf16(self, bits) -> np.ndarray:
        b = np.asarray(bits, dtype=np.uint16).reshape(-1)
        return np.array([self.lib.orc_bf16(int(v)) for v in b])

    def e4m3(self, codes) -> np.ndarray:
        c = np.asarray(codes, dtype=np.uint8).reshape(-1)
        return np.array([self.lib.orc_e4m3(int(v)) for v in c])

    def sigmoid(self, x: float) -> float:
        return self.lib.orc_sigmoid(float(x))

    # -- scores --------------------------------------------------------------
    def score_bf16(self, q, w, k) -> float:
        q = _c(q, np.uint16); w = _c(w, np.float32); k = _c(k, np.uint16)
        n_h, d = q.shape
        return self.lib.orc_score_bf16(_p(q, u16p), _p(w, f32p), _p(k, u16p), n_h, d)

    def score_fp8(self, q, w, k8, scale) -> float:
        q = _c(q, np.uint16); w = _c(w, np.float32); k8 = _c(k8, np.uint8)
        n_h, d = q.shape
        return self.lib.orc_score_fp8(_p(q, u16p), _p(w, f32p), _p(k8, u8p), float(scale), n_h, d)

    # -- Memory Indexer --------------------------------------------------------
    def memindex_logits(self, q, w, K) -> np.ndarray:
        """q [B,L,n_h,d] bf16 bits, w [B,L,n_h], K [B,L,S,d] bf16 bits -> x [B,L,S] fp64."""
        q = _c(q, np.uint16); w = _c(w, np.float32); K = _c(K, np.uint16)
        B, L, n_h, d = q.shape
        S = K.shape[2]
        x = np.empty((B, L, S), dtype=np.float64)
        self.lib.orc_memindex_logits(_p(q, u16p), _p(w, f32p), _p(K, u16p), L * S * d, S * d, B, L, S,
                                     n_h, d, _p(x, f64p))
        return x

    def memindex_logits_fp8(self, q, w, k8, scale) -> np.ndarray:
        """q [B,L,n_h,d] bf16 bits, w [B,L,n_h], k8 [B,L,S,d] E4M3 codes,
        scale [B,L,S] fp32 -> x [B,L,S] fp64."""
        q = _c(q, np.uint16); w = _c(w, np.float32); k8 = _c(k8, np.uint8); scale = _c(scale, np.float32)
        B, L, n_h, d = q.shape
        S = k8.shape[2]
        x = np.empty((B, L, S), dtype=np.float64)
        self.lib.orc_memindex_logits_fp8(_p(q, u16p), _p(w, f32p), _p(k8, u8p), _p(scale, f32p), L * S * d, S * d,
                                         L * S, S, B, L, S, n_h, d, _p(x, f64p))
        return x

    def memindex_select(self, x, thr: float = 0.5):
        """x [B,L,S] -> mask [B, ceil(S/32)] uint32, maxsig [B,S] fp64."""
        x = _c(x, np.float64)
        B, L, S = x.shape
        mask = np.empty((B, (S + 31) // 32), dtype=np.uint32)
        maxsig = np.empty((B, S), dtype=np.float64)
        self.lib.orc_memindex_select(_p(x, f64p), B, L, S, float(thr), _p(mask, u32p), _p(maxsig, f64p))
        return mask, maxsig

    def unpack_compressed_k(self, ck):
        """ck [..., d + 4] uint8 packed rows -> k8 [..., d] uint8, scale [...] fp32."""
        ck = _c(ck, np.uint8)
        d = ck.shape[-1] - 4
        n = ck.size // (d + 4)
        k8 = np.empty(ck.shape[:-1] + (d,), dtype=np.uint8)
        sc = np.empty(ck.shape[:-1], dtype=np.float32)
        self.lib.orc_unpack_compressed_k(_p(ck, u8p), n, d, _p(k8, u8p), _p(sc, f32p))
        return k8, sc

    # -- query projection chain -------------------------------------------------
    ROPE = dict(rope_dim=64, base=160000.0, factor=16.0, orig_len=65536.0, beta_fast=32.0, beta_slow=1.0)

    def rmsnorm(self, x, g, eps: float = 1e-6) -> np.ndarray:
        x = _c(x, np.float64); g = _c(g, np.uint16)
        y = np.empty_like(x)
        self.lib.orc_rmsnorm(_p(x, f64p), _p(g, u16p), len(x), float(eps), _p(y, f64p))
        return y

    def yarn_freq(self, i: int, rope_dim=64, base=160000.0, factor=16.0, orig_len=65536.0, beta_fast=32.0,
                  beta_slow=1.0) -> float:
        return self.lib.orc_yarn_freq(int(i), int(rope_dim), float(base), float(factor), float(orig_len),
                                      float(beta_fast), float(beta_slow))

    def rope_yarn(self, x, pos: int, rope_dim=64, base=160000.0, factor=16.0, orig_len=65536.0, beta_fast=32.0,
                  beta_slow=1.0) -> np.ndarray:
        y = _c(np.array(x, dtype=np.float64), np.float64)
        self.lib.orc_rope_yarn(_p(y, f64p), len(y), int(rope_dim), int(pos), float(base), float(factor),
                               float(orig_len), float(beta_fast), float(beta_slow))
        return y

    def hadamard(self, x) -> np.ndarray:
        x = _c(x, np.float64)
        y = np.empty_like(x)
        self.lib.orc_hadamard(_p(x, f64p), len(x), _p(y, f64p))
        return y

    def query_chain(self, hidden, wq_a, q_norm, wq_b, w_proj, pos, n_h: int, head_dim: int = 128,
                    eps: float = 1e-6, **rope):
        """hidden [T,dim] bf16 bits; wq_a [r,dim], q_norm [r], wq_b [n_h*head_dim, r],
        w_proj [n_h, dim] bf16 bits; pos [T] -> q [T,n_h,head_dim], w [T,n_h] fp64."""
        cfg = dict(self.ROPE, **rope)
        hidden = _c(hidden, np.uint16); wq_a = _c(wq_a, np.uint16); q_norm = _c(q_norm, np.uint16)
        wq_b = _c(wq_b, np.uint16); w_proj = _c(w_proj, np.uint16); pos = _c(pos, np.int64)
        T, dim = hidden.shape
        r = wq_a.shape[0]
        q = np.empty((T, n_h, head_dim), dtype=np.float64)
        w = np.empty((T, n_h), dtype=np.float64)
        self.lib.orc_query_chain(_p(hidden, u16p), _p(wq_a, u16p), _p(q_norm, u16p), _p(wq_b, u16p),
                                 _p(w_proj, u16p), _p(pos, i64p), T, dim, r, n_h, head_dim, cfg["rope_dim"],
                                 cfg["base"], cfg["factor"], cfg["orig_len"], cfg["beta_fast"], cfg["beta_slow"],
                                 float(eps), _p(q, f64p), _p(w, f64p))
        return q, w

    def memindex_ensemble(self, x, mode: int = 0, thr: float = 0.5):
        """x [B,L,S] -> mask [B, ceil(S/32)] uint32, ensembled score [B,S] fp64
        (mode 0: max over layers, mode 1: mean over layers of the sigmoids)."""
        x = _c(x, np.float64)
        B, L, S = x.shape
        mask = np.empty((B, (S + 31) // 32), dtype=np.uint32)
        ens = np.empty((B, S), dtype=np.float64)
        self.lib.orc_memindex_ensemble(_p(x, f64p), B, L, S, int(mode), float(thr), _p(mask, u32p), _p(ens, f64p))
        return mask, ens

    # -- top-k -------------------------------------------------------------------
    def topk(self, ids, x, k: int = 512):
        ids = _c(ids, np.int64); x = _c(x, np.float64)
        idx = np.empty(k, dtype=np.int32)
        sc = np.empty(k, dtype=np.float64)
        m = self.lib.orc_topk(_p(ids, i64p), _p(x, f64p), len(ids), k, _p(idx, i32p), _p(sc, f64p))
        return idx, sc, m

    def paged_topk(self, q, w, k8, scale, page_phys, page_logical, n_res=None, k: int = 512,
                   want_logits: bool = False, res_mask=None, mask_group: int = 1, id_mode: int = 0):
        """res_mask [rows, mask_ld] uint32 (row qi // mask_group per query) or
        None; id_mode 0 = logical chunk ids, 1 = reserve cells phys*64 + o."""
        q = _c(q, np.uint16); w = _c(w, np.float32); k8 = _c(k8, np.uint8); scale = _c(scale, np.float32)
        page_phys = _c(page_phys, np.int32); page_logical = _c(page_logical, np.int32)
        Q, n_h, d = q.shape
        R = page_phys.shape[1]
        page = k8.shape[1]
        nr = _c(n_res, np.int32) if n_res is not None else None
        idx = np.empty((Q, k), dtype=np.int32)
        sc = np.empty((Q, k), dtype=np.float64)
        lg = np.empty((Q, R * page), dtype=np.float64) if want_logits else None
        m = _c(np.atleast_2d(res_mask), np.uint32) if res_mask is not None else None
        mask_ld = m.shape[1] if m is not None else 0
        self.lib.orc_paged_topk_ex(_p(q, u16p), _p(w, f32p), _p(k8, u8p), _p(scale, f32p), _p(page_phys, i32p),
                                   _p(page_logical, i32p), _p(nr, i32p), Q, R, n_h, d, page, k, _p(m, u32p),
                                   mask_ld, mask_group, id_mode, _p(idx, i32p), _p(sc, f64p), _p(lg, f64p))
        return (idx, sc, lg) if want_logits else (idx, sc)

    def paged_topk_bf16(self, q, w, kbf, page_phys, page_logical, n_res=None, k: int = 512,
                        want_logits: bool = False, res_mask=None, mask_group: int = 1, id_mode: int = 0):
        """paged_topk over a pool of bf16 keys kbf [P, page, d] (bf16 bits, no scale)."""
        q = _c(q, np.uint16); w = _c(w, np.float32); kbf = _c(kbf, np.uint16)
        page_phys = _c(page_phys, np.int32); page_logical = _c(page_logical, np.int32)
        Q, n_h, d = q.shape
        R = page_phys.shape[1]
        page = kbf.shape[1]
        nr = _c(n_res, np.int32) if n_res is not None else None
        idx = np.empty((Q, k), dtype=np.int32)
        sc = np.empty((Q, k), dtype=np.float64)
        lg = np.empty((Q, R * page), dtype=np.float64) if want_logits else None
        m = _c(np.atleast_2d(res_mask), np.uint32) if res_mask is not None else None
        mask_ld = m.shape[1] if m is not None else 0
        self.lib.orc_paged_topk_bf16_ex(_p(q, u16p), _p(w, f32p), _p(kbf, u16p), _p(page_phys, i32p),
                                        _p(page_logical, i32p), _p(nr, i32p), Q, R, n_h, d, page, k, _p(m, u32p),
                                        mask_ld, mask_group, id_mode, _p(idx, i32p), _p(sc, f64p), _p(lg, f64p))
        return (idx, sc, lg) if want_logits else (idx, sc)

    def causal_limit(self, pos: int, S: int, ratio: int = 4) -> int:
        return self.lib.orc_causal_limit(int(pos), int(S), int(ratio))

    def prefill_logits(self, q, w, pos, K, ratio: int = 4) -> np.ndarray:
        """The prefill scores ([V4] sec. 3 CSA-1): Y[t,s] = sum_h w[t,h] ReLU(q[t,h].K[s])
        for s < causal_limit(pos[t]), -inf beyond.  q [T,n_h,d] bf16 bits,
        w [T,n_h], pos [T], K [S,d] bf16 bits -> [T,S] fp64.  The Memory
        Indexer's logits with every query row reading the same keys (request
        stride 0)."""
        q = _c(q, np.uint16); w = _c(w, np.float32); K = _c(K, np.uint16)
        T, n_h, d = q.shape
        S = K.shape[0]
        x = np.empty((T, 1, S), dtype=np.float64)
        self.lib.orc_memindex_logits(_p(q, u16p), _p(w, f32p), _p(K, u16p), 0, S * d, T, 1, S, n_h, d, _p(x, f64p))
        x = x[:, 0, :]
        for t in range(T):
            x[t, self.causal_limit(int(pos[t]), S, ratio):] = -np.inf
        return x

    def prefill_topk(self, q, w, pos, K, ratio: int = 4, k: int = 512):
        q = _c(q, np.uint16); w = _c(w, np.float32); pos = _c(pos, np.int64); K = _c(K, np.uint16)
        T, n_h, d = q.shape
        S = K.shape[0]
        idx = np.empty((T, k), dtype=np.int32)
        sc = np.empty((T, k), dtype=np.float64)
        self.lib.orc_prefill_topk(_p(q, u16p), _p(w, f32p), _p(pos, i64p), _p(K, u16p), T, S, n_h, d, ratio,
                                  k, _p(idx, i32p), _p(sc, f64p))
        return idx, sc

    def page_recall(self, mask, S: int, kmax: int, sink: int = 0, recent: int = 0, page_size: int = 64):
        """mask [B, ceil(S/32)] uint32 -> (pages [B,kmax] int32 ascending, -1 padded;
        density [B,kmax] int32, -1 padded; n [B] int32)."""
        mask = _c(np.atleast_2d(mask), np.uint32)
        B = mask.shape[0]
        pages = np.empty((B, kmax), np.int32)
        dens = np.empty((B, kmax), np.int32)
        n = np.empty(B, np.int32)
        self.lib.orc_page_recall(_p(mask, u32p), B, S, sink, recent, page_size, kmax,
                                 _p(pages, i32p), _p(dens, i32p), _p(n, i32p))
        return pages, dens, n

    def num_threads(self) -> int:
        return self.lib.orc_num_threads()

    def set_num_threads(self, n: int) -> None:
        self.lib.orc_set_num_threads(int(n))


_default = None


def get() -> Oracle:
    """The oracle compiled from oracle.c (rebuilt if the source is newer)."""
    global _default
    if _default is None:
        if not os.path.exists(SO) or os.path.getmtime(SRC) > os.path.getmtime(SO):
            build()
        _default = Oracle(SO)
    return _default
