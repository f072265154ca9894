"""Seeded synthetic workloads for the LSA c4 indexer (input generation only).

This module makes inputs; it holds none of the indexer's arithmetic.  Element
values come from the counter-based recipes in ``gen.h`` (SplitMix64 streams,
an Irwin-Hall(8) stand-in for normal variates, RNE rounding to bf16 / OCP
E4M3).  The host library (``gen_host.c``) and the device fill kernels
(``gen_cuda.cu``) compile the same recipes, so any sample of a device-filled
multi-GB tensor can be regenerated on the host bit for bit.

Workload recipes follow the indexer's five synthetic configurations:
q ~ N(0, 1) bf16, cold keys ~ N(0, 1/128), head weights w = +1 for heads 0-7
and -0.2 for heads 8-63 (decode configurations) or w ~ N(0, 1/64) (prefill),
planted hot chunks K_s = 3 * unit(mean(q_0..7)) + noise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(HERE, "libfm_gen_host.so")
CUDA_SO = os.path.join(HERE, "libfm_gen_cuda.so")
BASE_SEED = 20260606
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def build_host() -> str:
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11",
           "-o", HOST_SO, os.path.join(HERE, "gen_host.c"), "-lm"]
    subprocess.run(cmd, check=True)
    return HOST_SO


def build_cuda() -> str:
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    cmd = [nvcc, ARCH, "-O3", "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
           "-fmad=false", "-o", CUDA_SO, os.path.join(HERE, "gen_cuda.cu")]
    subprocess.run(cmd, check=True)
    return CUDA_SO


def _stale(so: str, *srcs: str) -> bool:
    if not os.path.exists(so):
        return True
    t = os.path.getmtime(so)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in srcs)


_host = None
_cuda = None

u16p = ctypes.POINTER(ctypes.c_uint16)
u8p = ctypes.POINTER(ctypes.c_uint8)
f32p = ctypes.POINTER(ctypes.c_float)
i32p = ctypes.POINTER(ctypes.c_int32)
i64p = ctypes.POINTER(ctypes.c_int64)
U64, I64, I32, U32, VP = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p


def host_lib():
    global _host
    if _host is None:
        if _stale(HOST_SO, "gen_host.c", "gen.h"):
            build_host()
        lib = ctypes.CDLL(HOST_SO)
        lib.gen_fill_q_bf16.argtypes = [U64, I64, I64, I32, I32, u16p]
        lib.gen_hot_dirs.argtypes = [u16p, I64, I64, I32, I32, f32p]
        lib.gen_k_bf16_rows.argtypes = [U64, I64, I64, i64p, I64, I32, U32, f32p, u16p]
        lib.gen_fill_k_bf16.argtypes = [U64, I64, I64, I64, I32, U32, f32p, u16p]
        lib.gen_planted_list.argtypes = [U64, I64, I64, I64, U32, u8p]
        lib.gen_k_fp8_rows.argtypes = [U64, I64, I64, i64p, I64, I32, U32, f32p, u8p, f32p]
        lib.gen_fill_w_normal.argtypes = [U64, I64, I32, f32p]
        lib.gen_sample_distinct.argtypes = [U64, U64, I64, I64, I32, I32, i32p, i32p]
        lib.gen_sample_distinct.restype = ctypes.c_int
        _host = lib
    return _host


def cuda_lib():
    global _cuda
    if _cuda is None:
        if not os.path.exists(CUDA_SO):
            build_cuda()
        lib = ctypes.CDLL(CUDA_SO)
        lib.gen_cuda_fill_k_bf16.argtypes = [U64, I64, I64, I64, I32, U32, VP, VP, I64, I64, VP]
        lib.gen_cuda_fill_k_fp8_pool.argtypes = [U64, I64, I32, I32, U32, VP, VP, I64, I64, VP, VP, VP]
        lib.gen_cuda_fill_q_bf16.argtypes = [U64, I64, I64, I32, I32, VP, VP]
        lib.gen_cuda_fill_k_bf16_pool.argtypes = [U64, I64, I32, I32, VP, VP, VP]
        for f in (lib.gen_cuda_fill_k_bf16, lib.gen_cuda_fill_k_fp8_pool, lib.gen_cuda_fill_q_bf16,
                  lib.gen_cuda_fill_k_bf16_pool):
            f.restype = ctypes.c_int
        _cuda = lib
    return _cuda


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(t)


def thr32(frac: float) -> int:
    return max(0, min(0xFFFFFFFF, int(frac * 4294967296.0)))


def w_pattern(n_h: int = 64) -> np.ndarray:
    """Decode head weights: +1 for heads 0-7, -0.2 for heads 8..n_h-1 (fp32)."""
    w = np.full(n_h, np.float32(-0.2), dtype=np.float32)
    w[: min(8, n_h)] = 1.0
    return w


# --------------------------------------------------------------------------
# Configurations
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class MemIndexCfg:
    """Memory Indexer workload: B requests x L indexer layers x S chunks."""
    name: str
    B: int
    L: int
    S: int
    n_h: int = 64
    d: int = 128
    hot_frac: float = 0.12
    seed: int = BASE_SEED

    @property
    def chunk_scores(self) -> int:
        return self.B * self.L * self.S


@dataclass(frozen=True)
class PagedCfg:
    """Native paged top-k: requests x layers queries, R resident pages of
    ``page`` chunks drawn from n_pages logical pages per request."""
    name: str
    requests: int
    layers: int
    n_pages: int
    R: int
    n_h: int = 64
    d: int = 128
    page: int = 64
    k: int = 512
    seed: int = BASE_SEED + 3

    @property
    def Q(self) -> int:
        return self.requests * self.layers

    @property
    def P(self) -> int:
        return self.Q * self.R

    @property
    def chunk_scores(self) -> int:
        return self.Q * self.R * self.page


@dataclass(frozen=True)
class PrefillCfg:
    """Prefill top-k: T query tokens at positions pos0.. against S chunks."""
    name: str
    T: int
    S: int
    pos0: int
    n_h: int = 64
    d: int = 128
    ratio: int = 4
    k: int = 512
    seed: int = BASE_SEED + 5

    @property
    def chunk_scores(self) -> int:
        return self.T * self.S


@dataclass(frozen=True)
class RecallCfg:
    """Page recall: B requests' resident masks over S chunks, KMAX densest
    pages recalled.  Mask recipe: hot runs of 64..256 consecutive chunks
    covering about hot_frac of the history (the planted, query-relevant
    regions) plus a fraction ``cold`` of the other chunks (cold chunks whose
    logit still passes the threshold)."""
    name: str
    B: int
    S: int
    kmax: int
    cold: float = 0.25
    hot_frac: float = 0.12
    seed: int = BASE_SEED + 6


TINY = MemIndexCfg("tiny_s4096", B=1, L=1, S=4096, seed=BASE_SEED + 0)
MEMINDEX_256K = MemIndexCfg("memindex_256k_b76_l3_s65536", B=76, L=3, S=65536, seed=BASE_SEED + 1)
MEMINDEX_1M = MemIndexCfg("memindex_1m_b30_l3_s262144", B=30, L=3, S=262144, seed=BASE_SEED + 2)
PAGED_512K = PagedCfg("paged_512k_q1260_r192", requests=60, layers=21, n_pages=2048, R=192,
                      seed=BASE_SEED + 3)
PAGED_1M = PagedCfg("paged_1m_q630_r384", requests=30, layers=21, n_pages=4096, R=384,
                    seed=BASE_SEED + 4)
# The trained retriever's Memory Indexer: 128 heads over packed compressed_k
# rows, at the 1M workload's sizes.
RETRIEVER_1M = MemIndexCfg("retriever_1m_b30_l3_s262144_h128", B=30, L=3, S=262144, n_h=128, seed=BASE_SEED + 10)
# Full-history native top-512 (the path without residency that LSA is
# compared against): every one of a 1M-token request's 4096 pages is listed.
PAGED_FULL_1M = PagedCfg("paged_full_1m_q630_r4096", requests=30, layers=21, n_pages=4096, R=4096,
                         seed=BASE_SEED + 9)
PREFILL = PrefillCfg("prefill_t4096_s65536", T=4096, S=65536, pos0=262144, seed=BASE_SEED + 5)
RECALL_256K = RecallCfg("recall_256k_b76_s65536_k96", B=76, S=65536, kmax=96)
RECALL_512K = RecallCfg("recall_512k_b60_s131072_k192", B=60, S=131072, kmax=192, seed=BASE_SEED + 7)
RECALL_1M = RecallCfg("recall_1m_b30_s262144_k384", B=30, S=262144, kmax=384, seed=BASE_SEED + 8)


def pack_mask(bits: np.ndarray) -> np.ndarray:
    """bool [B, S] -> uint32 [B, ceil(S/32)], bit s & 31 of word s >> 5 = chunk s."""
    bits = np.atleast_2d(bits)
    B, S = bits.shape
    words = (S + 31) // 32
    padded = np.zeros((B, words * 32), dtype=bool)
    padded[:, :S] = bits
    return np.packbits(padded, axis=-1, bitorder="little").view("<u4").reshape(B, words)


def recall_mask(cfg: RecallCfg) -> np.ndarray:
    """Seeded resident mask [B, ceil(S/32)] uint32 for a RecallCfg."""
    rng = np.random.default_rng(cfg.seed)
    bits = rng.random((cfg.B, cfg.S)) < cfg.cold
    for b in range(cfg.B):
        covered = 0
        while covered < cfg.hot_frac * cfg.S:
            run = int(rng.integers(64, 257))
            start = int(rng.integers(0, max(cfg.S - run, 1)))
            bits[b, start:start + run] = True
            covered += run
    return pack_mask(bits)


# --------------------------------------------------------------------------
# Memory Indexer inputs
# --------------------------------------------------------------------------


def memindex_qw(cfg: MemIndexCfg):
    """q [B,L,n_h,d] bf16 bits, w [B,L,n_h] fp32, hot [B,L,d] fp32 (host)."""
    lib = host_lib()
    q = np.empty((cfg.B, cfg.L, cfg.n_h, cfg.d), dtype=np.uint16)
    lib.gen_fill_q_bf16(cfg.seed, cfg.B, cfg.L, cfg.n_h, cfg.d, _p(q, u16p))
    hot = np.empty((cfg.B, cfg.L, cfg.d), dtype=np.float32)
    lib.gen_hot_dirs(_p(q, u16p), cfg.B, cfg.L, cfg.n_h, cfg.d, _p(hot, f32p))
    w = np.broadcast_to(w_pattern(cfg.n_h), (cfg.B, cfg.L, cfg.n_h)).copy()
    return q, w, hot


def memindex_keys_host(cfg: MemIndexCfg, hot: np.ndarray) -> np.ndarray:
    """Dense K [B,L,S,d] bf16 bits on the host (small workloads only)."""
    lib = host_lib()
    K = np.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=np.uint16)
    lib.gen_fill_k_bf16(cfg.seed, cfg.B, cfg.L, cfg.S, cfg.d, thr32(cfg.hot_frac), _p(hot, f32p),
                        _p(K, u16p))
    return K


def memindex_key_rows(cfg: MemIndexCfg, b: int, l: int, s_list, hot: np.ndarray) -> np.ndarray:
    """Keys K[b][l][s][:] for the listed chunk ids (host), bf16 bits [n, d]."""
    s = np.ascontiguousarray(np.asarray(s_list, dtype=np.int64))
    out = np.empty((len(s), cfg.d), dtype=np.uint16)
    h = np.ascontiguousarray(hot[b, l], dtype=np.float32)
    host_lib().gen_k_bf16_rows(cfg.seed, b, l, _p(s, i64p), len(s), cfg.d, thr32(cfg.hot_frac),
                               _p(h, f32p), _p(out, u16p))
    return out


def planted(cfg: MemIndexCfg, b: int, l: int) -> np.ndarray:
    out = np.empty(cfg.S, dtype=np.uint8)
    host_lib().gen_planted_list(cfg.seed, b, l, cfg.S, thr32(cfg.hot_frac), _p(out, u8p))
    return out.astype(bool)


def memindex_keys_device(cfg: MemIndexCfg, hot_dev_ptr: int, out_ptr: int, stride_b: int,
                         stride_l: int, stream: int = 0) -> None:
    """Fill K [B,L,S,d] bf16 on the device (same values as memindex_keys_host)."""
    rc = cuda_lib().gen_cuda_fill_k_bf16(cfg.seed, cfg.B, cfg.L, cfg.S, cfg.d, thr32(cfg.hot_frac),
                                         hot_dev_ptr, out_ptr, stride_b, stride_l, stream)
    if rc != 0:
        raise RuntimeError(f"gen_cuda_fill_k_bf16 failed: cuda error {rc}")


def memindex_fp8_key_rows(cfg: MemIndexCfg, b: int, l: int, s_list, hot: np.ndarray):
    """Compressed keys of (request b, layer l) for the listed chunk ids (host):
    E4M3 codes [n, d] and fp32 scales [n] -- the same planted / cold keys as
    the bf16 workload, quantised per chunk (scale = max|K_s| / 448)."""
    s = np.ascontiguousarray(np.asarray(s_list, dtype=np.int64))
    k8 = np.empty((len(s), cfg.d), dtype=np.uint8)
    sc = np.empty(len(s), dtype=np.float32)
    h = np.ascontiguousarray(hot[b, l], dtype=np.float32)
    host_lib().gen_k_fp8_rows(cfg.seed, b, l, _p(s, i64p), len(s), cfg.d, thr32(cfg.hot_frac), _p(h, f32p),
                              _p(k8, u8p), _p(sc, f32p))
    return k8, sc


def memindex_fp8_keys_host(cfg: MemIndexCfg, hot: np.ndarray):
    """Dense k8 [B,L,S,d] E4M3 codes and scale [B,L,S] fp32 (small workloads)."""
    k8 = np.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=np.uint8)
    sc = np.empty((cfg.B, cfg.L, cfg.S), dtype=np.float32)
    for b in range(cfg.B):
        for l in range(cfg.L):
            k8[b, l], sc[b, l] = memindex_fp8_key_rows(cfg, b, l, np.arange(cfg.S), hot)
    return k8, sc


def memindex_fp8_keys_device(cfg: MemIndexCfg, hot_dev_ptr: int, owner_dev_ptr: int, k8_ptr: int, scale_ptr: int,
                             stream: int = 0) -> None:
    """Fill dense k8 [B,L,S,d] and scale [B,L,S] on the device with the values
    of memindex_fp8_keys_host.  The dense layout is a pool of 64-chunk blocks:
    block (b*L + l)*(S/64) + j holds chunks 64j.. of (b, l); owner_dev_ptr
    points at memindex_fp8_owner(cfg) on the device.  Needs S % 64 == 0."""
    if cfg.S % 64:
        raise ValueError("memindex_fp8_keys_device needs S % 64 == 0")
    P = cfg.B * cfg.L * (cfg.S // 64)
    rc = cuda_lib().gen_cuda_fill_k_fp8_pool(cfg.seed, P, cfg.d, 64, thr32(cfg.hot_frac), owner_dev_ptr,
                                             hot_dev_ptr, cfg.L * cfg.d, cfg.d, k8_ptr, scale_ptr, stream)
    if rc != 0:
        raise RuntimeError(f"gen_cuda_fill_k_fp8_pool failed: cuda error {rc}")


def pack_compressed_k(k8: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """The retriever's packed rows: [..., 128] E4M3 codes and [...] fp32 scales
    -> [..., 132] bytes (codes, then the scale's little-endian bytes)."""
    sc = np.ascontiguousarray(scale, dtype="<f4")
    return np.concatenate([np.asarray(k8, dtype=np.uint8), sc.view(np.uint8).reshape(sc.shape + (4,))], axis=-1)


def query_chain_inputs(T: int, dim: int = 4096, r: int = 2048, n_h: int = 128, head_dim: int = 128,
                       seed: int = BASE_SEED + 11, pos=None):
    """Synthetic weights and inputs of one CSA layer's query chain (bf16 bits):
    hidden [T,dim] ~ N(0,1), wq_a [r,dim] ~ N(0,1/dim), q_norm [r] ~ U(0.5,1.5),
    wq_b [n_h*head_dim, r] ~ N(0,1/r), w_proj [n_h,dim] ~ N(0,1/dim); pos [T]
    int64 spread over a 1M-token context unless given."""
    rng = np.random.default_rng(seed)

    def bf16(a):
        u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    hidden = bf16(rng.standard_normal((T, dim)))
    wq_a = bf16(rng.standard_normal((r, dim)) / np.sqrt(dim))
    q_norm = bf16(rng.uniform(0.5, 1.5, r))
    wq_b = bf16(rng.standard_normal((n_h * head_dim, r)) / np.sqrt(r))
    w_proj = bf16(rng.standard_normal((n_h, dim)) / np.sqrt(dim))
    if pos is None:
        pos = rng.integers(0, 1 << 20, T)
        pos[: min(T, 3)] = [0, 65535, (1 << 20) - 1][: min(T, 3)]
    return hidden, wq_a, q_norm, wq_b, w_proj, np.asarray(pos, dtype=np.int64)


def memindex_fp8_owner(cfg: MemIndexCfg) -> np.ndarray:
    """owner [B*L*S/64, 3] int32: (request, layer, block) of each 64-chunk block."""
    nb = cfg.S // 64
    blk = np.arange(cfg.B * cfg.L * nb, dtype=np.int64)
    return np.stack([blk // (cfg.L * nb), (blk // nb) % cfg.L, blk % nb], axis=1).astype(np.int32)


# --------------------------------------------------------------------------
# Paged inputs
# --------------------------------------------------------------------------


def paged_tables(cfg: PagedCfg):
    """page_logical, page_phys [Q,R] int32 and owner [P,3] int32.

    Query qi = r * layers + j (request r, CSA layer j).  The R resident logical
    pages of request r are drawn uniformly without replacement from n_pages and
    shared by its layers; each (request, layer) page has its own physical pool
    page, placed by a seeded permutation of the pool.
    """
    lib = host_lib()
    Q, R = cfg.Q, cfg.R
    logical = np.empty((Q, R), dtype=np.int32)
    scratch = np.empty(max(cfg.n_pages, cfg.P), dtype=np.int32)
    row = np.empty(R, dtype=np.int32)
    for r in range(cfg.requests):
        rc = lib.gen_sample_distinct(cfg.seed, 5, r, 0, cfg.n_pages, R, _p(scratch, i32p), _p(row, i32p))
        if rc != 0:
            raise ValueError("R > n_pages")
        logical[r * cfg.layers:(r + 1) * cfg.layers] = row
    perm = np.empty(cfg.P, dtype=np.int32)
    lib.gen_sample_distinct(cfg.seed, 6, 0, 0, cfg.P, cfg.P, _p(scratch, i32p), _p(perm, i32p))
    phys = perm.reshape(Q, R).copy()
    owner = np.empty((cfg.P, 3), dtype=np.int32)
    qi = np.repeat(np.arange(Q, dtype=np.int32), R)
    owner[phys.reshape(-1), 0] = qi // cfg.layers
    owner[phys.reshape(-1), 1] = qi % cfg.layers
    owner[phys.reshape(-1), 2] = logical.reshape(-1)
    return logical, phys, owner


def paged_qw(cfg: PagedCfg):
    """q [Q,n_h,d] bf16 bits (stream (request, layer)), w [Q,n_h] fp32."""
    q = np.empty((cfg.requests, cfg.layers, cfg.n_h, cfg.d), dtype=np.uint16)
    host_lib().gen_fill_q_bf16(cfg.seed, cfg.requests, cfg.layers, cfg.n_h, cfg.d, _p(q, u16p))
    w = np.broadcast_to(w_pattern(cfg.n_h), (cfg.Q, cfg.n_h)).copy()
    return q.reshape(cfg.Q, cfg.n_h, cfg.d), w


def paged_pool_host(cfg: PagedCfg, owner: np.ndarray):
    """k8 [P,page,d] E4M3 codes and scale [P,page] fp32 on the host."""
    lib = host_lib()
    k8 = np.empty((cfg.P, cfg.page, cfg.d), dtype=np.uint8)
    scale = np.empty((cfg.P, cfg.page), dtype=np.float32)
    for p in range(cfg.P):
        a, b, lp = (int(v) for v in owner[p])
        s = np.arange(lp * cfg.page, (lp + 1) * cfg.page, dtype=np.int64)
        lib.gen_k_fp8_rows(cfg.seed, a, b, _p(s, i64p), cfg.page, cfg.d, 0, None,
                           _p(k8[p], u8p), _p(scale[p], f32p))
    return k8, scale


def paged_pool_rows(cfg: PagedCfg, logical: np.ndarray, phys: np.ndarray, queries=None, n_pool=None):
    """The pool pages that the listed queries' tables name, filled with the
    values of paged_pool_host: one host call per query (all its pages at once).

    queries: query ids (default all); phys: pool page per table entry (the
    caller may pass a remapped, local numbering).  Returns k8 [n_pool, page, d]
    and scale [n_pool, page]; pages no listed query names stay zero.
    """
    queries = range(cfg.Q) if queries is None else queries
    n_pool = cfg.P if n_pool is None else n_pool
    k8 = np.zeros((n_pool, cfg.page, cfg.d), dtype=np.uint8)
    scale = np.zeros((n_pool, cfg.page), dtype=np.float32)
    off = np.arange(cfg.page, dtype=np.int64)
    for qi in queries:
        a, b = int(qi) // cfg.layers, int(qi) % cfg.layers
        s = (logical[qi].astype(np.int64)[:, None] * cfg.page + off[None, :]).reshape(-1)
        rows, sc = paged_chunk_rows(cfg, a, b, s)
        k8[phys[qi]] = rows.reshape(-1, cfg.page, cfg.d)
        scale[phys[qi]] = sc.reshape(-1, cfg.page)
    return k8, scale


def paged_pool_rows_bf16(cfg: PagedCfg, logical: np.ndarray, phys: np.ndarray, queries=None, n_pool=None):
    """A pool of bf16 keys for the listed queries' tables (the same cold-key
    recipe, N(0, 1/128), rounded to bf16 instead of quantised to E4M3):
    kbf [n_pool, page, d] bf16 bits; pages no listed query names stay zero."""
    queries = range(cfg.Q) if queries is None else queries
    n_pool = cfg.P if n_pool is None else n_pool
    kbf = np.zeros((n_pool, cfg.page, cfg.d), dtype=np.uint16)
    off = np.arange(cfg.page, dtype=np.int64)
    for qi in queries:
        a, b = int(qi) // cfg.layers, int(qi) % cfg.layers
        s = np.ascontiguousarray((logical[qi].astype(np.int64)[:, None] * cfg.page + off[None, :]).reshape(-1))
        rows = np.empty((len(s), cfg.d), dtype=np.uint16)
        host_lib().gen_k_bf16_rows(cfg.seed, a, b, _p(s, i64p), len(s), cfg.d, 0, None, _p(rows, u16p))
        kbf[phys[qi]] = rows.reshape(-1, cfg.page, cfg.d)
    return kbf


def paged_chunk_rows(cfg: PagedCfg, a: int, b: int, s_list):
    """E4M3 codes [n,d] and scales [n] of chunks s_list of stream (request a, layer b)."""
    s = np.ascontiguousarray(np.asarray(s_list, dtype=np.int64))
    k8 = np.empty((len(s), cfg.d), dtype=np.uint8)
    sc = np.empty(len(s), dtype=np.float32)
    host_lib().gen_k_fp8_rows(cfg.seed, a, b, _p(s, i64p), len(s), cfg.d, 0, None, _p(k8, u8p),
                              _p(sc, f32p))
    return k8, sc


def paged_pool_device(cfg: PagedCfg, owner_dev_ptr: int, k8_ptr: int, scale_ptr: int,
                      stream: int = 0) -> None:
    rc = cuda_lib().gen_cuda_fill_k_fp8_pool(cfg.seed, cfg.P, cfg.d, cfg.page, 0, owner_dev_ptr, None,
                                             0, 0, k8_ptr, scale_ptr, stream)
    if rc != 0:
        raise RuntimeError(f"gen_cuda_fill_k_fp8_pool failed: cuda error {rc}")


def paged_pool_bf16_device(cfg: PagedCfg, owner_dev_ptr: int, kbf_ptr: int, stream: int = 0) -> None:
    """A bf16 key pool [P, page, d] on the device with the values of
    paged_pool_rows_bf16 (owner_dev_ptr: paged_tables' owner on the device)."""
    rc = cuda_lib().gen_cuda_fill_k_bf16_pool(cfg.seed, cfg.P, cfg.d, cfg.page, owner_dev_ptr, kbf_ptr, stream)
    if rc != 0:
        raise RuntimeError(f"gen_cuda_fill_k_bf16_pool failed: cuda error {rc}")


# --------------------------------------------------------------------------
# Prefill inputs
# --------------------------------------------------------------------------


def prefill_host(cfg: PrefillCfg, pos=None):
    """q [T,n_h,d] bf16 bits, w [T,n_h] fp32 ~ N(0,1/64), pos [T] int64,
    K [S,d] bf16 bits ~ N(0,1/128) (no planting)."""
    lib = host_lib()
    q = np.empty((cfg.T, 1, cfg.n_h, cfg.d), dtype=np.uint16)
    lib.gen_fill_q_bf16(cfg.seed, cfg.T, 1, cfg.n_h, cfg.d, _p(q, u16p))
    w = np.empty((cfg.T, cfg.n_h), dtype=np.float32)
    lib.gen_fill_w_normal(cfg.seed, cfg.T, cfg.n_h, _p(w, f32p))
    K = np.empty((1, 1, cfg.S, cfg.d), dtype=np.uint16)
    lib.gen_fill_k_bf16(cfg.seed, 1, 1, cfg.S, cfg.d, 0, None, _p(K, u16p))
    if pos is None:
        pos = cfg.pos0 + np.arange(cfg.T, dtype=np.int64)
    return q.reshape(cfg.T, cfg.n_h, cfg.d), w, np.ascontiguousarray(pos, dtype=np.int64), K.reshape(cfg.S, cfg.d)


__all__ = [
    "BASE_SEED", "MemIndexCfg", "PagedCfg", "PrefillCfg", "TINY", "MEMINDEX_256K", "MEMINDEX_1M",
    "PAGED_512K", "PAGED_1M", "PAGED_FULL_1M", "RETRIEVER_1M", "PREFILL", "memindex_qw", "memindex_keys_host", "memindex_key_rows",
    "memindex_keys_device", "planted", "pack_compressed_k", "query_chain_inputs", "paged_tables", "paged_qw", "paged_pool_host",
    "paged_chunk_rows", "paged_pool_rows", "paged_pool_rows_bf16", "paged_pool_device", "paged_pool_bf16_device", "prefill_host", "w_pattern", "thr32", "replace",
]
