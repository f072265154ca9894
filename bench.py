#!/usr/bin/env python3
"""Benchmark of the LSA c4 indexer hot path on GB300.

One step is one pass of the whole hot path over one batch of synthetic input
at 1M-token context:
  1. Memory Indexer (fm_memindex_score_mask): 30 requests x 3 indexer layers x
     262144 c4 chunks, bf16 keys, 12% planted -> OR-union resident bitmask and
     per-chunk max-sigmoid;
  2. native paged top-512 (fm_native_topk_paged): 30 requests x 21 CSA layers,
     384 resident 64-chunk E4M3 pages each (KMAX at 1M context);
  3. prefill top-512 (fm_index_prefill_topk): 4096 query tokens at positions
     262144.. against 65536 bf16 chunks under the causal limit.
value = chunk scores computed per second (all phases, all ranks);
queries_per_s = top-512 queries answered per second.

Inputs live in HBM before the timed region; the keys streamed per step
(6.04 GB + 2.04 GB) are far larger than the 129 MB L2, so no L2 flush is
needed between steps.  `e2e` repeats the step through the same calls with the
inputs in pinned host memory: the host->device copies of every input and the
device->host copies of every output are inside its timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, fp64) on a bounded sample of
the same workload on the host cores.  Under torchrun every rank runs its own
batch (weak scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "indexer chunk-scores/s + top-512 queries/s at 1M ctx; % of HBM roofline"
UNIT = "chunk-scores/s"
WORKLOAD = ("lsa_c4_indexer_1m: memindex 30x3x262144 bf16 (12% hot) + paged top-512 630 queries x 384 pages "
            "E4M3 + prefill top-512 4096 tokens x 65536 chunks")


PROFILE_CASES = {
    # phase: [(profile summary, kernel source files, units in the summary's case, units in the bench step)]
    "memindex": [("memindex_kernel_memindex_1m_b4_l3_s262144.md", ["memindex.cu", "fm_common.cuh"], 4, 30)],
    "paged_topk": [("paged_score_kernel_paged_1m_q84_r384.md", ["paged.cu", "fp8.cuh", "fm_common.cuh"], 84, 630),
                   ("topk_rows_kernel_paged_1m_q84_r384.md", ["topk.cu", "topk.cuh", "fm_common.cuh"], 84, 630)],
    "memindex_fp8": [("memindex_fp8_kernel_memindex_fp8_1m_b4_l3_s262144.md", ["memindex_fp8.cu", "fp8.cuh", "fm_common.cuh"],
                      4, 30)],
    "retriever": [("retriever_kernel_retriever_1m_b4_l3_s262144.md", ["retriever.cu", "fp8.cuh", "fm_common.cuh"], 4, 30)],
    "query_chain": [("proj_gemm_kernel_query_chain_t30.md", ["query_chain.cu", "fm_common.cuh"], 1, 1)],
    "prefill_scores": [("prefill_score_kernel_prefill_t4096_s65536_dram.md", ["prefill.cu", "fm_common.cuh"], 1, 1)],
    "prefill_topk": [("prefill_score_kernel_prefill_t512_s65536.md", ["prefill.cu", "fm_common.cuh"], 512, 4096),
                     ("topk_rows_segmax_kernel_prefill_t512_s65536.md", ["topk.cu", "topk.cuh", "fm_common.cuh"], 512,
                      4096)],
}


def kernel_traffic(name: str):
    """DRAM bytes (read + write) per launch of a full-size kernel launch from
    its committed one-pass ncu summary; None if its sources changed since."""
    return profiled_traffic(name)


def profiled_traffic(phase: str):
    """DRAM traffic (read + write bytes) of a phase's kernels per step, from the
    committed ncu summaries in profiles/, scaled from the captured case by the
    units processed; None if a kernel's source changed since its capture."""
    import hashlib
    import re
    total = 0.0
    for name, files, units_case, units_step in PROFILE_CASES.get(phase, []):
        path = os.path.join(ROOT, "profiles", name)
        if not os.path.exists(path):
            return None
        text = open(path).read()
        m_hash = re.search(r"first 16 hex\): `([0-9a-f]+)`", text)
        m_traf = re.findall(r"\| traffic \(read \+ write\) per launch \| ([0-9.]+) MB \|", text)
        if not m_hash or not m_traf:
            return None
        h = hashlib.sha256()
        for f in files:
            with open(os.path.join(ROOT, "sparse_attention_kv_c4_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest()[:16] != m_hash.group(1):
            return None
        total += sum(float(x) for x in m_traf) * 1e6 * units_step / units_case  # every launch of the summary
    return total or None


def profile_metric(name: str, files, metric: str):
    """One metric row of a committed ncu summary in profiles/ (a float), or
    None if the summary is missing or its kernel sources changed since."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"first 16 hex\): `([0-9a-f]+)`", text)
    m = re.search(r"\| " + re.escape(metric) + r" \| ([0-9.]+)", text)
    if not m_hash or not m:
        return None
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sparse_attention_kv_c4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return float(m.group(1)) if h.hexdigest()[:16] == m_hash.group(1) else None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# GB300's nominal HBM3e bandwidth: a read-dominated kernel can pass the
# measured copy peak, never this.
HBM_NOMINAL_GBS = 7900.0


def read_peak_gbs(torch, dev, gib: int = 4, reps: int = 10) -> float:
    """A read-only streaming rate for the read-dominated kernels (the Memory
    Indexer reads ~250 bytes for every byte it writes): torch's sum over a
    `gib` GiB fp32 buffer, best of `reps`, CUDA events.  MEASURED_PEAKS.json's
    hbm_gbs is a copy (read + write) and stays the roofline's denominator;
    this is reported beside it."""
    x = torch.ones((gib << 28,), dtype=torch.float32, device=dev)
    best = None
    for _ in range(reps + 2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        x.sum()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    del x
    return (gib << 30) / (best / 1e3) / 1e9


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s in sm if s > 0.5 * (max(smax) if smax else 1)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload construction
# ---------------------------------------------------------------------------


def workload_cfgs(small: bool):
    """The step's three configurations; `small` shrinks each one (fewer
    requests / queries / tokens, same per-unit shape) for ncu captures."""
    import gen
    mi, pg, pf = gen.MEMINDEX_1M, gen.PAGED_1M, gen.PREFILL
    if small:
        mi = gen.replace(mi, B=4)
        pg = gen.replace(pg, requests=4)
        pf = gen.replace(pf, T=512)
    return mi, pg, pf


def build_inputs(torch, dev, cfgs, only=None):
    import gen
    mi, pg, pf = cfgs
    W = {}
    if only not in (None, "memindex"):
        mi = None
    if only not in (None, "paged"):
        pg = None
    if only not in (None, "prefill"):
        pf = None
    if mi is None:
        return _build_rest(torch, dev, W, cfgs, pg, pf)
    q, w, hot = gen.memindex_qw(mi)
    W["mi_q"] = torch.from_numpy(q.view(np.int16)).to(dev)
    W["mi_w"] = torch.from_numpy(w).to(dev)
    hot_d = torch.from_numpy(hot).to(dev)
    W["mi_K"] = torch.empty((mi.B, mi.L, mi.S, mi.d), dtype=torch.int16, device=dev)
    gen.memindex_keys_device(mi, hot_d.data_ptr(), W["mi_K"].data_ptr(), mi.L * mi.S * mi.d, mi.S * mi.d)
    W["mi_mask"] = torch.empty((mi.B, (mi.S + 31) // 32), dtype=torch.int32, device=dev)
    W["mi_maxsig"] = torch.empty((mi.B, mi.S), dtype=torch.float32, device=dev)
    W["rc_pages"] = torch.empty((mi.B, KMAX), dtype=torch.int32, device=dev)
    W["rc_n"] = torch.empty((mi.B,), dtype=torch.int32, device=dev)
    return _build_rest(torch, dev, W, cfgs, pg, pf)


def _build_rest(torch, dev, W, cfgs, pg, pf):
    import gen
    if pg is None:
        return _build_prefill(torch, dev, W, cfgs, pf)
    logical, phys, owner = gen.paged_tables(pg)
    q, w = gen.paged_qw(pg)
    W["pg_q"] = torch.from_numpy(q.view(np.int16)).to(dev)
    W["pg_w"] = torch.from_numpy(w).to(dev)
    own_d = torch.from_numpy(owner).to(dev)
    W["pg_k8"] = torch.empty((pg.P, pg.page, pg.d), dtype=torch.uint8, device=dev)
    W["pg_scale"] = torch.empty((pg.P, pg.page), dtype=torch.float32, device=dev)
    gen.paged_pool_device(pg, own_d.data_ptr(), W["pg_k8"].data_ptr(), W["pg_scale"].data_ptr())
    W["pg_phys"] = torch.from_numpy(phys).to(dev)
    W["pg_logical"] = torch.from_numpy(logical).to(dev)
    W["pg_idx"] = torch.empty((pg.Q, pg.k), dtype=torch.int32, device=dev)
    W["pg_score"] = torch.empty((pg.Q, pg.k), dtype=torch.float32, device=dev)
    return _build_prefill(torch, dev, W, cfgs, pf)


def _build_prefill(torch, dev, W, cfgs, pf):
    import gen
    if pf is None:
        torch.cuda.synchronize()
        return W, cfgs
    q, w, pos, K = gen.prefill_host(pf)
    W["pf_q"] = torch.from_numpy(q.view(np.int16)).to(dev)
    W["pf_w"] = torch.from_numpy(w).to(dev)
    W["pf_pos"] = torch.from_numpy(pos).to(dev)
    W["pf_K"] = torch.from_numpy(K.view(np.int16)).to(dev)
    W["pf_idx"] = torch.empty((pf.T, pf.k), dtype=torch.int32, device=dev)
    W["pf_score"] = torch.empty((pf.T, pf.k), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    return W, cfgs


INPUT_KEYS = ["mi_q", "mi_w", "mi_K", "pg_q", "pg_w", "pg_k8", "pg_scale", "pg_phys", "pg_logical", "pf_q", "pf_w",
              "pf_pos", "pf_K"]
OUTPUT_KEYS = ["mi_mask", "mi_maxsig", "rc_pages", "rc_n", "pg_idx", "pg_score", "pf_idx", "pf_score"]
# Pages recalled per request after the Memory Indexer: the KMAX of 1M context
# (256K -> 96, 512K -> 192, 1M -> 384 densest 64-chunk pages).
KMAX = 384


def make_step(fm, W, cfgs, ws, events=None):
    mi, pg, pf = cfgs

    def step():
        if events is not None:
            events[0].record()
        if "mi_K" in W:
            fm.fm_memindex_score_mask(W["mi_q"], W["mi_w"], W["mi_K"], W["mi_mask"], W["mi_maxsig"])
        if events is not None:
            events[1].record()
        if "mi_K" in W:
            fm.fm_page_recall(W["mi_mask"], mi.S, KMAX, W["rc_pages"], None, W["rc_n"])
        if events is not None:
            events[4].record()
        if "pg_k8" in W:
            fm.fm_native_topk_paged(W["pg_q"], W["pg_w"], W["pg_k8"], W["pg_scale"], W["pg_phys"],
                                    W["pg_logical"], pg.k, W["pg_idx"], W["pg_score"], workspace=ws["pg"])
        if events is not None:
            events[2].record()
        if "pf_K" in W:
            fm.fm_index_prefill_topk(W["pf_q"], W["pf_w"], W["pf_pos"], W["pf_K"], pf.k, W["pf_idx"],
                                     W["pf_score"], workspace=ws["pf"])
        if events is not None:
            events[3].record()
    return step


KERNELS_PER_STEP = 1 + 1 + 3 + 3  # memindex; page recall; paged prep/score/top-k; prefill limits/score/top-k


def time_prefill_scores(fm, torch, W, ws, reps=10, warmup=2):
    """The step's dominant kernel, prefill_score_kernel, alone: one
    fm_index_prefill_scores call per launch (the prefill call's own score
    kernel, writing into the prefill workspace's logits, then the -inf fill
    past the causal limits, which has nothing to write at this workload),
    timed with CUDA events on the current stream; mean ms per call."""
    logits = ws["pf"][: W["pf_q"].shape[0] * W["pf_K"].shape[0] * 4].view(torch.float32).view(
        W["pf_q"].shape[0], W["pf_K"].shape[0])

    def call():
        fm.fm_index_prefill_scores(W["pf_q"], W["pf_w"], W["pf_pos"], W["pf_K"], logits)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        call()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def phase_figures(cfgs):
    mi, pg, pf = cfgs
    return {
        "memindex": {"chunk_scores": mi.chunk_scores, "queries": 0,
                     "bytes": mi.B * mi.L * mi.S * mi.d * 2 + mi.B * mi.S * 4 + mi.B * ((mi.S + 31) // 32) * 4,
                     "flops": mi.chunk_scores * mi.n_h * mi.d * 2, "bound": "hbm"},
        "page_recall": {"chunk_scores": 0, "queries": 0,
                        "bytes": mi.B * ((mi.S + 31) // 32) * 4 + mi.B * (KMAX + 1) * 4, "flops": 0,
                        "bound": "hbm"},
        "paged_topk": {"chunk_scores": pg.chunk_scores, "queries": pg.Q,
                       "bytes": pg.P * pg.page * (pg.d + 4) + pg.Q * pg.R * 8 + pg.Q * pg.k * 8,
                       "flops": pg.chunk_scores * pg.n_h * pg.d * 2, "bound": "hbm"},
        "prefill_topk": {"chunk_scores": pf.chunk_scores, "queries": pf.T,
                         "bytes": pf.T * pf.n_h * pf.d * 2 + pf.S * pf.d * 2 + pf.T * pf.k * 8,
                         "flops": pf.chunk_scores * pf.n_h * pf.d * 2, "bound": "tensor"},
    }


def resident_fraction(torch, mask, B, S):
    """Fraction of the B x S chunks set in a packed resident mask (a popcount
    through a byte table; a reported statistic, not part of the path)."""
    lut = torch.tensor([bin(i).count("1") for i in range(256)], dtype=torch.int64, device=mask.device)
    return float(lut[mask.contiguous().view(torch.uint8).long()].sum().item()) / (B * S)


def memindex_hot_variant(torch, dev, fm, W, mi, hot, pk, reps=10, warmup=3):
    """The 1M Memory-Indexer workload at another planted-hot fraction: the
    step's key buffer refilled in place (after the step), timed alone."""
    import gen
    cfg = gen.replace(mi, hot_frac=hot)
    q, w, hv = gen.memindex_qw(cfg)
    W["mi_q"].copy_(torch.from_numpy(q.view(np.int16)))
    W["mi_w"].copy_(torch.from_numpy(w))
    hot_d = torch.from_numpy(hv).to(dev)
    gen.memindex_keys_device(cfg, hot_d.data_ptr(), W["mi_K"].data_ptr(), cfg.L * cfg.S * cfg.d, cfg.S * cfg.d)
    call = lambda: fm.fm_memindex_score_mask(W["mi_q"], W["mi_w"], W["mi_K"], W["mi_mask"], W["mi_maxsig"])
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        call()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    nbytes = cfg.B * cfg.L * cfg.S * 256 + cfg.B * cfg.S * 4 + cfg.B * ((cfg.S + 31) // 32) * 4
    ach = nbytes / (ms / 1e3) / 1e9
    return {"ms": round(ms, 4), "chunk_scores_per_s": cfg.B * cfg.L * cfg.S / (ms / 1e3), "bound": "hbm",
            "achieved": round(ach, 2), "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
            "algorithmic_bytes": nbytes, "hot_frac": hot,
            "resident_fraction": round(resident_fraction(torch, W["mi_mask"], cfg.B, cfg.S), 4), "reps": reps,
            "workload": f"memindex {cfg.B}x{cfg.L}x{cfg.S} bf16, {int(round(hot * 100))}% planted hot"}


def sanity(torch, W, cfgs):
    mi, pg, pf = cfgs
    frac = resident_fraction(torch, W["mi_mask"], mi.B, mi.S)
    ok = bool((W["pg_idx"] >= 0).all().item()) and bool((W["pf_idx"] >= 0).all().item())
    recalled = float(W["rc_n"].float().mean().item())
    return {"resident_fraction": frac, "topk_full": ok, "pages_recalled_mean": recalled}


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------


class OracleSample:
    """A bounded sample of the step for the CPU oracle: one Memory-Indexer
    request over a chunk prefix, whole paged queries, whole prefill rows, in
    roughly the step's proportions of chunk scores."""

    def __init__(self, cfgs):
        import gen
        import oracle
        self.orc = oracle.get()
        mi, pg, pf = cfgs
        self.cfgs = cfgs
        n_mi = 8192
        q, w, hot = gen.memindex_qw(mi)
        s = np.arange(n_mi)
        self.mi = (q[:1], w[:1], np.stack([gen.memindex_key_rows(mi, 0, l, s, hot) for l in range(mi.L)])[None])
        n_pg = 1
        logical, phys, owner = gen.paged_tables(pg)
        qp, wp = gen.paged_qw(pg)
        k8s = np.empty((n_pg * pg.R, pg.page, pg.d), np.uint8)
        scs = np.empty((n_pg * pg.R, pg.page), np.float32)
        for i in range(n_pg):
            a, b = i // pg.layers, i % pg.layers
            for j in range(pg.R):
                lp = int(logical[i, j])
                k8s[i * pg.R + j], scs[i * pg.R + j] = gen.paged_chunk_rows(
                    pg, a, b, np.arange(lp * pg.page, (lp + 1) * pg.page))
        sub_phys = np.arange(n_pg * pg.R, dtype=np.int32).reshape(n_pg, pg.R)
        self.pg = (qp[:n_pg], wp[:n_pg], k8s, scs, sub_phys, logical[:n_pg])
        n_pf = 8
        self.pf = gen.prefill_host(gen.replace(pf, T=n_pf))
        self.chunk_scores = mi.L * n_mi + n_pg * pg.R * pg.page + n_pf * pf.S
        self.queries = n_pg + n_pf
        self.desc = (f"memindex 1 request x {mi.L} layers x {n_mi} chunks + paged {n_pg} query x {pg.R} pages + "
                     f"prefill {n_pf} tokens x {pf.S} chunks ({self.chunk_scores} chunk scores)")

    def run_once(self) -> float:
        mi, pg, pf = self.cfgs
        t0 = time.perf_counter()
        x = self.orc.memindex_logits(*self.mi)
        self.orc.memindex_select(x, 0.5)
        self.orc.paged_topk(*self.pg, k=pg.k)
        q, w, pos, K = self.pf
        self.orc.prefill_topk(q, w, pos, K, k=pf.k)
        return time.perf_counter() - t0

    def rate(self, min_seconds: float = 10.0, max_reps: int = 50):
        """Repeat the sample until at least min_seconds of CPU time."""
        dt, reps = 0.0, 0
        while dt < min_seconds and reps < max_reps:
            dt += self.run_once()
            reps += 1
        return self.chunk_scores * reps / dt, self.queries * reps / dt, dt, reps


# ---------------------------------------------------------------------------


def reduce_max(value: float, device, world: int) -> float:
    """MAX of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    import gen
    cfgs = (gen.MEMINDEX_1M, gen.PAGED_1M, gen.PREFILL)
    smp = OracleSample(cfgs)
    dt, reps = 0.0, 0
    for i in range(args.warmup + args.steps):
        t = smp.run_once()
        if i >= args.warmup:
            dt += t
            reps += 1
    value = smp.chunk_scores * reps / dt
    nq = smp.queries * reps
    threads = smp.orc.num_threads()
    desc = smp.desc
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / reps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "queries_per_s": nq / dt,
            "config": {"workload": WORKLOAD + " (bounded sample per step)", "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import sparse_attention_kv_c4_gb300 as fm
    fm.lib()

    if args.only == "prefill_scores":  # the dominant kernel alone at full size (one-pass DRAM capture)
        cfgs = workload_cfgs(False)
        W, cfgs = build_inputs(torch, dev, cfgs, "prefill")
        pf = cfgs[2]
        ws = {"pf": torch.empty(fm.fm_index_prefill_workspace(pf.T, pf.S), dtype=torch.uint8, device=dev)}
        ms = time_prefill_scores(fm, torch, W, ws, reps=max(1, args.steps), warmup=args.warmup)
        print(json.dumps({"profile_case": True, "only": args.only, "ms_per_step": ms,
                          "device_status": fm.fm_device_status(reset=True)}), flush=True)
        return
    if args.only == "recall":  # page recall alone: the 1M recall workload's masks (30 x 262144 chunks, KMAX 384)
        import gen
        rc = gen.RECALL_1M
        mask = torch.from_numpy(gen.recall_mask(rc).view(np.int32)).to(dev)
        pages = torch.empty((rc.B, rc.kmax), dtype=torch.int32, device=dev)
        n_out = torch.empty((rc.B,), dtype=torch.int32, device=dev)
        ms = time_call(torch, lambda: fm.fm_page_recall(mask, rc.S, rc.kmax, pages, None, n_out),
                       max(1, args.steps), args.warmup)
        print(json.dumps({"profile_case": True, "only": args.only, "ms_per_step": ms,
                          "device_status": fm.fm_device_status(reset=True)}), flush=True)
        return
    if args.only in ("memindex_fp8", "paged_full", "retriever", "query_chain"):
        v = {"memindex_fp8": Fp8MemIndex, "paged_full": FullHistoryPaged, "retriever": RetrieverMemIndex,
             "query_chain": QueryChain}[args.only](torch, dev, fm, small=args.small)
        r = v.measure(max(1, args.steps), args.warmup, peaks())
        print(json.dumps({"profile_case": True, "only": args.only, "small": args.small, "ms_per_step": r["ms"],
                          "device_status": fm.fm_device_status(reset=True)}), flush=True)
        return
    cfgs = workload_cfgs(args.small)
    W, cfgs = build_inputs(torch, dev, cfgs, args.only)
    mi, pg, pf = cfgs
    ws = {}
    if "pg_k8" in W:
        ws["pg"] = torch.empty(fm.fm_native_topk_paged_workspace(pg.Q, pg.R), dtype=torch.uint8, device=dev)
    if "pf_K" in W:
        ws["pf"] = torch.empty(fm.fm_index_prefill_workspace(pf.T, pf.S), dtype=torch.uint8, device=dev)
    if args.only is not None or args.small:
        return run_profile_case(args, fm, torch, W, cfgs, ws)
    stream = torch.cuda.current_stream()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    warm = make_step(fm, W, cfgs, ws)
    for _ in range(args.warmup):
        warm()
    torch.cuda.synchronize()
    if fm.fm_device_status(reset=True) != 0:
        raise RuntimeError("device status flagged an error during warm-up")

    # ---- device-resident timed region ----
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        make_step(fm, W, cfgs, ws, ev[i])()
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms_total = start.elapsed_time(end)
    phase_ms = {"memindex": [], "page_recall": [], "paged_topk": [], "prefill_topk": []}
    for e in ev:
        phase_ms["memindex"].append(e[0].elapsed_time(e[1]))
        phase_ms["page_recall"].append(e[1].elapsed_time(e[4]))
        phase_ms["paged_topk"].append(e[4].elapsed_time(e[2]))
        phase_ms["prefill_topk"].append(e[2].elapsed_time(e[3]))
    status = fm.fm_device_status(reset=True)
    chk = sanity(torch, W, cfgs)

    ms_total = reduce_max(ms_total, dev, world)
    ms_step = ms_total / K
    figs = phase_figures(cfgs)
    cs_step = sum(f["chunk_scores"] for f in figs.values())
    q_step = sum(f["queries"] for f in figs.values())
    value = world * cs_step * K / (ms_total / 1e3)
    pk = peaks()

    phases = {}
    for name, f in figs.items():
        m = statistics.mean(phase_ms[name])
        if f["bound"] == "hbm":
            ach = f["bytes"] / (m / 1e3) / 1e9
            peak, unit = pk["hbm_gbs"], "GB/s"
        else:
            ach = f["flops"] / (m / 1e3) / 1e12
            peak, unit = pk["bf16_tflops_sustained"], "TFLOP/s"
        phases[name] = {"ms": round(m, 4), "chunk_scores_per_s": f["chunk_scores"] / (m / 1e3),
                        "queries_per_s": (f["queries"] / (m / 1e3)) if f["queries"] else None,
                        "bound": f["bound"], "achieved": round(ach, 2), "peak": peak, "unit": unit,
                        "frac": round(ach / peak, 4), "algorithmic_bytes": f["bytes"], "flops": f["flops"]}
    read_gbs = read_peak_gbs(torch, dev)
    for name in ("memindex", "page_recall"):
        phases[name]["frac_of_read_peak"] = round(phases[name]["achieved"] / read_gbs, 4)
    for f in phases.values():
        if f["unit"] == "GB/s":
            f["frac_of_nominal"] = round(f["achieved"] / HBM_NOMINAL_GBS, 4)
    dom = max(phases, key=lambda n: phases[n]["ms"])
    d = phases[dom]
    for name in phases:
        phases[name]["traffic_bytes_est"] = profiled_traffic(name)
    # the dominant kernel (prefill_score_kernel, ~65% of the step's device time
    # per the ncu launch list) timed alone: timed alone, it is held to the
    # measured burst peak
    k_ms = time_prefill_scores(fm, torch, W, ws)
    k_flops = figs["prefill_topk"]["flops"]
    k_ach = k_flops / (k_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(k_ach, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(k_ach / pk["bf16_tflops"], 4), "traffic": kernel_traffic("prefill_scores"),
                "kernel": "prefill_score_kernel", "ms_per_launch": round(k_ms, 4), "flops_per_launch": k_flops,
                "peak_source": pk["source"] + " burst (kernel timed alone)",
                "frac_of_sustained": round(k_ach / pk["bf16_tflops_sustained"], 4),
                "scope": ("fm_index_prefill_scores on the step's prefill input (4096 tokens x 65536 chunks): one "
                          "launch of prefill_score_kernel (and an empty causal fill) per call, CUDA events over 10 "
                          "calls on the bench stream after the timed step region; the prefill call's own launch "
                          "also writes the segment entries for its top-k (within 0.2% of this time in the ncu "
                          "launch list)"),
                "dominant_phase": {"phase": dom, "frac": d["frac"], "ms": d["ms"]},
                # the tensor pipe's own busy fraction (ncu, --set full on the 512-token case), beside frac:
                # the burst peak above was measured by cuBLAS at a median 1470 MHz under load, while this
                # kernel runs at the clocks in "clocks" (2070 MHz max), so frac flatters it
                "tensor_pipe_active_pct": profile_metric(
                    "prefill_score_kernel_prefill_t512_s65536.md", ["prefill.cu", "fm_common.cuh"],
                    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed"),
                "peak_clock_mhz": json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get(
                    "clocks_under_load", {}).get("sm_mhz_median") if pk["source"] == "measured" else None}

    # ---- end to end through the same calls, inputs in pinned host memory ----
    # Every step copies its inputs from pinned host memory and reads its
    # results back; the copies of step i+1 run on a second stream into a
    # second set of input buffers while step i computes (the copy of a buffer
    # set waits until the step that last read it has finished).
    host_in = {k: W[k].to("cpu").pin_memory() for k in INPUT_KEYS}
    host_out = {k: torch.empty(W[k].shape, dtype=W[k].dtype).pin_memory() for k in OUTPUT_KEYS}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    e2e_steps = max(2, min(K, 4))
    sets = [W, dict(W, **{k: torch.empty_like(W[k]) for k in INPUT_KEYS})]
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    released = [None, None]

    def issue_copy(b):
        with torch.cuda.stream(copy_stream):
            if released[b] is not None:
                copy_stream.wait_event(released[b])
            for k in INPUT_KEYS:
                sets[b][k].copy_(host_in[k], non_blocking=True)
            copied[b].record(copy_stream)

    def e2e_run(n, start_event=None):
        if start_event is not None:
            copy_stream.wait_event(start_event)
        issue_copy(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                issue_copy(b ^ 1)
            stream.wait_event(copied[b])
            make_step(fm, sets[b], cfgs, ws)()
            ev = torch.cuda.Event()
            ev.record(stream)
            released[b] = ev
            for k in OUTPUT_KEYS:
                host_out[k].copy_(sets[b][k], non_blocking=True)

    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = reduce_max(e2e_ms, dev, world)
    e2e_value = world * cs_step / (e2e_ms / 1e3)

    # ---- variant rows, each timed alone on its own inputs after the step ----
    variants = None
    if not args.no_variants:
        del sets, host_in, host_out
        variants = {}
        for name, cls, reps in (("tiny", TinyConfig, 50), ("memindex_256k", MemIndex256K, 10),
                                ("paged_512k", Paged512K, 10), ("paged_bf16_1m", PagedBf16, 10)):
            v = cls(torch, dev, fm)
            variants[name] = v.measure(reps, 3, pk)
            del v
        v = Fp8MemIndex(torch, dev, fm)
        variants["memindex_fp8"] = v.measure(10, 3, pk)
        del v
        v = FullHistoryPaged(torch, dev, fm)
        variants["paged_full_history"] = v.measure(10, 3, pk)
        del v
        for mode, name in ((0, "retriever_max"), (1, "retriever_mean")):
            v = RetrieverMemIndex(torch, dev, fm, mode=mode)
            variants[name] = v.measure(10, 3, pk)
            del v
        v = QueryChain(torch, dev, fm)
        variants["query_chain"] = v.measure(20, 3, pk)
        del v
        for hot in (0.05, 0.25):  # the 1M workload's other hot fractions (the step runs 12%)
            variants[f"memindex_hot{int(round(hot * 100))}"] = memindex_hot_variant(torch, dev, fm, W, mi, hot, pk)
        for name in ("memindex_256k", "memindex_fp8", "retriever_max", "retriever_mean", "memindex_hot5",
                     "memindex_hot25"):
            variants[name]["frac_of_read_peak"] = round(variants[name]["achieved"] / read_gbs, 4)
        for f in variants.values():
            if f.get("unit") == "GB/s":
                f["frac_of_nominal"] = round(f["achieved"] / HBM_NOMINAL_GBS, 4)
        if fm.fm_device_status(reset=True) != 0:
            raise RuntimeError("device status flagged an error in the variant rows")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(cfgs)
        v, qv, dt, reps = smp.rate(min_seconds=args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": smp.orc.num_threads(), "kind": "oracle",
               "sample": f"{reps} x [{smp.desc}]", "seconds": round(dt, 2), "queries_per_s": qv}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
                "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16/e4m3 in, fp32 accumulate", "data": "synthetic",
                "config": {"workload": WORKLOAD, "global_batch": world * (mi.B + pg.Q + pf.T),
                           "seq_len": 4 * mi.S, "kmax": KMAX, "parallelism": f"replicas x{world} (request sharding)",
                           "l2": "inputs larger than L2 (8.1 GB of keys streamed per step); no flush"},
                "queries_per_s": world * q_step * K / (ms_total / 1e3),
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": e2e_ms},
                "gpu_launches": KERNELS_PER_STEP * K,
                "roofline": roofline, "phases": phases, "variants": variants, "clocks": clk, "cpu_baseline": cpu,
                "read_peak": {"value": round(read_gbs, 1), "unit": "GB/s",
                              "how": "torch sum over 4 GiB fp32, best of 10 (read-only); the HBM fractions above "
                                     "use the measured copy peak, frac_of_read_peak this one"},
                "device_status": status, "sanity": chk}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def time_call(torch, call, reps, warmup):
    """Mean device time of one call (ms): CUDA events around each of `reps`
    calls on the current stream, after `warmup` untimed calls."""
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


class TinyConfig:
    """The tiny workload (1 query, 1 indexer layer, S = 4096 chunks, 12%
    planted): the Memory Indexer's mask and logits, then the top-512 over all
    4096 chunks (fm_topk_select on the logits).  1 MB of keys: launch-bound,
    and L2-resident after the first call, so its fraction of the HBM roofline
    is not a bandwidth claim."""

    def __init__(self, torch, dev, fm):
        import gen
        self.torch, self.fm, self.cfg = torch, fm, gen.TINY
        c = self.cfg
        q, w, hot = gen.memindex_qw(c)
        K = gen.memindex_keys_host(c, hot)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.q, self.w, self.K = t(q.view(np.int16)), t(w), t(K.view(np.int16))
        self.mask = torch.empty((1, c.S // 32), dtype=torch.int32, device=dev)
        self.logits = torch.empty((1, 1, c.S), dtype=torch.float32, device=dev)
        self.idx = torch.empty((1, 512), dtype=torch.int32, device=dev)
        self.sc = torch.empty((1, 512), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()

    def call(self):
        self.fm.fm_memindex_score_mask(self.q, self.w, self.K, self.mask, None, self.logits)
        self.fm.fm_topk_select(self.logits[0], 512, self.idx, self.sc)

    def measure(self, reps, warmup, pk):
        c = self.cfg
        ms = time_call(self.torch, self.call, reps, warmup)
        nbytes = c.S * c.d * 2 + c.S * 4 * 2 + (c.S // 32) * 4 + 512 * 8
        ach = nbytes / (ms / 1e3) / 1e9
        return {"ms": round(ms, 5), "chunk_scores_per_s": c.S / (ms / 1e3), "queries_per_s": 1 / (ms / 1e3),
                "bound": "launch", "achieved": round(ach, 2), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 5), "algorithmic_bytes": nbytes, "launches": 2, "reps": reps,
                "workload": "tiny: 1 query x 1 layer x 4096 chunks bf16 (12% planted): mask + logits, then top-512"}


class MemIndex256K:
    """The Memory Indexer at 256K-token context: 76 requests x 3 layers x
    65536 chunks, bf16 keys, 12% planted (3.8 GB per call, far above L2),
    OR-union mask and max-sigmoid."""

    def __init__(self, torch, dev, fm):
        import gen
        self.torch, self.fm, self.cfg = torch, fm, gen.MEMINDEX_256K
        c = self.cfg
        q, w, hot = gen.memindex_qw(c)
        self.q = torch.from_numpy(q.view(np.int16)).to(dev)
        self.w = torch.from_numpy(w).to(dev)
        hot_d = torch.from_numpy(hot).to(dev)
        self.K = torch.empty((c.B, c.L, c.S, c.d), dtype=torch.int16, device=dev)
        gen.memindex_keys_device(c, hot_d.data_ptr(), self.K.data_ptr(), c.L * c.S * c.d, c.S * c.d)
        self.mask = torch.empty((c.B, (c.S + 31) // 32), dtype=torch.int32, device=dev)
        self.maxsig = torch.empty((c.B, c.S), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()

    def call(self):
        self.fm.fm_memindex_score_mask(self.q, self.w, self.K, self.mask, self.maxsig)

    def measure(self, reps, warmup, pk):
        c = self.cfg
        ms = time_call(self.torch, self.call, reps, warmup)
        nbytes = c.B * c.L * c.S * c.d * 2 + c.B * c.S * 4 + c.B * ((c.S + 31) // 32) * 4
        ach = nbytes / (ms / 1e3) / 1e9
        return {"ms": round(ms, 4), "chunk_scores_per_s": c.chunk_scores / (ms / 1e3), "bound": "hbm",
                "achieved": round(ach, 2), "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
                "algorithmic_bytes": nbytes, "launches": 1, "reps": reps,
                "resident_fraction": round(resident_fraction(self.torch, self.mask, c.B, c.S), 4),
                "workload": f"memindex 256K: {c.B}x{c.L}x{c.S} bf16 (12% planted), mask + max-sigmoid"}


class Paged512K:
    """The native paged top-512 at 512K-token context: 60 requests x 21 CSA
    layers = 1260 queries, 192 resident E4M3 pages each (2.0 GB of keys and
    scales per call)."""

    def __init__(self, torch, dev, fm):
        import gen
        self.torch, self.fm, self.cfg = torch, fm, gen.PAGED_512K
        c = self.cfg
        logical, phys, owner = gen.paged_tables(c)
        q, w = gen.paged_qw(c)
        self.q = torch.from_numpy(q.view(np.int16)).to(dev)
        self.w = torch.from_numpy(w).to(dev)
        own_d = torch.from_numpy(owner).to(dev)
        self.k8 = torch.empty((c.P, c.page, c.d), dtype=torch.uint8, device=dev)
        self.sc = torch.empty((c.P, c.page), dtype=torch.float32, device=dev)
        gen.paged_pool_device(c, own_d.data_ptr(), self.k8.data_ptr(), self.sc.data_ptr())
        del own_d
        self.phys = torch.from_numpy(phys).to(dev)
        self.logical = torch.from_numpy(logical).to(dev)
        self.idx = torch.empty((c.Q, c.k), dtype=torch.int32, device=dev)
        self.score = torch.empty((c.Q, c.k), dtype=torch.float32, device=dev)
        self.ws = torch.empty(fm.fm_native_topk_paged_workspace(c.Q, c.R), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def call(self):
        self.fm.fm_native_topk_paged(self.q, self.w, self.k8, self.sc, self.phys, self.logical, self.cfg.k,
                                     self.idx, self.score, workspace=self.ws)

    def measure(self, reps, warmup, pk):
        c = self.cfg
        ms = time_call(self.torch, self.call, reps, warmup)
        nbytes = c.P * c.page * (c.d + 4) + c.Q * c.R * 8 + c.Q * c.k * 8
        ach = nbytes / (ms / 1e3) / 1e9
        return {"ms": round(ms, 4), "chunk_scores_per_s": c.chunk_scores / (ms / 1e3),
                "queries_per_s": c.Q / (ms / 1e3), "bound": "hbm", "achieved": round(ach, 2), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "algorithmic_bytes": nbytes, "launches": 3,
                "reps": reps, "workload": f"paged top-{c.k} 512K: {c.Q} queries x {c.R} pages, E4M3 + fp32 scale"}


class PagedBf16:
    """The native paged top-512 over a pool of bf16 keys (key_dtype
    FM_DTYPE_BF16, no scale) at the 1M decode workload's sizes: 630 queries x
    384 resident pages, 4.0 GB of keys per call (twice the E4M3 pool's
    bytes)."""

    def __init__(self, torch, dev, fm):
        import gen
        self.torch, self.fm, self.cfg = torch, fm, gen.PAGED_1M
        c = self.cfg
        logical, phys, owner = gen.paged_tables(c)
        q, w = gen.paged_qw(c)
        self.q = torch.from_numpy(q.view(np.int16)).to(dev)
        self.w = torch.from_numpy(w).to(dev)
        own_d = torch.from_numpy(owner).to(dev)
        self.kbf = torch.empty((c.P, c.page, c.d), dtype=torch.int16, device=dev)
        gen.paged_pool_bf16_device(c, own_d.data_ptr(), self.kbf.data_ptr())
        del own_d
        self.phys = torch.from_numpy(phys).to(dev)
        self.logical = torch.from_numpy(logical).to(dev)
        self.idx = torch.empty((c.Q, c.k), dtype=torch.int32, device=dev)
        self.score = torch.empty((c.Q, c.k), dtype=torch.float32, device=dev)
        self.ws = torch.empty(fm.fm_native_topk_paged_workspace(c.Q, c.R), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def call(self):
        self.fm.fm_native_topk_paged(self.q, self.w, self.kbf, None, self.phys, self.logical, self.cfg.k, self.idx,
                                     self.score, workspace=self.ws)

    def measure(self, reps, warmup, pk):
        c = self.cfg
        ms = time_call(self.torch, self.call, reps, warmup)
        nbytes = c.P * c.page * c.d * 2 + c.Q * c.R * 8 + c.Q * c.k * 8
        ach = nbytes / (ms / 1e3) / 1e9
        return {"ms": round(ms, 4), "chunk_scores_per_s": c.chunk_scores / (ms / 1e3),
                "queries_per_s": c.Q / (ms / 1e3), "bound": "hbm", "achieved": round(ach, 2), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "algorithmic_bytes": nbytes, "launches": 3,
                "reps": reps, "workload": f"paged top-{c.k} over bf16 keys: {c.Q} queries x {c.R} pages"}


class Fp8MemIndex:
    """The Memory Indexer over compressed keys (fm_memindex_score_mask_fp8):
    the bench step's 30 requests x 3 layers x 262144 chunks with E4M3 codes
    and one fp32 scale per chunk (3.1 GB streamed per call, far above L2).
    Timed on its own after the step, not part of the step's value."""

    def __init__(self, torch, dev, fm, small=False):
        import gen
        self.torch, self.fm = torch, fm
        mi = gen.replace(gen.MEMINDEX_1M, B=4) if small else gen.MEMINDEX_1M
        self.cfg = mi
        q, w, hot = gen.memindex_qw(mi)
        self.q = torch.from_numpy(q.view(np.int16)).to(dev)
        self.w = torch.from_numpy(w).to(dev)
        hot_d = torch.from_numpy(hot).to(dev)
        own_d = torch.from_numpy(gen.memindex_fp8_owner(mi)).to(dev)
        self.k8 = torch.empty((mi.B, mi.L, mi.S, mi.d), dtype=torch.uint8, device=dev)
        self.sc = torch.empty((mi.B, mi.L, mi.S), dtype=torch.float32, device=dev)
        gen.memindex_fp8_keys_device(mi, hot_d.data_ptr(), own_d.data_ptr(), self.k8.data_ptr(), self.sc.data_ptr())
        self.mask = torch.empty((mi.B, (mi.S + 31) // 32), dtype=torch.int32, device=dev)
        self.maxsig = torch.empty((mi.B, mi.S), dtype=torch.float32, device=dev)
        self.ws = torch.empty(fm.fm_memindex_fp8_workspace(mi.B, mi.L), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def call(self):
        self.fm.fm_memindex_score_mask_fp8(self.q, self.w, self.k8, self.sc, self.mask, self.maxsig,
                                           workspace=self.ws)

    def bytes(self):
        mi = self.cfg
        return (mi.B * mi.L * mi.S * (mi.d + 4) + mi.B * mi.S * 4 + mi.B * ((mi.S + 31) // 32) * 4
                + mi.B * mi.L * mi.n_h * (mi.d * 2 + 4))

    def measure(self, reps, warmup, pk):
        torch = self.torch
        for _ in range(warmup):
            self.call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record()
            self.call()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        ach = self.bytes() / (ms / 1e3) / 1e9
        mi = self.cfg
        return {"ms": round(ms, 4), "chunk_scores_per_s": mi.chunk_scores / (ms / 1e3), "bound": "hbm",
                "achieved": round(ach, 2), "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
                "algorithmic_bytes": self.bytes(), "traffic_bytes_est": profiled_traffic("memindex_fp8"),
                "launches": 2, "reps": reps,
                "workload": f"memindex fp8 keys {mi.B}x{mi.L}x{mi.S}, E4M3 + per-chunk fp32 scale"}


class RetrieverMemIndex:
    """The trained retriever's Memory Indexer (fm_retriever_score_mask): the
    1M workload's 30 requests x 3 layers x 262144 chunks, 128 heads, keys in
    packed 132-byte compressed_k rows (3.1 GB per call), max or mean layer
    ensemble.  Timed on its own after the step."""

    def __init__(self, torch, dev, fm, small=False, mode=0):
        import gen
        self.torch, self.fm, self.mode = torch, fm, mode
        cfg = gen.replace(gen.RETRIEVER_1M, B=4) if small else gen.RETRIEVER_1M
        self.cfg = cfg
        q, w, hot = gen.memindex_qw(cfg)
        self.q = torch.from_numpy(q.view(np.int16)).to(dev)
        self.w = torch.from_numpy(w).to(dev)
        hot_d = torch.from_numpy(hot).to(dev)
        own_d = torch.from_numpy(gen.memindex_fp8_owner(cfg)).to(dev)
        k8 = torch.empty((cfg.B, cfg.L, cfg.S, cfg.d), dtype=torch.uint8, device=dev)
        sc = torch.empty((cfg.B, cfg.L, cfg.S), dtype=torch.float32, device=dev)
        gen.memindex_fp8_keys_device(cfg, hot_d.data_ptr(), own_d.data_ptr(), k8.data_ptr(), sc.data_ptr())
        self.ck = torch.cat([k8, sc.view(torch.uint8).view(cfg.B, cfg.L, cfg.S, 4)], dim=-1)
        del k8, sc
        self.mask = torch.empty((cfg.B, (cfg.S + 31) // 32), dtype=torch.int32, device=dev)
        self.ens = torch.empty((cfg.B, cfg.S), dtype=torch.float32, device=dev)
        self.ws = torch.empty(fm.fm_retriever_workspace(cfg.B, cfg.L, cfg.n_h), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def call(self):
        self.fm.fm_retriever_score_mask(self.q, self.w, self.ck, self.mask, self.ens, ensemble=self.mode,
                                        workspace=self.ws)

    def bytes(self):
        c = self.cfg
        return (c.B * c.L * c.S * (c.d + 4) + c.B * c.S * 4 + c.B * ((c.S + 31) // 32) * 4
                + c.B * c.L * c.n_h * (c.d * 2 + 4))

    def measure(self, reps, warmup, pk):
        torch = self.torch
        for _ in range(warmup):
            self.call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record()
            self.call()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        ach = self.bytes() / (ms / 1e3) / 1e9
        c = self.cfg
        return {"ms": round(ms, 4), "chunk_scores_per_s": c.chunk_scores / (ms / 1e3), "bound": "hbm",
                "achieved": round(ach, 2), "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
                "algorithmic_bytes": self.bytes(), "traffic_bytes_est": profiled_traffic("retriever"),
                "launches": 2, "reps": reps,
                "workload": (f"retriever {c.B}x{c.L}x{c.S}, {c.n_h} heads, packed 132-byte compressed_k rows, "
                             f"{'max' if self.mode == 0 else 'mean'} ensemble")}


class FullHistoryPaged:
    """Full-history native top-512 (fm_native_topk_paged with every page
    listed): 30 requests x 21 layers = 630 queries, each scoring all 4096
    pages (262144 chunks) of its 1M-token history -- the path without
    residency that the Memory Indexer's page recall replaces.  21.8 GB of
    E4M3 keys and scales per call.  Timed on its own after the step."""

    def __init__(self, torch, dev, fm, small=False):
        import gen
        self.torch, self.fm = torch, fm
        cfg = gen.replace(gen.PAGED_FULL_1M, requests=2) if small else gen.PAGED_FULL_1M
        self.cfg = cfg
        logical, phys, owner = gen.paged_tables(cfg)
        q, w = gen.paged_qw(cfg)
        self.q = torch.from_numpy(q.view(np.int16)).to(dev)
        self.w = torch.from_numpy(w).to(dev)
        own_d = torch.from_numpy(owner).to(dev)
        self.k8 = torch.empty((cfg.P, cfg.page, cfg.d), dtype=torch.uint8, device=dev)
        self.sc = torch.empty((cfg.P, cfg.page), dtype=torch.float32, device=dev)
        gen.paged_pool_device(cfg, own_d.data_ptr(), self.k8.data_ptr(), self.sc.data_ptr())
        del own_d
        self.phys = torch.from_numpy(phys).to(dev)
        self.logical = torch.from_numpy(logical).to(dev)
        self.idx = torch.empty((cfg.Q, cfg.k), dtype=torch.int32, device=dev)
        self.score = torch.empty((cfg.Q, cfg.k), dtype=torch.float32, device=dev)
        self.ws = torch.empty(fm.fm_native_topk_paged_workspace(cfg.Q, cfg.R), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def call(self):
        self.fm.fm_native_topk_paged(self.q, self.w, self.k8, self.sc, self.phys, self.logical, self.cfg.k,
                                     self.idx, self.score, workspace=self.ws)

    def bytes(self):
        c = self.cfg
        return c.P * c.page * (c.d + 4) + c.Q * c.R * 8 + c.Q * c.k * 8

    def measure(self, reps, warmup, pk):
        torch = self.torch
        for _ in range(warmup):
            self.call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record()
            self.call()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        ach = self.bytes() / (ms / 1e3) / 1e9
        c = self.cfg
        return {"ms": round(ms, 4), "chunk_scores_per_s": c.chunk_scores / (ms / 1e3),
                "queries_per_s": c.Q / (ms / 1e3), "bound": "hbm", "achieved": round(ach, 2), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "algorithmic_bytes": self.bytes(),
                "launches": 3, "reps": reps,
                "workload": f"full-history paged top-{c.k}: {c.Q} queries x {c.R} pages (all of a 1M-token history), E4M3"}


class QueryChain:
    """The query side of the retriever's three indexer layers (fm_query_chain:
    wq_a -> RMSNorm -> wq_b -> YaRN rotary -> Walsh-Hadamard, plus the head
    weights) for one decode token of each of the 1M workload's 30 requests.
    Each layer has its own synthetic weights (dim 4096, rank 2048, 128 heads of
    128): 86 MB of bf16 weights per layer, 258 MB per call over the three
    layers, above the 129 MB L2.  Timed on its own after the step."""

    def __init__(self, torch, dev, fm, small=False, T=30, layers=3):
        import gen
        self.torch, self.fm = torch, fm
        self.T, self.layers, self.dim, self.r, self.n_h = T, layers, 4096, 2048, 128
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).to(dev)
        self.sets = []
        for l in range(layers):
            ins = gen.query_chain_inputs(T, dim=self.dim, r=self.r, n_h=self.n_h, seed=gen.BASE_SEED + 600 + l)
            self.sets.append([t(a) for a in ins])
        # one call for the three layers: q [T, L, n_h, 128], w [T, L, n_h] (the retriever's q / w layout);
        # the layers share the tokens' positions
        self.q = torch.empty((T, layers, self.n_h, 128), dtype=torch.int16, device=dev)
        self.w = torch.empty((T, layers, self.n_h), dtype=torch.float32, device=dev)
        self.ws = torch.empty(fm.fm_query_chain_layers_workspace(layers, T, self.r, self.n_h), dtype=torch.uint8,
                              device=dev)
        torch.cuda.synchronize()

    def call(self):
        S = self.sets
        self.fm.fm_query_chain_layers([x[0] for x in S], [x[1] for x in S], [x[2] for x in S], [x[3] for x in S],
                                      [x[4] for x in S], S[0][5], self.q, self.w, workspace=self.ws)

    def bytes(self):
        T, dim, r, n_h = self.T, self.dim, self.r, self.n_h
        weights = (r * dim + r + n_h * 128 * r + n_h * dim) * 2
        io = T * dim * 2 + T * 8 + T * n_h * 128 * 2 + T * n_h * 4
        return self.layers * (weights + io)

    def measure(self, reps, warmup, pk):
        torch = self.torch
        for _ in range(warmup):
            self.call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record()
            self.call()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        ach = self.bytes() / (ms / 1e3) / 1e9
        return {"ms": round(ms, 4), "tokens_per_s": self.T * self.layers / (ms / 1e3), "bound": "hbm",
                "achieved": round(ach, 2), "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
                "algorithmic_bytes": self.bytes(), "traffic_bytes_est": profiled_traffic("query_chain"),
                "launches": "one fm_query_chain_layers call: 2 projection GEMMs + RMSNorm + rotary/Hadamard for all layers",
                "reps": reps,
                "workload": (f"query chain: {self.T} decode tokens x {self.layers} indexer layers, dim {self.dim}, "
                             f"rank {self.r}, {self.n_h} heads x 128 (bf16 weights, fp32 accumulate)")}


def run_profile_case(args, fm, torch, W, cfgs, ws):
    """--only / --small: run a reduced or single-phase case for ncu captures
    (prints the timing as one JSON line marked as a profiling case)."""
    step = make_step(fm, W, cfgs, ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": True, "only": args.only, "small": args.small,
                      "ms_per_step": e0.elapsed_time(e1) / max(1, args.steps),
                      "device_status": fm.fm_device_status(reset=True)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true", help="skip the variant rows timed after the step")
    ap.add_argument("--only", choices=["memindex", "paged", "prefill", "memindex_fp8", "paged_full", "retriever",
                                       "query_chain", "prefill_scores", "recall"], default=None,
                    help="profiling case: run one phase only")
    ap.add_argument("--small", action="store_true", help="profiling case: reduced sizes for ncu captures")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
