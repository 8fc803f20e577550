"""Benchmark: one decode step of the block-sparse paged-KV path on a GB300.

A step runs, for every (request, kv head) unit of the Llama-3-8B-layer workload
(batch 32, 32 q / 8 kv heads, context 32768, page 64, k = 64 with k_q = k_e = 32, 1% of key
rows scaled x20), all rows of the hot path through the C ABI:

  paged_kv_append -> score_blocks -> select_topk -> resident_setdiff -> lru_bucket_update
  -> sparse_decode_attn

(the three bookkeeping operations through select_resident_update, their one-kernel fused form).

``value`` is the step's algorithmic KV-cache bytes (pooled-key summaries scored + K/V pages
attended + bookkeeping tables) divided by the device time of the step; ``queries_per_s`` is
requests / step time.  ``roofline`` reports the dominant kernel (sparse_decode_attn) against
the measured HBM copy bandwidth.  ``e2e`` repeats the step through the public API with the
step's inputs copied from pinned host memory and its outputs read back inside the timed region.
``cpu_baseline`` times the fp64 oracle on the host cores.  ``--impl reference`` times only the
oracle (the reference arm of this comparison).
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

METRIC = "sparse decode-attn KV GB/s (% of GB300 HBM peak) and queries/s per GPU"
UNIT = "GB/s"
L2_FLUSH_BYTES = 256 << 20
PAGE_BYTES = 2 * 64 * 128 * 2          # K + V of one page of one head
SUMMARY_BYTES = 4 * 128 * 4            # fp32 pooled-key sums of one page of one head
N_SLOTS = 2048                         # resident pages per (request, kv head)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-lazy", action="store_true")
    ap.add_argument("--no-rag", action="store_true", help="skip the lazy-RoPE RAG sub-measurement")
    ap.add_argument("--no-prefill", action="store_true", help="skip the LazyAttention prefill sub-measurement")
    ap.add_argument("--no-bf16-summaries", action="store_true",
                    help="skip the step with bf16 pooled-key summaries")
    ap.add_argument("--no-colscore", action="store_true",
                    help="skip the PyramidKV-style column-score sub-measurement")
    ap.add_argument("--col-batch", type=int, default=16,
                    help="prompts of the column-score workload (5000 tokens, last 256 rows each)")
    ap.add_argument("--rag-batch", type=int, default=64,
                    help="requests of the lazy-RoPE RAG workload (64 = the workload; smaller for profiling)")
    ap.add_argument("--rag-docs", type=int, default=256,
                    help="cached documents of the RAG workload (256 = the workload; smaller for profiling)")
    ap.add_argument("--no-offload", action="store_true",
                    help="skip the offload sub-measurement (262k context, pool in pinned host memory)")
    ap.add_argument("--l2", default="none", choices=["none", "write"],
                    help="none: no flush, every step reads ~0.8 GB (> 129 MB L2); write: 256 MiB write "
                         "between timed steps")
    ap.add_argument("--bookkeeping", default="overlap", choices=["fused", "overlap"],
                    help="fused: selection + set-difference + LRU in one kernel before attention; "
                         "overlap: selection, then set-difference + LRU on a second stream beside attention")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the tiny and NOSA-trajectory workloads of the per-config report")
    ap.add_argument("--batch", type=int, default=32,
                    help="requests per step (32 = the Llama-3-8B-layer workload; smaller for profiling)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor throughput (TFLOP/s, burst) measured on this machine, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def rank_max(v: float, device) -> float:
    """Max of v over the ranks of the default process group (v itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, bytes_per_rank_step: float, ms_max: float) -> float:
    """Whole-job GB/s of `world` independent replicas, each moving bytes_per_rank_step per step,
    when the slowest rank takes ms_max per step (weak scaling: per-rank work is fixed)."""
    return world * bytes_per_rank_step / (ms_max * 1e-3) / 1e9


def measured_traffic():
    """DRAM bytes per full attention launch from the committed ncu summary, or None when the
    kernel source has changed since those counters were taken."""
    import hashlib
    import re
    prof = os.path.join(ROOT, "profiles", "attn_split_kernel_llama8b_B8_full.md")
    src = os.path.join(ROOT, "sparse_paged_kv_score_gb300", "csrc", "attn.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    m = re.search(r"bench-traffic: attn.cu=([0-9a-f]+) traffic_bytes_per_launch=(\d+)", open(prof).read())
    if not m or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != m.group(1):
        return None
    return int(m.group(2))


def step_bytes(w, k):
    """Algorithmic bytes of one step (one read of every operand, one write of every result)."""
    B, Hk, Hq, npm = w["B"], w["Hk"], w["Hq"], w["np_max"]
    U = B * Hk
    local = int((w["seq_len"][0] - 1) // 64)
    stride = k + 1
    b = {}
    b["append"] = U * 2 * 128 * 2 + U * 16 * 128 * 2 + U * SUMMARY_BYTES // 4
    b["score"] = U * local * SUMMARY_BYTES + B * npm * 4 + B * Hq * 128 * 2 + U * npm * 4
    b["select"] = U * npm * 4 * 2 + U * ((npm + 31) // 32) * 4 * 2 + U * stride * 4 + U * 4
    b["setdiff"] = U * N_SLOTS * 4 + U * stride * 4 * 4
    b["lru"] = U * N_SLOTS * 4 * 2 * 2 + U * stride * 4 * 3 + U * 64 * 4
    b["attn_kv"] = U * stride * PAGE_BYTES
    b["attn"] = b["attn_kv"] + B * Hq * 128 * (2 + 4) + B * Hq * 4 + U * stride * 4
    return b


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        else:
            self.lines = []

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle legs

def oracle_step(w, units, n_slots=N_SLOTS, residency=True, reps=1):
    """Times the fp64 oracle on one decode step of the listed units: block scores, dual top-k
    selection, sparse attention and (residency) the set-difference and LRU update against fresh
    resident tables of n_slots slots.  Returns (seconds per step, threads)."""
    import oracle
    nthreads = os.cpu_count() or 1
    k_q, k_e = w["k_q"], w["k_e"]
    alive = np.ones((w["B"], w["Hk"], w["np_max"]), np.uint8)
    stride = k_q + k_e + 1
    t0 = time.perf_counter()
    for _ in range(reps):
        s = oracle.score_batch(w["q"], w["k_pool"], w["page_table"], w["seq_len"], units=units,
                               nthreads=nthreads)
        sel, n_sel, _ = oracle.select_batch(s, w["evict"], alive, w["seq_len"], k_q, k_e, units=units,
                                            nthreads=nthreads)
        oracle.sparse_attn_batch(w["q"], w["k_pool"], w["v_pool"], w["page_table"], sel, n_sel,
                                 w["seq_len"], units=units, nthreads=nthreads)
        if residency:
            U = len(units)
            sel_u = sel.reshape(-1, stride)[units]
            n_u = n_sel.reshape(-1)[units]
            resident = np.full((U, n_slots), -1, np.int32)
            ts = np.full((U, n_slots), np.iinfo(np.int32).min, np.int32)
            miss, nm, slot = oracle.setdiff_batch(resident, sel_u, n_u, nthreads=nthreads)
            oracle.lru_batch(resident, ts, slot, n_u, miss, nm, 0, 1, nthreads=nthreads)
    return (time.perf_counter() - t0) / reps, nthreads


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import gen
    w = gen.llama8b(seed=0)
    units = np.arange(w["B"] * w["Hk"], dtype=np.int32)
    times = []
    thr = 1
    for i in range(args.warmup + args.steps):
        dt, thr = oracle_step(w, units)
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    b = step_bytes(w, w["k_q"] + w["k_e"])
    byts = sum(v for kk, v in b.items() if kk != "attn_kv")
    value = byts / (ms * 1e-3) / 1e9
    sample = ("the whole step, all 256 (request, kv head) units: block scores, dual top-k selection, sparse "
              "attention, set-difference and LRU update (2048 slots), fp64")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w["name"], "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU step

def _dev_helpers(dev):
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)

    return bf, i32


def _parts(b, names):
    return int(sum(b[n] for n in names))


def _cpu_line(dt, byts, thr, sample, reps=1):
    return {"value": byts / dt / 1e9, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample,
            "ms_per_step": dt * 1e3}


def _oracle_timed(fn, min_s=0.5):
    """Seconds per call of fn() (the fp64 oracle), repeated until min_s of work has run."""
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    reps = max(0, int(min_s / max(dt, 1e-6)) - 1)
    if reps:
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        dt = (time.perf_counter() - t0) / reps
    return dt


def tiny_leg(args, dev, timed, cap, peak, cpu_baseline):
    """The tiny sparse-decode workload (batch 1, 8 q / 2 kv heads, context 4096, k = 16): one step
    is the new token's append with the block scores (one launch), the dual top-k selection and
    the sparse attention, each step one CUDA graph."""
    import torch
    import gen
    import sparse_paged_kv_score_gb300 as spkv
    bf, i32 = _dev_helpers(dev)
    w = gen.tiny(seed=0)
    B, Hq, Hk, npm = w["B"], w["Hq"], w["Hk"], w["np_max"]
    k_q, k_e = w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    U = B * Hk
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.float32, device=dev)
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, i32(gen.page_counts(w)), max_units=U)
    pt, seq = i32(w["page_table"]), i32(w["seq_len"])
    n_iter = args.warmup + args.steps
    qs = [bf(gen.rows_bf16(0, 7000 + i, B * Hq).reshape(B, Hq, 128)) for i in range(n_iter)]
    evs = [torch.from_numpy(w["evict"]).to(dev) for _ in range(n_iter)]
    kn = [bf(gen.rows_bf16(0, 9000 + i, U).reshape(B, Hk, 128)) for i in range(n_iter)]
    vn = [bf(gen.rows_bf16(0, 9500 + i, U).reshape(B, Hk, 128)) for i in range(n_iter)]
    scores = torch.empty(B, Hk, npm, dtype=torch.float32, device=dev)
    alive = torch.full((B, Hk, (npm + 31) // 32), -1, dtype=torch.int32, device=dev)
    sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=dev)
    n_sel = torch.empty(B, Hk, dtype=torch.int32, device=dev)
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)

    def step(i):
        spkv.decode_append_score(cache, kn[i], vn[i], qs[i], pt, seq, scores)
        spkv.select_topk(cache, scores, evs[i], alive, seq, k_q, k_e, sel, n_sel)
        spkv.sparse_decode_attn(cache, qs[i], pt, sel, n_sel, seq, out, lse)

    for i in range(args.warmup):
        step(i)
    idx = list(range(args.warmup, n_iter))
    graphs = {}
    for i in idx:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(i)
        graphs[i] = g
    torch.cuda.synchronize()
    ms = statistics.median(timed(lambda i: graphs[i].replay(), idx))
    st, bits = spkv.get_device_error(cache)
    if st != 0:
        raise RuntimeError(f"device error bits {bits} in the tiny leg")
    cache.close()
    byts = _parts(step_bytes(w, k_q + k_e), ("append", "score", "select", "attn"))
    gbs = byts / (ms * 1e-3) / 1e9
    res = {"workload": w["name"], "step": "append+score, select, sparse attention (3 launches + combine)",
           "us_per_step": ms * 1e3, "bytes_per_step": byts, "GBps": gbs, "pct_hbm_peak": 100 * gbs / peak,
           "queries_per_s": B / (ms * 1e-3), "launch": "one CUDA graph per step", "stat": "median"}
    if cpu_baseline:
        units = np.arange(U, dtype=np.int32)
        thr = os.cpu_count() or 1
        dt = _oracle_timed(lambda: oracle_step(w, units, residency=False))
        res["cpu_baseline"] = _cpu_line(dt, byts, thr, "the whole step (both units), fp64")
    return res


def traj_leg(args, dev, timed, cap, peak, cpu_baseline):
    """The NOSA trajectory (batch 16, 32 q / 8 kv heads, context 65536 growing by one token per
    step, k = 64 with k_e = 48, k_q = 16): 64 consecutive decode steps, each the new token's append
    with the block scores, the dual top-k selection (eviction scores on a random walk) and the
    sparse attention, one CUDA graph per step.  The trajectory runs once untimed (warm-up), its
    state is reset, and runs again timed; the locality gamma(t) is read from the timed steps'
    selections afterwards."""
    import torch
    import gen
    import sparse_paged_kv_score_gb300 as spkv
    bf, i32 = _dev_helpers(dev)
    w = gen.nosa_traj(seed=0)
    B, Hq, Hk, npm, steps = w["B"], w["Hq"], w["Hk"], w["np_max"], w["steps"]
    k_q, k_e = w["k_q"], w["k_e"]
    k = k_q + k_e
    stride = k + 1
    U = B * Hk
    L0 = w["seq_len"].copy()
    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.float32, device=dev)
    cnt0 = i32(gen.page_counts(w))
    cnt = cnt0.clone()
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, cnt, max_units=U)
    pt = i32(w["page_table"])
    inps, e_walk = [], None
    for t in range(steps):
        inp = gen.traj_step_inputs(w, t, e_walk)
        e_walk = inp["evict"]
        inps.append(dict(q=bf(inp["q"]), ev=torch.from_numpy(e_walk.astype(np.float32)).to(dev),
                         kn=bf(inp["k_new"]), vn=bf(inp["v_new"]), seq=i32(L0 + t + 1)))
        if t == 0:
            inp0 = inp
    scores = torch.empty(B, Hk, npm, dtype=torch.float32, device=dev)
    alive = torch.full((B, Hk, (npm + 31) // 32), -1, dtype=torch.int32, device=dev)
    sels = [torch.empty(B, Hk, stride, dtype=torch.int32, device=dev) for _ in range(steps)]
    nsels = [torch.empty(B, Hk, dtype=torch.int32, device=dev) for _ in range(steps)]
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)

    def step(t):
        x = inps[t]
        spkv.decode_append_score(cache, x["kn"], x["vn"], x["q"], pt, x["seq"], scores)
        spkv.select_topk(cache, scores, x["ev"], alive, x["seq"], k_q, k_e, sels[t], nsels[t])
        spkv.sparse_decode_attn(cache, x["q"], pt, sels[t], nsels[t], x["seq"], out, lse)

    graphs = []
    for t in range(steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(t)
        graphs.append(g)
    torch.cuda.synchronize()
    for g in graphs:          # warm-up: the whole trajectory once
        g.replay()
    torch.cuda.synchronize()
    alive.fill_(-1)           # back to the initial state (the local page's summaries are never scored)
    cnt.copy_(cnt0)
    torch.cuda.synchronize()
    ms_all = timed(lambda t: graphs[t].replay(), range(steps))
    st, bits = spkv.get_device_error(cache)
    if st != 0:
        raise RuntimeError(f"device error bits {bits} in the trajectory leg")
    sel_h = [x.cpu().numpy() for x in sels]
    n_h = [x.cpu().numpy() for x in nsels]
    gammas = []
    for t in range(1, steps):
        local = (L0 + t) // 64
        for b in range(B):
            for h in range(Hk):
                prev = set(sel_h[t - 1][b, h, :n_h[t - 1][b, h]].tolist())
                cur = set(sel_h[t][b, h, :n_h[t][b, h]].tolist()) - {int(local[b])}
                gammas.append(len(cur & prev) / k)
    del graphs
    cache.close()
    wb = dict(w, seq_len=L0 + 1)
    byts = _parts(step_bytes(wb, k), ("append", "score", "select", "attn"))
    ms = statistics.mean(ms_all)
    gbs = byts / (ms * 1e-3) / 1e9
    res = {"workload": w["name"], "step": "append+score, select, sparse attention; 64 steps in a row",
           "ms_per_step": ms, "ms_per_step_median": statistics.median(ms_all), "bytes_per_step": byts,
           "GBps": gbs, "pct_hbm_peak": 100 * gbs / peak, "queries_per_s": B / (ms * 1e-3),
           "gamma_min": min(gammas), "gamma_mean": statistics.mean(gammas), "gamma_bound": k_e / k,
           "launch": "one CUDA graph per step"}
    if cpu_baseline:
        # the oracle on the trajectory's first step (its query, eviction scores and appended row)
        phys = w["page_table"][np.arange(B), L0 // 64]
        for b in range(B):
            w["k_pool"][:, phys[b], L0[b] % 64] = inp0["k_new"][b]
            w["v_pool"][:, phys[b], L0[b] % 64] = inp0["v_new"][b]
        w1 = dict(w, q=inp0["q"], evict=inp0["evict"], seq_len=L0 + 1)
        units = np.arange(U, dtype=np.int32)
        dt = _oracle_timed(lambda: oracle_step(w1, units, residency=False), min_s=0.0)
        res["cpu_baseline"] = _cpu_line(dt, byts, os.cpu_count() or 1,
                                        f"the trajectory's first step, all {U} units, fp64")
    del k_pool, v_pool, ksum
    torch.cuda.empty_cache()
    return res


def resident262k_leg(args, dev, timed, cap, peak, cpu_baseline, w, scache, qs, q_host0):
    """The 262k-context workload with its whole pool resident on the device (batch 8, 40 q / 8 kv
    heads, 4096 pages per request, k = 128): one step is the block scores, the selection with the
    set-difference against each unit's 2048-slot resident buffer and the 64-bucket LRU update
    (at this context: the selection, then the set-difference and the LRU update on a second stream
    beside the sparse attention, which does not read them, as in the Llama-3-8B step), and the
    sparse attention, one CUDA graph per step along the query walk.  The set-difference and the LRU
    update are also timed alone on further eager steps."""
    import torch
    import sparse_paged_kv_score_gb300 as spkv
    bf, i32 = _dev_helpers(dev)
    B, Hq, Hk, npm = w["B"], w["Hq"], w["Hk"], w["np_max"]
    U = B * Hk
    k_q, k_e = w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    ns = w["n_slots"]
    pt, seq = i32(w["page_table"]), i32(w["seq_len"])
    ev = torch.from_numpy(w["evict"].astype(np.float32)).to(dev)
    scores = torch.empty(B, Hk, npm, dtype=torch.float32, device=dev)
    alive = torch.full((B, Hk, (npm + 31) // 32), -1, dtype=torch.int32, device=dev)
    sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=dev)
    n_sel = torch.empty(B, Hk, dtype=torch.int32, device=dev)
    resident = torch.full((U, ns), -1, dtype=torch.int32, device=dev)
    ts = torch.full((U, ns), np.iinfo(np.int32).min, dtype=torch.int32, device=dev)
    missing, slot, victims = (torch.empty(U, stride, dtype=torch.int32, device=dev) for _ in range(3))
    n_missing = torch.empty(U, dtype=torch.int32, device=dev)
    hist = torch.empty(U, 64, dtype=torch.int32, device=dev)
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    n_iter = args.warmup + args.steps
    side = torch.cuda.Stream()

    def bookkeeping_beside(attn, i):
        """The selection's residency bookkeeping on a second stream beside the attention call."""
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            spkv.resident_setdiff(scache, resident, sel, n_sel, missing, n_missing, slot)
            spkv.lru_bucket_update(scache, resident, ts, slot, n_sel, missing, n_missing, i, 1, victims, hist)
        attn()
        main.wait_stream(side)

    def step(i):
        spkv.score_blocks(scache, qs[i], pt, seq, scores)
        spkv.select_topk(scache, scores, ev, alive, seq, k_q, k_e, sel, n_sel)
        bookkeeping_beside(lambda: spkv.sparse_decode_attn(scache, qs[i], pt, sel, n_sel, seq, out, lse), i)

    for i in range(args.warmup):
        step(i)
    idx = list(range(args.warmup, n_iter))
    graphs = {}
    for i in idx:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(i)
        graphs[i] = g
    torch.cuda.synchronize()
    ms_all = timed(lambda i: graphs[i].replay(), idx)
    del graphs
    # the bookkeeping alone, on further steps of the walk (events between the calls)
    sd_us, lru_us, miss = [], [], []
    st_ = torch.cuda.current_stream()
    for i in range(n_iter, n_iter + max(args.steps, 5)):
        spkv.score_blocks(scache, qs[i], pt, seq, scores)
        spkv.select_topk(scache, scores, ev, alive, seq, k_q, k_e, sel, n_sel)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(st_)
        spkv.resident_setdiff(scache, resident, sel, n_sel, missing, n_missing, slot)
        e[1].record(st_)
        spkv.lru_bucket_update(scache, resident, ts, slot, n_sel, missing, n_missing, i, 1, victims, hist)
        e[2].record(st_)
        torch.cuda.synchronize()
        sd_us.append(e[0].elapsed_time(e[1]) * 1e3)
        lru_us.append(e[1].elapsed_time(e[2]) * 1e3)
        miss.append(int(n_missing.sum().item()))
    # the same step with the page table as a two-level directory ([Spin] 2C): every segment on the
    # device tier, then every segment on the host tier (read in place over the host link)
    pdir = {}
    shift = 8
    n_segs = B * ((npm + (1 << shift) - 1) >> shift)
    for tier in ("device", "host"):
        pm = spkv.PageMap(B, npm, seg_shift=shift, n_dev_segs=n_segs if tier == "device" else 0)
        for b in range(B):
            pm.map(b, 0, w["page_table"][b])
            if tier == "device":
                for p0 in range(0, npm, 1 << shift):
                    pm.promote(b, p0)
        pm.sync()

        def dstep(i):
            spkv.score_blocks_dir(scache, qs[i], pm, seq, scores)
            spkv.select_topk(scache, scores, ev, alive, seq, k_q, k_e, sel, n_sel)
            bookkeeping_beside(lambda: spkv.sparse_decode_attn_dir(scache, qs[i], pm, sel, n_sel, seq, out, lse), i)

        dstep(0)
        graphs = {}
        for i in idx:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                dstep(i)
            graphs[i] = g
        torch.cuda.synchronize()
        dms = timed(lambda i: graphs[i].replay(), idx)
        sc_us = statistics.median(timed(lambda i: spkv.score_blocks_dir(scache, qs[i], pm, seq, scores), idx)) * 1e3
        del graphs
        dev_b, host_b = pm.nbytes()
        pdir[tier + "_tier"] = {"ms_per_step": statistics.mean(dms), "score_blocks_us": sc_us,
                                "metadata_device_bytes": dev_b, "metadata_host_bytes": host_b}
        pm.close()
    pdir["flat_page_table_bytes"] = B * npm * 4
    pdir["flat_score_blocks_us"] = statistics.median(
        timed(lambda i: spkv.score_blocks(scache, qs[i], pt, seq, scores), idx)) * 1e3
    pdir["segment_ids"] = 1 << shift
    st, bits = spkv.get_device_error(scache)
    if st != 0:
        raise RuntimeError(f"device error bits {bits} in the resident 262k leg")
    byts = _parts(step_bytes(w, k_q + k_e), ("score", "select", "setdiff", "lru", "attn"))
    ms = statistics.mean(ms_all)
    gbs = byts / (ms * 1e-3) / 1e9
    res = {"workload": w["name"] + ", pool resident on the device",
           "step": "score, select, set-difference + LRU (2048 slots) on a second stream beside the sparse attention",
           "ms_per_step": ms, "ms_per_step_median": statistics.median(ms_all), "bytes_per_step": byts,
           "GBps": gbs, "pct_hbm_peak": 100 * gbs / peak, "queries_per_s": B / (ms * 1e-3),
           "resident_setdiff_us": statistics.median(sd_us), "lru_bucket_update_us": statistics.median(lru_us),
           "missing_pages_per_step": statistics.mean(miss), "launch": "one CUDA graph per step",
           "page_directory": pdir}
    if cpu_baseline:
        units = np.arange(U, dtype=np.int32)
        w1 = dict(w, q=q_host0)
        dt = _oracle_timed(lambda: oracle_step(w1, units, n_slots=ns), min_s=0.0)
        res["cpu_baseline"] = _cpu_line(dt, byts, os.cpu_count() or 1,
                                        f"one whole step (all {U} units) at the walk's first query, fp64")
    return res


def offload_leg(args, dev, stream, timed, cap, peak, cpu_baseline):
    """Retrieve over the host link: the 262k-context workload (B8, Hq40/Hk8, 4096 pages per
    request, k = 128) with the whole K/V pool in pinned host memory and 2048 device slots per
    (request, kv head).  The pooled-key summaries stay on the device (built once from a device
    copy of the pool); every page that attention reads comes from a slot."""
    import torch
    import gen
    import sparse_paged_kv_score_gb300 as spkv

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)

    def pinned(a):
        t = torch.empty(a.shape, dtype=torch.int16, pin_memory=True)
        t.numpy()[...] = a.view(np.int16)
        return t.view(torch.bfloat16)

    w = gen.long262k(seed=0)
    B, Hq, Hk, npm = w["B"], w["Hq"], w["Hk"], w["np_max"]
    U = B * Hk
    k_q, k_e = w["k_q"], w["k_e"]
    stride = k_q + k_e + 1
    ns = w["n_slots"]
    dk, dv = bf(w["k_pool"]), bf(w["v_pool"])
    dks = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.float32, device=dev)
    scache = spkv.paged_kv_create(dk, dv, dks, i32(gen.page_counts(w)), max_units=U)   # summaries
    k_host, v_host = pinned(w["k_pool"]), pinned(w["v_pool"])
    k_slots = torch.zeros(Hk, B * ns, 64, 128, dtype=torch.bfloat16, device=dev)
    v_slots = torch.zeros_like(k_slots)
    slots = spkv.paged_kv_create(k_slots, v_slots, None, None, max_units=U)
    pt, seq = i32(w["page_table"]), i32(w["seq_len"])
    n_iter = args.warmup + args.steps
    walk = gen.walk_queries(w, 2 * n_iter + max(args.steps, 5) + 1)
    qs = [bf(q) for q in walk]   # eager steps, then graph-captured steps
    # the same workload with its pool resident on the device (the handle over the device pool)
    res_leg = resident262k_leg(args, dev, timed, cap, peak, cpu_baseline, w, scache, qs, walk[0])
    ev = torch.from_numpy(w["evict"].astype(np.float32)).to(dev)
    scores = torch.empty(B, Hk, npm, dtype=torch.float32, device=dev)
    alive = torch.full((B, Hk, (npm + 31) // 32), -1, dtype=torch.int32, device=dev)
    sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=dev)
    n_sel = torch.empty(B, Hk, dtype=torch.int32, device=dev)
    resident = torch.full((U, ns), -1, dtype=torch.int32, device=dev)
    ts = torch.full((U, ns), np.iinfo(np.int32).min, dtype=torch.int32, device=dev)
    missing = torch.empty(U, stride, dtype=torch.int32, device=dev)
    n_missing = torch.empty(U, dtype=torch.int32, device=dev)
    slot = torch.empty(U, stride, dtype=torch.int32, device=dev)
    victims = torch.empty(U, stride, dtype=torch.int32, device=dev)
    hist = torch.empty(U, 64, dtype=torch.int32, device=dev)
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)

    def select_and_plan(i):
        spkv.score_blocks(scache, qs[i], pt, seq, scores)
        spkv.select_resident_update(scache, scores, ev, alive, seq, k_q, k_e, sel, n_sel, resident, ts, i, 1,
                                    missing, n_missing, slot, victims, hist)

    def retrieve():
        spkv.retrieve_pages(slots, k_host, v_host, pt, missing, n_missing, victims, slot, n_sel, ns)

    def attend(i):
        spkv.sparse_decode_attn_slots(slots, qs[i], sel, slot.view(B, Hk, stride), n_sel, ns, seq, out, lse)

    # cold swap-in: every slot empty, so every selected page crosses the host link
    select_and_plan(0)
    slot0 = slot.clone()
    cold_pages = int(n_missing.sum().item())
    retrieve()
    attend(0)

    def cold(_):
        slot.copy_(slot0)    # the slot list is completed in place; restore it (outside the events)

    cold_ms = []
    for r in range(3 + args.steps):
        cold(r)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        retrieve()
        b_.record(stream)
        torch.cuda.synchronize()
        if r >= 3:
            cold_ms.append(a.elapsed_time(b_))
    cold_bytes = cold_pages * PAGE_BYTES
    cold_avg = statistics.mean(cold_ms)
    # copy-engine reference over the same link: one 1 GiB pinned -> device copy
    src = torch.empty(1 << 29, dtype=torch.int16, pin_memory=True)
    dst = torch.empty(1 << 29, dtype=torch.int16, device=dev)
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    ce_ms = statistics.mean(timed(lambda i: dst.copy_(src, non_blocking=True), range(5)))
    ce_gbs = (1 << 30) / (ce_ms * 1e-3) / 1e9
    del src, dst

    # steady offloaded decode steps (the query walks, so most selected pages stay resident)
    step_ms, ret_ms, att_ms, miss = [], [], [], []
    for i in range(1, n_iter + 1):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        select_and_plan(i)
        e[1].record(stream)
        retrieve()
        e[2].record(stream)
        attend(i)
        e[3].record(stream)
        torch.cuda.synchronize()
        if i > args.warmup:
            step_ms.append(e[0].elapsed_time(e[3]))
            ret_ms.append(e[1].elapsed_time(e[2]))
            att_ms.append(e[2].elapsed_time(e[3]))
            miss.append(int(n_missing.sum().item()))
    # the walk goes on with each step captured as one CUDA graph (no events between its calls)
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    gsteps = list(range(n_iter + 1, 2 * n_iter + 1))
    graphs = {}
    for i in gsteps:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            select_and_plan(i)
            retrieve()
            attend(i)
        graphs[i] = g
    torch.cuda.synchronize()
    gstep_ms, gmiss = [], []
    for i in gsteps:
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graphs[i].replay()
        b_.record(stream)
        torch.cuda.synchronize()
        if i > n_iter + args.warmup:
            gstep_ms.append(a.elapsed_time(b_))
            gmiss.append(int(n_missing.sum().item()))
    del graphs
    for c in (scache, slots):
        st, bits = spkv.get_device_error(c)
        if st != 0:
            raise RuntimeError(f"device error bits {bits} in the offload leg")
    scache.close()
    slots.close()
    ms = statistics.mean(step_ms)
    r_ms = statistics.mean(ret_ms)
    attn_bytes = int(n_sel.sum().item()) * PAGE_BYTES
    out_d = {
        "workload": w["name"] + ", K/V pool (8.6 GB) in pinned host memory, 2048 device slots per unit",
        "retrieve_cold": {"pages": cold_pages, "bytes": cold_bytes, "us": cold_avg * 1e3,
                          "GBps": cold_bytes / (cold_avg * 1e-3) / 1e9,
                          "bound": "host link (NVLink-C2C)", "peak": ce_gbs,
                          "peak_kind": "measured copy-engine pinned-host-to-device copy of 1 GiB",
                          "frac": cold_bytes / (cold_avg * 1e-3) / 1e9 / ce_gbs},
        "step": {"launch": "eager, one call per kernel", "ms_per_step": ms, "queries_per_s": B / (ms * 1e-3),
                 "missing_pages_per_step": statistics.mean(miss),
                 "retrieve_us": r_ms * 1e3,
                 "retrieve_GBps": statistics.mean(miss) * PAGE_BYTES / (r_ms * 1e-3) / 1e9,
                 "attn_slots_us": statistics.mean(att_ms) * 1e3,
                 "attn_slots_GBps": attn_bytes / (statistics.mean(att_ms) * 1e-3) / 1e9},
        "step_graph": {"launch": "one CUDA graph per step", "ms_per_step": statistics.mean(gstep_ms),
                       "queries_per_s": B / (statistics.mean(gstep_ms) * 1e-3),
                       "missing_pages_per_step": statistics.mean(gmiss)},
    }
    del dk, dv, dks, k_slots, v_slots, k_host, v_host
    torch.cuda.empty_cache()
    return out_d, res_leg


def run_native(args):
    import torch
    import gen
    import sparse_paged_kv_score_gb300 as spkv
    from sparse_paged_kv_score_gb300 import build as cuda_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    cuda_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    w = gen.llama8b(seed=rank, B=args.batch)
    B, Hq, Hk, npm = w["B"], w["Hq"], w["Hk"], w["np_max"]
    k_q, k_e = w["k_q"], w["k_e"]
    k = k_q + k_e
    stride = k + 1
    U = B * Hk
    L = int(w["seq_len"][0])

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)

    k_pool, v_pool = bf(w["k_pool"]), bf(w["v_pool"])
    ksum = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.float32, device=dev)
    cnt = i32(gen.page_counts(w))
    cache = spkv.paged_kv_create(k_pool, v_pool, ksum, cnt, max_units=U)
    pt, seq = i32(w["page_table"]), i32(w["seq_len"])
    n_iter = args.warmup + args.steps
    # per-step inputs: fresh query, eviction scores (random walk), the new token's K/V rows
    qs = [bf(gen.rows_bf16(rank, 7000 + i, B * Hq).reshape(B, Hq, 128)) for i in range(n_iter)]
    ev0 = w["evict"].astype(np.float64)
    evs, e = [], ev0
    for i in range(n_iter):
        e = e + 0.1 * gen.normal_f64(rank, 8000 + i, e.size).reshape(e.shape)
        evs.append(torch.from_numpy(e.astype(np.float32)).to(dev))
    knew = [bf(gen.rows_bf16(rank, 9000 + i, U).reshape(B, Hk, 128)) for i in range(n_iter)]
    vnew = [bf(gen.rows_bf16(rank, 9500 + i, U).reshape(B, Hk, 128)) for i in range(n_iter)]
    # the step's own token sits at position L-1 (the last row of the local page)

    scores = torch.empty(B, Hk, npm, dtype=torch.float32, device=dev)
    alive = torch.full((B, Hk, (npm + 31) // 32), -1, dtype=torch.int32, device=dev)
    sel = torch.empty(B, Hk, stride, dtype=torch.int32, device=dev)
    n_sel = torch.empty(B, Hk, dtype=torch.int32, device=dev)
    resident = torch.full((U, N_SLOTS), -1, dtype=torch.int32, device=dev)
    ts = torch.full((U, N_SLOTS), np.iinfo(np.int32).min, dtype=torch.int32, device=dev)
    missing = torch.empty(U, stride, dtype=torch.int32, device=dev)
    n_missing = torch.empty(U, dtype=torch.int32, device=dev)
    slot = torch.empty(U, stride, dtype=torch.int32, device=dev)
    victims = torch.empty(U, stride, dtype=torch.int32, device=dev)
    hist = torch.empty(U, 64, dtype=torch.int32, device=dev)
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    class _Flush:
        @staticmethod
        def zero_():
            if args.l2 == "write":
                flush_buf.zero_()

    flush = _Flush()
    stream = torch.cuda.current_stream()

    side = torch.cuda.Stream()

    def run_step(c, q, k_new, v_new, ev, al, res, tsr, t, o, ls):
        """One decode step through the public API on handle c."""
        # the new token's K/V row at position L-1 and the block scores, one launch
        spkv.decode_append_score(c, k_new, v_new, q, pt, seq, scores)
        if args.bookkeeping == "fused":
            # select_topk + resident_setdiff + lru_bucket_update, fused into one kernel
            spkv.select_resident_update(c, scores, ev, al, seq, k_q, k_e, sel, n_sel, res, tsr, t, 1, missing,
                                        n_missing, slot, victims, hist)
            spkv.sparse_decode_attn(c, q, pt, sel, n_sel, seq, o, ls)
        else:
            # the selection, then the residency bookkeeping (which attention does not read) on a
            # second stream while the pages stream; the step ends when both are done
            spkv.select_topk(c, scores, ev, al, seq, k_q, k_e, sel, n_sel)
            main = torch.cuda.current_stream()
            side.wait_stream(main)
            with torch.cuda.stream(side):
                spkv.resident_setdiff(c, res, sel, n_sel, missing, n_missing, slot)
                spkv.lru_bucket_update(c, res, tsr, slot, n_sel, missing, n_missing, t, 1, victims, hist)
            spkv.sparse_decode_attn(c, q, pt, sel, n_sel, seq, o, ls)
            main.wait_stream(side)

    def step(i):
        run_step(cache, qs[i], knew[i], vnew[i], evs[i], alive, resident, ts, i, out, lse)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            torch.cuda.synchronize()

    def timed(fn, idx):
        """Device time (ms) of fn(i) for i in idx, each bracketed by events, L2 flushed between."""
        ev = []
        for i in idx:
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(i)
            b_.record(stream)
            flush.zero_()
            ev.append((a, b_))
        torch.cuda.synchronize()
        return [a.elapsed_time(b_) for a, b_ in ev]

    for i in range(args.warmup):
        step(i)
        flush.zero_()
    st, bits = spkv.get_device_error(cache)
    if st != 0:
        raise RuntimeError(f"device error bits {bits} after warm-up")

    # one CUDA graph per timed step (each step has its own inputs and LRU time)
    timed_idx = list(range(args.warmup, args.warmup + args.steps))
    graphs = {}
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    for i in timed_idx:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(i)
        graphs[i] = g
    torch.cuda.synchronize()
    barrier()
    with Clocks(local_rank) as clk:
        step_ms = timed(lambda i: graphs[i].replay(), timed_idx)
        barrier()
    eager_ms = statistics.mean(timed(step, timed_idx))
    attn_ms = timed(lambda i: spkv.sparse_decode_attn(cache, qs[i], pt, sel, n_sel, seq, out, lse), timed_idx)
    ms = rank_max(statistics.mean(step_ms), dev)
    ms_median = rank_max(statistics.median(step_ms), dev)
    st, bits = spkv.get_device_error(cache)
    if st != 0:
        raise RuntimeError(f"device error bits {bits} in the timed region")

    byts = step_bytes(w, k)
    step_total = sum(v for kk, v in byts.items() if kk != "attn_kv")
    value = replica_throughput(world, step_total, ms)
    attn_avg = statistics.mean(attn_ms)
    peak, peak_kind = peaks()
    cpu_on = rank == 0 and world == 1 and not args.no_cpu_baseline
    achieved = byts["attn_kv"] / (attn_avg * 1e-3) / 1e9

    # ---- lazy-RoPE attention on the same selected pages (8 documents x 4096 tokens)
    lazy = None
    if not args.no_lazy:
        sel_h, n_h = sel.cpu().numpy(), n_sel.cpu().numpy()
        phys = np.zeros((B, Hk, stride), np.int32)
        valid = np.ones((B, Hk, stride), np.int32)
        dslot = np.zeros((B, Hk, stride), np.int32)
        for b in range(B):
            for h in range(Hk):
                pg = sel_h[b, h, :n_h[b, h]]
                phys[b, h, :len(pg)] = w["page_table"][b, pg]
                valid[b, h, :len(pg)] = np.minimum(64, L - 64 * pg)
                dslot[b, h, :len(pg)] = pg // 64
        words = spkv.pack_page_words(phys, valid, dslot)
        meta = torch.from_numpy(words.view(np.int32)).to(dev)
        n_pages = i32(np.full(B, stride, np.int32))
        doc_pos = i32(np.tile(np.arange(8, dtype=np.int32) * 4096, (B, 1)))
        qpos = i32(np.full(B, L - 1, np.int32))
        lout = torch.empty_like(out)
        llse = torch.empty_like(lse)

        def lazy_call(i):
            spkv.lazy_rope_decode_attn(cache, qs[i], qpos, meta, n_pages, doc_pos, 500000.0, lout, llse)

        timed(lazy_call, range(3))
        lazy_ms = statistics.mean(timed(lazy_call, timed_idx))
        lazy_gbs = byts["attn_kv"] / (lazy_ms * 1e-3) / 1e9
        lazy = {"kernel": "lazy_rope_decode_attn (same 65 pages/head as 8 docs x 4096 tokens)",
                "us": lazy_ms * 1e3, "achieved_GBps": lazy_gbs, "frac": lazy_gbs / peak,
                "vs_sparse_time": lazy_ms / attn_avg}

    # ---- lazy-RoPE dense decode over shared documents (64 requests x 8 Zipf-drawn documents)
    rag = None
    prefill = None
    if not args.no_rag and rank == 0:
        wr = gen.lazy_rag(seed=0, B=args.rag_batch, n_docs=args.rag_docs)
        Br, Hqr, Hkr = wr["B"], wr["Hq"], wr["Hk"]
        rk, rv = bf(wr["k_pool"]), bf(wr["v_pool"])
        rks = torch.zeros(Hkr, wr["n_phys"], 4, 128, dtype=torch.float32, device=dev)
        rcache = spkv.paged_kv_create(rk, rv, rks, i32(wr["page_cnt"]), max_units=Br * Hkr)
        ok = wr["phys"] >= 0
        wwords = np.zeros(wr["phys"].shape, np.uint32)
        wwords[ok] = spkv.pack_page_words(wr["phys"][ok], wr["valid"][ok], wr["slot"][ok])
        rmeta = torch.from_numpy(wwords.view(np.int32)).to(dev)
        rq, rqpos, rnp, rdoc = bf(wr["q"]), i32(wr["qpos"]), i32(wr["n_pages"]), i32(wr["doc_pos"])
        rout = torch.empty(Br, Hqr, 128, dtype=torch.float32, device=dev)
        rlse = torch.empty(Br, Hqr, dtype=torch.float32, device=dev)

        def rag_call(i):
            spkv.lazy_rope_decode_attn(rcache, rq, rqpos, rmeta, rnp, rdoc, wr["theta"], rout, rlse)

        timed(rag_call, range(3))
        rag_ms = statistics.mean(timed(rag_call, timed_idx))
        pages = int(wr["n_pages"].sum()) * Hkr
        logical = pages * PAGE_BYTES
        distinct = len(np.unique(wr["phys"][ok])) * Hkr * PAGE_BYTES
        # the same decode scheduled by document (a plan built once on the host for this batch)
        plan = spkv.DocPlan(rcache, Hqr, wr["picks"], wr["doc_first"])
        dwords = spkv.pack_page_words(wr["doc_phys"], wr["doc_valid"], np.zeros_like(wr["doc_phys"]))
        rdw = torch.from_numpy(dwords.view(np.int32)).to(dev)
        rdf = i32(wr["doc_first"])
        dout = torch.empty_like(rout)
        dlse = torch.empty_like(rlse)

        def docs_call(i):
            spkv.lazy_rope_decode_attn_docs(rcache, plan, rq, rqpos, rdw, rdf, rdoc, wr["theta"], dout, dlse)

        timed(docs_call, range(3))
        docs_ms = statistics.mean(timed(docs_call, timed_idx))
        if not torch.allclose(dout, rout, rtol=0, atol=1e-4):
            raise RuntimeError("document-major lazy decode differs from the per-request form")
        doc_jobs = plan.n_jobs
        plan.close()
        # LazyAttention prefill over the same cached documents: 128 new query rows per request
        if not args.no_prefill:
            Tq = 128
            pq = bf(gen.rows_bf16(0, 7700, Br * Tq * Hqr).reshape(Br, Tq, Hqr, 128))
            pout = torch.empty(Br, Tq, Hqr, 128, dtype=torch.float32, device=dev)
            plse = torch.empty(Br, Tq, Hqr, dtype=torch.float32, device=dev)

            def pre_call(i):
                spkv.lazy_rope_prefill_attn(rcache, pq, rqpos, rmeta, rnp, rdoc, wr["theta"], pout, plse)

            timed(pre_call, range(3))
            pre_ms = statistics.mean(timed(pre_call, timed_idx))
            keys = int(wr["qpos"].sum())          # cached tokens over all requests
            flops = 4.0 * 128 * Tq * Hqr * keys   # QK^T and PV, 2 flops per multiply-add each
            tflops = flops / (pre_ms * 1e-3) / 1e12
            tpeak, tkind = bf16_peak()
            # the same prefill for ALiBi models: unrotated keys, bias -slope * distance
            ok_pages = wr["phys"] >= 0
            pstart = np.where(ok_pages, wr["page_start"], 0).astype(np.int32)
            rps = i32(pstart)
            slopes = torch.from_numpy((2.0 ** (-8.0 * (np.arange(Hqr) + 1) / Hqr)).astype(np.float32)).to(dev)

            def alibi_call(i):
                spkv.lazy_alibi_prefill_attn(rcache, pq, rqpos, rmeta, rnp, rps, rdoc, slopes, pout, plse)

            timed(alibi_call, range(3))
            al_ms = statistics.mean(timed(alibi_call, timed_idx))
            al_tf = flops / (al_ms * 1e-3) / 1e12
            prefill = {"kernel": "lazy_rope_prefill_attn (tcgen05.mma, TMEM accumulators, TMA pages)",
                       "workload": f"the RAG documents above, 128 new query rows per request ({Br} x 128 x 32 heads)",
                       "us": pre_ms * 1e3, "flops": flops, "bound": "tensor", "achieved_TFLOPs": tflops,
                       "peak": tpeak, "peak_kind": tkind + " bf16 dense (cuBLAS burst)", "frac": tflops / tpeak,
                       "query_rows_per_s": Br * Tq / (pre_ms * 1e-3),
                       "alibi": {"kernel": "lazy_alibi_prefill_attn (same kernel, bias instead of rotation)",
                                 "slopes": "2^(-8 (h+1) / 32) per query head h", "us": al_ms * 1e3,
                                 "achieved_TFLOPs": al_tf, "frac": al_tf / tpeak}}
            del pq, pout, plse
        st, bits = spkv.get_device_error(rcache)
        if st != 0:
            raise RuntimeError(f"device error bits {bits} in the RAG leg")
        rcache.close()
        rag = {"workload": f"lazy-RoPE RAG decode B{Br} Hq32/Hk8, 8 Zipf(1.1) docs of 1024-4096 tokens "
                           f"(pool of {args.rag_docs} documents)",
               "us": rag_ms * 1e3, "logical_GBps": logical / (rag_ms * 1e-3) / 1e9,
               "distinct_page_GBps": distinct / (rag_ms * 1e-3) / 1e9,
               "distinct_page_frac": distinct / (rag_ms * 1e-3) / 1e9 / peak,
               "logical_bytes": logical, "distinct_page_bytes": distinct,
               "queries_per_s": Br / (rag_ms * 1e-3),
               "note": "logical = every (request, head, page) read; shared hot documents hit in L2",
               "by_document": {"kernel": "lazy_rope_decode_attn_docs (jobs of one document, one kv head and up "
                                         "to 4 requests; plan built once on the host)",
                               "jobs": doc_jobs, "us": docs_ms * 1e3,
                               "distinct_page_GBps": distinct / (docs_ms * 1e-3) / 1e9,
                               "distinct_page_frac": distinct / (docs_ms * 1e-3) / 1e9 / peak,
                               "queries_per_s": Br / (docs_ms * 1e-3)}}
        if cpu_on:
            import oracle
            su = np.sort(np.random.default_rng(0).choice(Br * Hkr, 64, replace=False)).astype(np.int32)
            thr = os.cpu_count() or 1
            dt = _oracle_timed(lambda: oracle.lazy_attn_batch(
                wr["q"], wr["k_pool"], wr["v_pool"], wr["phys"], wr["valid"], wr["slot"], wr["n_pages"], wr["qpos"],
                wr["doc_pos"], wr["theta"], materialise=False, units=su, nthreads=thr), min_s=0.0)
            su_bytes = int(wr["n_pages"][su // Hkr].sum()) * PAGE_BYTES
            rag["cpu_baseline"] = _cpu_line(dt, su_bytes, thr, "64 of the 512 (request, kv head) units, lazy form, "
                                                               "fp64; logical bytes of those units")
        del rk, rv, rks, rmeta

    # ---- cheaper scoring: the same step with bf16 pooled-key summaries (half the scoring bytes)
    bf16_sum = None
    if not args.no_bf16_summaries:
        ksum16 = torch.zeros(Hk, w["n_phys"], 4, 128, dtype=torch.bfloat16, device=dev)
        cache16 = spkv.paged_kv_create(k_pool, v_pool, ksum16, cnt, max_units=U)
        alive16 = alive.clone()
        res16, ts16 = resident.clone(), ts.clone()

        def step16(i):
            run_step(cache16, qs[i], knew[i], vnew[i], evs[i], alive16, res16, ts16, i, out, lse)

        for i in range(args.warmup):
            step16(i)
        graphs16 = {}
        for i in timed_idx:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                step16(i)
            graphs16[i] = g
        torch.cuda.synchronize()
        ms16 = statistics.mean(timed(lambda i: graphs16[i].replay(), timed_idx))
        sc16 = statistics.mean(timed(lambda i: spkv.score_blocks(cache16, qs[i], pt, seq, scores), timed_idx))
        sc32 = statistics.mean(timed(lambda i: spkv.score_blocks(cache, qs[i], pt, seq, scores), timed_idx))
        st16, bits16 = spkv.get_device_error(cache16)
        if st16 != 0:
            raise RuntimeError(f"device error bits {bits16} in the bf16-summary leg")
        total16 = step_total - byts["score"] // 2
        bf16_sum = {"workload": w["name"] + " with bf16 pooled-key summaries",
                    "ms_per_step": ms16, "queries_per_s": B / (ms16 * 1e-3),
                    "value_GBps": total16 / (ms16 * 1e-3) / 1e9, "bytes_per_step": int(total16),
                    "score_us": sc16 * 1e3, "score_GBps": byts["score"] / 2 / (sc16 * 1e-3) / 1e9,
                    "score_fp32_us": sc32 * 1e3, "launch": "one CUDA graph per step"}
        del graphs16
        cache16.close()

    # ---- PyramidKV-style column score S: prompts of 5000 tokens, window of the last 256 rows
    colsc = None
    if not args.no_colscore and rank == 0:
        Bc, nc, ac = args.col_batch, 5000, 256
        npc = (nc + 63) // 64
        ck = bf(gen.rows_bf16(0, 7800, Hk * Bc * npc * 64).reshape(Hk, Bc * npc, 64, 128))
        ccache = spkv.paged_kv_create(ck, ck, None, None)           # V is not read by the score
        cpt = i32(gen.permutation(0, 7801, Bc * npc).reshape(Bc, npc))
        cseq = i32(np.full(Bc, nc, np.int32))
        cq = bf(gen.rows_bf16(0, 7802, Bc * ac * Hq).reshape(Bc, ac, Hq, 128))
        cs = torch.empty(Bc, Hq, npc * 64, dtype=torch.float32, device=dev)

        def col_call(i):
            spkv.attn_column_scores(ccache, cq, cpt, cseq, cs)

        timed(col_call, range(3))
        col_ms = statistics.mean(timed(col_call, timed_idx))
        sums = cs.sum(-1)
        if not torch.allclose(sums, torch.full_like(sums, float(ac)), rtol=1e-3):
            raise RuntimeError("column scores do not sum to the window size")
        # the method's own work: one S = Q K^T over the window rows and every key (the rows' maximum
        # and sum come from the attention that already ran)
        cflops = 2.0 * 128 * ac * nc * Hq * Bc
        ctf = cflops / (col_ms * 1e-3) / 1e12
        tpeak, tkind = bf16_peak()
        # the form that takes each window row's log-sum-exp from that attention: the rows' LSE is
        # prepared here with plain torch on the device (input set-up, outside the timed region)
        kk = ck.view(Hk, Bc * npc * 64, 128)
        lse_in = torch.empty(Bc, ac, Hq, dtype=torch.float32, device=dev)
        pos = torch.arange(nc, device=dev)
        for b in range(Bc):
            rows = (cpt[b].long()[:, None] * 64 + torch.arange(64, device=dev)[None, :]).reshape(-1)[:nc]
            for h in range(Hk):
                kb = kk[h, rows].float()
                z = torch.einsum("ahd,kd->ahk", cq[b, :, h * (Hq // Hk):(h + 1) * (Hq // Hk)].float(), kb)
                z = z / float(np.sqrt(128.0))
                vis = pos[None, :] <= (nc - ac + torch.arange(ac, device=dev))[:, None]
                z = z.masked_fill(~vis[:, None, :], float("-inf"))
                lse_in[b, :, h * (Hq // Hk):(h + 1) * (Hq // Hk)] = torch.logsumexp(z, dim=-1)
        csl = torch.empty_like(cs)

        def col_lse_call(i):
            spkv.attn_column_scores_lse(ccache, cq, lse_in, cpt, cseq, csl)

        timed(col_lse_call, range(3))
        coll_ms = statistics.mean(timed(col_lse_call, timed_idx))
        if not torch.allclose(csl, cs, rtol=1e-3, atol=1e-5):
            raise RuntimeError("column scores from the given LSE differ from the two-pass form")
        st_c, bits_c = spkv.get_device_error(ccache)
        if st_c != 0:
            raise RuntimeError(f"device error bits {bits_c} in the column-score leg")
        ctf_l = cflops / (coll_ms * 1e-3) / 1e12
        colsc = {"kernel": "attn_column_scores (colscore_kernel pass 1: each row's LSE; colscore_lse_kernel: the "
                           "probabilities with keys as M; tcgen05.mma, TMA pages)",
                 "workload": f"{Bc} prompts x {nc} tokens, window of the last {ac} rows, Hq {Hq} / Hk {Hk}",
                 "us": col_ms * 1e3, "flops": cflops,
                 "flops_def": "2 * 128 * window rows * prompt tokens * Hq * prompts (one Q K^T pass)",
                 "bound": "tensor", "achieved_TFLOPs": ctf,
                 "peak": tpeak, "peak_kind": tkind + " bf16 dense (cuBLAS burst)", "frac": ctf / tpeak,
                 "prompts_per_s": Bc / (col_ms * 1e-3),
                 "launches": "two kernels (the LSE of both 128-row chunks in one grid, then the probability pass)",
                 "given_lse": {"kernel": "attn_column_scores_lse (colscore_lse_kernel: the probability pass alone)",
                               "us": coll_ms * 1e3, "achieved_TFLOPs": ctf_l, "frac": ctf_l / tpeak}}
        ccache.close()
        del ck, cq, cs, csl, lse_in

    # ---- offload: the 262k-context workload with its K/V pool in pinned host memory
    offload, resident262k = None, None
    if not args.no_offload and rank == 0:
        offload, resident262k = offload_leg(args, dev, stream, timed, cap, peak, cpu_on)

    # ---- the other workloads of the per-config report
    tiny, traj = None, None
    if not args.no_configs and rank == 0:
        tiny = tiny_leg(args, dev, timed, cap, peak, cpu_on)
        traj = traj_leg(args, dev, timed, cap, peak, cpu_on)

    # ---- end to end through the public API: pinned host inputs in, outputs back, every step.
    # A step's inputs (q, eviction scores, the new K and V rows) sit in one pinned host buffer
    # and its outputs (O, LSE) in one device buffer, so each direction is a single copy; the API
    # calls get typed views of the matching device buffers.
    in_shapes = [((B, Hq, 128), torch.bfloat16), ((B, Hk, npm), torch.float32), ((B, Hk, 128), torch.bfloat16),
                 ((B, Hk, 128), torch.bfloat16)]
    in_bytes = [int(np.prod(sh)) * torch.tensor([], dtype=dt).element_size() for sh, dt in in_shapes]
    in_off = np.concatenate([[0], np.cumsum(in_bytes)]).astype(int)   # every section a multiple of 256 B

    def views(buf, offs, shapes):
        return [buf[offs[j]:offs[j + 1]].view(dt).view(sh) for j, (sh, dt) in enumerate(shapes)]

    in_h = [torch.empty(int(in_off[-1]), dtype=torch.uint8).pin_memory() for _ in range(2)]
    for s_ in range(2):
        for dst, src in zip(views(in_h[s_], in_off, in_shapes), (qs[s_], evs[s_], knew[s_], vnew[s_])):
            dst.copy_(src.cpu())
    in_d = torch.empty(int(in_off[-1]), dtype=torch.uint8, device=dev)
    q_d, e_d, k_d, v_d = views(in_d, in_off, in_shapes)
    out_shapes = [((B, Hq, 128), torch.float32), ((B, Hq), torch.float32)]
    out_off = np.array([0, B * Hq * 128 * 4, B * Hq * 129 * 4])
    res_d = torch.empty(int(out_off[-1]), dtype=torch.uint8, device=dev)
    res_h = torch.empty(int(out_off[-1]), dtype=torch.uint8).pin_memory()
    out_e, lse_e = views(res_d, out_off, out_shapes)
    h2d = int(in_off[-1])
    d2h = int(out_off[-1])

    def e2e_step(i):
        in_d.copy_(in_h[i % 2], non_blocking=True)
        run_step(cache, q_d, k_d, v_d, e_d, alive, resident, ts, 1000 + i, out_e, lse_e)
        res_h.copy_(res_d, non_blocking=True)

    def e2e_timed(run):
        """Device time of each step from the first copy in to the result on the host; the host
        waits for every step's result before it starts the next."""
        eev = []
        for i in range(args.steps):
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run(i)
            b_.record(stream)
            b_.synchronize()
            flush.zero_()
            eev.append((a, b_))
        return statistics.mean(a.elapsed_time(b_) for a, b_ in eev)

    for i in range(args.warmup):
        e2e_step(i)
        flush.zero_()
    barrier()
    e2e_eager_ms = rank_max(e2e_timed(e2e_step), dev)
    # the same calls captured as one CUDA graph per step, the copies from and to pinned host
    # memory included (each step keeps its own LRU time, as in the device-timed step)
    e2e_graphs = {}
    for i in range(args.steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            e2e_step(i)
        e2e_graphs[i] = g
    torch.cuda.synchronize()
    for i in range(min(args.warmup, args.steps)):
        e2e_graphs[i].replay()
    barrier()
    e2e_ms = rank_max(e2e_timed(lambda i: e2e_graphs[i].replay()), dev)
    e2e_value = replica_throughput(world, step_total, e2e_ms)
    del e2e_graphs

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        units = np.arange(U, dtype=np.int32)
        dt, thr = oracle_step(w, units)
        cpu = {"value": step_total / dt / 1e9, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": (f"one whole step (all {U} units): block scores, dual top-k selection, sparse attention, "
                          f"set-difference and LRU update ({N_SLOTS} slots), fp64"),
               "ms_per_step": dt * 1e3}

    cache.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": ms_median,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "queries_per_s": world * B / (ms * 1e-3),
            "pct_hbm_peak": 100.0 * (step_total / (ms * 1e-3) / 1e9) / peak,
            "config": {"workload": w["name"], "batch": B, "q_heads": Hq, "kv_heads": Hk, "context": L,
                       "page": 64, "subblock": 16, "k_q": k_q, "k_e": k_e, "resident_slots": N_SLOTS,
                       "step": "append+score+select+setdiff+lru+sparse_attn",
                       "launch": ("one CUDA graph per step (kernels chained by programmatic dependent launch); "
                                  "append + score as one kernel; " +
                                  ("select + setdiff + lru as one fused kernel" if args.bookkeeping == "fused" else
                                   "select, then setdiff + lru on a second stream beside the attention")),
                       "bytes_per_step": {kk: int(v) for kk, v in byts.items()},
                       "l2": ("no flush: each step reads ~0.81 GB of K/V pages and pooled-key sums, more "
                              "than the 129 MB L2, through evict-first loads" if args.l2 == "none" else
                              "256 MiB write between timed steps (outside the events)"),
                       "parallelism": f"replicas x{world}"},
            "roofline": {"kernel": "sparse_decode_attn (attn_split_kernel)", "bound": "hbm",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "us": attn_avg * 1e3,
                         "bytes_per_launch": byts["attn_kv"],
                         "traffic": measured_traffic() if B == 32 else None},
            "lazy_attn": lazy,
            "lazy_rag": rag,
            "lazy_prefill": prefill,
            "bf16_summaries": bf16_sum,
            "column_scores": colsc,
            "offload": offload,
            "per_config": {
                "1_tiny": tiny,
                "2_llama8b": {"workload": w["name"], "ms_per_step": ms, "GBps": value,
                              "pct_hbm_peak": 100.0 * (step_total / (ms * 1e-3) / 1e9) / peak,
                              "queries_per_s": world * B / (ms * 1e-3), "sparse_decode_attn_us": attn_avg * 1e3,
                              "sparse_decode_attn_frac": achieved / peak,
                              "lazy_rope_decode_attn_frac": lazy["frac"] if lazy else None,
                              "cpu_baseline": cpu},
                "3_lazy_rag": rag,
                "4_long262k_resident": resident262k,
                "5_nosa_traj": traj,
            },
            "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "launch": "one CUDA graph per step: copies in from pinned host memory, the API calls, "
                              "copies out; the host waits for each step's result",
                    "eager_ms_per_step": e2e_eager_ms},
            "gpu_launches": (4 if args.bookkeeping == "fused" else 6) * args.steps,
            "eager_ms_per_step": eager_ms,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
