#!/usr/bin/env python3
"""Decode-attention benchmark of the MOIRA sparse-decode library on GB300.

One step = every layer's selection + attention (the library's
moira_decode_step: score -> select -> attend per layer, 32 layers), captured
once in a CUDA graph and replayed.  Workload: a single Llama-3-8B-shaped
request at 131072 tokens (32 layers, 32 query / 8 KV heads, head dim 128,
16-token pages), seeded synthetic keys with planted high-mass pages.

Printed (rank 0, one JSON line): microseconds per step at gamma = 0.99 and
the achieved HBM GB/s on the bytes the step must read, next to the same
library at gamma = 0.98 and at gamma = 1 (dense, the same split-KV kernel
over every page), the attention kernel's roofline fraction, an end-to-end
figure through the host-buffer entry point, sampled SM clocks, and the
fp64 CPU oracle timed on a bounded sample of the same workload.

`--impl reference` times only the oracle (the CPU reference) on the host.
Under torchrun each rank runs an independent replica (the path has no
exchange step); the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/decode-attn step & achieved HBM GB/s at 128k ctx, γ=0.99 vs γ=1 dense"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) that the attention kernel moves per list entry,
# i.e. per kept (page, KV head) with its 4 KB of K and 4 KB of V, from
# one-pass ncu captures of dense launches (dram__bytes_read.sum +
# dram__bytes_write.sum divided by the entries), for k_attend's two block
# shapes (below 64 lists and from 64 lists on).  The digest names the kernel
# sources the captures were taken on; once they change the figure is withheld
# (traffic = null).
ATTEND_TRAFFIC = {"sources_sha256": "f19d2fe360e2296397ffc5eb05a5aadff974da4c2134f1ed150a30a38d29bfe8",
                  "many_lists_from": 64,
                  "dram_bytes_per_entry": {"few_lists": 8243.1, "many_lists": 8217.0}}
ATTEND_SOURCES = ("attend_core.cuh", "attend.cu", "moira_device.cuh", "moira_launch.h")   # k_attend's own

# The other configurations reported next to the headline (γ = 0.99 each).
OTHER_WORKLOADS = ("llama8b_32k", "serving_ragged", "stress_regimes")


def attend_sources_digest() -> str:
    h = hashlib.sha256()
    for f in ATTEND_SOURCES:
        with open(os.path.join(ROOT, "sparse_long_context_page_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (x itself when running alone)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 20 ms; stop() keeps those stamped inside the
    timed window (host wall clock, bracketing the timed region)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]),
                             {nm for nm, v in zip(names, parts[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        where = "inside the timed region"
        sel = rows
        if window is not None:
            sel = [r for r in rows if window[0] <= r[0] <= window[1]]
            if not sel:                      # region shorter than the sampling period
                sel = sorted(rows, key=lambda r: min(abs(r[0] - window[0]), abs(r[0] - window[1])))[:2]
                where = "nearest samples to a timed region shorter than the sampling period"
        reasons = set().union(*[r[3] for r in sel]) if sel else set()
        return {"sm_mhz": float(np.median([r[1] for r in sel])) if sel else None,
                "sm_max_mhz": float(max(r[2] for r in sel)) if sel else None,
                "samples": len(sel), "where": where, "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- bytes

def step_bytes(w, lengths: np.ndarray, gamma: float, summ_page_bytes: int | None = None):
    """Algorithmic bytes of one step: summaries of every full page (gamma < 1;
    bf16 rows unless a record size per page is given), K and V of the listed
    tokens, q in and fp32 out.  lengths: [L][B][Hkv]."""
    sp = w.spec
    d, S = sp.head_dim, sp.page_size
    L = w.seq_lens.astype(np.int64)
    F, T = L // S, (L % S != 0).astype(np.int64)
    tail_tok = L % S
    page_summ = sp.kv_heads * d * 2 if summ_page_bytes is None else summ_page_bytes
    per_layer_summ = int(F.sum()) * page_summ if gamma < 1.0 else 0
    lens = lengths.astype(np.int64)                                   # [L][B][Hkv]
    tokens = (lens - T[None, :, None]) * S + (T * tail_tok)[None, :, None]
    kv = tokens * d * 2 * 2                                           # K + V bf16
    q_b = sp.batch * sp.q_heads * d * 2
    o_b = sp.batch * sp.q_heads * d * 4
    layer = kv.sum(axis=(1, 2)) + per_layer_summ + q_b + o_b          # [L]
    pages_read = float(lens.sum()) / float((F + T).sum() * sp.kv_heads * sp.layers)
    return layer, int(layer.sum()), pages_read, {
        "summaries": per_layer_summ * sp.layers, "kv": int(kv.sum()),
        "q": q_b * sp.layers, "out": o_b * sp.layers}


# --------------------------------------------------------------------------- oracle timing

def oracle_sample(w, layers, gamma):
    """Host copies of the given layers and the oracle's own summaries."""
    from oracle import oracle
    idx = torch.tensor(layers, device=w.k_pool.device)

    def u16(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    k = u16(w.k_pool.index_select(0, idx))
    v = u16(w.v_pool.index_select(0, idx))
    q = u16(w.q.index_select(0, idx))
    summ = oracle.summaries(k.reshape(-1, 16, 128)).reshape(k.shape[0], k.shape[1], k.shape[2], 128)
    return q, summ, k, v


def time_oracle(w, layers, gamma, threads=0):
    from oracle import oracle
    q, summ, k, v = oracle_sample(w, layers, gamma)
    t0 = time.perf_counter()
    _, _, used = oracle.decode_step(q, summ, k, v, w.page_table, w.seq_lens, gamma, w.sm_scale,
                                    n_threads=threads)
    return time.perf_counter() - t0, used


# --------------------------------------------------------------------------- our arm

def workload_config(args, w, head):
    sp = w.spec
    return {"workload": f"{args.workload}: {sp.batch} request(s) x {int(w.seq_lens.max())} "
                        f"tokens, {sp.layers} layers, {sp.q_heads} q / {sp.kv_heads} kv heads, "
                        f"d=128, 16-token pages",
            "gamma": round(head, 4), "seed": args.seed, "summaries": args.summaries,
            "l2": "inputs larger than L2 (each step reads >5 GB of K/V)",
            "graph": f"whole {sp.layers}-layer step in one CUDA graph, replayed"}


def capture_step(st, gamma):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        st.step(gamma)                                   # eager warm-up outside capture
        with torch.cuda.graph(g, stream=s):
            st.step(gamma)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def time_graph(g, steps, warmup, world):
    for _ in range(warmup):
        g.replay()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    return e0.elapsed_time(e1) / steps, (t0, t1)         # ms per step, host window


def time_parts(st, gamma, steps, warmup):
    """In-graph durations of the two halves of a layer: select (score +
    select kernels) and attend.  Each half is captured for all layers in its
    own CUDA graph (per-layer lists kept apart) and replayed between CUDA
    events on the capturing stream.  Returns ms per layer for each."""
    L = st.layers
    lists_all = torch.zeros((L,) + tuple(st.lists.shape), dtype=torch.int32, device=st.device)
    graphs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for l in range(L):                                   # eager pass fills the lists
            st.select_layer(l, gamma, lists_all[l], st.lengths[l])
        for part in ("select", "attend"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for l in range(L):
                    if part == "select":
                        st.select_layer(l, gamma, lists_all[l], st.lengths[l])
                    else:
                        st.attend_layer(l, lists_all[l], st.lengths[l])
            graphs.append(g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    out = []
    for g in graphs:
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / steps / L)
    del graphs, lists_all
    return out[0], out[1]


def time_summaries(st, w, spb, peak, reps=3):
    """The page-summary kernel (off the decode step: once per layer after
    prefill): every page of every layer, CUDA events around the layers'
    launches; bytes = the keys read plus the summaries written."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st.summarize()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        st.summarize()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps / st.layers
    layer_bytes = w.k_pool[0].numel() * 2 + w.num_phys_pages * spb
    gbs = layer_bytes / (us * 1e3)
    return {"kernel": "k_summarize", "us_per_layer": round(us, 2), "bytes_per_layer": int(layer_bytes),
            "achieved": round(gbs, 1), "peak": peak[0], "unit": "GB/s", "frac": round(gbs / peak[0], 4),
            "peak_source": peak[1], "how": f"{st.layers} layers x {reps} repetitions between CUDA events"}


def time_score(st, steps, warmup):
    """In-graph duration of the page-scoring kernel alone, per layer: the
    layers' k_score launches captured in one CUDA graph and replayed between
    CUDA events on the capturing stream."""
    g = capture_fn(lambda: [st.score_layer(l) for l in range(st.layers)])
    ms, _ = time_graph(g, steps, warmup, 1)
    del g
    return ms / st.layers


def kernel_roofline(st, w, head, lengths, spb, peak, steps, warmup, two_launch=None):
    """The step's dominant kernel (k_attend: the decode step runs k_score,
    k_select and k_attend per layer), its algorithmic bytes per launch (K and
    V of the kept tokens, q, out) and its average in-graph launch duration,
    timed in a graph of attention launches alone (two_launch = time_parts'
    result)."""
    sp = w.spec
    per_layer, _, _, parts = step_bytes(w, lengths, head, spb)
    att_bytes = per_layer - parts["summaries"] / sp.layers      # K/V of kept tokens + q + out
    entries = float(lengths.reshape(sp.layers, -1).sum(axis=1).mean())     # list entries per launch
    score_ms = time_score(st, steps, warmup)
    if two_launch is None:
        two_launch = time_parts(st, head, steps, warmup)
    kernel, dur_ms = "k_attend", two_launch[1]
    shape = "many_lists" if sp.batch * sp.kv_heads >= ATTEND_TRAFFIC["many_lists_from"] else "few_lists"
    gbs = float(att_bytes.mean() / (dur_ms * 1e6))
    per_entry = ATTEND_TRAFFIC["dram_bytes_per_entry"].get(shape)
    traffic = None
    if per_entry and ATTEND_TRAFFIC["sources_sha256"] == attend_sources_digest():
        traffic = int(round(per_entry * entries))
    how = "graph of the layers' attention launches alone, CUDA events"
    return {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": peak[0], "unit": "GB/s",
            "frac": round(gbs / peak[0], 4), "peak_source": peak[1], "traffic": traffic,
            "traffic_how": (f"ncu DRAM bytes per list entry of a dense launch of the same kernel "
                            f"({shape.replace('_', ' ')}) x entries per launch" if traffic is not None else
                            "null: no ncu capture of the current attention sources"),
            "entries_per_launch": round(entries, 1), "bytes_per_launch": int(att_bytes.mean()),
            "duration_us": round(dur_ms * 1e3, 2), "duration_how": how,
            "score_us_per_layer": round(score_ms * 1e3, 2)}


def time_clustered_select(st, gamma, steps, warmup):
    """Per-layer duration of moira_select_clustered (the score and the cut in
    one launch, a thread-block cluster per list) where the batch fits the
    device's clusters, else None: the layers' calls captured in one CUDA
    graph, CUDA events.  A comparison only: the step selects with k_score +
    k_select."""
    import sparse_long_context_page_gb300 as moira
    if st.fmt != moira.SUMM_BF16 or not moira.select_cluster_size(st.shape, st.batch, st.max_pages):
        return None
    lists = torch.zeros_like(st.lists)
    lengths = torch.zeros_like(st.lengths)
    g = capture_fn(lambda: [st.select_layer_clustered(l, gamma, lists, lengths[l]) for l in range(st.layers)])
    ms, _ = time_graph(g, steps, warmup, 1)
    del g
    return ms / st.layers


def time_single_launch(st, gamma, steps, warmup):
    """Per-layer duration of moira_select_attend when it takes its one-launch
    form for this batch (k_score, then k_select_attend), else None: the
    layers' calls captured in one CUDA graph, CUDA events.  A comparison
    only: the decode step runs three launches per layer."""
    import sparse_long_context_page_gb300 as moira
    if not moira.select_attend_is_fused(st.shape, st.batch, st.max_pages):
        return None
    lists = torch.zeros_like(st.lists)
    out = torch.zeros_like(st.out)
    g = capture_fn(lambda: [st.select_attend_layer(l, gamma, lists, st.lengths[l], out[l])
                            for l in range(st.layers)])
    ms, _ = time_graph(g, steps, warmup, 1)
    del g
    return ms / st.layers


def load_balance(st, w, gamma):
    """Per-block attention times of one step, from the load-balance build of
    the library (the same kernels with %globaltimer stamps): per attention
    launch, the blocks' time from their plan to the end of their merges;
    max / mean over the blocks that hold pages, and the launch's span from
    the first start to the last end.  One eager step; median over layers."""
    import sparse_long_context_page_gb300 as moira
    from sparse_long_context_page_gb300 import build as B
    nb = moira.attend_grid_blocks()
    buf = torch.zeros((w.spec.layers, nb, 2), dtype=torch.int64, device=st.device)
    try:
        with moira._binding.library_variant(B.LIB_CTA_TIMES):
            moira._binding.set_cta_times(buf, w.spec.layers)
            try:
                st.step(gamma)
                torch.cuda.synchronize()
            finally:
                moira._binding.set_cta_times(None, 0)
    except moira.MoiraError as e:
        return {"error": str(e)}
    t = buf.cpu().numpy()
    ratios, spans = [], []
    for l in range(w.spec.layers):
        s, e = t[l, :, 0], t[l, :, 1]
        ok = s > 0
        d = (e[ok] - s[ok]).astype(np.float64)
        if len(d):
            ratios.append(float(d.max() / d.mean()))
            spans.append(float(e[ok].max() - s[ok].min()) / 1e3)
    return {"max_over_mean_block_time": round(float(np.median(ratios)), 4),
            "max_over_mean_worst_layer": round(float(np.max(ratios)), 4),
            "launch_span_us_median": round(float(np.median(spans)), 2),
            "how": "load-balance build (libmoira_cta_times.so): per attention launch, each block's time "
                   "from its plan to the end of its merges; max/mean over blocks with pages; median over layers"}


def other_workload(name, args, peak, local):
    """One more configuration at gamma = 0.99: the step (one graph) and the
    dense step, the step's HBM rate on the bytes it must read, and the
    dominant kernel's roofline."""
    import sparse_long_context_page_gb300 as moira
    from sparse_long_context_page_gb300 import workloads as W
    from sparse_long_context_page_gb300.state import DecodeState
    t0 = time.time()
    w = W.make_workload(name, seed=args.seed, device=f"cuda:{local}")
    st = DecodeState(w)
    st.summarize()
    spb = moira.summary_page_bytes(st.shape, moira.SUMM_BF16)
    torch.cuda.synchronize()
    gen_s = time.time() - t0
    head = float(np.float32(0.99))
    out = {}
    steps = max(3, args.steps // 2)
    for gm in (1.0, head):
        g = capture_step(st, gm)
        ms, _ = time_graph(g, steps, args.warmup, 1)
        del g
        out[gm] = ms
    assert moira.read_device_status(st.ws) == 0, f"device status word set during {name}"
    lengths = st.lengths.cpu().numpy()          # the gamma = 0.99 step ran last
    _, total, frac, _ = step_bytes(w, lengths, head, spb)
    roof = kernel_roofline(st, w, head, lengths, spb, peak, steps, args.warmup)
    res = {"workload": f"{name}: {w.spec.batch} request(s), {int(w.seq_lens.min())}..{int(w.seq_lens.max())} "
                       f"tokens, {w.spec.layers} layer(s), 32 q / 8 kv heads",
           "us_per_step": round(out[head] * 1e3, 2), "dense_us_per_step": round(out[1.0] * 1e3, 2),
           "speedup_vs_dense": round(out[1.0] / out[head], 3), "pages_read_fraction": round(frac, 4),
           "step_hbm_gbs": round(total / out[head] / 1e6, 1),
           "step_hbm_frac_of_measured": round(total / out[head] / 1e6 / peak[0], 4),
           "roofline": roof,
           "load_balance": load_balance(st, w, head)}
    log(f"[bench] {name}: generated in {gen_s:.1f}s; {out[head] * 1e3:.1f} us/step "
        f"({res['step_hbm_frac_of_measured']:.3f} of peak), dense {out[1.0] * 1e3:.1f}, "
        f"{roof['kernel']} {roof['frac']:.3f}")
    del st, w
    torch.cuda.empty_cache()
    return res


def capture_fn(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        fn()                                             # eager warm-up outside capture
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def compare_rules(st, w, head, results, args):
    """Coverage (gamma = head) against top-k and top-delta at equal pages read.
    k is the coverage rule's mean full pages per unit; delta is bisected (in
    log space) until the total pages match within 0.5%.  Each rule's step is
    captured and timed like the headline step; its output is compared with
    the dense (gamma = 1) step's: relative L2 per (layer, request, query head)."""
    import sparse_long_context_page_gb300 as moira
    sp = w.spec
    st.step(1.0)
    torch.cuda.synchronize()
    dense_out = st.out.clone()
    full = (st.seq_lens // 16).to(torch.float64)                         # full pages per request
    tails = int((st.seq_lens % 16 != 0).sum()) * sp.kv_heads * sp.layers

    def pages_of(rule, param):
        for l in range(sp.layers):
            st.select_layer_rule(l, rule, param, st.lists, st.lengths[l])
        torch.cuda.synchronize()
        return int(st.lengths.sum())

    target = pages_of(moira.RULE_COVERAGE, head)
    units = sp.layers * sp.batch * sp.kv_heads
    k = int(round((target - tails) / units))
    lo, hi = 1e-12, 1.0
    delta = 1e-3
    for _ in range(40):                                   # pages fall as delta grows
        delta = math.sqrt(lo * hi)
        n = pages_of(moira.RULE_TOPDELTA, delta)
        if abs(n - target) <= 0.005 * target:
            break
        if n > target:
            lo = delta
        else:
            hi = delta
    out = {}
    for name, rule, param in (("coverage", moira.RULE_COVERAGE, head), ("topk", moira.RULE_TOPK, float(k)),
                              ("topdelta", moira.RULE_TOPDELTA, delta)):
        g = capture_fn(lambda: st.step_rule(rule, param))
        ms, _ = time_graph(g, max(3, args.steps // 2), args.warmup, 1)
        g.replay()
        torch.cuda.synchronize()
        pages = int(st.lengths.sum())
        err = (st.out - dense_out).norm(dim=-1) / dense_out.norm(dim=-1).clamp_min(1e-30)
        err = err.flatten().double().cpu().numpy()
        out[name] = {"param": round(float(param), 8), "pages_read": pages,
                     "pages_fraction": round(pages / float(full.sum() * sp.kv_heads * sp.layers + tails), 4),
                     "us_per_step": round(ms * 1e3, 2),
                     "out_rel_l2_vs_dense": {"mean": float(np.mean(err)), "p99": float(np.percentile(err, 99)),
                                             "max": float(np.max(err))}}
        del g
    return out


def compare_summaries(w, head, args):
    """The headline step with each page-summary format: the bf16 mean key and
    its 8-bit and 2-bit mid-rise codes.  Per format: step time (graph), the
    in-graph selection and attention halves per layer, pages read, summary
    bytes per step, and the attention output against the dense (gamma = 1)
    step's (relative L2 per (layer, request, query head))."""
    import sparse_long_context_page_gb300 as moira
    from sparse_long_context_page_gb300.state import DecodeState
    sp = w.spec
    out = {}
    dense_out = None
    full = int((torch.from_numpy(w.seq_lens.astype(np.int64)) // 16).sum())     # full pages, one layer
    for name, fmt in (("bf16", moira.SUMM_BF16), ("q8", moira.SUMM_Q8), ("q2", moira.SUMM_Q2)):
        st = DecodeState(w, fmt=fmt)
        st.summarize()
        if dense_out is None:
            st.step(1.0)
            torch.cuda.synchronize()
            dense_out = st.out.clone()
        g = capture_fn(lambda: st.step(head))
        ms, _ = time_graph(g, max(3, args.steps // 2), args.warmup, 1)
        g.replay()
        torch.cuda.synchronize()
        assert moira.read_device_status(st.ws) == 0
        pages = int(st.lengths.sum())
        tails = int((st.seq_lens % 16 != 0).sum()) * sp.kv_heads * sp.layers
        err = (st.out - dense_out).norm(dim=-1) / dense_out.norm(dim=-1).clamp_min(1e-30)
        err = err.flatten().double().cpu().numpy()
        sel_ms, att_ms = time_parts(st, head, max(3, args.steps // 4), args.warmup)
        out[name] = {"us_per_step": round(ms * 1e3, 2),
                     "per_layer_us": {"select": round(sel_ms * 1e3, 2), "attend": round(att_ms * 1e3, 2)},
                     "summary_bytes_per_step": full * sp.layers * moira.summary_page_bytes(st.shape, fmt),
                     "pages_fraction": round(pages / float(full * sp.kv_heads * sp.layers + tails), 4),
                     "out_rel_l2_vs_dense": {"mean": float(np.mean(err)), "p99": float(np.percentile(err, 99)),
                                             "max": float(np.max(err))}}
        log(f"[bench] summaries {name}: {ms * 1e3:.1f} us/step, select {sel_ms * 1e3:.2f} us/layer, "
            f"pages {out[name]['pages_fraction']:.4f}, rel-L2 mean {np.mean(err):.4f}")
        del g, st
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import sparse_long_context_page_gb300 as moira
    from sparse_long_context_page_gb300 import workloads as W
    from sparse_long_context_page_gb300.state import DecodeState

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    moira.load_library()
    peak, peak_src = hbm_peak()
    t0 = time.time()
    over = {"layers": args.layers} if args.layers else {}
    if args.batch:
        over["batch"] = args.batch
        ctx = W.spec(args.workload).context
        if len(ctx) > 1:                      # per-request lengths: the first `batch` of them
            over["context"] = tuple(ctx[:args.batch])
    w = W.make_workload(args.workload, seed=args.seed, device=f"cuda:{local}", **over)
    fmt = {"bf16": moira.SUMM_BF16, "q8": moira.SUMM_Q8, "q2": moira.SUMM_Q2}[args.summaries]
    st = DecodeState(w, fmt=fmt)
    st.summarize()
    spb = moira.summary_page_bytes(st.shape, fmt)
    torch.cuda.synchronize()
    summ_kernel = time_summaries(st, w, spb, (peak, peak_src))
    log(f"[bench] workload {args.workload} generated in {time.time() - t0:.1f}s, "
        f"P={w.num_phys_pages} pages, KV {2 * w.k_pool.numel() * 2 / 2**30:.1f} GiB")
    sp = w.spec
    gammas = [float(np.float32(g)) for g in (args.gamma, 0.98, 1.0)]
    head = gammas[0]
    results = {}
    for gm in gammas:
        g = capture_step(st, gm)
        clocks = ClockSampler(local) if gm == head else None
        ms, window = time_graph(g, args.steps if gm == head else max(3, args.steps // 2), args.warmup, world)
        clk = clocks.stop(window) if clocks else None
        ms = max_over_ranks(ms, world)
        lengths = st.lengths.cpu().numpy()
        per_layer, total, frac, parts = step_bytes(w, lengths, gm, spb)
        results[gm] = dict(ms=ms, bytes=total, frac=frac, parts=parts, per_layer=per_layer,
                           lengths=lengths, clocks=clk)
        log(f"[bench] gamma={gm:.4f}: {ms * 1e3:.1f} us/step, {total / ms / 1e6:.0f} GB/s, "
            f"pages read {frac:.3f}")
        del g
    assert moira.read_device_status(st.ws) == 0, "device status word set during the benchmark"

    # dominant kernel and the layer's split (in-graph, CUDA events)
    two = time_parts(st, head, max(3, args.steps // 2), args.warmup)
    roof = kernel_roofline(st, w, head, results[head]["lengths"], spb, (peak, peak_src),
                           max(3, args.steps // 2), args.warmup, two_launch=two)
    sel_ms, att_ms = two
    single_ms = time_single_launch(st, head, max(3, args.steps // 2), args.warmup)
    clustered_ms = time_clustered_select(st, head, max(3, args.steps // 2), args.warmup)
    balance = load_balance(st, w, head)

    # the same step under the fixed-budget and relative-threshold rules, tuned
    # to read the same pages as coverage at the headline gamma; quality is the
    # attention output against the dense step's
    rules = compare_rules(st, w, head, results, args) if not args.no_rules else None
    formats = compare_summaries(w, head, args) if not args.no_rules else None

    # end to end: host q in, host out back, through moira_decode_step_host
    # (bf16 summaries; the low-bit formats are a profiling option here)
    e2e_ms = eager_ms = None
    q_host = out_host = None
    if fmt == moira.SUMM_BF16:
        q_host = w.q.cpu().pin_memory()
        out_host = torch.empty(st.out.shape, dtype=torch.float32).pin_memory()
        q_dev, out_dev = torch.empty_like(w.q), torch.empty_like(st.out)

        def host_step():
            moira.decode_step_host(st.shape, q_host, q_dev, w.k_pool, w.v_pool, st.summ, st.page_table,
                                   st.seq_lens, head, st.sm_scale, st.lists, st.lengths, out_dev,
                                   out_host, st.ws)

        # eager: the host enqueues the copies and the 3 x layers launches every step
        for _ in range(args.warmup):
            host_step()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            host_step()
        e1.record()
        torch.cuda.synchronize()
        eager_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
        # the same public call captured once (H2D copy of q from pinned memory, the
        # step, D2H copy of out) and replayed: how a serving loop runs it
        g_host = capture_fn(host_step)
        e2e_ms, _ = time_graph(g_host, args.steps, args.warmup, world)
        e2e_ms = max_over_ranks(e2e_ms, world)
        del g_host

    # CPU baseline: the oracle on a bounded sample of the same step (rank 0 only)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and fmt == moira.SUMM_BF16:
        n = max(1, min(sp.layers, args.cpu_layers))
        sample = list(range(n))
        secs, used = time_oracle(w, sample, head)
        secs1, _ = time_oracle(w, sample[:1], head, threads=1)
        cpu = {"value": secs / n * sp.layers * 1e6, "unit": "us/step", "cores": used,
               "kind": "oracle",
               "sample": f"layers {sample[0]}..{sample[-1]} of {sp.layers} (all {sp.kv_heads} KV heads, "
                         f"every request's full context) at gamma={head:.2f}; value = "
                         f"measured seconds x {sp.layers}/{n}; summaries precomputed (off-step)",
               "single_core": {"value": secs1 * sp.layers * 1e6, "unit": "us/step", "cores": 1,
                               "sample": f"layer {sample[0]} only, x {sp.layers}"}}

    hd = results[head]
    dense = results[1.0]
    launches_per_step = sp.layers * 3          # k_score, k_select, k_attend per layer

    line = {
        "metric": METRIC,
        "value": round(hd["ms"] * 1e3, 2),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(hd["ms"], 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded q/K/V, keys of 1-5% of pages per (layer, KV head) planted as "
                "c*qhat+N(0,1) with c~U[0,4] (stands in for RULER at 128k)",
        "config": workload_config(args, w, head),
        "hbm_gbs": round(hd["bytes"] / hd["ms"] / 1e6, 1),
        "hbm_frac_of_measured": round(hd["bytes"] / hd["ms"] / 1e6 / peak, 4),
        "hbm_frac_of_8tbs_nominal": round(hd["bytes"] / hd["ms"] / 1e6 / 8000.0, 4),
        "bytes_per_step": hd["bytes"],
        "bytes_parts": hd["parts"],
        "pages_read_fraction": {f"{g:.2f}": round(results[g]["frac"], 4) for g in gammas},
        "dense": {"gamma": 1.0, "us_per_step": round(dense["ms"] * 1e3, 2),
                  "hbm_gbs": round(dense["bytes"] / dense["ms"] / 1e6, 1),
                  "speedup_of_headline": round(dense["ms"] / hd["ms"], 3)},
        "gamma_0.98": {"us_per_step": round(results[gammas[1]]["ms"] * 1e3, 2),
                       "hbm_gbs": round(results[gammas[1]]["bytes"] / results[gammas[1]]["ms"] / 1e6, 1),
                       "speedup_vs_dense": round(dense["ms"] / results[gammas[1]]["ms"], 3)},
        "per_layer_us": {"step": round(hd["ms"] * 1e3 / sp.layers, 2),
                         "score": roof["score_us_per_layer"],
                         "select": round(sel_ms * 1e3, 2), "attend": round(att_ms * 1e3, 2),
                         "single_launch_layer": round(single_ms * 1e3, 2) if single_ms is not None else None,
                         "clustered_select": round(clustered_ms * 1e3, 2) if clustered_ms is not None else None,
                         "how": "in-graph, CUDA events: the step graph; graphs of the layers' scoring "
                                "launches alone; of their selections (k_score + k_select) and of their "
                                "attentions (k_attend) alone; and, for comparison (neither is used by the "
                                "step), moira_select_attend's one-launch layer and moira_select_clustered's "
                                "one-launch selection where the batch takes them"},
        "roofline": roof,
        "load_balance": balance,
        "summaries_kernel": summ_kernel,
        "e2e": ({"value": round(e2e_ms * 1e3, 2), "unit": "us/step",
                 "h2d_bytes_per_step": int(q_host.numel() * 2),
                 "d2h_bytes_per_step": int(out_host.numel() * 4),
                 "how": "moira_decode_step_host (q copied in from pinned host memory, out copied back) "
                        "captured in a CUDA graph and replayed; CUDA events",
                 "eager_value": round(eager_ms * 1e3, 2)} if e2e_ms is not None else None),
        "gpu_launches": args.steps * launches_per_step,
        "clocks": hd["clocks"],
        "cpu_baseline": cpu,
        "rules_at_equal_pages": rules,
        "summary_formats": formats,
        "other_workloads": None,
    }
    # the other configurations (the headline's buffers are freed first)
    if not args.no_others and world == 1:
        del st, w, q_host, out_host
        torch.cuda.empty_cache()
        line["other_workloads"] = [other_workload(nm, args, (peak, peak_src), local) for nm in OTHER_WORKLOADS
                                   if nm != args.workload]
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The fp64 oracle on the host cores, one bounded sample per step."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    from sparse_long_context_page_gb300 import workloads as W
    from oracle import oracle
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = W.make_workload(args.workload, seed=args.seed, device=dev)
    sp = w.spec
    head = float(np.float32(args.gamma))
    from oracle import oracle as O
    n_cached = min(sp.layers, 4)                 # host copies of 4 layers, every step
    q, summ, k, v = oracle_sample(w, list(range(n_cached)), head)
    times = []
    used = 1
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        _, _, used = O.decode_step(q, summ, k, v, w.page_table, w.seq_lens, head, w.sm_scale)
        if i >= args.warmup:
            times.append((time.perf_counter() - t0) * sp.layers / n_cached)
    v = float(np.mean(times)) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same generator and seed)",
        "config": workload_config(args, w, head),
        "cpu_baseline": {"value": round(v, 1), "unit": "us/step", "cores": used, "kind": "oracle",
                         "sample": f"layers 0..{n_cached - 1} (all KV heads, full context) per step, "
                                   f"x{sp.layers}/{n_cached} for a {sp.layers}-layer step"},
        "e2e": {"value": round(v, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b_128k")
    ap.add_argument("--gamma", type=float, default=0.99)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-layers", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rules", action="store_true",
                    help="skip the comparisons: top-k / top-delta at equal pages, and the summary formats")
    ap.add_argument("--layers", type=int, default=0,
                    help="fewer layers than the workload's (small profiling cases only)")
    ap.add_argument("--summaries", default="bf16", choices=["bf16", "q8", "q2"],
                    help="page-summary format of the measured step (bf16 is the headline; the "
                         "low-bit formats are for profiling: no e2e or CPU legs)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the other configurations (32k, serving, stress) after the headline")
    ap.add_argument("--batch", type=int, default=0,
                    help="fewer requests than the workload's (small profiling cases only)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)          # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
