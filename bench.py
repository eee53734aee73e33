"""Benchmark of the sparse-MLA layer hot path on one GB300 (or N, one process per GPU).

One step = one pass of the whole hot path over one batch: hs_indexer_scores -> hs_topk ->
hs_sparse_mla_fwd. The default line is the long prefill: one step is one 131,072-token sequence
as 64 sequential chunks of 2,048 tokens (64 x 128-d FP8 index heads, top-2048, 64 MLA heads,
paged FP8 KV), i.e. 192 launches; it also reports the per-chunk curve, the chunk where the indexer
overtakes attention, and the MTP-decode (64 requests x (1+3) tokens, contexts 16K-64K; indexer
and top-k as the one call hs_indexer_topk), chunked-prefill (2,048 tokens after 65,536) and
mixed-residency (32 requests, contexts 256K-1M with the older rows in pinned host memory; resolve
+ sparse MLA, 50 steps) workloads as extra keys. Other workloads are available for analysis with
--config 1|2|3|5, --kv-append, --kv-offload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 4]

Timing: W untimed steps, then K steps; before each timed step a 256 MB buffer is written so L2
(126 MB) holds nothing of the previous step; launches are bracketed by CUDA events on the
launching stream; the reported time is the mean per step, max over ranks. Per-kernel events give
each kernel's duration for the roofline. `e2e` repeats the step through the same API with the
step's inputs copied from pinned host memory and the outputs copied back inside the timed region.
`cpu_baseline` times the CPU oracle (test infrastructure, never on the product path) on a bounded
sample of the same workload. `--impl reference` times only that oracle, which is the reference
implementation here.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA layer tokens/s (indexer+top-k+attn); % of GB300 roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0   # dense e4m3 / bf16 tensor rate: nominal, and the per-MMA rate measured on GB300 (below)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ------------------------------------------------------------------------ distributed -------

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(base: int, rank: int) -> int:
    """Each rank decodes its own batch (weak scaling): a distinct, reproducible seed."""
    return base + 1000 * rank


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------ clocks ------------

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU works."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append({"sm": float(f[2]), "max": float(f[3]), "power": float(f[4]),
                             "hw": f[6], "hwt": f[7], "swt": f[8], "pcap": f[9]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["power"] > 0.5 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy), "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------------------------ traffic record -----

def kernel_source_digest(kernel: str) -> str:
    src = {"indexer": "indexer.cu", "topk": "topk.cu", "mla": "mla.cu", "resolve": "resolve.cu", "append": "append.cu"}[kernel]
    h = hashlib.sha256()
    for f in (src, "common.cuh"):
        with open(os.path.join(ROOT, "dsa_sparse_mla_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on this workload,
    or None if there is none or the kernel's source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "%s.%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    d = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != kernel_source_digest(kernel):
        return None
    return float(m.group(1))


# ------------------------------------------------------------------------ workloads ---------

def build_workload(config: int, seed: int, requests: int = 64):
    from dsa_sparse_mla_gb300 import inputs
    if config == 1:
        return inputs.config1(seed=seed)
    if config == 2:
        return inputs.config2(seed=seed, B=requests)
    if config == 3:
        return inputs.config3(seed=seed)
    raise SystemExit("--config %d: use 1, 2 or 3 for the indexer/top-k/MLA step (4, 5: analysis modes)" % config)


def final_tokens(w):
    """Index of each request's final query token (the one that sees the most tokens)."""
    return np.array([np.flatnonzero(w.token_req == r)[np.argmax(w.token_kvlen[w.token_req == r])]
                     for r in np.unique(w.token_req)])


def work_of(w, shared=False):
    """Algorithmic work per step. With shared index sets the indexer and top-k run for each
    request's final token only; attention rows are counted as min(n_t, k) per token either way
    (with a shared set a token may see up to three fewer)."""
    from dsa_sparse_mla_gb300 import costmodel as cm
    sel = final_tokens(w) if shared else np.arange(w.T)
    kvsum = int(w.token_kvlen[sel].astype(np.int64).sum())
    ctxsum = int(w.ctx.astype(np.int64).sum())
    rows = int(np.minimum(w.token_kvlen, w.topk).astype(np.int64).sum())
    return {"indexer": cm.indexer_work(w.Hi, w.Di, kvsum, ctxsum, len(sel)),
            "topk": cm.topk_work(kvsum, len(sel), w.topk), "mla": cm.mla_work(w.H, rows, w.T)}


# ------------------------------------------------------------------------ CPU oracle ---------

def oracle_sample(w, tokens, threads=0, shared=False):
    """Runs the CPU oracle (indexer -> top-k -> sparse MLA) on the given query tokens; returns
    the wall time in seconds. With shared index sets the indexer and top-k run for the final
    token of each request among them, and every token attends its request's set."""
    import oracle
    rows = np.asarray(tokens)
    sl = lambda a: np.ascontiguousarray(a[rows])
    sel = rows
    if shared:
        fin = set(final_tokens(w).tolist())
        sel = np.array([t for t in rows if t in fin])
    sf = lambda a: np.ascontiguousarray(a[sel])
    t0 = time.perf_counter()
    s = oracle.indexer_scores(sf(w.q_idx), sf(w.q_scale), sf(w.weights), w.k_cache, w.k_scale, w.block_table,
                              sf(w.token_req), sf(w.token_kvlen), ld=w.ld, threads=threads)
    idx = oracle.topk(s, sf(w.token_kvlen), w.topk, threads=threads)
    if shared:
        idx = oracle.shared_index_sets(idx, np.searchsorted(w.token_req[sel], w.token_req[rows]), sl(w.token_kvlen))
    oracle.sparse_mla(sl(w.q_mla), w.kv_pool, idx, w.softmax_scale, w.block_table, sl(w.token_req), threads=threads)
    return time.perf_counter() - t0


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------------------ GPU arm -----------

def run_ours(args):
    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import dsa_sparse_mla_gb300 as hs
    from dsa_sparse_mla_gb300.pipeline import DeviceWorkload, HotPath, SharedSetHotPath

    hs.load()
    peaks, peaks_kind = load_peaks()
    w = build_workload(args.config, rank_seed(args.config, rank), args.requests)
    dw = DeviceWorkload.from_host(w, dev)
    Path = SharedSetHotPath if args.shared_sets else HotPath
    # decode batches (the MTP-decode workload) run indexer and top-k as the one call hs_indexer_topk
    fused = args.config == 2 and not args.separate
    hp = Path(dw, fused=fused)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    work = work_of(w, args.shared_sets)
    wl_name = w.name + ("-shared-sets" if args.shared_sets else "")

    for _ in range(args.warmup):
        hp.step()
    torch.cuda.synchronize()
    if hs.hs_check_flag(hp.err):
        raise SystemExit("device error flag set during warm-up: 0x%x" % hs.hs_check_flag(hp.err))

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        e = ev[i]
        e[0].record(stream)
        if fused:
            hp.indexer_topk()
            e[1].record(stream)
            e[2].record(stream)
        else:
            hp.indexer()
            e[1].record(stream)
            hp.topk()
            e[2].record(stream)
        hp.mla()
        e[3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    t_step = [ev[i][0].elapsed_time(ev[i][3]) for i in range(K)]
    t_mla = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K)]
    ms_step = max_over_ranks(float(np.mean(t_step)), world, dev)
    fused_info = None
    if fused:
        # the per-kernel split (and the roofline of each) from the same steps run as separate calls
        t_it = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 0xFF)
            ev2[i][0].record(stream)
            hp.indexer()
            ev2[i][1].record(stream)
            hp.topk()
            ev2[i][2].record(stream)
        torch.cuda.synchronize()
        t_idx = [ev2[i][0].elapsed_time(ev2[i][1]) for i in range(K)]
        t_topk = [ev2[i][1].elapsed_time(ev2[i][2]) for i in range(K)]
        fused_info = {"indexer_topk_ms": round(float(np.mean(t_it)), 4),
                      "separate_calls_ms": round(float(np.mean(t_idx)) + float(np.mean(t_topk)), 4),
                      "note": "the step runs hs_indexer_topk (scores kept in L2 between the two kernels); "
                              "kernels.indexer and kernels.topk come from the same steps run as the two "
                              "separate calls"}
    else:
        t_idx = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
        t_topk = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    flag = hs.hs_check_flag(hp.err)

    # ---- end to end through host buffers (pinned), same API. Every step's inputs are copied in
    # from pinned host memory and its outputs copied back; the copies run on a second stream with
    # two buffer sets, so step i + 1's inputs and step i - 1's outputs move while step i computes,
    # as a serving loop would run them. No L2 flush: the K cache and KV pool are larger than L2.
    import dataclasses
    names_in = ("q_idx", "q_scale", "weights", "q_mla", "token_req", "token_kvlen")
    h_in = [t.cpu().pin_memory() for t in hp.step_inputs()]
    dws = [dw, dataclasses.replace(dw, **{nm: torch.empty_like(getattr(dw, nm)) for nm in names_in})]
    hps = [hp, Path(dws[1], fused=fused)]
    h_out = [[torch.empty_like(hp.out, device="cpu").pin_memory(), torch.empty_like(hp.lse, device="cpu").pin_memory()]
             for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    K2 = max(2, min(K, 200))
    cstream = torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]   # inputs of buffer set s copied in
    step_done = [torch.cuda.Event() for _ in range(2)]  # the step on set s finished
    out_done = [torch.cuda.Event() for _ in range(2)]   # outputs of set s copied out

    def copy_in(i):
        st = i & 1
        with torch.cuda.stream(cstream):
            if i >= 2:
                cstream.wait_event(step_done[st])  # step i - 2 read this set's inputs
            for dst, h in zip(hps[st].step_inputs(), h_in):
                dst.copy_(h, non_blocking=True)
            in_ready[st].record(cstream)

    def copy_out(i):
        st = i & 1
        with torch.cuda.stream(cstream):
            cstream.wait_event(step_done[st])
            h_out[st][0].copy_(hps[st].out, non_blocking=True)
            h_out[st][1].copy_(hps[st].lse, non_blocking=True)
            out_done[st].record(cstream)

    e2e_t = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier(world)
    torch.cuda.synchronize()
    e2e_t[0].record(stream)
    cstream.wait_event(e2e_t[0])
    copy_in(0)
    for i in range(K2):
        st = i & 1
        if i + 1 < K2:
            copy_in(i + 1)
        stream.wait_event(in_ready[st])
        if i >= 2:
            stream.wait_event(out_done[st])  # step i - 2's outputs are on the host before reuse
        hps[st].step(stream)
        step_done[st].record(stream)
        copy_out(i)
    stream.wait_event(out_done[0])
    stream.wait_event(out_done[1])
    e2e_t[1].record(stream)
    torch.cuda.synchronize()
    assert torch.equal(h_out[(K2 - 1) & 1][0].view(torch.int16), hp.out.cpu().view(torch.int16)), "e2e outputs differ"
    ms_e2e = max_over_ranks(e2e_t[0].elapsed_time(e2e_t[1]) / K2, world, dev)
    clk = clocks.stop() if rank == 0 else None

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    tokens = w.T * world
    ms = {"indexer": float(np.mean(t_idx)), "topk": float(np.mean(t_topk)), "mla": float(np.mean(t_mla))}
    hbm = float(peaks["hbm_gbs"])
    fp8 = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * FP8_PER_BF16
    bf16 = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    kern = {}
    for name in ("indexer", "topk", "mla"):
        wk = work[name]
        t = ms[name] * 1e-3
        gbs = wk.bytes / t / 1e9
        tf = wk.flops / t / 1e12
        t_roof = max(wk.bytes / (hbm * 1e9), wk.flops / ((fp8 if name == "indexer" else bf16) * 1e12))
        kern[name] = {"ms": round(ms[name], 4), "share": None, "bytes": wk.bytes, "flops": wk.flops,
                      "gbs": round(gbs, 1), "tflops": round(tf, 1), "roofline_ms": round(t_roof * 1e3, 4),
                      "roofline_frac": round(t_roof / t, 4)}
    tot = sum(ms.values())
    for name in kern:
        kern[name]["share"] = round(ms[name] / tot, 4)
    dom = max(ms, key=ms.get)
    wk = work[dom]
    t_dom = ms[dom] * 1e-3
    bytes_bound = wk.bytes / (hbm * 1e9) >= wk.flops / ((fp8 if dom == "indexer" else bf16) * 1e12)
    if bytes_bound:
        roof = {"bound": "hbm", "achieved": round(wk.bytes / t_dom / 1e9, 1), "peak": hbm, "unit": "GB/s"}
    else:
        pk = fp8 if dom == "indexer" else bf16
        roof = {"bound": "tensor", "achieved": round(wk.flops / t_dom / 1e12, 1), "peak": pk, "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["kernel"] = dom
    roof["peak_source"] = ("%s (MEASURED_PEAKS.json)" % peaks_kind) + (
        "; fp8 = sustained bf16 x 2 (an e4m3 M128N256K32 and a bf16 M128N256K16 tcgen05.mma both take "
        "128.4 cycles, so e4m3 does twice the MACs per cycle)" if (dom == "indexer" and not bytes_bound) else "")
    roof["traffic"] = recorded_traffic(dom, wl_name)
    layer_roof_ms = sum(kern[n]["roofline_ms"] for n in kern)

    # ---- CPU baseline: the oracle on a bounded sample of the same workload
    cpu = None
    if not args.no_cpu_baseline and world == 1:   # rank 0 at N = 1 only
        import oracle
        threads = oracle.num_threads(0)
        # bounded sample: whole passes over the batch's query tokens until about 10 s of CPU work
        sample = list(range(w.T))
        wall_cpu, passes = 0.0, 0
        while passes < 4 and (passes == 0 or wall_cpu < 10.0):
            wall_cpu += oracle_sample(w, sample, threads=0, shared=args.shared_sets)
            passes += 1
        cpu = {"value": round(passes * len(sample) / wall_cpu, 3), "unit": "tokens/s",
               "cores": min(threads, len(sample)), "kind": "oracle",
               "sample": "%d pass(es) over the batch's %d query tokens, full indexer+top-k+MLA in float64; "
                         "%.1f s wall on %s" % (passes, len(sample), wall_cpu, cpu_model())}
        # and on one core: the query tokens of the first request
        one = [int(t) for t in np.flatnonzero(w.token_req == w.token_req[0])]
        t1 = oracle_sample(w, one, threads=1, shared=args.shared_sets)
        cpu["single_thread"] = {"value": round(len(one) / t1, 3), "unit": "tokens/s",
                                "sample": "the first request's %d query tokens on one thread; %.1f s wall"
                                          % (len(one), t1)}

    line = {"metric": METRIC, "value": round(tokens / (ms_step * 1e-3), 1), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+bf16", "data": "synthetic",
            "config": {"workload": wl_name, "requests": w.B, "query_tokens": w.T,
                       "ctx": "U{16384..65536}" if args.config == 2 else int(w.ctx.max()),
                       "index_heads": w.Hi, "index_dim": w.Di, "topk": w.topk, "mla_heads": w.H, "page": 64,
                       "l2": "256 MB write between timed steps (inputs also > L2)", "parallelism": "dp%d" % world,
                       "indexer_topk": "one call (hs_indexer_topk)" if fused else "two calls",
                       "index_sets": ("shared: each request's final query token's top-k, reused by its other query "
                                      "tokens up to their own visible length") if args.shared_sets else "per query token"},
            "roofline": roof,
            "layer_roofline_frac": round(layer_roof_ms / tot, 4),
            "kernels": kern,
            "indexer_topk_fused": fused_info,
            "e2e": {"value": round(tokens / (ms_e2e * 1e-3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4), "steps": K2,
                    "overlap": "inputs of step i+1 in and outputs of step i-1 out on a second stream during step i "
                               "(two buffer sets)", "l2": "no flush (K cache and KV pool > L2)"},
            "gpu_launches": 3 * K, "cpu_baseline": cpu, "clocks": clk, "wall_s_timed_region": round(wall, 3),
            "device_flag": flag}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------------ peaks ---------------

def measure_fp8_peak(seconds: float = 3.0):
    """Dense e4m3 GEMM rate of this GPU through cuBLASLt (torch._scaled_mm, 8192^3, unit scales,
    bf16 output, 2 n^3 FLOPs): the best of 10 launches (burst) and launches back to back for about
    `seconds` (sustained, under the power cap). None if the call is unavailable."""
    import torch
    n = 8192
    try:
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn).t()   # column-major B
        one = torch.ones((), dtype=torch.float32, device="cuda")
        f = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
    except (RuntimeError, AttributeError, TypeError) as e:  # pragma: no cover - depends on the build
        return {"error": str(e).splitlines()[0][:200]}
    flop = 2.0 * n ** 3
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        f()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    count = 0
    t0 = time.perf_counter()
    e0.record()
    while time.perf_counter() - t0 < seconds:
        for _ in range(10):
            f()
        count += 10
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    del a, b
    return {"fp8_tflops": round(flop / (best * 1e-3) / 1e12, 1),
            "fp8_tflops_sustained": round(flop * count / (e0.elapsed_time(e1) * 1e-3) / 1e12, 1),
            "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3 (2 n^3 FLOPs): best of 10 (burst) and "
                   "%d launches back to back (sustained)" % count}


def kernel_rooflines(works, ms, hbm, fp8, bf16):
    """Per kernel: algorithmic bytes and FLOPs summed over `works` (one dict of costmodel Work per
    launch group), measured ms (summed likewise), roofline ms (per launch the slower of bytes at
    HBM bandwidth and FLOPs at the kernel's tensor peak, summed) and the bound that dominates."""
    out = {}
    for name in ("indexer", "topk", "mla"):
        peak = fp8 if name == "indexer" else bf16
        b = sum(w[name].bytes for w in works)
        fl = sum(w[name].flops for w in works)
        t_bytes = sum(w[name].bytes / (hbm * 1e9) for w in works)
        t_flops = sum(w[name].flops / (peak * 1e12) for w in works)
        t_roof = sum(max(w[name].bytes / (hbm * 1e9), w[name].flops / (peak * 1e12)) for w in works)
        t = ms[name] * 1e-3
        out[name] = {"ms": round(ms[name], 4), "bytes": b, "flops": fl, "gbs": round(b / t / 1e9, 1),
                     "tflops": round(fl / t / 1e12, 1), "roofline_ms": round(t_roof * 1e3, 4),
                     "roofline_frac": round(t_roof / t, 4), "bound": "hbm" if t_bytes >= t_flops else "tensor"}
    tot = sum(ms.values())
    for name in out:
        out[name]["share"] = round(ms[name] / tot, 4)
    return out


def measure_hot_path(w, steps: int, warmup: int, dev, peaks, fused: bool = False):
    """One workload's step (indexer -> top-k -> sparse MLA on all its query tokens): mean time per
    step and per kernel over `steps` timed steps, a 256 MB L2 flush before each. With `fused`
    (decode batches) the step's value is also measured with hs_indexer_topk in place of the two
    calls."""
    import torch
    import dsa_sparse_mla_gb300 as hs
    from dsa_sparse_mla_gb300.pipeline import DeviceWorkload, HotPath
    hp = HotPath(DeviceWorkload.from_host(w, dev), fused=fused)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        hp.step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 0xFF)
        e = ev[i]
        e[0].record(stream)
        hp.indexer()
        e[1].record(stream)
        hp.topk()
        e[2].record(stream)
        hp.mla()
        e[3].record(stream)
    torch.cuda.synchronize()
    ms = {n: float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)]))
          for j, n in enumerate(("indexer", "topk", "mla"))}
    step_ms = float(np.mean([ev[i][0].elapsed_time(ev[i][3]) for i in range(steps)]))
    kern = kernel_rooflines([work_of(w)], ms, peaks["hbm"], peaks["fp8"], peaks["bf16"])
    out = {"value": round(w.T / (step_ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(step_ms, 4),
           "steps": steps, "query_tokens": w.T, "kernels": kern,
           "layer_roofline_frac": round(sum(k["roofline_ms"] for k in kern.values()) / sum(ms.values()), 4)}
    if fused:
        evf = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 0xFF)
            evf[i][0].record(stream)
            hp.indexer_topk()
            evf[i][1].record(stream)
            hp.mla()
            evf[i][2].record(stream)
        torch.cuda.synchronize()
        f_step = float(np.mean([evf[i][0].elapsed_time(evf[i][2]) for i in range(steps)]))
        f_it = float(np.mean([evf[i][0].elapsed_time(evf[i][1]) for i in range(steps)]))
        out["indexer_topk_fused"] = {"value": round(w.T / (f_step * 1e-3), 1), "unit": "tokens/s",
                                     "ms_per_step": round(f_step, 4), "indexer_topk_ms": round(f_it, 4),
                                     "separate_calls_ms": round(ms["indexer"] + ms["topk"], 4),
                                     "note": "the same step with hs_indexer_topk (scores kept in L2) in place "
                                             "of hs_indexer_scores + hs_topk"}
    out["device_flag"] = hs.hs_check_flag(hp.err)
    del hp, flush
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------ analysis modes ----

def _timed(fn, flush, reps):
    """Median device time (ms) of fn() over reps runs, L2 flushed before each, CUDA events."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    fn()
    torch.cuda.synchronize()
    for a, b in ev:
        flush.fill_(1)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return float(statistics.median(a.elapsed_time(b) for a, b in ev))


def long_prefill_cpu_sample(chunks, threads=0):
    """The CPU oracle on a stratified sample of the long-prefill pass: 16 query tokens evenly spaced
    in each of 8 evenly spaced chunks (3, 11, ..., 59), so that the sampled positions' mean cost is
    the pass's mean cost per token. Returns (tokens, wall seconds)."""
    picks = [c for c in range(3, len(chunks), 8)]
    tok = np.linspace(0, chunks[0].T - 1, 16).round().astype(int).tolist()
    wall = 0.0
    for c in picks:
        wall += oracle_sample(chunks[c], tok, threads=threads)
    return len(picks) * len(tok), wall


def run_long_prefill_pass(args):
    """The benchmark line: one step is one long-prefill pass, 131,072 tokens of one sequence as 64
    sequential chunks of 2,048, each chunk through hs_indexer_scores -> hs_topk ->
    hs_sparse_mla_fwd (192 launches). The cache and every chunk's query inputs are resident in
    HBM when the timed region starts; each chunk's queries see every earlier token and themselves.
    Reports whole-pass tokens/s, the per-chunk time curve with the chunk at which the indexer
    overtakes attention, the roofline of the dominant kernel over the pass, the MTP-decode and
    chunked-prefill workloads as extra keys, e2e through host buffers and the CPU oracle."""
    import dataclasses
    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import dsa_sparse_mla_gb300 as hs
    from dsa_sparse_mla_gb300 import inputs
    from dsa_sparse_mla_gb300.pipeline import LongPrefillPass

    hs.load()
    peaks, peaks_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    bf16 = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    fp8m = measure_fp8_peak() if (rank == 0 and not args.no_peak) else None
    if fp8m and "fp8_tflops_sustained" in fp8m:
        fp8, fp8_src = fp8m["fp8_tflops_sustained"], "measured in this run (sustained e4m3 GEMM)"
    else:
        fp8, fp8_src = bf16 * FP8_PER_BF16, "derived: sustained bf16 x 2 (no e4m3 GEMM available)"
    pk = {"hbm": hbm, "fp8": fp8, "bf16": bf16}

    t0 = time.perf_counter()
    only = sorted(set(int(c) for c in args.chunks.split(","))) if args.chunks else None
    chunks = inputs.config4_pass(seed=rank_seed(4, rank), chunks=only)
    chunk_ids = only if only else list(range(len(chunks)))
    gen_s = time.perf_counter() - t0
    n, T = len(chunks), chunks[0].T
    total_tokens = n * T
    lp = LongPrefillPass(chunks, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    works = [work_of(w) for w in chunks]

    for _ in range(args.warmup):
        lp.step()
    torch.cuda.synchronize()
    if hs.hs_check_flag(lp.err):
        raise SystemExit("device error flag set during warm-up: 0x%x" % hs.hs_check_flag(lp.err))

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(1 + 3 * n)] for _ in range(K)]
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        e = ev[i]
        e[0].record(stream)
        for c in range(n):
            lp.indexer(c)
            e[1 + 3 * c].record(stream)
            lp.topk(c)
            e[2 + 3 * c].record(stream)
            lp.mla(c)
            e[3 + 3 * c].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    t_pass = [ev[i][0].elapsed_time(ev[i][3 * n]) for i in range(K)]
    per = np.array([[[ev[i][3 * c + j].elapsed_time(ev[i][3 * c + j + 1]) for j in range(3)] for c in range(n)]
                    for i in range(K)]).mean(axis=0)          # [chunk, kernel] ms
    ms_step = max_over_ranks(float(np.mean(t_pass)), world, dev)
    flag = hs.hs_check_flag(lp.err)

    # ---- end to end: every chunk's query inputs copied in from pinned host memory and its output
    # and LSE copied back, chunk by chunk, on two copy streams (in, out) with two device buffer
    # sets, so chunk c + 1's inputs and chunk c - 1's outputs move while chunk c computes
    h_in = [[t.cpu().pin_memory() for t in lp.step_inputs(c)] for c in range(n)]
    h_out = [(torch.empty_like(lp.out[c], device="cpu").pin_memory(),
              torch.empty_like(lp.lse[c], device="cpu").pin_memory()) for c in range(n)]
    d_in = [[torch.empty_like(t) for t in lp.step_inputs(0)] for _ in range(2)]
    d_out = [(torch.empty_like(lp.out[0]), torch.empty_like(lp.lse[0])) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for row in h_in for t in row)
    d2h = sum(a.numel() * a.element_size() + b.numel() * b.element_size() for a, b in h_out)
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    # timing events of each chunk's copies, to report the achieved copy rates
    t_in = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    t_out = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]

    def copy_in(c):
        st = c & 1
        with torch.cuda.stream(cin):
            if c >= 2:
                cin.wait_event(done[st])          # chunk c - 2 has finished reading this set
            t_in[c][0].record(cin)
            for dst, h in zip(d_in[st], h_in[c]):
                dst.copy_(h, non_blocking=True)
            t_in[c][1].record(cin)
            in_ready[st].record(cin)

    def copy_out(c):
        st = c & 1
        with torch.cuda.stream(cout):
            cout.wait_event(done[st])
            t_out[c][0].record(cout)
            h_out[c][0].copy_(d_out[st][0], non_blocking=True)
            h_out[c][1].copy_(d_out[st][1], non_blocking=True)
            t_out[c][1].record(cout)
            out_done[st].record(cout)

    e2e_t = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier(world)
    torch.cuda.synchronize()
    e2e_t[0].record(stream)
    cin.wait_event(e2e_t[0])
    copy_in(0)
    for c in range(n):
        st = c & 1
        if c + 1 < n:
            copy_in(c + 1)
        stream.wait_event(in_ready[st])
        if c >= 2:
            stream.wait_event(out_done[st])       # chunk c - 2's outputs are on the host
        q_idx, q_scale, weights, q_mla, kvlen = d_in[st]
        lp.indexer(c, q_idx=q_idx, q_scale=q_scale, weights=weights, token_kvlen=kvlen)
        lp.topk(c, token_kvlen=kvlen)
        lp.mla(c, q_mla=q_mla, out=d_out[st][0], lse=d_out[st][1])
        done[st].record(stream)
        copy_out(c)
    stream.wait_event(out_done[0])
    stream.wait_event(out_done[1])
    e2e_t[1].record(stream)
    torch.cuda.synchronize()
    assert torch.equal(h_out[n - 1][0].view(torch.int16), lp.out[n - 1].cpu().view(torch.int16)), "e2e outputs differ"
    ms_e2e = max_over_ranks(e2e_t[0].elapsed_time(e2e_t[1]), world, dev)
    ms_in = sum(a.elapsed_time(b) for a, b in t_in)
    ms_out = sum(a.elapsed_time(b) for a, b in t_out)
    clk = clocks.stop() if rank == 0 else None
    del h_in, h_out, d_in, d_out

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    ms = {name: float(per[:, j].sum()) for j, name in enumerate(("indexer", "topk", "mla"))}
    kern = kernel_rooflines(works, ms, hbm, fp8, bf16)
    dom = max(ms, key=ms.get)
    kd = kern[dom]
    if kd["bound"] == "hbm":
        roof = {"bound": "hbm", "achieved": kd["gbs"], "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": kd["tflops"], "peak": fp8 if dom == "indexer" else bf16,
                "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["kernel"] = dom
    roof["achieved_over"] = "the kernel's 64 launches of one pass: algorithmic work / summed launch time"
    roof["peak_source"] = ("HBM and bf16 %s (MEASURED_PEAKS.json); e4m3 %s" % (peaks_kind, fp8_src))
    tr = recorded_traffic(dom, "long-prefill-chunk63") if chunk_ids[-1] == 63 else None
    roof["traffic"] = tr
    if tr is not None:
        roof["traffic_launch"] = "chunk 63 (2048 queries over up to 131,072 keys), one launch"
        roof["algorithmic_bytes_launch"] = works[-1][dom].bytes
    curve = [{"chunk": chunk_ids[c], "ctx_end": int((chunk_ids[c] + 1) * T), "indexer_ms": round(float(per[c, 0]), 4),
              "topk_ms": round(float(per[c, 1]), 4), "mla_ms": round(float(per[c, 2]), 4),
              "indexer_tflops": round(works[c]["indexer"].flops / (per[c, 0] * 1e9), 1),
              "mla_gbs": round(works[c]["mla"].bytes / (per[c, 2] * 1e6), 1)} for c in range(n)]
    cross = next((e["chunk"] for e in curve if e["indexer_ms"] > e["mla_ms"]), None)

    # ---- the other workloads of the same hot path, measured in the same run
    others = {}
    if not args.no_extra:
        for cfg, steps in ((2, 200), (3, 20)):
            w = build_workload(cfg, rank_seed(cfg, 0))
            others[w.name] = measure_hot_path(w, steps, 3, dev, pk, fused=cfg == 2)
            del w
        if world == 1:  # the mixed-residency decode (its host tier is 13 GB of pinned memory per process)
            hsp = measure_hisparse(32, 50)
            others[hsp["workload"]] = hsp

    # ---- CPU baseline: the oracle on a stratified sample of the pass
    cpu = None
    if not args.no_cpu_baseline and world == 1 and only is None:
        import oracle
        threads = oracle.num_threads(0)
        ntok, wall_cpu = long_prefill_cpu_sample(chunks)
        cpu = {"value": round(ntok / wall_cpu, 3), "unit": "tokens/s", "cores": min(threads, 16), "kind": "oracle",
               "sample": "16 query tokens evenly spaced in each of chunks 3, 11, ..., 59 of the pass (%d tokens, "
                         "their mean cost is the pass's), full indexer+top-k+MLA in float64; %.1f s wall on %s"
                         % (ntok, wall_cpu, cpu_model())}

    line = {"metric": METRIC, "value": round(total_tokens * world / (ms_step * 1e-3), 1), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+bf16",
            "data": "synthetic",
            "config": {"workload": "long-prefill-128K" if only is None else "long-prefill-chunks-" + args.chunks,
                       "sequence_tokens": total_tokens, "chunks": n,
                       "chunk_tokens": T, "index_heads": chunks[0].Hi, "index_dim": chunks[0].Di,
                       "topk": chunks[0].topk, "mla_heads": chunks[0].H, "page": 64,
                       "step": "one whole pass: 64 chunks x (indexer, top-k, sparse MLA)",
                       "l2": "256 MB write before each timed pass (each pass reads 10.8 GB of query inputs)",
                       "parallelism": "dp%d" % world},
            "roofline": roof,
            "layer_roofline_frac": round(sum(k["roofline_ms"] for k in kern.values()) / sum(ms.values()), 4),
            "kernels": kern,
            "peaks": dict(fp8m or {}, hbm_gbs=hbm, bf16_tflops_sustained=bf16),
            "chunk_curve": curve, "indexer_overtakes_attention_at_chunk": cross,
            "crossover_ctx_tokens": None if cross is None else (cross + 1) * T,
            "other_workloads": others,
            "e2e": {"value": round(total_tokens * world / (ms_e2e * 1e-3), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4), "steps": 1,
                    "copies": {"h2d_ms": round(ms_in, 2), "d2h_ms": round(ms_out, 2),
                               "h2d_gbs": round(h2d / (ms_in * 1e6), 1), "d2h_gbs": round(d2h / (ms_out * 1e6), 1),
                               "note": "summed durations of the chunks' copies on their own streams (they overlap "
                                       "the kernels, so a sum above ms_per_step of the device pass means the "
                                       "pass is copy-bound)"},
                    "overlap": "chunk c+1's inputs in and chunk c-1's outputs out on two copy streams while chunk c "
                               "computes (two device buffer sets)"},
            "gpu_launches": 3 * n * K, "cpu_baseline": cpu, "clocks": clk, "wall_s_timed_region": round(wall, 3),
            "inputs_generated_s": round(gen_s, 1), "device_flag": flag}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_kv_append(args):
    """FP8 KV append of N new tokens (512-d latent + 64-d RoPE + 128-d indexer key, bf16) spread over
    64 requests of a paged pool with a random block table; median device time with an L2 flush
    before each launch. Algorithmic bytes per token: reads 1024 + 128 + 256 (inputs) + 12
    (request, position, block entry), writes 656 (row) + 128 (key) + 4 (key scale)."""
    import torch
    import dsa_sparse_mla_gb300 as hs
    torch.cuda.set_device(0)
    hs.load()
    N, B = args.kv_append, 64
    pages = (N + B * 64 - 1) // (B * 64)
    nblk = B * pages
    g = torch.Generator(device="cuda").manual_seed(0)
    latent = torch.randn(N, 512, device="cuda", generator=g).to(torch.bfloat16)
    rope = torch.randn(N, 64, device="cuda", generator=g).to(torch.bfloat16)
    key = torch.randn(N, 128, device="cuda", generator=g).to(torch.bfloat16)
    bt = torch.randperm(nblk, device="cuda", generator=g).view(B, pages).int()
    ar = torch.arange(N, device="cuda", dtype=torch.int32)
    req, pos = (ar % B).contiguous(), (ar // B).contiguous()
    kv = torch.empty((nblk * 64, 656), dtype=torch.uint8, device="cuda")
    kc = torch.empty((nblk, 64, 128), dtype=torch.uint8, device="cuda")
    ks = torch.empty((nblk, 64), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fn = lambda: hs.hs_kv_append(req, pos, bt, err, latent=latent, rope=rope, kv_pool=kv, index_key=key, k_cache=kc,
                                 k_scale=ks)
    t = _timed(fn, flush, max(args.reps, 5))
    per_tok = 1024 + 128 + 256 + 12 + 656 + 128 + 4
    gbs = N * per_tok / (t * 1e6)
    peaks, kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    line = {"metric": "FP8 KV append (quantise + paged write) tokens/s", "tokens": N, "requests": B,
            "value": round(N / (t * 1e-3), 1), "unit": "tokens/s", "ms": round(t, 4),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                         "bytes_per_token": per_tok, "peak_source": "%s (MEASURED_PEAKS.json)" % kind,
                         "traffic": recorded_traffic("append", "kv-append-%d" % N)},
            "device_flag": hs.hs_check_flag(err), "l2": "256 MB write before each timed launch", "data": "synthetic"}
    print(json.dumps(line), flush=True)


def run_kv_offload(args):
    """HiSparse write side: N complete pages (64 rows x 656 B) spread over 8 layers x 32 requests,
    copied from the device pools into pinned host rows by hs_kv_offload; median device time with an
    L2 flush before each launch. For context, the copy engine's rate on one contiguous
    device-to-host copy of the same bytes is measured in the same run."""
    import torch
    import dsa_sparse_mla_gb300 as hs
    from dsa_sparse_mla_gb300.pipeline import pinned_uint8
    torch.cuda.set_device(0)
    hs.load()
    L, B = 8, 32
    pages = max(1, (args.kv_offload + L * B - 1) // (L * B))
    n = L * B * pages
    g = torch.Generator(device="cuda").manual_seed(0)
    nblk = B * pages
    pools = [torch.randint(0, 256, (nblk * 64, 656), dtype=torch.uint8, device="cuda", generator=g) for _ in range(L)]
    bt = torch.randperm(nblk, device="cuda", generator=g).view(B, pages).int()
    hosts = [pinned_uint8(pages * 64 * 656) for _ in range(L * B)]
    ar = torch.arange(n, device="cuda", dtype=torch.int32)
    layer, req, page = (ar // (B * pages)).contiguous(), ((ar // pages) % B).contiguous(), (ar % pages).contiguous()
    seq = torch.full((B,), pages * 64, dtype=torch.int32, device="cuda")
    pp = torch.tensor([p.data_ptr() for p in pools], dtype=torch.int64, device="cuda")
    hp = torch.tensor([h.ctypes.data for h in hosts], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fn = lambda: hs.hs_kv_offload(pp, hp, layer, req, page, bt, seq, err, R=nblk * 64)
    t = _timed(fn, flush, max(args.reps, 5))
    nbytes = n * 64 * 656
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    t_ce = _timed(lambda: host.copy_(dev, non_blocking=True), flush, 5)
    line = {"metric": "KV offload (device pages -> pinned host) GB/s", "pages": n, "layers": L, "requests": B,
            "bytes": nbytes, "ms": round(t, 4), "value": round(nbytes / (t * 1e6), 1), "unit": "GB/s",
            "copy_engine_gbs": round(nbytes / (t_ce * 1e6), 1), "frac_of_copy_engine": round(t_ce / t, 3),
            "device_flag": hs.hs_check_flag(err), "l2": "256 MB write before each timed launch", "data": "synthetic"}
    print(json.dumps(line), flush=True)


def run_hisparse(args):
    """HiSparse mixed-residency decode: 32 requests, contexts U{262144..1048576}, the last 4,096
    tokens resident, older rows in pinned host memory, 4,096 hot slots per request; 50 steps of
    resolve + sparse MLA over the Zipf(1.1) index stream with 80 % step-to-step overlap."""
    import torch
    torch.cuda.set_device(0)
    line = {"metric": "HiSparse decode tokens/s (resolve+attn)"}
    line.update(measure_hisparse(args.hisparse_requests, args.hisparse_steps))
    print(json.dumps(line), flush=True)


def measure_hisparse(requests: int, nsteps: int) -> dict:
    """The mixed-residency decode measured on the current device (see run_hisparse)."""
    import torch
    import dsa_sparse_mla_gb300 as hs
    from dsa_sparse_mla_gb300 import costmodel as cm, inputs
    from dsa_sparse_mla_gb300.pipeline import DeviceHiSparse, pinned_uint8
    hs.load()
    t0 = time.perf_counter()
    hw = inputs.config5(B=requests, steps=nsteps, host_alloc=pinned_uint8)
    gen_s = time.perf_counter() - t0
    dh = DeviceHiSparse(hw)
    stream = torch.cuda.current_stream()
    # one-time setup: the GPU's first read of each host page is slow, so the tier is mapped first
    t_touch = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    t_touch[0].record(stream)
    dh.touch_host()
    t_touch[1].record(stream)
    steps = hw.idx.shape[0]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    counters = []
    torch.cuda.synchronize()
    for st in range(steps):
        e = ev[st]
        e[0].record(stream)
        dh.resolve(st)
        e[1].record(stream)
        dh.mla(st)
        e[2].record(stream)
        counters.append(dh.counters.sum(0))
    torch.cuda.synchronize()
    cnt = torch.stack(counters).cpu().numpy()          # [steps, 3] resident, hit, miss
    t_res = np.array([e[0].elapsed_time(e[1]) for e in ev])
    t_mla = np.array([e[1].elapsed_time(e[2]) for e in ev])
    # the host link's measured rate: one 1 GiB copy-engine copy from pinned host memory, best of 5
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    best = float("inf")
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    link_gbs = (1 << 30) / (best * 1e6)
    del src, dst
    warm = slice(1, steps)
    miss_bytes = cnt[:, 2].astype(np.float64) * 656
    mla_w = cm.mla_work(hw.H, hw.B * hw.k, hw.B)
    line = {"workload": hw.name, "requests": hw.B,
            "steps": steps, "topk": hw.k, "hot_slots": hw.S, "mla_heads": hw.H,
            "value": round(hw.B * (steps - 1) / ((t_res[warm] + t_mla[warm]).sum() * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step_warm": round(float((t_res[warm] + t_mla[warm]).mean()), 4),
            "resolve_ms_warm": round(float(t_res[warm].mean()), 4), "mla_ms_warm": round(float(t_mla[warm].mean()), 4),
            "step0_cold": {"resolve_ms": round(float(t_res[0]), 4), "mla_ms": round(float(t_mla[0]), 4),
                           "misses": int(cnt[0, 2]), "host_read_gbs": round(miss_bytes[0] / (t_res[0] * 1e6), 1)},
            "resolve_ms_steps": [round(float(x), 3) for x in t_res[:12]],
            "resolve_ms_warm_p50": round(float(np.percentile(t_res[warm], 50)), 4),
            "resolve_ms_warm_p95": round(float(np.percentile(t_res[warm], 95)), 4),
            "host_link": {"copy_engine_h2d_gbs": round(link_gbs, 1),
                          "how": "one 1 GiB copy from pinned host memory to the device, best of 5",
                          "resolve_frac_warm": round(float((miss_bytes[warm] / (t_res[warm] * 1e6)).mean()) / link_gbs, 4),
                          "resolve_frac_step0": round(miss_bytes[0] / (t_res[0] * 1e6) / link_gbs, 4)},
            "per_step_warm": {"hits": round(float(cnt[warm, 1].mean()), 1), "misses": round(float(cnt[warm, 2].mean()), 1),
                              "resident": round(float(cnt[warm, 0].mean()), 1),
                              "host_read_gbs": round(float((miss_bytes[warm] / (t_res[warm] * 1e6)).mean()), 1)},
            "mla_hbm_gbs_warm": round(mla_w.bytes / (float(t_mla[warm].mean()) * 1e6), 1),
            "host_tier": {"gb": round(sum(h.nbytes for h in hw.host_rows) / 1e9, 2),
                          "touch_ms": round(t_touch[0].elapsed_time(t_touch[1]), 2),
                          "note": "hs_hisparse_touch_host once before step 0 (setup, not in value)"},
            "device_flag": hs.hs_check_flag(dh.err), "inputs_generated_s": round(gen_s, 1), "data": "synthetic",
            "l2": "no flush (consecutive decode steps)"}
    del dh, hw
    torch.cuda.empty_cache()
    return line


# ------------------------------------------------------------------------ reference arm -----

def run_reference(args):
    """The CPU oracle timed as the reference implementation, on the same workload and metric. On
    the long-prefill pass a step is 16 query tokens evenly spaced in one chunk, the chunks cycling
    through 3, 11, ..., 59 (their mean cost per token is the pass's); on the other workloads a
    step is one query token per core."""
    rank, world, local = dist_info()
    if rank != 0:
        return
    import oracle
    from dsa_sparse_mla_gb300 import inputs
    oracle.build()
    threads = oracle.num_threads(0)
    if args.config == 4:
        picks = list(range(3, 64, 8))
        ws = inputs.config4_pass(seed=rank_seed(4, 0), chunks=picks)
        tok = np.linspace(0, ws[0].T - 1, 16).round().astype(int).tolist()
        plan = [(ws[i % len(ws)], tok) for i in range(len(ws))]
        name = "long-prefill-128K"
    else:
        w = build_workload(args.config, rank_seed(args.config, 0), args.requests)
        per_step = max(4, threads)
        plan = [(w, [(i * per_step + j) % w.T for j in range(per_step)]) for i in range(max(1, w.T // per_step))]
        name = w.name
    # size the sample so that warm-up + timed steps stay within about three minutes
    probe = oracle_sample(plan[0][0], plan[0][1], threads=0)
    budget = 180.0
    steps_timed = max(1, min(args.steps, int(budget / max(probe, 1e-3)) - args.warmup))
    t = 0.0
    ntok = 0
    for i in range(steps_timed):
        w, toks = plan[i % len(plan)]
        t += oracle_sample(w, toks, threads=0)
        ntok += len(toks)
    value = ntok / t
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "steps_timed": steps_timed, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t / steps_timed, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "query_tokens_per_step": len(plan[0][1])},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle", "cores": threads,
                             "sample": "%d query tokens per step (indexer+top-k+MLA, float64) of %s, %d timed steps "
                                       "(the probe step untimed) on %s" % (len(plan[0][1]), name, steps_timed,
                                                                           cpu_model())},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 5 long-prefill passes, else 1000)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", type=int, default=4,
                    help="4 (default): the long-prefill pass; 1, 2, 3: one step of that workload; 5: HiSparse decode")
    ap.add_argument("--requests", type=int, default=64, help="decode batch size (profiling runs use fewer)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="--config 4: skip the MTP-decode, chunked-prefill and mixed-residency keys")
    ap.add_argument("--chunks", default="", help="--config 4: run only these chunks of the pass (comma list; profiling)")
    ap.add_argument("--no-peak", action="store_true", help="--config 4: skip the e4m3 GEMM peak measurement (profiling)")
    ap.add_argument("--reps", type=int, default=5, help="--kv-append / --kv-offload: timed launches")
    ap.add_argument("--hisparse-steps", type=int, default=50, help="--config 5: decode steps")
    ap.add_argument("--hisparse-requests", type=int, default=32, help="--config 5: requests (profiling runs use fewer)")
    ap.add_argument("--kv-append", type=int, default=0, help="time hs_kv_append on this many new tokens instead")
    ap.add_argument("--kv-offload", type=int, default=0, help="time hs_kv_offload on about this many pages instead")
    ap.add_argument("--separate", action="store_true",
                    help="--config 2: run indexer and top-k as two calls in the step, not hs_indexer_topk")
    ap.add_argument("--shared-sets", action="store_true",
                    help="the query tokens of a request share its final token's index set (indexer and top-k "
                         "run for final tokens only)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.steps is None:
        args.steps = 5 if (args.config == 4 and args.impl == "ours") else 1000
    if args.impl == "reference":
        run_reference(args)
    elif args.kv_append > 0:
        run_kv_append(args)
    elif args.kv_offload > 0:
        run_kv_offload(args)
    elif args.config == 4:
        run_long_prefill_pass(args)
    elif args.config == 5:
        run_hisparse(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
