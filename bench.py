#!/usr/bin/env python3
"""Benchmark of the eviction step (one kvc_evict over the whole cache) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
                    [--row-agg max|mean] [--group-agg max|sum] [--head-budget given|entropy] [--entropy]

Prints ONE JSON line. A step is one pass of the whole hot path (beacons, scores, selection,
in-place compaction) over every (layer, sequence, KV head) of the workload. Inputs are
resident in HBM; between timed steps the cache is restored from a pristine copy and L2 is
flushed (both untimed); each step is bracketed by CUDA events on the launch stream.

value = cached tokens per second = B * N / step time (a token spans all layers and heads),
summed over ranks. For N > 1 (torchrun) every rank runs an independent replica on its own
GPU: the step has no cross-GPU exchange, so there is no collective on the data path.
``--impl reference`` times the CPU oracle (the reference arm) on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "eviction-step cached tokens/sec and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "cached tokens/s"
DEFAULT_CONFIG = "qwen3-14b-long"
SINGLE_CORE_CONFIGS = ("tiny", "qwen3-4b")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------


class L2Flush:
    """Evicts the step's inputs from L2 between timed steps (untimed): a 512 MB write (four times
    the 129 MB L2), then a 512 MB read of another buffer, so that the write's dirty lines are
    written back before the next step rather than inside it. Each step starts with a clean L2
    that holds none of its inputs."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(128 << 20, dtype=torch.int32, device=dev)
        self.amax = torch.amax
        self.sink = None

    def __call__(self):
        self.w.zero_()
        self.sink = self.amax(self.r)

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(x: float, world: int) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region (read-only)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(1.0)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except ValueError:
                continue
            rows.append((ts, parts))
        lo, hi = (self.t0 or 0) - 1.0, (self.t1 or 1e18) + 1.0
        inwin = [p for ts, p in rows if lo <= ts <= hi] or [p for _, p in rows]
        sm = [float(p[2]) for p in inwin if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for p in inwin if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inwin for i in range(4) if p[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inwin)}


def src_hash(files=None) -> str:
    """Hash of CUDA sources (the given files under csrc/, else all of them); an ncu traffic figure is
    only reported while the sources of the kernel it was taken from are unchanged."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "decoding_kv_cache_gb300", "csrc")
    names = sorted(files) if files else sorted(f for f in os.listdir(d) if f.endswith((".cu", ".cuh")))
    for f in names:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str, phase: str):
    """DRAM bytes (read + write) per launch of the phase's dominant kernel, from profiles/traffic.json."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(config, {}).get(phase)
    if not e or e.get("src_hash") != src_hash(e.get("sources")):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def variant_of(args) -> str:
    """'' for the default step, else e.g. 'mean,sum' / 'max,max+entropy' / 'max,max+entropy-budgets'."""
    v = f"{args.row_agg},{args.group_agg}"
    if args.head_budget == "entropy":
        v += "+entropy-budgets"
    elif args.entropy:
        v += "+entropy"
    return "" if v == "max,max" else v


def workload_desc(config: str, variant: str = "", layers: int = 0) -> str:
    """The workload's name and shape from its spec (no tensors), the same string in both arms."""
    from decoding_kv_cache_gb300.inputs import CONFIGS, EPIKV_CONFIGS
    if config in EPIKV_CONFIGS:
        sp = EPIKV_CONFIGS[config]
        L = layers or sp["L"]
        return (f"{config} EPIKV eviction step: L{L} B{sp['B']} Hkv{sp['Hkv']} D{sp['D']} {sp['dtype']} "
                f"N{sp['N']}->{(7 * sp['N']) // 8}, hidden size {sp['dm']} (band layers A, B), window "
                f"{sp['window']}, eps {sp['eps']:g}")
    sp = CONFIGS[config]
    L = layers or sp["L"]
    keep = "per-head budgets" if sp["cfg"] == 4 else f"{(7 * sp['N']) // 8}"
    d = (f"{config} eviction step: L{L} B{sp['B']} Hq{sp['Hq']} Hkv{sp['Hkv']} D{sp['D']} {sp['dtype']} "
         f"N{sp['N']}->{keep}, obs {sp['n_r']} recent + {sp['n_b']} beacons (buffer {sp['qmax']})")
    if variant:
        d += (f"; aggregation {variant.split('+')[0]} (rows, GQA group)" +
              ("; budgets reallocated per layer by attention entropy" if "budgets" in variant else "") +
              ("; entropy output" if variant.endswith("+entropy") else ""))
    return d


def pinned_like(t):
    """A page-locked host copy of a device tensor (one host allocation, filled by a D2H copy)."""
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def h2d_anchor(hosts, devs, stream, reps: int = 3):
    """A plain pinned host-to-device copy of the same tensors the e2e step copies (CUDA events on the
    launch stream, best of ``reps``): the copy engines' rate that bounds the e2e figure."""
    import torch
    nbytes = sum(h.numel() * h.element_size() for h in hosts)
    best = None
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for h, d in zip(hosts, devs):
            d.copy_(h, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    return {"bytes": nbytes, "ms": best, "gbs": nbytes / (best / 1e3) / 1e9,
            "note": "plain pinned H2D copies of the e2e inputs, no kernel, best of %d" % reps}


def algorithmic_bytes(inp, kept_idx, kept_len):
    """K read once for scoring + K and V read and written for every kept token that moves."""
    import torch
    es = 2 if inp.dtype == "bf16" else 4
    row = inp.D * es
    k_read = inp.heads * inp.N * row
    n = kept_idx.shape[-1]
    ar = torch.arange(n, device=kept_idx.device, dtype=torch.int32)
    valid = ar < kept_len[..., None]
    moved = int(((kept_idx != ar) & valid).sum().item())
    return k_read, moved * 4 * row, moved


def score_flop(inp):
    """Tensor work of the scoring passes as the BeaconKV write-up's score defines it ("打分时的 RoPE
    对齐": every observation row against every cached key, softmax over the keys before the max):
    QK^T over the M = G (n_r + n_b) observation rows of each KV head, once to find each row's
    log-sum-exp and once more to take the max, i.e. 4 M D FLOP per cached key. Zero for fp32
    caches, which are not scored on the tensor cores."""
    if inp.dtype != "bf16":
        return 0
    M = (inp.Hq // inp.Hkv) * (inp.n_r + inp.n_b)
    return 4 * M * inp.D * inp.heads * inp.N


def bounds(nbytes, flop, ms, pk):
    """The HBM and tensor-pipe times of a piece of work and the one that governs it (the larger), with
    the fraction of it that ``ms`` achieves. The tensor peak is the measured burst figure: every
    timed region here is a single step or phase of a few ms at most."""
    hbm_ms = nbytes / (float(pk["hbm_gbs"]) * 1e9) * 1e3
    tensor_ms = flop / (float(pk["bf16_tflops"]) * 1e12) * 1e3
    gov = "tensor" if tensor_ms > hbm_ms else "hbm"
    return {"hbm_ms": hbm_ms, "tensor_ms": tensor_ms, "governing": gov,
            "frac": max(hbm_ms, tensor_ms) / ms if ms > 0 else 0.0}


def append_timing(inp, dev, stream, reps: int = 20):
    """Per-decode-step kvc_append over every query head of the workload (the step that feeds the
    eviction's observation state), on copies of its buffers. One fill/compress cycle is captured as
    two CUDA graphs: the qmax/2 - 1 calls that only append, and the call that fills the buffers and
    compresses them; the graphs are replayed alternately with CUDA events around each replay, so
    the times are the GPU's (kernel plus inter-kernel latency), not the host's launch overhead."""
    import torch
    from decoding_kv_cache_gb300 import kvc
    qb, cnt, ring = inp.qbuf.clone(), inp.count.clone(), inp.q_recent.clone()
    nq = inp.L * inp.B * inp.Hq
    g = torch.Generator(device=dev).manual_seed(1234)
    pool = [torch.randn((inp.L, inp.B, inp.Hq, inp.D), generator=g, device=dev).to(inp.K.dtype) for _ in range(8)]
    m = inp.qmax // 2
    cs = torch.cuda.Stream(device=dev)
    cs.wait_stream(stream)
    res = {}
    for post in (False, True):  # ring row by rotation, then from a given post-RoPE query
        kw = lambda i: dict(q_post=pool[(i + 3) % 8] if post else None)
        with torch.cuda.stream(cs):
            cnt.fill_(m)
            for i in range(m):  # warm-up: one cycle outside the graphs
                kvc.kvc_append(pool[i % 8], qb, cnt, ring, inp.t + 1 + i, inp.theta, **kw(i))
            ga, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(ga, stream=cs):
                for i in range(m - 1):
                    kvc.kvc_append(pool[i % 8], qb, cnt, ring, inp.t + 1 + i, inp.theta, **kw(i))
            with torch.cuda.graph(gb, stream=cs):
                kvc.kvc_append(pool[(m - 1) % 8], qb, cnt, ring, inp.t + m, inp.theta, **kw(m - 1))
            ev = []
            for r in range(reps + 2):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record(cs)
                ga.replay()
                e[1].record(cs)
                gb.replay()
                e[2].record(cs)
                if r >= 2:
                    ev.append(e)
        torch.cuda.synchronize()
        plain = statistics.median(e[0].elapsed_time(e[1]) for e in ev) / (m - 1)
        comp = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
        res["post_given" if post else "rotated"] = (plain, comp, (plain * (m - 1) + comp) / m)
        del ga, gb
    stream.wait_stream(cs)
    es = 2 if inp.dtype == "bf16" else 4
    row = inp.D * es
    b_plain = nq * (3 * row + 8)                      # q_pre read, buffer row and ring row written, count
    b_comp = b_plain + nq * (inp.qmax - 1 + m) * row  # + the buffer staged and the survivors written back
    pr, cr, avg = res["rotated"]
    return {"query_heads": nq, "replays": reps, "us_plain": 1e3 * pr, "us_compress": 1e3 * cr,
            "us_per_step_avg": 1e3 * avg, "us_plain_post_given": 1e3 * res["post_given"][0],
            "bytes_plain": b_plain, "bytes_compress_max": b_comp, "gbs_plain": b_plain / (pr / 1e3) / 1e9,
            "note": "kvc_append per decode step, CUDA-graph replays of one fill/compress cycle; ring row by "
                    "rotation unless post_given; bound: latency"}


def gpu_arm(args, rank, world, local_rank):
    import torch
    from decoding_kv_cache_gb300 import build as kbuild
    from decoding_kv_cache_gb300 import kvc
    from decoding_kv_cache_gb300.inputs import make_inputs

    if not kbuild.up_to_date():
        kbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    over = {"L": args.layers} if args.layers else {}
    inp = make_inputs(args.config, device=dev, **over)
    stream = torch.cuda.current_stream(dev)
    K0, V0 = inp.K.clone(), inp.V.clone()
    cache = kvc.Cache(inp.K, inp.V, inp.Hq)
    shape = (inp.L, inp.B, inp.Hkv)
    kept_len = torch.zeros(shape, dtype=torch.int32, device=dev)
    kept_idx = torch.zeros(shape + (inp.N,), dtype=torch.int32, device=dev)
    scores = torch.zeros(shape + (inp.N,), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(kvc.kvc_evict_workspace_size(cache, inp.n_r, inp.n_b), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)

    def reset():
        inp.K.copy_(K0)
        inp.V.copy_(V0)
        flush()

    variant = variant_of(args)
    ent = torch.zeros(shape, dtype=torch.float32, device=dev) if (args.entropy or args.head_budget == "entropy") \
        else None
    vkw = dict(row_agg=args.row_agg, group_agg=args.group_agg)

    def evict():
        kvc.kvc_evict(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, inp.prefix, inp.recent,
                      kept_len, budget=inp.budget, budget_all=inp.budget_all, kept_idx=kept_idx, scores=None,
                      status=status, workspace=ws, head_budget=args.head_budget, entropy=ent, **vkw)

    for _ in range(args.warmup):
        reset()
        evict()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {status.item()} after warm-up")
    k_read, moved_bytes, moved = algorithmic_bytes(inp, kept_idx, kept_len)
    alg = k_read + moved_bytes

    # ---- headline: K timed steps of kvc_evict ------------------------------------------
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("t0")
    for i in range(args.steps):
        reset()
        ev[i][0].record(stream)
        evict()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world)
    clk = clocks.stop() if rank == 0 else None
    ms_per_step = total_ms / args.steps
    tokens = inp.B * inp.N
    value = world * tokens * args.steps / (total_ms / 1e3)

    # ---- phase split (same work through the three entry points) to find the dominant kernel
    phase_ms = {"kvc_score": 0.0, "kvc_select": 0.0, "kvc_compact": 0.0}
    nph = max(3, min(args.steps, 50))
    sc_ws = torch.empty(kvc.kvc_score_workspace_size(cache, inp.n_r, inp.n_b), dtype=torch.uint8, device=dev)
    hb_out = torch.zeros(shape, dtype=torch.int32, device=dev)
    evs = []
    for i in range(nph):
        reset()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        kvc.kvc_score(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, scores, workspace=sc_ws,
                      entropy=ent, **vkw)
        e[1].record(stream)
        if args.head_budget == "entropy":  # the reallocation runs inside the selection kernel in kvc_evict
            kvc.kvc_head_budget(ent, inp.N, inp.prefix, inp.recent, hb_out, budget=inp.budget,
                                budget_all=inp.budget_all)
        kvc.kvc_select(scores, inp.prefix, inp.recent, kept_idx, kept_len,
                       budget=hb_out if args.head_budget == "entropy" else inp.budget, budget_all=inp.budget_all)
        e[2].record(stream)
        kvc.kvc_compact(cache, kept_idx, kept_len, status=status)
        e[3].record(stream)
        evs.append(e)
    torch.cuda.synchronize()
    for e in evs:
        phase_ms["kvc_score"] += e[0].elapsed_time(e[1]) / nph
        phase_ms["kvc_select"] += e[1].elapsed_time(e[2]) / nph
        phase_ms["kvc_compact"] += e[2].elapsed_time(e[3]) / nph
    phase_bytes = {"kvc_score": k_read, "kvc_select": 0, "kvc_compact": moved_bytes}
    dom = max(phase_ms, key=phase_ms.get)

    # ---- end to end: host buffers in, step, result out ------------------------------------
    hK, hV, hqr, hqb, hc = (pinned_like(t) for t in (K0, V0, inp.q_recent, inp.qbuf, inp.count))
    hkl, hki = torch.empty_like(kept_len, device="cpu").pin_memory(), torch.empty_like(kept_idx, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hK, hV, hqr, hqb, hc))
    anchor = h2d_anchor((hK, hV), (inp.K, inp.V), stream)
    d2h = hkl.numel() * 4 + hki.numel() * 4
    n_e2e = max(3, min(args.steps, 20))
    ee = []
    for i in range(n_e2e):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        inp.K.copy_(hK, non_blocking=True)
        inp.V.copy_(hV, non_blocking=True)
        inp.q_recent.copy_(hqr, non_blocking=True)
        inp.qbuf.copy_(hqb, non_blocking=True)
        inp.count.copy_(hc, non_blocking=True)
        evict()
        hkl.copy_(kept_len, non_blocking=True)
        hki.copy_(kept_idx, non_blocking=True)
        b.record(stream)
        ee.append((a, b))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ee) / n_e2e, world)

    app = append_timing(inp, dev, stream)

    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    dom_ms = phase_ms[dom]
    achieved = phase_bytes[dom] / (dom_ms / 1e3) / 1e9 if phase_bytes[dom] else 0.0
    step_gbs = alg / (ms_per_step / 1e3) / 1e9
    flop = score_flop(inp)
    phase_flop = {"kvc_score": flop, "kvc_select": 0, "kvc_compact": 0}
    hbm_view = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_source": pk_kind,
                "traffic": None if args.layers else recorded_traffic(args.config + (f"/{variant}" if variant else ""),
                                                                     dom)}
    if hbm_view["traffic"]:
        # the same launch's rate on the DRAM bytes ncu counted (writes still in L2 at the end and re-reads
        # make it differ from the algorithmic rate)
        hbm_view["achieved_dram"] = hbm_view["traffic"] / (dom_ms / 1e3) / 1e9
        hbm_view["frac_dram"] = hbm_view["achieved_dram"] / hbm
    dom_bounds = bounds(phase_bytes[dom], phase_flop[dom], dom_ms, pk)
    if dom_bounds["governing"] == "tensor":
        # the dominant phase does more tensor work than HBM time: its roofline is the tensor pipe's
        tf = float(pk["bf16_tflops"])
        ach_t = phase_flop[dom] / (dom_ms / 1e3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": ach_t, "peak": tf, "unit": "TFLOP/s",
                    "frac": ach_t / tf, "peak_source": pk_kind + " (bf16 burst)", "traffic": hbm_view["traffic"],
                    "flop_per_launch": phase_flop[dom], "hbm_view": hbm_view}
    else:
        roofline = hbm_view
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": inp.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(args.config, variant, args.layers), "l2": "flushed between steps (512 MB write, then a 512 MB read so no dirty line is left), cache restored "
                   "from a pristine copy between steps; both untimed", "parallelism": f"replicas x{world}",
                   "timing": "CUDA events around each kvc_evict on the launch stream"},
        "head_tokens_per_s": world * inp.heads * inp.N * args.steps / (total_ms / 1e3),
        "achieved_gbs": step_gbs, "step_roofline_frac": step_gbs / hbm,
        "algorithmic_bytes_per_step": {"k_read": k_read, "kv_moved": moved_bytes, "moved_tokens": moved},
        "score_flop_per_step": flop,
        "step_bounds": bounds(alg, flop, ms_per_step, pk),
        "roofline": roofline,
        "phases_ms": phase_ms,
        "e2e": {"value": world * tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "h2d_copy_anchor": anchor},
        "append": app,
        "gpu_launches": args.steps * kvc.kvc_evict_launch_count(cache, inp.n_r, inp.n_b),
        "clocks": clk,
    }
    return res, inp


def epikv_arm(args, rank, world, local_rank):
    """The EPIKV eviction step (EPIKV write-up, "方法论：EPIKV"): signals from two layers' hidden states,
    rolling z-score, one selection per sequence, compaction of every layer and KV head. Same metric;
    the algorithmic bytes are the hidden states read once plus K and V of every moved token."""
    import torch
    from decoding_kv_cache_gb300 import build as kbuild
    from decoding_kv_cache_gb300 import kvc
    from decoding_kv_cache_gb300.inputs import make_epikv_inputs

    if not kbuild.up_to_date():
        kbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    over = {"L": args.layers} if args.layers else {}
    inp = make_epikv_inputs(args.config, device=dev, **over)
    stream = torch.cuda.current_stream(dev)
    K0, V0 = inp.K.clone(), inp.V.clone()
    cache = kvc.Cache(inp.K, inp.V, inp.Hq)
    kept_len = torch.zeros((inp.B,), dtype=torch.int32, device=dev)
    kept_idx = torch.zeros((inp.B, inp.N), dtype=torch.int32, device=dev)
    scores = torch.zeros((inp.B, inp.N), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(kvc.kvc_epikv_workspace_size(inp.B, inp.N), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)

    def reset():
        inp.K.copy_(K0)
        inp.V.copy_(V0)
        flush()

    def evict():
        kvc.kvc_epikv_evict(cache, inp.hA, inp.hB, inp.window, inp.eps, inp.prefix, inp.recent, kept_len,
                            budget_all=inp.budget_all, kept_idx=kept_idx, scores=scores, status=status, workspace=ws)

    for _ in range(args.warmup):
        reset()
        evict()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {status.item()} after warm-up")
    es = 2 if inp.dtype == "bf16" else 4
    h_read = 2 * inp.B * inp.N * inp.dm * es
    ar = torch.arange(inp.N, device=dev, dtype=torch.int32)
    moved = int((((kept_idx != ar) & (ar < kept_len[:, None])).sum().item())) * inp.L * inp.Hkv
    moved_bytes = moved * 4 * inp.D * es
    alg = h_read + moved_bytes

    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("t0")
    for i in range(args.steps):
        reset()
        ev[i][0].record(stream)
        evict()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier(world)
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world)
    clk = clocks.stop() if rank == 0 else None
    ms_per_step = total_ms / args.steps

    # phases: the score alone, then the whole step (the difference is selection + compaction)
    nph = max(3, min(args.steps, 20))
    g = torch.zeros((2, inp.B, inp.N), device=dev)
    ph = []
    for i in range(nph):
        reset()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        kvc.kvc_epikv_score(inp.hA, inp.hB, inp.window, inp.eps, scores, g=g, workspace=ws)
        e[1].record(stream)
        ph.append(e)
    torch.cuda.synchronize()
    score_ms = sum(a.elapsed_time(b) for a, b in ph) / nph
    rest_ms = max(ms_per_step - score_ms, 1e-9)
    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    dom, dom_bytes, dom_ms = ("kvc_epikv_score", h_read, score_ms) if score_ms >= rest_ms else \
        ("select+compact", moved_bytes, rest_ms)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9

    hK, hV, hA, hB = (pinned_like(t) for t in (K0, V0, inp.hA, inp.hB))
    hkl, hki = torch.empty_like(kept_len, device="cpu").pin_memory(), torch.empty_like(kept_idx, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hK, hV, hA, hB))
    anchor = h2d_anchor((hK, hV), (inp.K, inp.V), stream)
    d2h = hkl.numel() * 4 + hki.numel() * 4
    ee = []
    for i in range(max(3, min(args.steps, 10))):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        inp.K.copy_(hK, non_blocking=True)
        inp.V.copy_(hV, non_blocking=True)
        inp.hA.copy_(hA, non_blocking=True)
        inp.hB.copy_(hB, non_blocking=True)
        evict()
        hkl.copy_(kept_len, non_blocking=True)
        hki.copy_(kept_idx, non_blocking=True)
        b.record(stream)
        ee.append((a, b))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ee) / len(ee), world)
    tokens = inp.B * inp.N
    step_gbs = alg / (ms_per_step / 1e3) / 1e9
    res = {
        "metric": METRIC, "value": world * tokens * args.steps / (total_ms / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": inp.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(args.config, "", args.layers),
                   "l2": "flushed between steps (512 MB write, then a 512 MB read so no dirty line is left), cache restored from a pristine copy between steps; "
                         "both untimed", "parallelism": f"replicas x{world}",
                   "timing": "CUDA events around each kvc_epikv_evict on the launch stream"},
        "achieved_gbs": step_gbs, "step_roofline_frac": step_gbs / hbm,
        "algorithmic_bytes_per_step": {"hidden_read": h_read, "kv_moved": moved_bytes, "moved_head_tokens": moved},
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": pk_kind, "traffic": None},
        "phases_ms": {"kvc_epikv_score": score_ms, "select+compact": rest_ms},
        "e2e": {"value": world * tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "h2d_copy_anchor": anchor},
        "gpu_launches": args.steps * 5,  # signal, prefix sums, z-score, select, compact
        "clocks": clk,
    }
    return res, inp


def oracle_epikv_sample(config: str, budget_s: float = 12.0):
    """The oracle's EPIKV step (scores, per-sequence selection, gather of every head) on a bounded
    sample of the workload's sequences; tokens/s scaled linearly to the full step."""
    from decoding_kv_cache_gb300.inputs import EPIKV_CONFIGS, make_epikv_inputs
    from oracle import oracle as O
    import numpy as np
    spec = EPIKV_CONFIGS[config]
    cores = O.set_threads(os.cpu_count() or 1)

    def run(inp):
        bits = lambda t: t.view(__import__("torch").int16).numpy().view(np.uint16) if inp.dtype == "bf16" else t.numpy()
        _, sc = O.epikv_score(bits(inp.hA), bits(inp.hB), inp.window, inp.eps, inp.dtype)
        K = bits(inp.K)
        V = bits(inp.V)
        for b in range(inp.B):
            kept = O.select(sc[b].astype(np.float32), inp.prefix, inp.recent, inp.budget_all)
            _ = K[:, b, :, kept], V[:, b, :, kept]

    probe = make_epikv_inputs(config, L=spec["L"], B=1, N=min(spec["N"], 512))
    t0 = time.perf_counter()
    run(probe)
    per_tok = (time.perf_counter() - t0) / probe.N
    n_tok = int(max(512, min(spec["N"], budget_s / max(per_tok, 1e-9))))
    samp = make_epikv_inputs(config, B=1, N=n_tok)
    t0 = time.perf_counter()
    run(samp)
    dt = time.perf_counter() - t0
    full_s = dt * (spec["B"] * spec["N"]) / n_tok
    tok = spec["B"] * spec["N"] / full_s
    return tok, cores, (f"oracle on 1 of {spec['B']} sequences, {n_tok} of {spec['N']} tokens, all layers, {dt:.2f} s "
                        f"wall on {cores} threads, scaled linearly to the full step"), dt


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(config: str, budget_s: float = 12.0, threads: int = 0, **variant):
    """Time the oracle, as it stands, on a bounded sample of the workload's heads (``variant``:
    the oracle's row_agg / group_agg / head_budget keywords; ``threads`` 0 = every core).
    Returns (tokens/s scaled to the full step, cores, sample description, seconds)."""
    from decoding_kv_cache_gb300.inputs import make_inputs
    from oracle import oracle as O
    from decoding_kv_cache_gb300.inputs import CONFIGS
    spec = CONFIGS[config]
    cores = O.set_threads(threads or os.cpu_count() or 1)
    heads_full = spec["L"] * spec["B"] * spec["Hkv"]
    # one layer of one sequence first, to size the sample
    probe = make_inputs(config, L=1, B=1)
    t0 = time.perf_counter()
    O.evict(probe, **variant)
    dt = time.perf_counter() - t0
    per_head = dt / probe.heads
    want_heads = max(probe.heads, min(heads_full, int(budget_s / max(per_head, 1e-9))))
    L = max(1, min(spec["L"], want_heads // (spec["B"] * spec["Hkv"])))
    B = spec["B"] if L > 1 else max(1, min(spec["B"], want_heads // spec["Hkv"]))
    samp = make_inputs(config, L=L, B=B)
    # a sample that is the whole step is run again while another run fits in the budget (at most
    # 64 runs), so that the figure rests on seconds of work
    reps = 0
    t0 = time.perf_counter()
    while True:
        O.evict(samp, **variant)
        reps += 1
        dt = time.perf_counter() - t0
        if samp.heads < heads_full or dt + dt / reps > budget_s or reps >= 64:
            break
    full_s = dt / reps * heads_full / samp.heads
    tok = spec["B"] * spec["N"] / full_s
    desc = (f"oracle on {samp.heads} of {heads_full} heads (L={L}, B={B}) of {config}"
            + (f", {reps} runs" if reps > 1 else "") + f", {dt:.2f} s wall on {cores} threads, scaled linearly to "
            "the full step")
    return tok, cores, desc, dt


def oracle_variant(args):
    return dict(row_agg=args.row_agg, group_agg=args.group_agg, head_budget=args.head_budget)


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    from decoding_kv_cache_gb300.inputs import CONFIGS, EPIKV_CONFIGS
    epikv = args.config in EPIKV_CONFIGS
    sample = (lambda budget_s: oracle_epikv_sample(args.config, budget_s)) if epikv else \
        (lambda budget_s: oracle_sample(args.config, budget_s, **oracle_variant(args)))
    vals, descs = [], []
    if args.warmup > 0:
        sample(2.0)
    for _ in range(args.steps):
        tok, cores, desc, _ = sample(min(12.0, 120.0 / max(args.steps, 1)))
        vals.append(tok)
        descs.append(desc)
    value = statistics.mean(vals)
    spec = (EPIKV_CONFIGS if epikv else CONFIGS)[args.config]
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": spec["B"] * spec["N"] / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(args.config, "" if epikv else variant_of(args))},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores,
                                                                 "kind": "oracle", "sample": descs[-1]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: run the workload with only this many layers (0 = all)")
    ap.add_argument("--row-agg", default="max", choices=["max", "mean"],
                    help="aggregation over a query head's observation rows")
    ap.add_argument("--group-agg", default="max", choices=["max", "sum"],
                    help="aggregation over the query heads of a KV head")
    ap.add_argument("--head-budget", default="given", choices=["given", "entropy"],
                    help="entropy: reallocate each layer's budget over its heads by attention entropy")
    ap.add_argument("--entropy", action="store_true", help="also output each head's attention entropy")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            dist.init_process_group("nccl")
    if args.impl == "reference":
        out = reference_arm(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    from decoding_kv_cache_gb300.inputs import EPIKV_CONFIGS
    epikv = args.config in EPIKV_CONFIGS
    res, _ = (epikv_arm if epikv else gpu_arm)(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            tok, cores, desc, _ = oracle_epikv_sample(args.config) if epikv else \
                oracle_sample(args.config, **oracle_variant(args))
            res["cpu_baseline"] = {"value": tok, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
            if args.config in SINGLE_CORE_CONFIGS:  # the two small workloads also on one core
                tok1, c1, desc1, _ = oracle_sample(args.config, threads=1, **oracle_variant(args))
                res["cpu_baseline_1core"] = {"value": tok1, "unit": UNIT, "cores": c1, "kind": "oracle",
                                             "sample": desc1}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
