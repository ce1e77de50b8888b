"""Benchmark of the sparse MLA forward on GB300 (one JSON line on stdout).

Default workload: decode bf16 — 64 sequences x 1 query row, H=16,
D_qk=D_v=512, paged 64-slot blocks, 131072-token contexts (8,388,608 slots,
8.6 GB bf16 pool), top-k 2048 distinct uniform indices per row. A step is one
sparse_mla_fwd call over the 64 rows (the whole path: index read, gather,
QK, masked online softmax, PV, split partials and LSE merge; one kernel).

Metric: gathered-KV GB/s = sum_t valid_t * D_qk * bytes_per_elem / step time
(higher is better); query rows/s is reported beside it.

Timing: W warm-up steps, then exactly K steps timed with CUDA events on the
launching stream, replayed from a CUDA graph of R consecutive calls that
rotate over R independent (q, indices) sets whose gathered bytes together
exceed 4x the L2 (the pool stays resident; every call gathers more than L2).
SM clocks are sampled with nvidia-smi during the timed region.

--impl reference times the fp64 CPU oracle on the host cores instead: each
step is one query row of the same workload (all heads), so K steps finish in
minutes; its line carries "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

from sparse_mla_attention_04_gb300 import inputs

FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_bf16", choices=sorted(inputs.CONFIGS) + ["producer"],
                    help="an attention workload, or `producer`: the fused RoPE + q concat + cache write step")
    ap.add_argument("--rotations", type=int, default=0, help="index/q sets (0 = enough for 4x L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="the per-call sweep: rows x fan-out grid (H=16, D=512, bf16), automatic vs fixed splits")
    ap.add_argument("--sinks", action="store_true",
                    help="give every head a sink logit (seeded, uniform in [-2, 4])")
    ap.add_argument("--bf16-dots", action="store_true",
                    help="E4M3 workloads: keep q in bf16 and dot it with the cache values (dot_precision bf16)")
    ap.add_argument("--q8", action="store_true",
                    help="E4M3 workloads: pass q pre-quantized (codes + a per-tensor scale) to sparse_mla_fwd_q8")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--ctx", type=int, default=0,
                    help="override the per-row context (pool size) of a decode workload, for profiling")
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "basic"],
                    help="kernel choice of the forward (auto: the library's; mma: the warp-MMA kernel; basic: the "
                         "tcgen05 kernels that take a whole SM per CTA)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --workload (skip the other configurations, the ceilings and the L2 probe)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; timing reduction only)
# ----------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(seed: int, r: int, rank: int) -> int:
    """Seed of input set r on `rank`: every rank draws its own rows (weak scaling)."""
    return seed + 1 + r + 1000 * rank


def job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job units per second: each of `world` ranks processed
    `units_per_rank` in the timed region, which took the slowest rank ms_max."""
    return units_per_rank * world / (ms_max * 1e-3)


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s)"


FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0   # nominal dense E4M3 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


def measured_bf16_tflops():
    """Burst bf16 tensor peak (a kernel timed on its own)."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16)"


def roofline(w, per_launch_bytes, valid_per_launch, sec_per_launch, traffic, l2_gbs=None):
    """The bound of one launch: HBM (gathered bytes / copy bandwidth) or the
    tensor cores (QK at 2*H*D_qk and PV at 2*H*D_v FLOP per valid index, QK
    at the E4M3 rate for an fp8 cache, PV at the bf16 rate), whichever takes
    longer; achieved and peak in that bound's unit."""
    hbm, hbm_src = measured_peaks()
    bf16, bf16_src = measured_bf16_tflops()
    qk_flop = 2.0 * w.H * w.D_qk * valid_per_launch
    pv_flop = 2.0 * w.H * w.D_v * valid_per_launch
    qk_peak = bf16 * (FP8_OVER_BF16 if w.kv_fp8 else 1.0)
    t_tensor = qk_flop / (qk_peak * 1e12) + pv_flop / (bf16 * 1e12)
    t_hbm = per_launch_bytes / (hbm * 1e9)
    if l2_gbs is not None:
        # the pool sits in L2: the gathered bytes move L2 -> SM, bound by the
        # L2 read bandwidth this run measured; the HBM formula rides along
        t_l2 = per_launch_bytes / (l2_gbs * 1e9)
        if t_l2 >= t_tensor:
            achieved = per_launch_bytes / sec_per_launch / 1e9
            return {"bound": "l2", "achieved": round(achieved, 2), "peak": round(l2_gbs, 1), "unit": "GB/s",
                    "frac": round(achieved / l2_gbs, 4), "traffic": traffic,
                    "peak_source": "measured in this run (smla_l2_read_probe: L2 -> SM streaming read)",
                    "algorithmic_bytes_per_launch": per_launch_bytes,
                    "hbm_formula_frac": round(per_launch_bytes / sec_per_launch / 1e9 / hbm, 4),
                    "tensor_frac": round(t_tensor / sec_per_launch, 4)}
    if t_tensor > t_hbm:
        flop = qk_flop + pv_flop
        peak = flop / t_tensor / 1e12   # the mix's peak: fp8 QK share at 2x
        achieved = flop / sec_per_launch / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": bf16_src + (" x %.0f for the E4M3 QK share" % FP8_OVER_BF16 if w.kv_fp8 else ""),
                "algorithmic_flop_per_launch": flop, "algorithmic_bytes_per_launch": per_launch_bytes,
                "hbm_frac": round(per_launch_bytes / sec_per_launch / 1e9 / hbm, 4)}
    achieved = per_launch_bytes / sec_per_launch / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": hbm_src,
            "algorithmic_bytes_per_launch": per_launch_bytes}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def _code_only(text: str) -> str:
    """C/CUDA source without comments, trailing blanks or empty lines (a
    comment-only edit leaves the kernels, and so their counters, unchanged)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_mla_attention_04_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        if n.endswith((".cu", ".cuh", ".h")):
            h.update(n.encode())
            h.update(_code_only(open(os.path.join(csrc, n), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else null)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        d = json.load(open(p))[workload]
    except Exception:
        return None
    return float(d["bytes_per_launch"]) if d.get("kernel_hash") == kernel_source_hash() else None


# ----------------------------------------------------------------------------
# workload construction
# ----------------------------------------------------------------------------

def build_workload(name: str, seed: int, rotations: int, device, rank: int, ctx: int = 0):
    from sparse_mla_attention_04_gb300 import binding
    w = inputs.CONFIGS[name](seed=seed)
    if ctx and w.kind in ("decode", "wide"):
        w.ctx = ctx
        w.num_slots = w.T * ctx
    src = inputs.make_kv_source(w, device=device)
    if w.kv_fp8:
        cache, kvs = binding.build_fp8_cache(src)
    else:
        cache, kvs = src, None
    torch.cuda.synchronize()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    sets = []
    total = 0
    r = 0
    while True:
        s = rank_seed(seed, r, rank)
        idx = inputs.make_indices(w, seed=s)
        q = inputs.make_q(w, seed=s, device=device)
        gathered = inputs.valid_count(idx) * w.D_qk * w.kv_bytes_per_elem
        sets.append(dict(q=q, idx_np=idx, idx=torch.from_numpy(idx).to(device), bytes=gathered))
        total += gathered
        r += 1
        if rotations and r >= rotations:
            break
        if not rotations and total >= 4 * l2 and r >= 2:
            break
        if r >= 64:
            break
    return w, src, cache, kvs, sets, l2


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def forward_setup(binding, w, cache, kvs, sets, dev, stream, args, sinks=None, num_splits=0):
    """Buffers, split plan and the call of one workload (call(i) runs the
    forward on input set i % R on `stream`; num_splits 0 = the library's
    automatic plan)."""
    R = len(sets)
    dot = "fp8" if w.kv_fp8 else "auto"
    if args.bf16_dots:
        if not w.kv_fp8 or args.q8:
            raise SystemExit("--bf16-dots needs an E4M3 workload and a bf16 q")
        dot = "bf16"
    if args.q8:
        if not w.kv_fp8:
            raise SystemExit("--q8 needs an E4M3 workload")
        for s in sets:   # q quantized once per set, outside the timed region, by the library's kernels
            s["q8"], s["qs"] = quantize_q_per_tensor(binding, s["q"])
    T, H = w.T, w.H
    kernel = getattr(args, "kernel", "auto")
    out = torch.empty((T, H, w.D_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    # the library's automatic plan (0); the split count it takes is reported
    planned = binding.smla_plan_num_splits(T, H, w.D_qk, w.topk, int(w.kv_fp8),
                                           torch.cuda.get_device_properties(dev).multi_processor_count)
    splits = num_splits
    need = binding.sparse_mla_fwd_workspace_size(T, H, w.D_qk, w.D_v, w.topk, int(w.kv_fp8), splits)
    ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=dev)

    def call(i):
        s = sets[i % R]
        if args.q8:
            binding.sparse_mla_fwd_q8(s["q8"], s["qs"], cache, s["idx"], w.scale, kv_scale=kvs, D_v=w.D_v,
                                      out=out, lse=lse, workspace=ws, num_splits=splits, stream=stream, sinks=sinks,
                                      kernel=kernel)
        else:
            binding.sparse_mla_fwd(s["q"], cache, s["idx"], w.scale, kv_scale=kvs, dot_precision=dot, D_v=w.D_v,
                                   out=out, lse=lse, workspace=ws, num_splits=splits, stream=stream, sinks=sinks,
                                   kernel=kernel)
    return call, dot, planned


def graph_of(call, R, warmup, stream):
    """W warm-up calls, then a CUDA graph of R consecutive calls (replayed once)."""
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            call(i)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(R):
                call(i)
        graph.replay()
        stream.synchronize()
    return graph


def time_steps(graph, call, R, K, stream):
    """Device milliseconds of exactly K calls (whole graphs, then the rest)."""
    reps, rem = divmod(K, R)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            graph.replay()
        for i in range(rem):
            call(i)
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def time_isolated(call, stream, flush, n=9):
    """Median device time of single calls, each after a write of a buffer
    larger than L2 (cold L2, nothing else in flight), with CUDA events on the
    launching stream."""
    times = []
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(n):
            flush.zero_()
            a.record(stream)
            call(i)
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
    return statistics.median(times)



def shared_gpu_splits(binding, w, sms):
    """The split count for calls that share a GPU of `sms` SMs with another
    call in flight: the library's plan for half the SMs (0, the automatic
    plan, for the 128-head path, whose explicit splits change its kernel)."""
    if w.kind == "wide":
        return 0
    return binding.smla_plan_num_splits(w.T, w.H, w.D_qk, w.topk, int(w.kv_fp8), max(1, sms // 2))


def concurrent_steps(binding, w, cache, kvs, sets, dev, stream, args, sinks=None, lanes=3, reps=20):
    """Device milliseconds per step with `lanes` independent steps in flight
    (as a server runs independent batches): step i runs on lane i % lanes,
    each lane its own stream with its own output and workspace buffers, each
    call planned for a shared GPU (shared_gpu_splits); the lanes fork from
    and join back into the timing stream inside one CUDA graph. Returns (ms
    per step, steps timed, splits)."""
    R = len(sets)
    S = shared_gpu_splits(binding, w, torch.cuda.get_device_properties(dev).multi_processor_count)
    ls = [torch.cuda.Stream(device=dev) for _ in range(lanes)]
    calls = [forward_setup(binding, w, cache, kvs, sets, dev, s_, args, sinks, num_splits=S)[0] for s_ in ls]
    G = R * lanes * max(1, 40 // (R * lanes))

    def seq():
        fork = torch.cuda.Event()
        fork.record(stream)
        for s_ in ls:
            s_.wait_event(fork)
        for i in range(G):
            calls[i % lanes](i)
        for s_ in ls:
            join = torch.cuda.Event()
            join.record(s_)
            stream.wait_event(join)

    with torch.cuda.stream(stream):
        seq()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        seq()
    graph.replay()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            graph.replay()
        b.record(stream)
    b.synchronize()
    del graph
    return a.elapsed_time(b) / (reps * G), reps * G, S


def ceiling_configs(row_bytes: int):
    """(CTAs per SM, stages, pair mode, issue warps, copy mode) of the
    gather-ceiling sweep: for each CTA count the most 64-row tiles that fit (as
    the probe pads its CTAs), filled by TMA gather4 copies (copy mode 0) issued
    as the first forward kernels did (issue warps 0) and spread evenly over
    more warps (a warp issues its lanes' copies one after another), or by
    16-byte cp.async copies from eight warps (copy mode 1); and CTA pairs that
    share each tile (1: cluster multicast, 2: bulk copy into the peer)."""
    boxes = (row_bytes + 127) // 128
    tile = 64 * 128 * boxes
    copies = 16 * boxes
    out = []
    for k in (1, 2, 3, 4):
        st = min(8, (233472 // k - 1024 - 1024 - 256) // tile)
        if st >= 1:
            out.append((k, st, 0, 0, 0))
            out.append((k, st, 0, max(-(-copies // 32), max(2, 8 // k)), 0))
            out.append((k, st, 0, 0, 1))
    for pm in (1, 2):
        out.append((1, min(8, (233472 - 1024 - 1024 - 256) // tile), pm, 0, 0))
    return out


def gather_ceiling(binding, cache, sets, stream, reps: int = 4):
    """The pure indexed-row copy probe on this workload's own pool and index
    sets, for 1-4 CTAs per SM and both copy methods: rows/s and GB/s of the
    valid rows."""
    row_bytes = cache.shape[1] * cache.element_size()
    valid = sum(int((s["idx_np"] != -1).sum()) for s in sets)
    sms = torch.cuda.get_device_properties(cache.device).multi_processor_count
    res = []
    for k, st, pm, iw, cm in ceiling_configs(row_bytes):
        ck = torch.zeros(sms * k, dtype=torch.int32, device=cache.device)

        def probe(i, k=k, st=st, pm=pm, iw=iw, cm=cm, ck=ck):
            binding.smla_gather_probe(cache, sets[i % len(sets)]["idx"], ctas_per_sm=k, stages=st, pair_mode=pm,
                                      issue_warps=iw, copy_mode=cm, checksum=ck, stream=stream)
        g = graph_of(probe, len(sets), 3, stream)
        ms = time_steps(g, probe, len(sets), reps * len(sets), stream)
        sec = ms * 1e-3 / reps
        res.append({"ctas_per_sm": k, "stages": st, "pair_mode": pm, "issue_warps": iw,
                    "copy": "cp.async" if cm else "tma_gather4",
                    "rows_per_s": round(valid / sec, 1), "gbs": round(valid * row_bytes / sec / 1e9, 1)})
    best = max((r for r in res if not r["pair_mode"]), key=lambda r: r["gbs"])
    return {"row_bytes": row_bytes, "best_gbs": best["gbs"], "best_rows_per_s": best["rows_per_s"],
            "best": [best["ctas_per_sm"], best["stages"], best["issue_warps"], best["copy"]], "sweep": res,
            "kernel": "smla_gather_probe (TMA tile::gather4 or 16-byte cp.async into a shared-memory ring, "
                      "64-row tiles, no arithmetic)"}


def l2_read_gbs(binding, dev, stream, mb: int = 32, reps: int = 16):
    """L2 -> SM streaming read bandwidth (best of several launches over an
    L2-resident buffer)."""
    buf = torch.ones(mb << 18, dtype=torch.int32, device=dev)   # mb MiB
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ck = torch.zeros(sms * 4, dtype=torch.int32, device=dev)
    best = 0.0
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(8):
            a.record(stream)
            binding.smla_l2_read_probe(buf, reps, sms * 4, checksum=ck, stream=stream)
            b.record(stream)
            b.synchronize()
            if i >= 2:
                best = max(best, buf.numel() * 4 * reps / (a.elapsed_time(b) * 1e-3) / 1e9)
    return best


def measure_config(binding, name, args, dev, stream, flush, l2_gbs):
    """One configuration timed in this process (the same way as the headline)
    with its roofline, isolated-launch time and gather ceiling."""
    w, src, cache, kvs, sets, l2 = build_workload(name, args.seed, 0, dev, 0)
    R = len(sets)
    call, dot, splits = forward_setup(binding, w, cache, kvs, sets, dev, stream, args)
    graph = graph_of(call, R, args.warmup, stream)
    K = max(args.steps, 2 * R)
    ms = time_steps(graph, call, R, K, stream)
    reps, rem = divmod(K, R)
    b_per = [s["bytes"] for s in sets]
    v_per = [int((s["idx_np"] != -1).sum()) for s in sets]
    nbytes = reps * sum(b_per) + sum(b_per[:rem])
    nvalid = reps * sum(v_per) + sum(v_per[:rem])
    sec = ms * 1e-3 / K
    iso = time_isolated(call, stream, flush)
    flop = 2.0 * w.H * (w.D_qk + w.D_v) * nvalid / K
    ceil = gather_ceiling(binding, cache, sets, stream)
    gbs = nbytes / K / sec / 1e9
    ms2, _, s2 = concurrent_steps(binding, w, cache, kvs, sets, dev, stream, args, reps=10)
    entry = {
        "config": {"workload": w.name, "T": w.T, "H": w.H, "D_qk": w.D_qk, "D_v": w.D_v, "topk": w.topk,
                   "num_slots": w.num_slots, "kv_dtype": "e4m3" if w.kv_fp8 else "bf16", "dot_precision": dot,
                   "context_per_row": w.ctx, "splits": splits, "rotating_sets": R,
                   "gathered_bytes_per_call": nbytes / K},
        "steps": K, "ms_per_call": round(ms / K, 6), "ms_isolated_launch": round(iso, 6),
        "gathered_gbs": round(gbs, 2), "query_rows_per_s": round(w.T / sec, 1),
        "tflops": round(flop / sec / 1e12, 2),
        "roofline": roofline(w, nbytes / K, nvalid / K, sec, ncu_traffic(w.name),
                             l2_gbs=l2_gbs if w.kind == "prefill" else None),
        "gather_ceiling": ceil,
        "frac_of_gather_ceiling": round(gbs / ceil["best_gbs"], 4),
        "gpu_launches_per_call": 2 if (w.kind == "wide" and not args.bf16_dots) else 1,
        "concurrent": {"streams": 3, "splits": s2, "ms_per_call": round(ms2, 6),
                       "gathered_gbs": round(nbytes / K / (ms2 * 1e-3) / 1e9, 2),
                       "note": "three independent calls in flight (three streams), per-call device time of the job"},
    }
    if w.kind == "prefill":
        entry["l2_bound"] = {"l2_read_gbs": round(l2_gbs, 1), "bound_ms": round(nbytes / K / (l2_gbs * 1e9) * 1e3, 4),
                             "note": "the %.0f MiB pool is L2-resident: gathered bytes / measured L2 read bandwidth"
                                     % (w.num_slots * w.D_qk * w.kv_bytes_per_elem / 2 ** 20)}
    del graph, sets, cache, src, kvs
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return entry


PER_CONFIG = ("decode_bf16", "decode_fp8", "prefill_bf16", "wide_fp8")


def run_ours(args):
    from sparse_mla_attention_04_gb300 import binding
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    w, src, cache, kvs, sets, l2 = build_workload(args.workload, args.seed, args.rotations, dev, rank, args.ctx)
    R = len(sets)
    sinks = None
    if args.sinks:
        g = np.random.default_rng(args.seed + 7)
        sinks = torch.from_numpy(g.uniform(-2.0, 4.0, w.H).astype(np.float32)).to(dev)
    stream = torch.cuda.Stream(device=dev)
    T, H = w.T, w.H
    call, dot, splits = forward_setup(binding, w, cache, kvs, sets, dev, stream, args, sinks)
    graph = graph_of(call, R, args.warmup, stream)

    K = args.steps
    reps, rem = divmod(K, R)
    bytes_per_step = [s["bytes"] for s in sets]
    total_bytes = reps * sum(bytes_per_step) + sum(bytes_per_step[:rem])
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    ms = time_steps(graph, call, R, K, stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms_max = max_over_ranks(ms, world, dev)
    ms_per_step = ms_max / K
    rows = sum(int((s["idx_np"] != -1).any(axis=1).sum()) for s in sets) / R   # rows with work (all, here)
    gbs = job_rate(total_bytes, world, ms_max) / 1e9
    per_launch_bytes = total_bytes / K
    valid_per_step = [int((s["idx_np"] != -1).sum()) for s in sets]
    valid_per_launch = (reps * sum(valid_per_step) + sum(valid_per_step[:rem])) / K

    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    iso = time_isolated(call, stream, flush)
    per_config = (world == 1 and not args.no_per_config and not (args.q8 or args.bf16_dots or args.sinks)
                  and args.ctx == 0)
    ceil = gather_ceiling(binding, cache, sets, stream) if per_config else None

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(w, cache, kvs, sets, dot,
                      shared_gpu_splits(binding, w, torch.cuda.get_device_properties(dev).multi_processor_count),
                      dev, stream, K, world, q8=args.q8)
    ms2, k2, s2 = concurrent_steps(binding, w, cache, kvs, sets, dev, stream, args, sinks)
    ms2 = max_over_ranks(ms2, world, dev)
    gbs2 = job_rate(per_launch_bytes, world, ms2) / 1e9
    two = {"streams": 3, "splits": s2, "ms_per_step": round(ms2, 6), "value": round(gbs2, 2), "unit": "GB/s",
           "steps": k2,
           "frac_of_hbm_peak": round(gbs2 / measured_peaks()[0], 4), "peak_source": measured_peaks()[1],
           "note": "the same steps with three independent steps in flight (three streams, as a server runs "
                   "independent batches; each call planned for half the SMs); value above is one step at a time"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, src, sets[0])

    pcs = None
    if per_config:
        del graph, sets, cache, src, kvs
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        l2_gbs = l2_read_gbs(binding, dev, stream)
        pcs = {"l2_read_gbs": round(l2_gbs, 1)}
        for name in PER_CONFIG:
            if name != args.workload:
                pcs[name] = measure_config(binding, name, args, dev, stream, flush, l2_gbs)

    if rank == 0:
        line = {
            "metric": "sparse MLA fwd gathered-KV GB/s (%s%s%s)" % (
                w.name, ", pre-quantized q" if args.q8 else (", bf16 dots" if args.bf16_dots else ""),
                ", sinks" if args.sinks else ""),
            "value": round(gbs, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": K,
            "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms_per_step, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("bf16 q . e4m3 codes as fp16 QK / fp16 PV" if args.bf16_dots else "fp8-e4m3 QK / fp16 PV") if w.kv_fp8
                     else "bf16",
            "data": "synthetic (seeded N(0,1) bf16 q and KV, uniform distinct top-k over paged contexts)",
            "config": {
                "workload": w.name, "T": T, "H": H, "D_qk": w.D_qk, "D_v": w.D_v, "topk": w.topk,
                "num_slots": w.num_slots, "kv_dtype": "e4m3" if w.kv_fp8 else "bf16",
                "context_per_row": w.ctx, "splits": splits, "rotating_sets": R,
                "gathered_bytes_per_step": per_launch_bytes,
                "l2": "inputs larger than L2: each step gathers %.0f MB, %d rotating index sets (%.0f MB, L2 %.0f MB)"
                      % (per_launch_bytes / 1e6, R, sum(bytes_per_step) / 1e6, l2 / 1e6),
                "parallelism": "dp%d (independent rows per GPU, no collective)" % world,
                "timing": "CUDA graph of %d calls replayed; CUDA events on the launching stream" % R,
            },
            "query_rows_per_s": round(job_rate(rows * K, world, ms_max), 1),
            "gpu_launches": K * (2 if (w.kind == "wide" and not args.bf16_dots) else 1),
            "roofline": roofline(w, per_launch_bytes, valid_per_launch, ms / K * 1e-3, ncu_traffic(w.name),
                                 l2_gbs=l2_read_gbs(binding, dev, stream) if w.kind == "prefill" else None),
            "ms_isolated_launch": round(iso, 6),
            "clocks": clk,
            "e2e": e2e,
            "concurrent": two,
            "cpu_baseline": cpu,
        }
        if ceil is not None:
            line["gather_ceiling"] = ceil
            line["frac_of_gather_ceiling"] = round(gbs / ceil["best_gbs"], 4)
        if pcs is not None:
            line["per_config"] = pcs
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def quantize_q_per_tensor(binding, q):
    """E4M3 codes of q / s with one per-tensor scale s = amax/448, by the
    library's own scale and quantizing-write kernels (as a producer would)."""
    T, H, D = q.shape
    qs = binding.smla_compute_fp8_scale(q)
    q8 = torch.empty((T * H, D), dtype=torch.uint8, device=q.device)
    rows = torch.arange(T * H, dtype=torch.int64, device=q.device)
    binding.smla_fp8_cache_write(q.reshape(T * H, D), rows, qs, q8)
    return q8.view(T, H, D), qs


def run_e2e(w, cache, kvs, sets, dot, splits, dev, stream, K, world, q8=False, slots=8):
    """Same metric through the public API with host buffers: every step copies
    that step's q and indices from pinned host memory and reads out and lse
    back into pinned host memory, inside the timed region.

    The steps are pipelined as a serving loop would run them: `slots` sets of
    device buffers, each with its own stream on which a step's host->device
    copies, its call and its device->host reads run in order; step i uses slot
    i % slots, so the slots' steps (their copies and calls) overlap one another
    and stream order alone keeps a slot's buffers from being reused early."""
    from sparse_mla_attention_04_gb300 import binding
    R = len(sets)
    NB = slots
    qkey = "q8" if q8 else "q"
    hq = [s[qkey].cpu().pin_memory() for s in sets]
    hi = [s["idx"].cpu().pin_memory() for s in sets]
    ho = [torch.empty((w.T, w.H, w.D_v), dtype=torch.bfloat16).pin_memory() for _ in range(NB)]
    hl = [torch.empty((w.T, w.H), dtype=torch.float32).pin_memory() for _ in range(NB)]
    dq = [torch.empty_like(sets[0][qkey]) for _ in range(NB)]
    di = [torch.empty_like(sets[0]["idx"]) for _ in range(NB)]
    out = [torch.empty((w.T, w.H, w.D_v), dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    lse = [torch.empty((w.T, w.H), dtype=torch.float32, device=dev) for _ in range(NB)]
    need = binding.sparse_mla_fwd_workspace_size(w.T, w.H, w.D_qk, w.D_v, w.topk, int(w.kv_fp8), splits)
    ws = [torch.zeros(max(need, 1), dtype=torch.uint8, device=dev) for _ in range(NB)]
    ss = [torch.cuda.Stream(device=dev) for _ in range(NB)]

    def step(i):
        k = i % NB
        with torch.cuda.stream(ss[k]):
            dq[k].copy_(hq[i % R], non_blocking=True)
            di[k].copy_(hi[i % R], non_blocking=True)
            if q8:
                binding.sparse_mla_fwd_q8(dq[k], sets[i % R]["qs"], cache, di[k], w.scale, kv_scale=kvs, D_v=w.D_v,
                                          out=out[k], lse=lse[k], workspace=ws[k], num_splits=splits, stream=ss[k])
            else:
                binding.sparse_mla_fwd(dq[k], cache, di[k], w.scale, kv_scale=kvs, dot_precision=dot, D_v=w.D_v,
                                       out=out[k], lse=lse[k], workspace=ws[k], num_splits=splits, stream=ss[k])
            ho[k].copy_(out[k], non_blocking=True)
            hl[k].copy_(lse[k], non_blocking=True)

    def sequence(n):
        # fork the slot streams off the timing stream, run n steps, join them back
        fork = torch.cuda.Event()
        fork.record(stream)
        for s_ in ss:
            s_.wait_event(fork)
        for i in range(n):
            step(i)
        for s_ in ss:
            join = torch.cuda.Event()
            join.record(s_)
            stream.wait_event(join)

    # the host issues ~6 CUDA operations per step, more than a call's device
    # time: the pipelined sequence is captured once as a CUDA graph and replayed
    G = R * NB * max(1, 40 // (R * NB))
    sequence(G)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sequence(G)
    graph.replay()
    torch.cuda.synchronize(dev)
    reps_g = max(1, -(-min(K, 4000) // G))
    steps = reps_g * G
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps_g):
            graph.replay()
        b.record(stream)
    b.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    # the results each slot read back last (step G - NB + k of the sequence)
    # against the same call on device-resident inputs, bit for bit
    verified = True
    for k in range(NB):
        i = G - NB + k
        ref_o = torch.empty_like(out[k])
        ref_l = torch.empty_like(lse[k])
        if q8:
            binding.sparse_mla_fwd_q8(sets[i % R][qkey], sets[i % R]["qs"], cache, sets[i % R]["idx"], w.scale,
                                      kv_scale=kvs, D_v=w.D_v, out=ref_o, lse=ref_l, workspace=ws[k],
                                      num_splits=splits, stream=stream)
        else:
            binding.sparse_mla_fwd(sets[i % R][qkey], cache, sets[i % R]["idx"], w.scale, kv_scale=kvs,
                                   dot_precision=dot, D_v=w.D_v, out=ref_o, lse=ref_l, workspace=ws[k],
                                   num_splits=splits, stream=stream)
        stream.synchronize()
        verified &= bool(torch.equal(ho[k], ref_o.cpu()) and torch.equal(hl[k], ref_l.cpu()))
    reps, rem = divmod(steps, R)
    nbytes = reps * sum(s["bytes"] for s in sets) + sum(s["bytes"] for s in sets[:rem])
    h2d = sets[0][qkey].numel() * sets[0][qkey].element_size() + sets[0]["idx"].numel() * 4
    d2h = out[0].numel() * 2 + lse[0].numel() * 4
    return {"value": round(job_rate(nbytes, world, ms) / 1e9, 2), "unit": "GB/s", "steps": steps,
            "ms_per_step": round(ms / steps, 6), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "results_match_device_call": verified, "splits": splits,
            "pipelining": "%d buffer slots, each with its own stream running a step's copies in, call and "
                          "copies out in order; the slots' steps overlap one another, each call planned for "
                          "half the SMs (splits 0 = the automatic plan); sequences of %d steps replayed from a "
                          "CUDA graph" % (NB, G)}


# ----------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------

def oracle_scale(src):
    """The oracle's per-tensor fp8 scale of the whole bf16 source (chunked amax)."""
    import oracle
    amax = 0.0
    for r0 in range(0, src.shape[0], 1 << 20):
        amax = max(amax, oracle.amax_bf16(src[r0:r0 + (1 << 20)].cpu()))
    return float(oracle.fp8_scale_from_amax(amax))


def oracle_inputs(w, src, s, rows, kvs_val):
    """Rows `rows` of a set, with the source rows their indices name gathered
    from the device pool and renumbered densely (the oracle reads a host array;
    an fp8 cache is encoded by the oracle itself from the bf16 source)."""
    import oracle
    idx = s["idx_np"][rows]
    uniq = np.unique(idx[idx >= 0])
    remap = np.where(idx >= 0, np.searchsorted(uniq, np.maximum(idx, 0)), -1).astype(np.int32)
    kv_rows = src[torch.from_numpy(uniq).to(src.device)].cpu()
    if w.kv_fp8:
        kv_rows = oracle.fp8_quantize(kv_rows, kvs_val)
    q = s["q"][torch.from_numpy(np.asarray(rows)).to(s["q"].device)].cpu()
    nbytes = int((idx != -1).sum()) * w.D_qk * w.kv_bytes_per_elem
    return q, kv_rows, remap, nbytes


def time_oracle(w, q, kv_rows, remap, kvs_val, nthreads: int = 0):
    import oracle
    t0 = time.perf_counter()
    oracle.sparse_mla(q, kv_rows, remap, w.scale, kv_fp8=w.kv_fp8, kv_scale=kvs_val, D_v=w.D_v,
                      q_mode=1 if w.kv_fp8 else 0, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(w, src, s, budget_s: float = 10.0):
    import oracle
    cores = oracle.max_threads()
    kvs_val = oracle_scale(src) if w.kv_fp8 else 1.0
    rows = list(range(w.T))
    q, kv_rows, remap, nbytes = oracle_inputs(w, src, s, rows, kvs_val)
    done, el, reps = 0, 0.0, 0
    while el < budget_s and reps < 50:
        el += time_oracle(w, q, kv_rows, remap, kvs_val)
        done += nbytes
        reps += 1
    # the same oracle on one core, over a few rows of the same set
    rows1 = list(range(min(8, w.T)))
    q1, kv1, remap1, nbytes1 = oracle_inputs(w, src, s, rows1, kvs_val)
    done1, el1, reps1 = 0, 0.0, 0
    while el1 < budget_s / 4 and reps1 < 20:
        el1 += time_oracle(w, q1, kv1, remap1, kvs_val, nthreads=1)
        done1 += nbytes1
        reps1 += 1
    return {"value": round(done / el / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d pass(es) over all %d rows of one index set (%d heads, fp64 C + OpenMP), %.1f s"
                      % (reps, w.T, w.H, el),
            "value_1core": round(done1 / el1 / 1e9, 4),
            "sample_1core": "%d pass(es) over %d rows of the same set on 1 thread, %.1f s" % (reps1, len(rows1), el1)}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    dev = torch.device("cuda", local) if torch.cuda.is_available() else None
    if dev is None:
        print(json.dumps({"impl": "reference", "unavailable": "no CUDA device to build the workload on"}))
        return
    torch.cuda.set_device(dev)
    w, src, cache, kvs, sets, l2 = build_workload(args.workload, args.seed, max(args.rotations, 1), dev, 0)
    kvs_val = oracle_scale(src) if w.kv_fp8 else 1.0
    s = sets[0]
    # one query row (all heads) per step
    prepared = [oracle_inputs(w, src, s, [t], kvs_val) for t in range(w.T)]
    for i in range(max(args.warmup, 3)):
        p = prepared[i % w.T]
        time_oracle(w, p[0], p[1], p[2], kvs_val)
    K = args.steps
    el, nbytes = 0.0, 0
    for i in range(K):
        p = prepared[i % w.T]
        el += time_oracle(w, p[0], p[1], p[2], kvs_val)
        nbytes += p[3]
    value = nbytes / el / 1e9
    line = {
        "impl": "reference",
        "metric": "sparse MLA fwd gathered-KV GB/s (%s)" % w.name,
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(el * 1e3 / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (same seeded workload as the GPU arm)",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "D_qk": w.D_qk, "topk": w.topk,
                   "step": "one query row (all %d heads) of the workload" % w.H},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": "one query row per step, %d steps" % K},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the fused producer step (RoPE on q_pe / k_pe, q concat, cache write)
# ----------------------------------------------------------------------------

PRODUCER_T, PRODUCER_H, PRODUCER_POS = 4096, 128, 8192
PRODUCER_Q_SCALE, PRODUCER_KV_SCALE = 0.0137, 0.0211


def producer_bytes(T: int, H: int, cache_rows: int) -> int:
    """Algorithmic bytes of one call with E4M3 q_out and cache: bf16 ql_nope,
    q_pe, kv_c, k_pe, the positions and slots, one cos/sin row per token read;
    q_out and the cache rows written."""
    reads = T * H * 576 * 2 + T * 576 * 2 + T * 8 * 2 + T * 64 * 4
    writes = T * H * 576 + cache_rows * 576
    return reads + writes


def run_producer(args):
    from sparse_mla_attention_04_gb300 import binding
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    T, H, P = PRODUCER_T, PRODUCER_H, PRODUCER_POS
    ql, qp, kc, kp, pos, slots, ns = inputs.producer_inputs(T, H, rank_seed(args.seed, 0, rank), P, num_slots=2 * T)
    cs = inputs.rope_cos_sin_cache(P)
    nbytes = producer_bytes(T, H, T)
    cfg = {"workload": "producer", "T": T, "H": H, "D_latent": 512, "D_rope": 64, "max_position": P,
           "q_out": "e4m3", "kv_cache": "e4m3", "rope": "neox", "num_slots": ns,
           "bytes_per_step": nbytes,
           "l2": "inputs larger than L2: each step reads %.0f MB and writes %.0f MB"
                 % ((nbytes - T * H * 576 - T * 576) / 1e6, (T * H * 576 + T * 576) / 1e6),
           "parallelism": "dp%d (independent tokens per GPU, no collective)" % world}
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(producer_reference(args, ql, qp, kc, kp, pos, slots, cs, ns, cfg)), flush=True)
        return
    d = [x.to(dev) for x in (ql, qp, kc, kp, pos, slots, cs)]
    cache = torch.zeros((ns, 576), dtype=torch.uint8, device=dev)
    q_out = torch.empty((T, H, 576), dtype=torch.uint8, device=dev)
    kvs = torch.tensor([PRODUCER_KV_SCALE], dtype=torch.float32, device=dev)
    qs = torch.tensor([PRODUCER_Q_SCALE], dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call():
        binding.smla_fused_qk_rope_cache(d[0], d[1], d[2], d[3], d[4], d[6], d[5], cache, is_neox=True,
                                         kv_scale=kvs, q_out=q_out, q_out_fp8=True, q_scale=qs, stream=stream)

    G = 10
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            call()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(G):
                call()
        graph.replay()
        stream.synchronize()
    K = max(G, (args.steps // G) * G)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(K // G):
            graph.replay()
        end.record(stream)
    end.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, world, dev)
    gbs = job_rate(nbytes * K, world, ms_max) / 1e9
    hbm, hbm_src = measured_peaks()
    per_launch = ms / K * 1e-3
    e2e = None
    if not args.no_e2e:
        e2e = producer_e2e(binding, (ql, qp, kc, kp), d, cache, q_out, kvs, qs, stream, nbytes, world, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = producer_reference(args, ql, qp, kc, kp, pos, slots, cs, ns, cfg, cpu_leg=True)
    if rank == 0:
        achieved = nbytes / per_launch / 1e9
        line = {
            "metric": "fused producer step GB/s (RoPE + q concat + cache write, producer)",
            "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms_max / K, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in, e4m3 out (binary32 rotation)",
            "data": "synthetic (seeded N(0,1) bf16 inputs, uniform positions, distinct slots)",
            "config": dict(cfg, timing="CUDA graph of %d calls replayed; CUDA events on the launching stream" % G),
            "tokens_per_s": round(job_rate(T * K, world, ms_max), 1),
            "gpu_launches": K,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "traffic": ncu_traffic("producer"),
                         "peak_source": hbm_src, "algorithmic_bytes_per_launch": nbytes},
            "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def producer_e2e(binding, host_in, d, cache, q_out, kvs, qs, stream, nbytes, world, dev):
    """The step through the public API with pinned host buffers: the four bf16
    inputs copied in and q_out read back every step (positions, slots and the
    cos/sin table stay resident), timed together."""
    hin = [x.pin_memory() for x in host_in]
    hout = torch.empty(q_out.shape, dtype=q_out.dtype).pin_memory()
    steps = 10
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(steps + 1):
            if i == 1:
                a.record(stream)
            for h, x in zip(hin, d[:4]):
                x.copy_(h, non_blocking=True)
            binding.smla_fused_qk_rope_cache(d[0], d[1], d[2], d[3], d[4], d[6], d[5], cache, is_neox=True,
                                             kv_scale=kvs, q_out=q_out, q_out_fp8=True, q_scale=qs, stream=stream)
            hout.copy_(q_out, non_blocking=True)
        b.record(stream)
    b.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    h2d = sum(x.numel() * x.element_size() for x in hin)
    d2h = hout.numel() * hout.element_size()
    return {"value": round(job_rate(nbytes * steps, world, ms) / 1e9, 2), "unit": "GB/s", "steps": steps,
            "ms_per_step": round(ms / steps, 6), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def producer_reference(args, ql, qp, kc, kp, pos, slots, cs, ns, cfg, cpu_leg: bool = False):
    """The oracle (binary32 mirror, OpenMP) on a bounded sample: 16 tokens with
    all heads per step; the value is scaled to bytes per second of the same
    per-token work."""
    import oracle
    oracle.build()
    T, H = ql.shape[0], ql.shape[1]
    n = 16
    cache = np.zeros((ns, 576), dtype=np.uint8)
    chunks = []
    for i in range(0, T, n):
        chunks.append((ql[i:i + n], qp[i:i + n], kc[i:i + n], kp[i:i + n], pos[i:i + n], slots[i:i + n]))
    K = 3 if cpu_leg else max(1, args.steps)
    W = 1 if cpu_leg else max(args.warmup, 3)

    def one(c):
        oracle.fused_qk_rope_cache(c[0], c[1], c[2], c[3], c[4], cs, True, c[5], cache, cache_fp8=True,
                                   kv_scale=PRODUCER_KV_SCALE, q_out_fp8=True, q_scale=PRODUCER_Q_SCALE, mode=1)

    for i in range(W):
        one(chunks[i % len(chunks)])
    t0 = time.perf_counter()
    for i in range(K):
        one(chunks[i % len(chunks)])
    el = time.perf_counter() - t0
    value = producer_bytes(n, H, n) * K / el / 1e9
    sample = "%d step(s) of %d tokens x %d heads (fp32-mirror C + OpenMP)" % (K, n, H)
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
           "sample": sample}
    if cpu_leg:
        return cpu
    return {"impl": "reference", "metric": "fused producer step GB/s (RoPE + q concat + cache write, producer)",
            "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": W,
            "ms_per_step": round(el * 1e3 / K, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 mirror", "data": "synthetic (same seeded workload as the GPU arm)",
            "config": dict(cfg, step="%d tokens (all %d heads) of the workload" % (n, H)),
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------
# the per-call sweep (rows x fan-out), automatic split plan against fixed ones
# ----------------------------------------------------------------------------

SWEEP_ROWS = (2, 16, 256, 512, 1024, 2048, 16384)
SWEEP_FANOUT = (128, 512, 2048)
SWEEP_SPLITS = (1, 2, 3, 4, 6, 8, 16)
SWEEP_POOL = 2 * 1024 * 1024


def run_sweep(args):
    """Per-call device time over the grid the pages measure per call (16 heads,
    D=512, bf16 cache; each row gathers `fan-out` uniform random slots of a
    shared 2M-slot pool), for the automatic split plan and for fixed split
    counts; reports where the plan is not the fastest."""
    from sparse_mla_attention_04_gb300 import binding
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    H, D = 16, 512
    scale = 1.0 / math.sqrt(D)
    pool = inputs.normal_bf16((SWEEP_POOL, D), 11, dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.Stream(device=dev)
    points = []
    for rows in SWEEP_ROWS:
        q = inputs.normal_bf16((rows, H, D), 12 + rows, dev)
        out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((rows, H), dtype=torch.float32, device=dev)
        for fan in SWEEP_FANOUT:
            g = torch.Generator(device=dev)
            g.manual_seed(rows * 7919 + fan)
            # uniform random slots per row (a duplicate, rare here, counts with multiplicity)
            idx = torch.randint(0, SWEEP_POOL, (rows, fan), generator=g, device=dev)
            idx = idx.to(torch.int32).contiguous()
            auto_s = binding.smla_plan_num_splits(rows, H, D, fan, 0, sms)
            choices = sorted(set(SWEEP_SPLITS) | {auto_s})
            times = {}
            for S in choices:
                try:
                    need = binding.sparse_mla_fwd_workspace_size(rows, H, D, D, fan, 0, S)
                except binding.SmlaError:
                    continue   # more than 8 splits need rows * H / 16 <= 4096
                ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=dev)

                def call():
                    binding.sparse_mla_fwd(q, pool, idx, scale, out=out, lse=lse, workspace=ws, num_splits=S,
                                           stream=stream)
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        call()
                    stream.synchronize()
                    reps = max(3, min(50, int(2e9 / max(1, rows * fan * D * 2))))
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for _ in range(reps):
                        call()
                    b.record(stream)
                b.synchronize()
                times[S] = a.elapsed_time(b) / reps * 1000.0
            best = min(times, key=times.get)
            points.append({"rows": rows, "fanout": fan, "auto_splits": auto_s,
                           "us_auto": round(times[auto_s], 2), "best_splits": best,
                           "us_best": round(times[best], 2),
                           "auto_over_best": round(times[auto_s] / times[best], 3),
                           "us_by_splits": {str(k): round(v, 2) for k, v in times.items()},
                           "gbs_auto": round(rows * fan * D * 2 / (times[auto_s] * 1e-6) / 1e9, 1)})
    worst = max(points, key=lambda p: p["auto_over_best"])
    line = {"metric": "sparse MLA fwd per-call time sweep (H=16, D=512, bf16)", "unit": "us",
            "higher_is_better": False, "n_gpus": 1, "points": points,
            "auto_over_best_worst": worst["auto_over_best"], "worst_point": [worst["rows"], worst["fanout"]],
            "config": {"workload": "sweep", "rows": list(SWEEP_ROWS), "fanout": list(SWEEP_FANOUT),
                       "splits_tried": list(SWEEP_SPLITS), "pool_slots": SWEEP_POOL,
                       "timing": "CUDA events around repeated calls on one stream after 3 warm-up calls"}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.sweep:
        run_sweep(args)
        return
    if args.workload == "producer":
        run_producer(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
