#!/usr/bin/env python
"""Benchmark: one step = forward (o, lse) + backward (Delta, dK/dV, dQ) of
causal / sliding-window GQA attention over one synthetic workload, through
the C ABI, on each GPU of one node.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Prints ONE JSON line on rank 0.  `value` is useful TFLOP/s summed over all
ranks: in-band (query, key) pairs x (4 D forward + 10 D backward) flops,
divided by the device time of the K timed steps (max over ranks).  Each rank
runs its own independent copy of the workload (weak scaling, no collective on
the data path).  L2 is flushed (256 MiB write) before every timed step and
the flush is outside the timed events.

The default workload is the wide-head global layer at 16,384 tokens (B 1,
32 query heads, 4 kv heads, D 512, causal).  The two windowed head-dim-256
layers (8,192 tokens, and the ragged 30,553-token step with outlier keys)
are measured after it, the same way, and reported in the same line under
`sub_workloads`, each with its own value, split, roofline and workspace.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# the wide-head global layer at 16,384 tokens; the two windowed D = 256 layers
# the metric is quoted for run as sub-records of the same line
DEFAULT_WORKLOAD = "global_l16384_d512"
DEFAULT_SUB_WORKLOADS = ("sliding_l8192_d256_w1024", "ragged_l30553_d256_w1024_outliers")
METRIC = "windowed attn fwd+bwd useful TFLOP/s & % bf16 TC peak; peak workspace GB"
SM_COUNT = 152
FP32_LANES_PER_SM = 128

# per-kernel flops the tensor cores ISSUE per in-band (query, key) pair, in
# units of D (the backward recomputes S and dP in both of its passes)
KERNEL_FLOPS_PER_PAIR_D = {
    "fwd_tc": 4,          # S = Q K^T, O += P V (tcgen05)
    "fwd_simt": 4,        # S = Q K^T, O += P V
    "bwd_dkdv_simt": 8,   # S, dP recomputed; dV += P^T dO; dK += dS^T Q
    "bwd_dq_simt": 6,     # S, dP recomputed; dQ += dS K
    "bwd_dkdv_tc": 8,     # S^T, dP^T recomputed; dV += P^T dO; dK += dS^T Q (tcgen05)
    "bwd_dq_tc": 6,       # S, dP recomputed; dQ += dS K (tcgen05)
}
# the backward's two passes, launched on two streams that run concurrently
CONCURRENT_BWD = ("bwd_dkdv_tc", "bwd_dq_tc")
# USEFUL flops per in-band pair, in units of D: forward Q K^T and P V (4 D);
# backward S, dP, dV, dQ, dK once each (10 D, the convention the metric uses)
USEFUL_FWD_PER_PAIR_D = 4
USEFUL_BWD_PER_PAIR_D = 10
HBM_KERNELS = {"bwd_delta", "convert_f16", "bwd_prep", "bwd_dscale", "fwd_decode"}
# the backward's launches before its two concurrent passes
BWD_PREP_KERNELS = ("bwd_dscale", "bwd_prep")
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--seq-len", type=int, default=0,
                   help="override the workload's sequence length (smaller cases for profiler captures)")
    p.add_argument("--sub-workloads", default=None,
                   help="comma-separated workloads measured after the main one and reported in its line under "
                        "sub_workloads ('' for none; default: the two windowed D = 256 layers when the main "
                        "workload is the default)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target length of the CPU baseline sample")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, sm_max_mhz=2070.0,
                source="fallback")


# source file that defines each kernel (for matching ncu counters to the current code)
KERNEL_SOURCE = {
    "fwd_simt": "simt_kernels.cu", "bwd_delta": "simt_kernels.cu", "bwd_dkdv_simt": "simt_kernels.cu",
    "bwd_dq_simt": "simt_kernels.cu", "fwd_tc": "tc_fwd.cu", "convert_f16": "tc_fwd.cu",
    "bwd_prep": "tc_bwd.cu", "bwd_dscale": "tc_bwd.cu", "bwd_dkdv_tc": "tc_bwd.cu", "bwd_dq_tc": "tc_bwd.cu",
}
# head dim 512: the tensor-core launches of the forward and backward come from the cluster kernels
KERNEL_SOURCE_D512 = {"fwd_tc": "tc_fwd512.cu", "bwd_dkdv_tc": "tc_bwd512.cu", "bwd_dq_tc": "tc_bwd512.cu"}


def source_digest(kernel: str, D: int = 0) -> str:
    """First 16 hex digits of the sha256 of the kernel's source file."""
    name = (KERNEL_SOURCE_D512.get(kernel) if D == 512 else None) or KERNEL_SOURCE.get(kernel)
    if name is None:
        return "unknown"
    with open(os.path.join(ROOT, "sliding_window_attention_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def unit_times(kernels: dict, bwd_ms: float, steps: int) -> dict:
    """Launch name -> (launches, total ms), with the tensor-core backward's
    dK/dV and dQ passes as one unit ("bwd_dkdv_tc+bwd_dq_tc").  The two run
    side by side (two streams, or one launched early beside the other on one
    stream), so their own spans overlap; the unit is timed from the end of
    the backward prep to the end of the backward call: `bwd_ms` minus the
    average launch times of the prep kernels, per step.  The units then do
    not overlap, and their totals divide into the step."""
    if not (all(n in kernels for n in CONCURRENT_BWD) and "bwd_prep" in kernels and bwd_ms):
        return dict(kernels)
    group_ms = bwd_ms - sum(kernels[n][1] / kernels[n][0] for n in BWD_PREP_KERNELS if n in kernels)
    units = {n: v for n, v in kernels.items() if n not in CONCURRENT_BWD}
    units["+".join(CONCURRENT_BWD)] = (kernels[CONCURRENT_BWD[0]][0], group_ms * steps)
    return units


def dominant_unit(kernels: dict, bwd_ms: float, steps: int):
    """(name, average ms per launch) of the unit with the most time per step
    (`unit_times`: the concurrent dK/dV and dQ passes count as one unit)."""
    name, (launches, total) = max(unit_times(kernels, bwd_ms, steps).items(), key=lambda kv: kv[1][1])
    return name, total / launches


def ncu_traffic(kernel: str, workload: str, D: int = 0):
    """DRAM bytes per launch recorded by an ncu capture (profiles/ncu_traffic.txt),
    or None when absent or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(kernel, D)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            if parts[3] == digest:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                     hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.tmp.name)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower() in ("active", "0x1", "1"):
                    reasons.add(name)
        loaded = [r["sm"] for r in rows if r["power"] > 0] or [r["sm"] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, max_ms: float) -> float:
    """Work of all ranks (each runs its own copy of the workload) over the slowest rank's time."""
    return world * flops_per_step * steps / (max_ms / 1e3) / 1e12


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local_rank


def _sample_q_rows(w, Ls):
    """Query rows of an oracle sample over the first Ls key positions: the
    workload's suffix fraction of Ls (all Ls for self-attention)."""
    return Ls if w.q_rows == w.L else max(1, round(Ls * w.q_rows / w.L))


def _sample_prefix(w, Ls):
    """The shared-prefix plan of an oracle sample over the first Ls tokens:
    the workload's prompt and chosen lengths scaled by Ls / L (None without
    a plan)."""
    if not w.prefix:
        return None
    P = round(w.prompt_len * Ls / w.L)
    Rc = min(Ls - P, round(w.chosen_len * Ls / w.L))
    return P, Rc


def _sample_pairs(w, Ls):
    from sliding_window_attention_gb300.inputs import band_pairs, band_pairs_ex, band_pairs_prefix

    if w.prefix:
        return band_pairs_prefix(Ls, w.window, *_sample_prefix(w, Ls))
    if w.q_rows == w.L and w.causal:
        return band_pairs(Ls, w.window)
    return band_pairs_ex(_sample_q_rows(w, Ls), Ls, w.window, w.causal)


def _oracle_sample_inputs(w, Ls, group=0):
    from sliding_window_attention_gb300.inputs import make_inputs

    G = w.Hq // w.Hkv
    q, k, v, dO = make_inputs(1, G, 1, Ls, w.D, w.seed + 104729 * group, w.do_scale, w.outlier_frac,
                              w.outlier_mult)
    nq = _sample_q_rows(w, Ls)
    if nq < Ls:
        q, dO = (t[:, :, Ls - nq:].contiguous() for t in (q, dO))
    return q, k, v, dO


def oracle_sample_seconds(w, Ls, inputs=None):
    """Seconds the fp64 oracle takes for its complete forward + backward (band
    mode) on one kv-head group (G query heads) over the first Ls tokens."""
    import oracle

    q, k, v, dO = inputs if inputs is not None else _oracle_sample_inputs(w, Ls)
    t0 = time.perf_counter()
    plan = _sample_prefix(w, q.shape[2])
    if w.fwd_only:
        oracle.forward(q, k, v, w.window, w.scale, band_only=True, causal=w.causal, prefix=plan)
    else:
        oracle.backward(q, k, v, dO, w.window, w.scale, band_only=True, causal=w.causal, prefix=plan)
    return time.perf_counter() - t0


def oracle_sample_length(w, target_s: float) -> int:
    """Sequence length Ls whose oracle sample takes about target_s seconds
    (cost model: proportional to the in-band pair count)."""
    import oracle

    oracle.build()
    Ls = min(256, w.L)
    t = oracle_sample_seconds(w, Ls)
    for _ in range(4):
        if t >= 0.6 * target_s or Ls >= w.L:
            break
        want_pairs = _sample_pairs(w, Ls) * target_s / max(t, 1e-3)
        lo, hi = Ls, w.L
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if _sample_pairs(w, mid) <= want_pairs:
                lo = mid
            else:
                hi = mid - 1
        if lo <= Ls:
            break
        Ls = lo
        t = oracle_sample_seconds(w, Ls)
    return Ls


def oracle_useful_flops(w, Ls) -> int:
    return (4 if w.fwd_only else 14) * w.D * (w.Hq // w.Hkv) * _sample_pairs(w, Ls)


def cpu_oracle_sample(w, target_s: float):
    """(useful TFLOP/s, seconds, Ls, threads, groups) of one oracle sample of
    about target_s: the first Ls tokens of one kv-head group, and when one
    group over the whole sequence ends early, further kv-head groups (each
    with its own seeded inputs) until the sample reaches about target_s."""
    import oracle

    Ls = oracle_sample_length(w, target_s)
    secs = oracle_sample_seconds(w, Ls)
    groups = 1
    while Ls >= w.L and secs < 0.8 * target_s and groups < w.B * w.Hkv:
        secs += oracle_sample_seconds(w, Ls, _oracle_sample_inputs(w, Ls, groups))
        groups += 1
    return groups * oracle_useful_flops(w, Ls) / secs / 1e12, secs, Ls, oracle.num_threads(), groups


def run_reference(args, w, world, rank):
    """The reference arm: the fp64 CPU oracle on the host cores, each step a
    bounded sample of the same workload (one kv-head group, first Ls tokens)."""
    if rank != 0:
        return 0
    import oracle

    steps, warm = args.steps, args.warmup
    per_step = max(0.5, min(8.0, 150.0 / max(1, steps + warm)))
    Ls = oracle_sample_length(w, per_step)
    inputs = _oracle_sample_inputs(w, Ls)
    secs = []
    for it in range(warm + steps):
        t = oracle_sample_seconds(w, Ls, inputs)
        if it >= warm:
            secs.append(t)
    flops = oracle_useful_flops(w, Ls)
    value = flops * steps / sum(secs) / 1e12
    G = w.Hq // w.Hkv
    sample = (f"fp64 oracle fwd+bwd (band mode) on 1 kv-head group ({G} query heads) x first {Ls} tokens "
              f"({_sample_q_rows(w, Ls)} query rows) of {w.name} per step; useful flops counted as on the GPU")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(1e3 * sum(secs) / steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) inputs rounded to bf16)",
        "config": dict({"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "L": w.L, "D": w.D,
                        "window": w.window}, **_variant_keys(w)),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _band_keys(w):
    """Keys that some query row of the workload sees (the decode kernel's range)."""
    off = w.L - w.q_rows
    win = w.window if 0 < w.window < w.L else 0
    lo = max(0, off - win + 1) if win else 0
    last = w.L - 1  # the last query row sits at key position L - 1
    hi = last if w.causal else (min(w.L - 1, last + win - 1) if win else w.L - 1)
    return hi - lo + 1


def _variant_keys(w):
    """Config keys of a band variant (queries a suffix of the keys, or non-causal)."""
    out = {}
    if w.q_rows != w.L:
        out["Lq"] = w.q_rows
    if not w.causal:
        out["causal"] = False
    if w.fwd_only:
        out["step"] = "forward only (decode)"
    if w.prefix:
        out["prompt_len"], out["chosen_len"] = w.prefix
        out["rejected_len"] = w.L - sum(w.prefix)
    return out


def roofline_record(kname: str, avg_ms: float, w, peaks: dict) -> dict:
    """Roofline entry of the dominant unit `kname` (one kernel, or the
    backward's two concurrent passes joined by '+') at `avg_ms` per launch.

    Tensor-core units count USEFUL flops: 4 D per in-band pair for the
    forward and 10 D for the backward (S, dP, dV, dQ, dK once each), so frac
    is the useful-flop fraction of the bf16 peak.  What the kernels issue (the
    backward recomputes S and dP in each pass) is reported beside it as
    issued_flops_per_pair_d.  HBM-bound units count their algorithmic bytes."""
    B, Hq, Hkv, L, D, Lq = w.B, w.Hq, w.Hkv, w.L, w.D, w.q_rows
    avg_s = avg_ms / 1e3
    if kname in HBM_KERNELS:
        if kname == "bwd_delta":
            alg = B * Hq * Lq * (D * 4 + D * 2 + 4)
        elif kname == "bwd_prep":  # q, k, v, dO: bf16 read + fp16 write; o (fp32) and lse read; stats written
            alg = 4 * D * B * (2 * Hq * Lq + 2 * Hkv * L) + B * Hq * Lq * (4 * D + 4 + 8)
        elif kname == "bwd_dscale":  # dO (bf16) read once
            alg = 2 * D * B * Hq * Lq
        elif kname == "fwd_decode":  # the K and V rows in band (bf16) once per kv head, q in, o and lse out
            alg = B * Hkv * _band_keys(w) * D * 2 * 2 + B * Hq * Lq * (D * 2 + D * 4 + 4)
        else:  # convert_f16 (forward): bf16 read + fp16 write of v
            alg = 4 * D * B * Hkv * L
        achieved = alg / avg_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "bytes_per_launch": alg}
    else:
        names = kname.split("+")

        issued = sum(KERNEL_FLOPS_PER_PAIR_D.get(n, 4) for n in names)
        if names[0].startswith("fwd"):
            useful = USEFUL_FWD_PER_PAIR_D
        elif tuple(names) == CONCURRENT_BWD or set(names) == {"bwd_dkdv_simt", "bwd_dq_simt"}:
            useful = USEFUL_BWD_PER_PAIR_D
        else:  # one backward pass on its own: its share of the useful work is not defined; count issued
            useful = issued
        achieved = useful * D * w.pairs() / avg_s / 1e12
        if kname.endswith("_simt"):
            peak = SM_COUNT * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
            roof = {"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 1), "unit": "TFLOP/s",
                    "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 flop x max SM clock"}
        else:
            roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "peak_source": f"{peaks['source']} bf16 dense (burst)"}
        roof["flops_per_pair_d"] = useful
        roof["issued_flops_per_pair_d"] = issued
        roof["pairs"] = w.pairs()
    roof["kernel"] = kname
    roof["ms_per_launch"] = round(avg_ms, 5)
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    parts = [ncu_traffic(n, w.name, D) for n in kname.split("+")]
    roof["traffic"] = None if None in parts else sum(parts)
    return roof


def split_record(w, fwd_ms: float, bwd_ms: float, peaks: dict) -> dict:
    """Forward and backward separately, from events on the caller's stream
    around each call: forward at 4 D useful flops per pair, backward at 10 D
    (and at 8 D, the count without the S / dP recompute)."""
    pk = peaks["bf16_tflops"]
    split = {"fwd": {"ms": round(fwd_ms, 4), "tflops": round(w.fwd_flops() / (fwd_ms * 1e9), 2) if fwd_ms else None}}
    split["fwd"]["pct_bf16_peak"] = round(100 * split["fwd"]["tflops"] / pk, 2) if fwd_ms else None
    if not w.fwd_only and bwd_ms:
        t10 = w.bwd_flops() / (bwd_ms * 1e9)
        t8 = 8 * w.D * w.pairs() / (bwd_ms * 1e9)
        split["bwd"] = {"ms": round(bwd_ms, 4), "tflops_10d": round(t10, 2),
                        "pct_bf16_peak_10d": round(100 * t10 / pk, 2), "tflops_8d": round(t8, 2),
                        "pct_bf16_peak_8d": round(100 * t8 / pk, 2)}
    return split


def measure_workload(args, w, world, rank, local_rank, dist, peaks):
    """Time K steps (after W warm-up steps) of workload `w` on this rank's GPU
    and the same through pinned host buffers (e2e); returns the fields of one
    bench record (rank 0's view, timings already maxed over ranks)."""
    import torch

    import sliding_window_attention_gb300 as swa
    from sliding_window_attention_gb300.inputs import make_inputs

    dev = torch.device(f"cuda:{local_rank}")
    # each rank: one independent copy of the workload (seed offset by rank)
    q_h, k_h, v_h, dO_h = make_inputs(w.B, w.Hq, w.Hkv, w.L, w.D, w.seed + 7919 * rank, w.do_scale,
                                      w.outlier_frac, w.outlier_mult)
    B, Hq, Hkv, L, D, W = w.B, w.Hq, w.Hkv, w.L, w.D, w.window
    Lq = w.q_rows  # query rows: the last Lq of the L key positions
    variant = Lq != L or not w.causal
    if Lq < L:
        q_h, dO_h = (t[:, :, L - Lq:].contiguous() for t in (q_h, dO_h))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    q, k, v, dO = (t.to(dev) for t in (q_h, k_h, v_h, dO_h))
    f32 = dict(dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    base_mem = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    o = torch.empty((B, Hq, Lq, D), **f32)
    lse = torch.empty((B, Hq, Lq), **f32)
    if w.fwd_only:  # a decode step has no backward
        dq = dk = dv = None
    else:
        dq = torch.empty((B, Hq, Lq, D), **f32)
        dk = torch.empty((B, Hkv, L, D), **f32)
        dv = torch.empty((B, Hkv, L, D), **f32)
    plan = w.prefix
    if plan:
        fws_b = swa.fwd_workspace_bytes_prefix(B, Hq, Hkv, L, D, W, *plan)
        bws_b = swa.bwd_workspace_bytes_prefix(B, Hq, Hkv, L, D, W, *plan)
    elif variant:
        fws_b = swa.fwd_workspace_bytes_ex(B, Hq, Hkv, Lq, L, D, W, w.causal)
        bws_b = 0 if w.fwd_only else swa.bwd_workspace_bytes_ex(B, Hq, Hkv, Lq, L, D, W, w.causal)
    else:
        fws_b = swa.fwd_workspace_bytes(B, Hq, Hkv, L, D, W)
        bws_b = swa.bwd_workspace_bytes(B, Hq, Hkv, L, D, W)
    fws = torch.empty(max(fws_b, 256), dtype=torch.uint8, device=dev)
    bws = torch.empty(max(bws_b, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(mid=None, after_fwd=None):
        # `mid`: an event recorded on the caller's stream between the forward
        # and the backward call, which splits the step's time between them;
        # `after_fwd`: called on the host between the two calls
        if w.fwd_only:
            swa.swa_attn_fwd_ex(q, k, v, o, lse, W, w.causal, w.scale, fws, stream)
        elif plan:
            swa.swa_attn_fwd_prefix(q, k, v, o, lse, W, plan[0], plan[1], w.scale, fws, stream)
            if mid is not None:
                mid.record(stream)
            if after_fwd is not None:
                after_fwd()
            swa.swa_attn_bwd_prefix(q, k, v, o, lse, dO, dq, dk, dv, W, plan[0], plan[1], w.scale, bws, stream)
        elif variant:
            swa.swa_attn_fwd_ex(q, k, v, o, lse, W, w.causal, w.scale, fws, stream)
            if mid is not None:
                mid.record(stream)
            if after_fwd is not None:
                after_fwd()
            swa.swa_attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, W, w.causal, w.scale, bws, stream)
        else:
            swa.swa_attn_fwd(q, k, v, o, lse, W, w.scale, fws, stream)
            if mid is not None:
                mid.record(stream)
            if after_fwd is not None:
                after_fwd()
            swa.swa_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, W, w.scale, bws, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    status = swa.swa_attn_get_status(stream)
    if status != 0:
        raise RuntimeError(f"{w.name}: device status after warm-up: {swa.strerror(status)}")
    peak_above_inputs = torch.cuda.max_memory_allocated(dev) - base_mem - L2_FLUSH_BYTES

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    swa.profile_begin()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step(mids[i])
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    kernels = swa.profile_end()
    if dist is not None:
        dist.barrier()
    clock_info = clocks.stop() if clocks else None
    status = swa.swa_attn_get_status(stream)
    if status != 0:
        raise RuntimeError(f"{w.name}: device status after timed steps: {swa.strerror(status)}")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if w.fwd_only:
        fwd_ms, bwd_ms = sum(step_ms) / args.steps, 0.0
    else:
        fwd_ms = sum(s.elapsed_time(m) for s, m in zip(starts, mids)) / args.steps
        bwd_ms = sum(m.elapsed_time(e) for m, e in zip(mids, ends)) / args.steps
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, dist, dev)
    useful = w.fwd_flops() + (0 if w.fwd_only else w.bwd_flops())
    value = whole_job_tflops(world, useful, args.steps, total_ms)
    launches = sum(n for n, _ in kernels.values())

    # end to end through the public API: pinned host inputs in, results out
    pin = lambda t: t.pin_memory()  # noqa: E731
    hq, hk, hv, hdO = (pin(t) for t in (q_h, k_h, v_h, dO_h))
    results = (o, lse) if w.fwd_only else (o, lse, dq, dk, dv)
    outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in results]
    ins = ((q, hq), (k, hk), (v, hv)) if w.fwd_only else ((q, hq), (k, hk), (v, hv), (dO, hdO))
    h2d = sum(h.numel() * h.element_size() for _, h in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    e2e_steps = max(3, min(args.steps, 10))
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # Every step copies all of its inputs in and all of its results out.  With
    # a backward, two of the copies run on a copy stream beside the kernels:
    # dO's upload beside the forward, and the download of o and lse beside
    # the backward.  The step ends when every copy has.
    cs = torch.cuda.Stream(dev)
    ev_dO, ev_fwd = torch.cuda.Event(), torch.cuda.Event()

    def e2e_step():
        for dst, src in ins:
            if w.fwd_only or dst is not dO:
                dst.copy_(src, non_blocking=True)
        if w.fwd_only:
            step()
            for dst, src in zip(outs_h, results):
                dst.copy_(src, non_blocking=True)
            return
        cs.wait_stream(stream)  # the previous step's backward has read dO
        with torch.cuda.stream(cs):
            dO.copy_(hdO, non_blocking=True)
        ev_dO.record(cs)

        def between():
            stream.wait_event(ev_dO)
            ev_fwd.record(stream)
            cs.wait_event(ev_fwd)
            with torch.cuda.stream(cs):
                for dst, src in zip(outs_h[:2], results[:2]):  # o, lse
                    dst.copy_(src, non_blocking=True)

        step(after_fwd=between)
        for dst, src in zip(outs_h[2:], results[2:]):  # dq, dk, dv
            dst.copy_(src, non_blocking=True)
        stream.wait_stream(cs)

    e2e_step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e2e_ms = 0.0
    for _ in range(e2e_steps):
        flush.zero_()
        es.record(stream)
        e2e_step()
        ee.record(stream)
        torch.cuda.synchronize()
        e2e_ms += es.elapsed_time(ee)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = whole_job_tflops(world, useful, e2e_steps, e2e_ms)
    status = swa.swa_attn_get_status(stream)
    if status != 0:
        raise RuntimeError(f"{w.name}: device status after the e2e steps: {swa.strerror(status)}")

    # roofline of the dominant kernel (or concurrent pair of kernels)
    kname, avg_ms = dominant_unit(kernels, bwd_ms, args.steps)
    roof = roofline_record(kname, avg_ms, w, peaks)
    units = unit_times(kernels, bwd_ms, args.steps)
    per_kernel = {n: {"launches": c, "avg_ms": round(ms / c, 4), "share": round(ms / sum(x[1] for x in
                  units.values()), 4)} for n, (c, ms) in units.items()}
    rec = {
        "value": round(value, 3), "ms_per_step": round(total_ms / args.steps, 4),
        "dtype": "f32" if kname.endswith("_simt") else "f16",
        "config": dict({"workload": w.name, "B": B, "Hq": Hq, "Hkv": Hkv, "L": L, "D": D, "window": W,
                        "scale": round(w.scale, 6), "parallelism": f"replicas x{world} (one workload per GPU)",
                        "l2": "flushed before every step (256 MiB write), flush outside the timed events"},
                       **_variant_keys(w)),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "pinned host memory; q, k, v in before the forward and dq, dk, dv out after the "
                          "backward on the compute stream" + ("" if w.fwd_only else
                          "; dO in beside the forward and o, lse out beside the backward on a copy stream")},
        "gpu_launches": launches,
        "clocks": clock_info,
        "kernels": per_kernel,
        "split": split_record(w, fwd_ms, bwd_ms, peaks),
        "workspace_gb": {"fwd": round(fws_b / 1e9, 4), "bwd": round(bws_b / 1e9, 4),
                         "peak_above_inputs": round(peak_above_inputs / 1e9, 4)},
        "pct_bf16_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
        "wall_s": round(wall, 3),
    }
    del q, k, v, dO, o, lse, dq, dk, dv, fws, bws, flush, outs_h, hq, hk, hv, hdO
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args, w, world, rank, local_rank, subs=()):
    import torch

    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    torch.cuda.set_device(local_rank)
    peaks = load_peaks()
    main_rec = measure_workload(args, w, world, rank, local_rank, dist, peaks)
    sub_recs = [measure_workload(args, s, world, rank, local_rank, dist, peaks) for s in subs]

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            tf, secs, Ls, threads, groups = cpu_oracle_sample(w, args.cpu_seconds)
            G = w.Hq // w.Hkv
            cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"fp64 oracle fwd+bwd (band mode), {groups} kv-head group(s) ({G} query heads each) "
                             f"x first {Ls} tokens ({_sample_q_rows(w, Ls)} query rows) of {w.name}, {secs:.1f} s; "
                             f"useful flops counted as on the GPU"}
        line = {
            "metric": METRIC, "value": main_rec["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": main_rec["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": main_rec["dtype"],
            "data": "synthetic (seeded N(0,1) inputs rounded to bf16)",
            "config": main_rec["config"],
            "roofline": main_rec["roofline"],
            "cpu_baseline": cpu,
        }
        for key in ("e2e", "gpu_launches", "clocks", "kernels", "split", "workspace_gb", "pct_bf16_peak",
                    "wall_s"):
            line[key] = main_rec[key]
        if sub_recs:
            line["sub_workloads"] = sub_recs
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    from sliding_window_attention_gb300.inputs import WORKLOADS

    if args.workload not in WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(WORKLOADS)}")
    w = WORKLOADS[args.workload]
    if args.seq_len > 0:
        import dataclasses

        lq = max(1, round(w.Lq * args.seq_len / w.L)) if w.Lq else 0  # keep the suffix fraction
        w = dataclasses.replace(w, name=f"{w.name}@L{args.seq_len}", L=args.seq_len, Lq=lq)
    world, rank, local_rank = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, w, world, rank)
    subs = ()
    if args.sub_workloads is None:
        if args.workload == DEFAULT_WORKLOAD and args.seq_len <= 0:
            subs = tuple(WORKLOADS[n] for n in DEFAULT_SUB_WORKLOADS)
    elif args.sub_workloads:
        subs = tuple(WORKLOADS[n] for n in args.sub_workloads.split(","))
    return run_ours(args, w, world, rank, local_rank, subs)


if __name__ == "__main__":
    sys.exit(main())
