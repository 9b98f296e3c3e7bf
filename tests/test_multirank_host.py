"""Multi-rank host logic of bench.py, on CPU with gloo (world size 2).

On the GPU machine bench.py runs one rank per GPU over NCCL; each rank runs its
own copy of the workload and the only collectives are a barrier and the
max-over-ranks of the timings.  These tests run that aggregation with gloo
processes on the CPU, plus the reference arm under two ranks (rank 0 times
the oracle, the other rank exits at once without work).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local_ms = [12.5, 20.0][rank]
    dist.barrier()
    m = bench.max_over_ranks(local_ms, dist, "cpu")
    v = bench.whole_job_tflops(world, 1e12, 10, m)
    out_q.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == 20.0  # every rank sees the slowest rank's time
        # 2 ranks x 1e12 flop x 10 steps / 20 ms = 1000 TFLOP/s
        assert abs(v - 1000.0) < 1e-9


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert abs(bench.whole_job_tflops(1, 2e12, 5, 10.0) - 1000.0) < 1e-9


def test_reference_arm_two_ranks_rank0_only():
    """torchrun-style environment, 2 ranks: rank 1 prints nothing and exits 0;
    rank 0 prints one JSON line with impl=reference."""
    outs = []
    for rank in (1, 0):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(_free_port()))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                            "--steps", "1", "--warmup", "0", "--workload", "tiny_l256_d64_w64"],
                           env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip())
    assert outs[0] == ""
    line = json.loads(outs[1].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_dominant_unit_groups_the_concurrent_backward_passes():
    import bench

    # two steps: forward 0.12 ms, prep 0.03 ms, dK/dV and dQ overlapping
    # inside a 0.36 ms backward (their own spans add up to more than that)
    k = {"convert_f16": (2, 0.02), "fwd_tc": (2, 0.24), "bwd_prep": (2, 0.06),
         "bwd_dkdv_tc": (2, 0.54), "bwd_dq_tc": (2, 0.64)}
    name, ms = bench.dominant_unit(k, 0.36, 2)
    assert name == "bwd_dkdv_tc+bwd_dq_tc"
    assert abs(ms - 0.33) < 1e-12
    # a forward that outweighs the backward's pair stays the dominant unit
    name, ms = bench.dominant_unit(dict(k, fwd_tc=(2, 0.80)), 0.36, 2)
    assert (name, ms) == ("fwd_tc", 0.40)
    # without the pair (the SIMT backward) each launch stands alone
    s = {"fwd_simt": (2, 1.0), "bwd_delta": (2, 0.1), "bwd_dkdv_simt": (2, 4.0), "bwd_dq_simt": (2, 3.0)}
    assert bench.dominant_unit(s, 3.55, 2) == ("bwd_dkdv_simt", 2.0)


def test_unit_times_count_the_concurrent_backward_passes_once():
    import bench

    # two steps: forward 0.12 ms, prep 0.03 ms, dK/dV and dQ overlapping
    # inside a 0.36 ms backward: one unit of 0.33 ms per step
    k = {"convert_f16": (2, 0.02), "fwd_tc": (2, 0.24), "bwd_prep": (2, 0.06),
         "bwd_dkdv_tc": (2, 0.54), "bwd_dq_tc": (2, 0.64)}
    u = bench.unit_times(k, 0.36, 2)
    assert set(u) == {"convert_f16", "fwd_tc", "bwd_prep", "bwd_dkdv_tc+bwd_dq_tc"}
    assert u["bwd_dkdv_tc+bwd_dq_tc"][0] == 2 and abs(u["bwd_dkdv_tc+bwd_dq_tc"][1] - 0.66) < 1e-12
    # the units add up to the steps' time
    assert abs(sum(ms for _, ms in u.values()) - 2 * (0.01 + 0.12 + 0.36)) < 1e-12
    # both passes bracketed together (their spans equal): the same unit
    k2 = dict(k, bwd_dkdv_tc=(2, 0.66), bwd_dq_tc=(2, 0.66))
    assert bench.unit_times(k2, 0.36, 2) == u
    # without the pair (the SIMT backward) the launches stand alone
    s = {"fwd_simt": (2, 1.0), "bwd_delta": (2, 0.1), "bwd_dkdv_simt": (2, 4.0), "bwd_dq_simt": (2, 3.0)}
    assert bench.unit_times(s, 3.55, 2) == s


def test_cpu_baseline_adds_kv_groups_up_to_the_workload():
    import dataclasses

    import bench
    from sliding_window_attention_gb300.inputs import WORKLOADS

    # a whole-sequence sample of one group far shorter than the target: more
    # kv-head groups are added, at most B * Hkv of them
    w = dataclasses.replace(WORKLOADS["tiny_l256_d64_w64"], B=2, Hq=4, Hkv=2)
    tf, secs, Ls, threads, groups = bench.cpu_oracle_sample(w, 30.0)
    assert Ls == w.L and groups == w.B * w.Hkv and secs > 0 and tf > 0 and threads >= 1
    # the rate counts every group's flops over the summed time
    one = bench.oracle_useful_flops(w, Ls)
    assert abs(tf - groups * one / secs / 1e12) <= 1e-9 * tf
    # each added group draws its own inputs
    a = bench._oracle_sample_inputs(w, Ls, 0)[0]
    b = bench._oracle_sample_inputs(w, Ls, 1)[0]
    assert not (a == b).all()


def test_roofline_counts_useful_flops_of_the_backward_pair():
    """The backward pair's frac is pairs x 10 D over (backward - prep) over the
    peak; the flops the passes issue (14 D; 16 D at head dim 256) are a
    separate field."""
    import bench
    from sliding_window_attention_gb300.inputs import WORKLOADS

    peaks = dict(hbm_gbs=6789.0, bf16_tflops=1897.1, bf16_tflops_sustained=1690.9, sm_max_mhz=2070.0,
                 source="measured")
    w = WORKLOADS["global_l16384_d512"]
    k = {"convert_f16": (2, 0.2), "fwd_tc": (2, 14.8), "bwd_dscale": (2, 0.16), "bwd_prep": (2, 1.2),
         "bwd_dkdv_tc": (2, 25.0), "bwd_dq_tc": (2, 40.0)}
    name, ms = bench.dominant_unit(k, 22.39, 2)
    assert name == "bwd_dkdv_tc+bwd_dq_tc" and abs(ms - 21.71) < 1e-9
    roof = bench.roofline_record(name, ms, w, peaks)
    want = w.pairs() * 10 * w.D / (21.71e-3) / 1e12 / 1897.1
    assert abs(roof["frac"] - want) < 1e-4
    assert roof["flops_per_pair_d"] == 10 and roof["issued_flops_per_pair_d"] == 14
    assert roof["pairs"] == w.pairs()
    s = WORKLOADS["sliding_l8192_d256_w1024"]
    # D = 256 dK/dV on CTA pairs forms S^T once (S^T, dP^T, dV, dK), as at D <= 128
    assert bench.roofline_record(name, 1.0, s, peaks)["issued_flops_per_pair_d"] == 14
    f = bench.roofline_record("fwd_tc", 7.4, w, peaks)
    assert f["flops_per_pair_d"] == 4 and abs(f["achieved"] - w.fwd_flops() / 7.4e-3 / 1e12) < 0.01


def test_split_record_backward_at_10d():
    import bench
    from sliding_window_attention_gb300.inputs import WORKLOADS

    peaks = dict(bf16_tflops=1897.1)
    w = WORKLOADS["sliding_l8192_d256_w1024"]
    s = bench.split_record(w, 0.375, 1.38, peaks)
    assert abs(s["bwd"]["pct_bf16_peak_10d"] - 100 * w.bwd_flops() / 1.38e9 / 1897.1) < 0.01
    assert abs(s["fwd"]["tflops"] - w.fwd_flops() / 0.375e9) < 0.01


def test_prefix_pair_count_brute_force():
    """band_pairs_prefix counts the pairs the shared-prefix mask keeps
    (causal AND NOT rejected->chosen, window on logical positions), checked
    by enumerating every (row, key) on small sequences."""
    import itertools

    from sliding_window_attention_gb300.inputs import band_pairs_prefix

    def brute(L, W, P, Rc):
        R = P + Rc
        lp = lambda x: x - Rc if x >= R else x  # noqa: E731
        return sum(1 for i in range(L) for j in range(i + 1)
                   if not (i >= R and P <= j < R) and not (W and W < L and lp(i) - lp(j) >= W))

    for L, W, P, Rc in itertools.product([1, 9, 40], [0, 1, 3, 7, 50], [0, 2, 5], [0, 1, 4]):
        if P + Rc <= L:
            assert band_pairs_prefix(L, W, P, Rc) == brute(L, W, P, Rc), (L, W, P, Rc)


def test_prefix_sample_plan_scales_with_the_sample():
    import bench
    from sliding_window_attention_gb300.inputs import WORKLOADS

    w = WORKLOADS["prefix_p6144_c1024_r1024_d256_w1024"]
    assert bench._sample_prefix(w, w.L) == (6144, 1024)
    P, Rc = bench._sample_prefix(w, 1024)
    assert (P, Rc) == (768, 128) and bench._sample_pairs(w, 1024) > 0
