"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs.

Small shapes are compared element by element over every output; the named
full-size workloads are compared on sampled rows (o, lse, dq) and key rows
(dk, dv) that the oracle computes one by one, plus properties that hold at
any size.  The bar is in helpers.py.
"""
import math

import numpy as np
import pytest
import torch

from helpers import assert_close, assert_lse_close, errors, gpu_fwd_bwd
from sliding_window_attention_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

SMALL = [
    # B, Hq, Hkv, L, D, window
    (1, 2, 1, 256, 64, 64),
    (2, 4, 2, 300, 64, 0),
    (1, 4, 1, 129, 128, 7),
    (1, 2, 2, 1, 64, 0),
    (1, 2, 1, 2, 128, 1),
    (1, 4, 2, 127, 256, 128),
    (1, 2, 1, 383, 512, 129),
    (1, 8, 2, 515, 128, 1000),
    (1, 4, 4, 1000, 64, 127),
    (2, 2, 1, 257, 256, 1),
    (1, 4, 2, 700, 512, 0),
    (1, 2, 1, 1100, 128, 300),
    (1, 4, 1, 2048, 512, 0),
    (1, 2, 2, 300, 512, 0),  # one query head per kv head: a key pair with a single step
    (1, 2, 1, 700, 256, 0),  # causal at head dim 256: up to 11 dQ key steps over two K/V stages
]


@pytest.mark.parametrize("B,Hq,Hkv,L,D,window", SMALL)
def test_small_shapes_elementwise(oracle_mod, B, Hq, Hkv, L, D, window):
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=1000 + L + D + window)
    scale = 1.0 / math.sqrt(D)
    ref = oracle_mod.backward(q, k, v, dO, window, scale, band_only=True)
    got = gpu_fwd_bwd(q, k, v, dO, window, scale)
    assert_lse_close(got["lse"].numpy(), ref["lse"])
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, got[n].numpy(), ref[n])


def test_tiny_workload_elementwise(oracle_mod):
    w = WORKLOADS["tiny_l256_d64_w64"]
    q, k, v, dO = workload_inputs(w)
    ref = oracle_mod.backward(q, k, v, dO, w.window, w.scale)
    got = gpu_fwd_bwd(q, k, v, dO, w.window, w.scale)
    assert_lse_close(got["lse"].numpy(), ref["lse"])
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, got[n].numpy(), ref[n])


# ---------------------------------------------------------------------------
# full-size workloads: sampled outputs + any-size properties


def _sample_rows(L, window, rng, n_random=6):
    cand = {0, 1, 63, 64, 127, 128, 129, L // 2, L - 2, L - 1, L - (L % 128 or 128)}
    if window:
        cand |= {window - 1, window, window + 1}
    cand |= set(int(x) for x in rng.integers(0, L, n_random))
    return sorted(i for i in cand if 0 <= i < L)


def _sample_keys(w, rng):
    """Key rows whose oracle cost stays within seconds: the key's column needs
    every query row that sees it, so for long causal rows keep keys late."""
    L = w.L
    if w.window or w.q_rows < L or not w.causal:
        lo = 0
    else:
        # rows [lo, L) each cost up to L keys; keep G * D * (L^2 - lo^2) bounded
        budget = 4.0e9
        G = w.Hq // w.Hkv
        lo2 = max(0.0, L * L - budget / (G * w.D) * 2)
        lo = int(math.sqrt(lo2))
    cand = {lo, lo + 1, L - 1, L - 2, L - 129, L - 128, (lo + L) // 2}
    cand |= set(int(x) for x in rng.integers(lo, L, 5))
    return sorted(j for j in cand if lo <= j < L)


@pytest.fixture(scope="module", params=[n for n in WORKLOADS if not n.startswith("tiny")])
def full_run(request):
    w = WORKLOADS[request.param]
    q, k, v, dO = workload_inputs(w)
    got = gpu_fwd_bwd(q, k, v, dO, w.window, w.scale, causal=w.causal, prefix=w.prefix)
    return w, (q, k, v, dO), got


def _log_errors(workload, what, errs):
    """Append the measured errors of one parity check to the file named by
    SWA_PARITY_LOG (one JSON object per line), when that is set."""
    import json
    import os

    path = os.environ.get("SWA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"workload": workload, "check": what, **errs}) + "\n")


def test_full_workload_sampled(oracle_mod, full_run):
    w, (q, k, v, dO), got = full_run
    rng = np.random.default_rng(w.seed)
    G = w.Hq // w.Hkv
    for name in ("o", "dq", "dk", "dv", "lse"):
        assert torch.isfinite(got[name]).all(), name
    heads = sorted({0, w.Hq - 1, G, w.Hq // 2})
    rows = _sample_rows(w.q_rows, w.window, rng)
    if w.prefix:  # both sides of the prompt / chosen / rejected boundaries
        P, Rc = w.prefix
        rows = sorted(set(rows) | {P - 1, P, P + Rc - 1, P + Rc, P + Rc + 1})
    worst = {}

    def keep(name, ma_rf):
        ma, rf = ma_rf if isinstance(ma_rf, tuple) else (ma_rf, 0.0)
        a, r = worst.get(name, (0.0, 0.0))
        worst[name] = (max(a, ma), max(r, rf))

    for h in heads:
        r = oracle_mod.rows(q, k, v, dO, w.window, w.scale, 0, h, rows, band_only=True, causal=w.causal,
                            prefix=w.prefix)
        keep("lse", assert_lse_close(got["lse"][0, h, rows].numpy(), r["lse"]))
        keep("o", assert_close(f"o[h={h}]", got["o"][0, h, rows].numpy(), r["o"]))
        keep("dq", assert_close(f"dq[h={h}]", got["dq"][0, h, rows].numpy(), r["dq"]))
    keys = _sample_keys(w, rng)
    if w.prefix:
        P, Rc = w.prefix
        keys = sorted(set(keys) | {P - 1, P, P + Rc - 1, P + Rc})
    for kvh in sorted({0, w.Hkv - 1}):
        r = oracle_mod.key_rows(q, k, v, dO, w.window, w.scale, 0, kvh, keys, band_only=True, causal=w.causal,
                                prefix=w.prefix)
        keep("dk", assert_close(f"dk[kvh={kvh}]", got["dk"][0, kvh, keys].numpy(), r["dk"]))
        keep("dv", assert_close(f"dv[kvh={kvh}]", got["dv"][0, kvh, keys].numpy(), r["dv"]))
    _log_errors(w.name, "sampled rows and keys",
                {n: {"max_abs": a, "rel_fro": f} for n, (a, f) in sorted(worst.items())})


@pytest.mark.parametrize("name", ["causal_gqa_l8192_d128",
                                  pytest.param("global_l16384_d512", marks=pytest.mark.slow)])
def test_full_workload_first_key_tile(oracle_mod, name):
    """Keys 0..127 of a causal workload accumulate dK and dV over every query
    row of every head of their group: the longest sums the dK/dV pass forms
    (at 16,384 tokens and 8 heads per kv head, 1,024 steps of 128 rows).
    Every element of that key tile against the oracle.  The oracle's cost is
    one row pass per query row, the same as for key 0 alone."""
    w = WORKLOADS[name]
    q, k, v, dO = workload_inputs(w)
    got = gpu_fwd_bwd(q, k, v, dO, w.window, w.scale, causal=w.causal)
    keys = list(range(128))
    errs = {}
    for kvh in sorted({0, w.Hkv - 1}) if w.D <= 128 else (0,):
        r = oracle_mod.key_rows(q, k, v, dO, w.window, w.scale, 0, kvh, keys, band_only=True, causal=w.causal)
        errs[f"dk[kvh={kvh}]"] = assert_close(f"dk[kvh={kvh}]", got["dk"][0, kvh, keys].numpy(), r["dk"])
        errs[f"dv[kvh={kvh}]"] = assert_close(f"dv[kvh={kvh}]", got["dv"][0, kvh, keys].numpy(), r["dv"])
    _log_errors(name, "keys 0..127", {n: {"max_abs": a, "rel_fro": f} for n, (a, f) in errs.items()})


def test_full_workload_properties(full_run):
    """Any-size identities of the exact result: rows of P sum to one, so
    sum_j dv_j = sum over the group's heads and all rows of dO; rows of dS sum
    to zero, so sum_j dk_j = 0."""
    w, (q, k, v, dO), got = full_run
    G = w.Hq // w.Hkv
    dv_sum = got["dv"].double().sum(2)                                  # [B, Hkv, D]
    want = dO.double().view(w.B, w.Hkv, G, w.q_rows, w.D).sum((2, 3))   # [B, Hkv, D]
    ma, rf = errors(dv_sum.numpy(), want.numpy())
    assert rf <= 1e-3, (ma, rf)
    dk_sum = got["dk"].double().sum(2)
    scale_ref = got["dk"].double().abs().sum(2).max().item()
    assert dk_sum.abs().max().item() <= 1e-3 * scale_ref


# ---------------------------------------------------------------------------
# invariants on the GPU


def test_wide_group_elementwise_and_deterministic(oracle_mod):
    # causal, eight query heads on one kv head (G = 8) at head dim 64: the
    # dK/dV pass of each key tile runs up to 64 steps over the whole group
    q, k, v, dO = make_inputs(1, 8, 1, 1024, 64, seed=4242)
    scale = 0.125
    ref = oracle_mod.backward(q, k, v, dO, 0, scale, band_only=True)
    a = gpu_fwd_bwd(q, k, v, dO, 0, scale)
    for n in ("dq", "dk", "dv"):
        assert_close(n, a[n].numpy(), ref[n])
    b = gpu_fwd_bwd(q, k, v, dO, 0, scale)
    for n in a:
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("D,L,W", [(128, 777, 100), (512, 700, 0)])
def test_backward_on_user_stream_and_in_cuda_graph(D, L, W):
    # The backward forks its dK/dV pass onto an internal stream and joins it
    # back before returning.  On a caller's non-default stream, and captured
    # into a CUDA graph and replayed, it must give the eager result bit for bit.
    import sliding_window_attention_gb300 as swa

    B, Hq, Hkv, scale = 1, 4, 2, 1.0 / math.sqrt(D)
    q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, L, D, seed=77))
    o, lse = swa.forward(q, k, v, W, scale)
    ref = swa.backward(q, k, v, o, lse, dO, W, scale)
    torch.cuda.synchronize()
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = [torch.full((B, Hq, L, D), float("nan"), **f32), torch.full((B, Hkv, L, D), float("nan"), **f32),
            torch.full((B, Hkv, L, D), float("nan"), **f32)]
    ws = torch.empty(swa.bwd_workspace_bytes(B, Hq, Hkv, L, D, W), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        swa.swa_attn_bwd(q, k, v, o, lse, dO, *outs, W, scale, ws, side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for a, b, n in zip(outs, ref, ("dq", "dk", "dv")):
        assert torch.equal(a, b), n
    for t in outs:
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        swa.swa_attn_bwd(q, k, v, o, lse, dO, *outs, W, scale, ws)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    for a, b, n in zip(outs, ref, ("dq", "dk", "dv")):
        assert torch.equal(a, b), n


@pytest.mark.parametrize("Hq,Hkv,L,D,W", [(4, 2, 777, 128, 100), (2, 1, 700, 256, 0), (4, 2, 700, 512, 0)])
def test_deterministic_bitwise(Hq, Hkv, L, D, W):
    # the outputs are written without atomics, each element by one CTA in a
    # fixed order, also while the dK/dV and dQ passes run side by side
    q, k, v, dO = make_inputs(1, Hq, Hkv, L, D, seed=5)
    scale = 1.0 / math.sqrt(D)
    a = gpu_fwd_bwd(q, k, v, dO, W, scale)
    b = gpu_fwd_bwd(q, k, v, dO, W, scale)
    for n in a:
        assert torch.equal(a[n], b[n]), n


def test_outputs_fully_overwritten():
    import sliding_window_attention_gb300 as swa

    B, Hq, Hkv, L, D, W = 1, 4, 2, 333, 64, 50
    q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, L, D, seed=6))
    nan = float("nan")
    o = torch.full((B, Hq, L, D), nan, device="cuda")
    lse = torch.full((B, Hq, L), nan, device="cuda")
    fws = torch.full((max(256, swa.fwd_workspace_bytes(B, Hq, Hkv, L, D, W)),), 0xFF, dtype=torch.uint8,
                     device="cuda")
    swa.swa_attn_fwd(q, k, v, o, lse, W, 0.125, fws)
    dq = torch.full((B, Hq, L, D), nan, device="cuda")
    dk = torch.full((B, Hkv, L, D), nan, device="cuda")
    dv = torch.full((B, Hkv, L, D), nan, device="cuda")
    ws = torch.full((swa.bwd_workspace_bytes(B, Hq, Hkv, L, D, W),), 0xFF, dtype=torch.uint8, device="cuda")
    swa.swa_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, W, 0.125, ws)
    torch.cuda.synchronize()
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("window", [0, 9])
def test_exact_zero_gradient_off_band(window):
    B, Hq, Hkv, L, D = 1, 2, 1, 300, 64
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=7)
    i0, h0 = 200, 1
    dO = torch.zeros_like(dO)
    dO[0, h0, i0] = torch.linspace(-1, 1, D).to(torch.bfloat16)
    got = gpu_fwd_bwd(q, k, v, dO, window, 0.125)
    band = [j for j in range(L) if j <= i0 and (window == 0 or i0 - j < window)]
    off = [j for j in range(L) if j not in band]
    assert (got["dk"][0, 0, off] == 0).all() and (got["dv"][0, 0, off] == 0).all()
    others = [i for i in range(L) if i != i0]
    assert (got["dq"][0, h0, others] == 0).all() and (got["dq"][0, 1 - h0] == 0).all()


def test_causality_bitwise():
    q, k, v, dO = make_inputs(1, 2, 1, 400, 128, seed=8)
    a = gpu_fwd_bwd(q, k, v, dO, 0, 0.1)
    k2, v2 = k.clone(), v.clone()
    k2[0, 0, 260:] = 30.0
    v2[0, 0, 260:] = -50.0
    b = gpu_fwd_bwd(q, k2, v2, dO, 0, 0.1)
    assert torch.equal(a["o"][:, :, :260], b["o"][:, :, :260])
    assert torch.equal(a["lse"][:, :, :260], b["lse"][:, :, :260])


def test_window_at_least_L_equals_causal_bitwise():
    q, k, v, dO = make_inputs(1, 2, 1, 200, 64, seed=9)
    a = gpu_fwd_bwd(q, k, v, dO, 0, 0.125)
    for w in (200, 5000):
        b = gpu_fwd_bwd(q, k, v, dO, w, 0.125)
        for n in a:
            assert torch.equal(a[n], b[n]), (w, n)


def test_gqa_equals_repeated_kv():
    B, Hq, Hkv, L, D, W = 1, 8, 2, 260, 128, 70
    G = Hq // Hkv
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=10)
    a = gpu_fwd_bwd(q, k, v, dO, W, 0.088)
    b = gpu_fwd_bwd(q, k.repeat_interleave(G, 1).contiguous(), v.repeat_interleave(G, 1).contiguous(), dO, W, 0.088)
    for n in ("o", "dq"):
        assert_close(n, a[n].numpy(), b[n].numpy(), max_abs=1e-4, rel_fro=1e-5)
    for n in ("dk", "dv"):
        assert_close(n, a[n].numpy(), b[n].view(B, Hkv, G, L, D).sum(2).numpy(), max_abs=1e-4, rel_fro=1e-5)


def test_errors_raise_through_binding():
    import sliding_window_attention_gb300 as swa

    q = torch.zeros((1, 3, 16, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(swa.SwaError) as ei:
        swa.forward(q, k, k, 0, 0.125)
    assert ei.value.code == -3
    assert swa.swa_attn_get_status() == 0


def test_device_timeout_is_reported_and_context_survives(oracle_mod):
    """A bounded device wait that runs out (a barrier nothing completes)
    latches SWA_ERR_DEVICE_TIMEOUT in the status word; reading it clears it,
    and the library keeps working on the same context."""
    import sliding_window_attention_gb300 as swa

    assert swa.swa_attn_get_status() == 0
    swa.swa_attn_selftest_timeout()
    torch.cuda.synchronize()
    code = swa.swa_attn_get_status()
    assert code == -11, code
    assert "timeout" in swa.strerror(code).lower() or "wait" in swa.strerror(code).lower()
    assert swa.swa_attn_get_status() == 0
    q, k, v, dO = make_inputs(1, 2, 1, 130, 64, seed=12)
    got = gpu_fwd_bwd(q, k, v, dO, 0, 0.125)  # asserts a clean status afterwards
    ref = oracle_mod.backward(q, k, v, dO, 0, 0.125, band_only=True)
    assert_lse_close(got["lse"].numpy(), ref["lse"])
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, got[n].numpy(), ref[n])


# ---------------------------------------------------------------------------
# queries that are a suffix of the keys (qL < kL), non-causal windows
# ("Lab 028 lab detail: Off NVIDIA, you fix the platform yourself", "What I
# changed, in plain terms" items 3-6 and "Gradient parity")

SUFFIX = [
    # B, Hq, Hkv, Lq, Lk, D, window, causal
    (1, 2, 1, 200, 700, 64, 0, True),
    (1, 4, 2, 129, 1000, 128, 128, True),   # keys 0 .. ~742 seen by no query
    (2, 2, 1, 1, 300, 64, 50, True),        # one decode step over a cache
    (1, 8, 2, 1, 2049, 128, 0, True),
    (1, 2, 1, 300, 300, 128, 100, False),   # non-causal self-attention window
    (1, 4, 2, 250, 777, 64, 0, False),      # unmasked
    (1, 2, 2, 333, 900, 256, 129, False),
    (1, 4, 2, 127, 400, 256, 0, True),
    (1, 2, 1, 300, 1100, 512, 200, True),
    (1, 2, 1, 260, 600, 512, 0, False),
    (1, 2, 1, 130, 1030, 512, 100, False),  # non-causal window, unreached keys on both sides
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,D,window,causal", SUFFIX)
def test_suffix_and_noncausal_elementwise(oracle_mod, B, Hq, Hkv, Lq, Lk, D, window, causal):
    import sliding_window_attention_gb300 as swa

    q, k, v, dO = make_inputs(B, Hq, Hkv, Lk, D, seed=2000 + Lq + Lk + D + window)
    q, dO = q[:, :, Lk - Lq:].contiguous(), dO[:, :, Lk - Lq:].contiguous()
    scale = 1.0 / math.sqrt(D)
    ref = oracle_mod.backward(q, k, v, dO, window, scale, band_only=True, causal=causal)
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, dO))
    o, lse = swa.forward(qd, kd, vd, window, scale, causal=causal)
    dq, dk, dv = swa.backward(qd, kd, vd, o, lse, gd, window, scale, causal=causal)
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    assert_lse_close(lse.cpu().numpy(), ref["lse"])
    got = dict(o=o, dq=dq, dk=dk, dv=dv)
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, got[n].cpu().numpy(), ref[n])
    # keys that no query sees: exact zeros
    dead = [j for j in range(Lk) if not np.any(ref["dv"][:, :, j]) and not np.any(ref["dk"][:, :, j])]
    if dead:
        assert (dk[:, :, dead] == 0).all() and (dv[:, :, dead] == 0).all()


def test_suffix_rows_equal_full_problem_rows():
    """The suffix call gives the rows of the self-attention call over all Lk
    positions (same band per row), up to the order of tile visits."""
    import sliding_window_attention_gb300 as swa

    B, Hq, Hkv, Lk, D, W, Lq = 1, 4, 2, 640, 128, 200, 256
    q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, Lk, D, seed=77))
    o_full, lse_full = swa.forward(q, k, v, W, 0.09)
    o_suf, lse_suf = swa.forward(q[:, :, Lk - Lq:].contiguous(), k, v, W, 0.09, causal=True)
    torch.cuda.synchronize()
    assert torch.allclose(o_suf, o_full[:, :, Lk - Lq:], atol=2e-6, rtol=0)
    assert torch.allclose(lse_suf, lse_full[:, :, Lk - Lq:], atol=2e-6, rtol=0)


# ---------------------------------------------------------------------------
# decode steps: at most 16 query rows per kv head (G * Lq <= 16) run on the
# decode kernel (bf16 cache read once per kv head, chunks merged at the end)

DECODE = [
    # B, Hq, Hkv, Lq, Lk, D, window, causal
    (1, 32, 4, 1, 16384, 512, 0, True),     # global layer, one token, many chunks
    (2, 32, 16, 4, 9000, 256, 1024, True),  # sliding layer, 4-token suffix
    (1, 8, 4, 3, 5000, 128, 100, False),    # non-causal window
    (1, 16, 1, 1, 777, 64, 0, True),        # 16 heads per kv head: M = 16
    (1, 4, 1, 4, 130, 128, 0, True),        # M = 16 from Lq x G
    (3, 6, 3, 1, 1, 64, 0, True),           # a cache of one key
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,D,window,causal", DECODE)
def test_decode_elementwise(oracle_mod, B, Hq, Hkv, Lq, Lk, D, window, causal):
    import sliding_window_attention_gb300 as swa

    q, k, v, dO = make_inputs(B, Hq, Hkv, Lk, D, seed=3000 + Lq + Lk + D + window)
    q = q[:, :, Lk - Lq:].contiguous()
    scale = 1.0 / math.sqrt(D)
    o_ref, lse_ref = oracle_mod.forward(q, k, v, window, scale, band_only=True, causal=causal)
    o, lse = swa.forward(q.cuda(), k.cuda(), v.cuda(), window, scale, causal=causal)
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    assert_lse_close(lse.cpu().numpy(), lse_ref)
    assert_close("o", o.cpu().numpy(), o_ref)


def test_decode_then_backward_matches_oracle(oracle_mod):
    """The backward of a decode-shaped call (tensor-core path) takes the
    decode forward's o and lse."""
    B, Hq, Hkv, Lq, Lk, D, W = 1, 8, 2, 2, 1500, 128, 300
    q, k, v, dO = make_inputs(B, Hq, Hkv, Lk, D, seed=41)
    q, dO = q[:, :, Lk - Lq:].contiguous(), dO[:, :, Lk - Lq:].contiguous()
    ref = oracle_mod.backward(q, k, v, dO, W, 0.1, band_only=True)
    got = gpu_fwd_bwd(q, k, v, dO, W, 0.1)
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, got[n].numpy(), ref[n])


# ---------------------------------------------------------------------------
# fp16 operand range: the backward scales its fp16 copy of dO by a power of
# two from max |dO|; q, k and v outside fp16's range latch a status code


@pytest.mark.parametrize("D,L,W", [(128, 300, 0), (256, 333, 100), (512, 300, 0)])
def test_do_power_of_two_scaling_bitwise_and_against_oracle(oracle_mod, D, L, W):
    """The backward is linear in dO.  With dO scaled by 2^-20 (cotangents far
    below fp16's normal range) and by 2^12, dq, dk and dv are the unscaled
    results times the same power of two, bit for bit, and 2^20 times the
    tiny-cotangent result matches the oracle on the unscaled dO."""
    q, k, v, dO = make_inputs(1, 4, 2, L, D, seed=31 + D)
    scale = 1.0 / math.sqrt(D)
    base = gpu_fwd_bwd(q, k, v, dO, W, scale)
    ref = oracle_mod.backward(q, k, v, dO, W, scale, band_only=True)
    for e in (-20, 12):
        dOs = (dO.float() * 2.0 ** e).to(torch.bfloat16)  # exact: a power of two
        assert torch.equal(dOs.float(), dO.float() * 2.0 ** e)
        got = gpu_fwd_bwd(q, k, v, dOs, W, scale)
        for n in ("dq", "dk", "dv"):
            assert torch.equal(got[n], base[n] * 2.0 ** e), (e, n)
        if e == -20:
            for n in ("dq", "dk", "dv"):
                assert_close(f"2^20 {n}", got[n].double().numpy() * 2.0 ** 20, ref[n])


@pytest.mark.parametrize("D", [64, 512])
def test_large_do_entry_needs_no_status(oracle_mod, D):
    """A dO entry of 1e5 (above fp16's largest finite value) is scaled into
    range with the rest of dO: no status, finite results, and the oracle's
    gradients within the parity bar relative to their size."""
    import sliding_window_attention_gb300 as swa

    L, W = 260, 0
    q, k, v, dO = make_inputs(1, 2, 1, L, D, seed=33 + D)
    dO[0, 1, 100, 7] = 1e5
    scale = 1.0 / math.sqrt(D)
    got = gpu_fwd_bwd(q, k, v, dO, W, scale)  # asserts a clean status
    ref = oracle_mod.backward(q, k, v, dO, W, scale, band_only=True)
    for n in ("dq", "dk", "dv"):
        assert torch.isfinite(got[n]).all(), n
        big = float(np.abs(ref[n]).max())
        assert_close(n, got[n].numpy() / big, ref[n] / big)
    assert swa.swa_attn_get_status() == 0


@pytest.mark.parametrize("D", [128, 512])
def test_fp16_range_status_then_clean_call(oracle_mod, D):
    """A bf16 v entry of 1e5 overflows the forward's fp16 copy of v, and a q
    entry of 1e5 the backward's copy of q: each call still returns SWA_OK
    (the check runs on the device), the status word reads
    SWA_ERR_FP16_RANGE (-14), reading it clears it, and a following call on
    clean inputs matches the oracle."""
    import sliding_window_attention_gb300 as swa

    B, Hq, Hkv, L, W = 1, 2, 1, 256, 0
    scale = 1.0 / math.sqrt(D)
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=35 + D)
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, dO))
    assert swa.swa_attn_get_status() == 0
    v_bad = vd.clone()
    v_bad[0, 0, 17, 3] = 1e5
    swa.forward(qd, kd, v_bad, W, scale)
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == -14
    assert swa.swa_attn_get_status() == 0
    assert "fp16" in swa.strerror(-14)
    o, lse = swa.forward(qd, kd, vd, W, scale)
    q_bad = qd.clone()
    q_bad[0, 1, 40, 5] = -1e5
    swa.backward(q_bad, kd, vd, o, lse, gd, W, scale)
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == -14
    assert swa.swa_attn_get_status() == 0
    got = gpu_fwd_bwd(q, k, v, dO, W, scale)  # asserts a clean status
    ref = oracle_mod.backward(q, k, v, dO, W, scale, band_only=True)
    assert_lse_close(got["lse"].numpy(), ref["lse"])
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, got[n].numpy(), ref[n])


# ---------------------------------------------------------------------------
# head dim 512: two backwards overlapping on two streams (the tile scratch is
# per SM, and no two CTAs of these kernels share an SM)


def test_d512_backwards_overlap_on_two_streams():
    import sliding_window_attention_gb300 as swa

    B, Hq, Hkv, L, D, W = 1, 8, 2, 2048, 512, 0
    scale = 1.0 / math.sqrt(D)
    runs = []
    for seed in (51, 52):
        q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, L, D, seed=seed))
        o, lse = swa.forward(q, k, v, W, scale)
        ref = swa.backward(q, k, v, o, lse, dO, W, scale)
        torch.cuda.synchronize()
        outs = [torch.full_like(t, float("nan")) for t in ref]
        ws = torch.empty(swa.bwd_workspace_bytes(B, Hq, Hkv, L, D, W), dtype=torch.uint8, device="cuda")
        runs.append(((q, k, v, o, lse, dO), ref, outs, ws))
    assert swa.swa_attn_get_status() == 0
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(3):
        for (ins, _, outs, ws), s in zip(runs, streams):
            with torch.cuda.stream(s):
                swa.swa_attn_bwd(*ins, *outs, W, scale, ws, s)
    for s in streams:
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    for _, ref, outs, _ in runs:
        for a, b, n in zip(outs, ref, ("dq", "dk", "dv")):
            assert torch.equal(a, b), n


# head dim 512: two forwards overlapping on two streams.  Both grids are
# persistent clusters that draw work items from a counter in their own
# workspace, so the two calls share nothing but the per-SM tile scratch.


def test_d512_forwards_overlap_on_two_streams():
    import sliding_window_attention_gb300 as swa

    shapes = [(1, 8, 2, 2048, 512, 0), (1, 4, 1, 1500, 512, 300)]  # different item counts and band lengths
    runs = []
    for seed, (B, Hq, Hkv, L, D, W) in zip((53, 54), shapes):
        q, k, v, _ = (t.cuda() for t in make_inputs(B, Hq, Hkv, L, D, seed=seed))
        scale = 1.0 / math.sqrt(D)
        o_ref, lse_ref = swa.forward(q, k, v, W, scale)
        torch.cuda.synchronize()
        o, lse = torch.full_like(o_ref, float("nan")), torch.full_like(lse_ref, float("nan"))
        ws = torch.empty(swa.fwd_workspace_bytes(B, Hq, Hkv, L, D, W), dtype=torch.uint8, device="cuda")
        runs.append(((q, k, v), (o, lse), (o_ref, lse_ref), ws, W, scale))
    assert swa.swa_attn_get_status() == 0
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(3):
        for (ins, outs, _, ws, W, scale), s in zip(runs, streams):
            with torch.cuda.stream(s):
                swa.swa_attn_fwd(*ins, *outs, W, scale, ws, s)
    for s in streams:
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    for _, outs, refs, _, _, _ in runs:
        for a, b, n in zip(outs, refs, ("o", "lse")):
            assert torch.equal(a, b), n


# ---------------------------------------------------------------------------
# shared prompt prefix: one pass over [prompt; chosen; rejected] with the
# mask "causal AND NOT rejected->chosen" and a window on logical positions
# ("Training -- design (ORPO, flash-CCE head, prefix sharing, segmented
# backward)", section 5.4 "Shared prompt-prefix forward")

PREFIX = [
    # B, Hq, Hkv, P, Rc, Rr, D, window
    (1, 2, 1, 300, 150, 200, 64, 0),
    (1, 4, 2, 257, 60, 190, 128, 100),   # chosen shorter than a tile: prompt, chosen and rejected keys share tiles
    (2, 2, 1, 0, 130, 140, 64, 50),      # no prompt: rejected rows see only their own response
    (1, 8, 2, 1000, 300, 400, 128, 0),
    (1, 4, 2, 500, 200, 300, 128, 256),
    (1, 2, 1, 200, 100, 150, 256, 0),
    (1, 4, 2, 333, 77, 210, 256, 129),
    (1, 2, 1, 300, 130, 270, 512, 0),
    (1, 4, 1, 260, 40, 300, 512, 200),
    (1, 2, 2, 700, 5, 3, 128, 64),       # three rejected rows, five chosen
]


@pytest.mark.parametrize("B,Hq,Hkv,P,Rc,Rr,D,window", PREFIX)
def test_prefix_plan_elementwise(oracle_mod, B, Hq, Hkv, P, Rc, Rr, D, window):
    import sliding_window_attention_gb300 as swa

    L = P + Rc + Rr
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=6000 + L + D + window)
    scale = 1.0 / math.sqrt(D)
    ref = oracle_mod.backward(q, k, v, dO, window, scale, band_only=True, prefix=(P, Rc))
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, dO))
    o, lse = swa.forward(qd, kd, vd, window, scale, prefix=(P, Rc))
    dq, dk, dv = swa.backward(qd, kd, vd, o, lse, gd, window, scale, prefix=(P, Rc))
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    assert_lse_close(lse.cpu().numpy(), ref["lse"])
    got = dict(o=o, dq=dq, dk=dk, dv=dv)
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, got[n].cpu().numpy(), ref[n])


@pytest.mark.parametrize("D", [128, 256, 512])
def test_prefix_plan_exact_zeros_and_deterministic(D):
    """dO only on the rejected rows: the chosen keys' dk and dv are exactly
    zero (no rejected row sees them), dq is exactly zero on every other row,
    and two runs agree bit for bit."""
    import sliding_window_attention_gb300 as swa

    P, Rc, Rr, W = 260, 150, 200, 0
    L = P + Rc + Rr
    q, k, v, dO = (t.cuda() for t in make_inputs(1, 4, 2, L, D, seed=6100 + D))
    dO[:, :, :P + Rc] = 0
    scale = 1.0 / math.sqrt(D)
    runs = []
    for _ in range(2):
        o, lse = swa.forward(q, k, v, W, scale, prefix=(P, Rc))
        runs.append((o, lse) + swa.backward(q, k, v, o, lse, dO, W, scale, prefix=(P, Rc)))
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    o, lse, dq, dk, dv = runs[0]
    assert (dk[:, :, P:P + Rc] == 0).all() and (dv[:, :, P:P + Rc] == 0).all()
    assert (dq[:, :, :P + Rc] == 0).all()
    assert dk[:, :, :P].abs().max() > 0 and dv[:, :, P + Rc:].abs().max() > 0
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)


def test_prefix_degenerate_plan_is_the_plain_call():
    """A plan without a chosen response runs the plain causal window."""
    import sliding_window_attention_gb300 as swa

    B, Hq, Hkv, L, D, W = 1, 4, 2, 500, 128, 100
    q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, L, D, seed=6200))
    o, lse = swa.forward(q, k, v, W, 0.1)
    o2, lse2 = swa.forward(q, k, v, W, 0.1, prefix=(300, 0))
    a = swa.backward(q, k, v, o, lse, dO, W, 0.1)
    b = swa.backward(q, k, v, o2, lse2, dO, W, 0.1, prefix=(300, 0))
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ---------------------------------------------------------------------------
# attention sinks: one logit per query head in every row's softmax normaliser
# (the backward primitive's "sinks" parameter, "Lab 028 lab detail: Off
# NVIDIA, you fix the platform yourself", "What I changed, in plain terms"
# item 2; the reading is stated in include/swa_attn.h)

SINKS = [
    # B, Hq, Hkv, Lq, Lk, D, window, causal
    (1, 4, 2, 300, 300, 64, 64, True),
    (2, 4, 1, 129, 129, 128, 0, True),
    (1, 4, 2, 257, 257, 256, 100, True),
    (1, 4, 2, 300, 300, 512, 0, True),
    (1, 2, 1, 100, 400, 128, 64, True),    # queries a suffix of the keys
    (1, 4, 2, 200, 200, 128, 50, False),   # non-causal window
    (2, 8, 1, 1, 700, 128, 0, True),       # decode step (8 rows per kv head)
    (1, 8, 2, 2, 1500, 512, 0, True),      # decode step at head dim 512
]


def _sink_values(Hq):
    base = [-math.inf, -1.5, 0.5, 4.0, -0.25, 2.0, 7.0, -3.0]
    return [base[h % len(base)] for h in range(Hq)]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,D,window,causal", SINKS)
def test_sinks_elementwise(oracle_mod, B, Hq, Hkv, Lq, Lk, D, window, causal):
    import sliding_window_attention_gb300 as swa

    q, k, v, dO = make_inputs(B, Hq, Hkv, Lk, D, seed=4000 + Lq + D + window)
    q, dO = q[:, :, Lk - Lq:].contiguous(), dO[:, :, Lk - Lq:].contiguous()
    scale = 1.0 / math.sqrt(D)
    sinks = _sink_values(Hq)
    ref = oracle_mod.backward(q, k, v, dO, window, scale, causal=causal, sinks=sinks)
    sd = torch.tensor(sinks, dtype=torch.float32, device="cuda")
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, dO))
    o, lse = swa.forward(qd, kd, vd, window, scale, causal=causal, sinks=sd)
    dq, dk, dv, dsinks = swa.backward(qd, kd, vd, o, lse, gd, window, scale, causal=causal, sinks=sd)
    torch.cuda.synchronize()
    assert swa.swa_attn_get_status() == 0
    assert_lse_close(lse.cpu().numpy(), ref["lse"])
    for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(n, t.cpu().numpy(), ref[n])
    got = dsinks.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    # dc_h sums exp(c_h - lse_i) Delta_i over B Lq rows, terms of either sign:
    # the bar is relative to the sum of the terms' magnitudes
    c = np.asarray(sinks).reshape(1, Hq, 1)
    mag = np.sum(np.exp(c - ref["lse"]) * np.abs(ref["delta"]), axis=(0, 2))
    assert np.all(np.abs(got - ref["dsinks"]) <= 2e-3 * mag + 1e-5), (got, ref["dsinks"], mag)
    assert got[0] == 0.0  # head 0 has a sink of -inf


@pytest.mark.parametrize("Lq,Lk,D,window", [(300, 300, 128, 64), (257, 257, 256, 0), (300, 300, 512, 0),
                                            (1, 700, 128, 0)])
def test_sinks_of_minus_infinity_equal_the_plain_call_bitwise(Lq, Lk, D, window):
    import sliding_window_attention_gb300 as swa

    Hq, Hkv = 8, 2
    q, k, v, dO = make_inputs(1, Hq, Hkv, Lk, D, seed=4100 + D)
    q, dO = q[:, :, Lk - Lq:].contiguous(), dO[:, :, Lk - Lq:].contiguous()
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, dO))
    scale = 1.0 / math.sqrt(D)
    sd = torch.full((Hq,), -math.inf, dtype=torch.float32, device="cuda")
    o0, l0 = swa.forward(qd, kd, vd, window, scale)
    o1, l1 = swa.forward(qd, kd, vd, window, scale, sinks=sd)
    g0 = swa.backward(qd, kd, vd, o0, l0, gd, window, scale)
    g1 = swa.backward(qd, kd, vd, o1, l1, gd, window, scale, sinks=sd)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    for a, b in zip(g0, g1[:3]):
        assert torch.equal(a, b)
    assert torch.all(g1[3] == 0)
