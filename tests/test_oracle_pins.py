"""Pins for the fp64 CPU oracle: each test checks it against something other
than itself -- a hand-worked example, the pages' mask rule, closed forms,
finite differences, torch's own softmax / matmul autograd, and invariants.

A plausible mistake anywhere in the oracle (dropped term, wrong sign, wrong
index, transposed operand, off-by-one window) fails at least one of these.
"""
import math
import os

import numpy as np
import pytest
import torch

from sliding_window_attention_gb300.inputs import make_inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand64(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, dtype=torch.float64, generator=g) * scale).contiguous()


def _torch_reference(q, k, v, dO, window, scale):
    """Independent path: torch CPU fp64 masked softmax + matmul + autograd."""
    q = q.double().clone().requires_grad_(True)
    k = k.double().clone().requires_grad_(True)
    v = v.double().clone().requires_grad_(True)
    B, Hq, L, D = q.shape
    G = Hq // k.shape[1]
    kr = k.repeat_interleave(G, dim=1)
    vr = v.repeat_interleave(G, dim=1)
    s = scale * torch.matmul(q, kr.transpose(-1, -2))
    i = torch.arange(L).view(L, 1)
    j = torch.arange(L).view(1, L)
    keep = j <= i
    if window > 0:
        keep = keep & (i - j < window)
    s = s.masked_fill(~keep, float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.matmul(p, vr)
    lse = torch.logsumexp(s, dim=-1)
    (o * dO.double()).sum().backward()
    return dict(o=o.detach(), lse=lse.detach(), dq=q.grad, dk=k.grad, dv=v.grad)


def _read_golden(name):
    vals = {}
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        vals[key] = [float(x) for x in rest]
    return vals


# ---------------------------------------------------------------------------
# worked examples from the pages' rules


def test_hand_worked_two_tokens(oracle_mod):
    g = _read_golden("hand_worked_l2.txt")
    t = {n: torch.tensor(g[n], dtype=torch.float64).view(1, 1, 2, 1) for n in ("q", "k", "v", "dO")}
    r = oracle_mod.backward(t["q"], t["k"], t["v"], t["dO"], int(g["window"][0]), g["scale"][0])
    for n in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[n].reshape(-1), g[n], rtol=1e-15, atol=1e-15, err_msg=n)


def test_window_mask_matches_pages_rule(oracle_mod):
    """With V = identity (D = L), o_i is row i of P; its zero pattern is the mask."""
    lines = [l for l in open(os.path.join(GOLD, "window_mask_l8_w3.txt")) if l.strip() and not l.startswith("#")]
    window = int(lines[0].split()[1])
    mask = np.array([[int(x) for x in l.split()] for l in lines[1:]])
    L = mask.shape[0]
    q = _rand64((1, 1, L, L), 1)
    k = _rand64((1, 1, L, L), 2)
    v = torch.eye(L, dtype=torch.float64).view(1, 1, L, L).contiguous()
    o, _ = oracle_mod.forward(q, k, v, window, 0.3)
    P = o[0, 0]
    assert np.array_equal(P != 0.0, mask == 1)
    np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-14)


# ---------------------------------------------------------------------------
# closed forms


@pytest.mark.parametrize("G", [1, 2])
def test_window_one_closed_form(oracle_mod, G):
    """Window 1: each query sees only itself, so o = v, lse = scale q.k, and
    dQ, dK are exactly zero ("Lab 028 lab detail", "Gradient parity")."""
    B, Hkv, L, D = 2, 2, 19, 8
    Hq = G * Hkv
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=11)
    scale = 0.37
    r = oracle_mod.backward(q, k, v, dO, 1, scale)
    qd, kd, vd, gd = (t.double().numpy() for t in (q, k, v, dO))
    kv_of = np.arange(Hq) // G
    np.testing.assert_array_equal(r["o"], vd[:, kv_of])
    np.testing.assert_allclose(r["lse"], scale * np.einsum("bhld,bhld->bhl", qd, kd[:, kv_of]), rtol=1e-15, atol=1e-15)
    assert np.all(r["dq"] == 0.0) and np.all(r["dk"] == 0.0)
    np.testing.assert_allclose(r["dv"], gd.reshape(B, Hkv, G, L, D).sum(2), rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("window", [0, 1, 4, 13])
def test_zero_queries_uniform(oracle_mod, window):
    """q = 0: every in-band score is 0, so P is uniform over the band,
    lse_i = ln |band(i)| and o_i is the mean of v over the band."""
    B, Hq, Hkv, L, D = 1, 2, 1, 17, 5
    q = torch.zeros((B, Hq, L, D), dtype=torch.float64)
    k = _rand64((B, Hkv, L, D), 3)
    v = _rand64((B, Hkv, L, D), 4)
    o, lse = oracle_mod.forward(q, k, v, window, 1.0)
    for i in range(L):
        j0 = 0 if window == 0 else max(0, i - window + 1)
        n = i - j0 + 1
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-14
        np.testing.assert_allclose(o[0, 1, i], v[0, 0, j0:i + 1].numpy().mean(0), rtol=1e-13, atol=1e-14)


def test_single_token(oracle_mod):
    q, k, v, dO = (_rand64((1, 3, 1, 4), s) for s in (5, 6, 7, 8))
    k, v = k[:, :1].contiguous(), v[:, :1].contiguous()
    r = oracle_mod.backward(q, k, v, dO, 0, 0.5)
    np.testing.assert_array_equal(r["o"], np.broadcast_to(v.numpy(), r["o"].shape))
    np.testing.assert_allclose(r["lse"][0, :, 0], 0.5 * (q[0, :, 0] * k[0, 0, 0]).sum(-1).numpy(), rtol=1e-15)
    assert np.all(r["dq"] == 0) and np.all(r["dk"] == 0)


# ---------------------------------------------------------------------------
# library routine: torch fp64 softmax / matmul autograd on tiny shapes


@pytest.mark.parametrize(
    "B,Hq,Hkv,L,D,window",
    [(1, 2, 1, 33, 16, 0), (2, 4, 2, 37, 8, 5), (1, 6, 2, 40, 12, 1), (1, 3, 3, 29, 4, 29), (2, 2, 1, 50, 8, 100),
     (1, 8, 2, 64, 16, 17)],
)
def test_matches_torch_autograd(oracle_mod, B, Hq, Hkv, L, D, window):
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=100 + L + window)
    scale = 1.0 / math.sqrt(D)
    r = oracle_mod.backward(q, k, v, dO, window, scale)
    ref = _torch_reference(q, k, v, dO, window, scale)
    for n in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[n], ref[n].numpy(), rtol=1e-10, atol=1e-12, err_msg=n)


# ---------------------------------------------------------------------------
# finite differences on loss = sum(dO * O)


@pytest.mark.parametrize("window,G", [(0, 1), (3, 2), (7, 1), (1, 2)])
def test_finite_differences(oracle_mod, window, G):
    B, Hkv, L, D = 1, 2, 14, 6
    Hq = G * Hkv
    q = _rand64((B, Hq, L, D), 21)
    k = _rand64((B, Hkv, L, D), 22)
    v = _rand64((B, Hkv, L, D), 23)
    dO = _rand64((B, Hq, L, D), 24)
    scale = 0.45
    r = oracle_mod.backward(q, k, v, dO, window, scale)

    def loss(qq, kk, vv):
        o, _ = oracle_mod.forward(qq, kk, vv, window, scale)
        return float((o * dO.numpy()).sum())

    rng = np.random.default_rng(7)
    eps = 1e-6
    for name, grad in (("q", r["dq"]), ("k", r["dk"]), ("v", r["dv"])):
        base = {"q": q, "k": k, "v": v}
        t = base[name]
        for _ in range(12):
            idx = tuple(int(rng.integers(0, s)) for s in t.shape)
            plus = t.clone()
            plus[idx] += eps
            minus = t.clone()
            minus[idx] -= eps
            args_p = dict(base, **{name: plus})
            args_m = dict(base, **{name: minus})
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


# ---------------------------------------------------------------------------
# invariants


def test_rows_of_P_sum_to_one(oracle_mod):
    q, k, _, _ = make_inputs(1, 2, 1, 70, 16, seed=31)
    v = torch.ones((1, 1, 70, 16), dtype=torch.bfloat16)
    for window in (0, 9):
        o, _ = oracle_mod.forward(q, k, v, window, 0.25)
        assert np.max(np.abs(o - 1.0)) <= 1e-12


@pytest.mark.parametrize("window", [0, 6])
def test_dv_equals_PT_dO(oracle_mod, window):
    B, Hq, Hkv, L, D = 1, 4, 2, 31, 8
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=41)
    scale = 0.3
    r = oracle_mod.backward(q, k, v, dO, window, scale)
    qd, kd, gd = q.double().numpy(), k.double().numpy(), dO.double().numpy()
    G = Hq // Hkv
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    keep = (j <= i) & ((window == 0) | (i - j < window))
    dv = np.zeros_like(r["dv"])
    for h in range(Hq):
        s = scale * qd[0, h] @ kd[0, h // G].T
        P = np.where(keep, np.exp(s - r["lse"][0, h][:, None]), 0.0)
        dv[0, h // G] += P.T @ gd[0, h]
    np.testing.assert_allclose(r["dv"], dv, rtol=1e-11, atol=1e-12)


def test_delta_two_forms_agree(oracle_mod):
    q, k, v, dO = make_inputs(1, 4, 2, 45, 16, seed=51)
    r = oracle_mod.backward(q, k, v, dO, 8, 0.25)
    assert r["delta_gap"] <= 1e-12
    np.testing.assert_allclose(r["delta"], np.einsum("bhld,bhld->bhl", dO.double().numpy(), r["o"]), atol=1e-12)


def test_window_at_least_L_is_causal_bitwise(oracle_mod):
    q, k, v, dO = make_inputs(1, 2, 1, 40, 8, seed=61)
    a = oracle_mod.backward(q, k, v, dO, 0, 0.35)
    for w in (40, 41, 1000):
        b = oracle_mod.backward(q, k, v, dO, w, 0.35)
        for n in ("o", "lse", "dq", "dk", "dv"):
            assert np.array_equal(a[n], b[n]), (w, n)


@pytest.mark.parametrize("window", [0, 5])
def test_gqa_equals_repeated_kv(oracle_mod, window):
    B, Hq, Hkv, L, D = 1, 6, 2, 27, 8
    G = Hq // Hkv
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=71)
    a = oracle_mod.backward(q, k, v, dO, window, 0.4)
    kr = k.repeat_interleave(G, dim=1).contiguous()
    vr = v.repeat_interleave(G, dim=1).contiguous()
    b = oracle_mod.backward(q, kr, vr, dO, window, 0.4)
    for n in ("o", "lse", "dq"):
        np.testing.assert_allclose(a[n], b[n], rtol=1e-12, atol=1e-13)
    for n in ("dk", "dv"):
        np.testing.assert_allclose(a[n], b[n].reshape(B, Hkv, G, L, D).sum(2), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("window", [0, 4])
def test_masked_positions_get_exact_zero_gradient(oracle_mod, window):
    B, Hq, Hkv, L, D = 1, 2, 1, 23, 8
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=81)
    i0, h0 = 13, 1
    dO = torch.zeros_like(dO)
    dO[0, h0, i0] = torch.linspace(-1, 1, D).to(torch.bfloat16)
    r = oracle_mod.backward(q, k, v, dO, window, 0.3)
    band = [j for j in range(L) if j <= i0 and (window == 0 or i0 - j < window)]
    off = [j for j in range(L) if j not in band]
    assert np.all(r["dk"][0, 0, off] == 0.0) and np.all(r["dv"][0, 0, off] == 0.0)
    others = [i for i in range(L) if i != i0]
    assert np.all(r["dq"][0, h0, others] == 0.0) and np.all(r["dq"][0, 1 - h0] == 0.0)
    assert np.any(r["dq"][0, h0, i0] != 0.0) and np.any(r["dk"][0, 0, band] != 0.0)


def test_causality_bitwise(oracle_mod):
    q, k, v, _ = make_inputs(1, 2, 1, 30, 8, seed=91)
    o1, l1 = oracle_mod.forward(q, k, v, 6, 0.3)
    k2, v2 = k.clone(), v.clone()
    k2[0, 0, 20:] = 3.0
    v2[0, 0, 20:] = -5.0
    o2, l2 = oracle_mod.forward(q, k2, v2, 6, 0.3)
    assert np.array_equal(o1[:, :, :20], o2[:, :, :20]) and np.array_equal(l1[:, :, :20], l2[:, :, :20])
    assert not np.array_equal(o1[:, :, 20:], o2[:, :, 20:])


# ---------------------------------------------------------------------------
# the oracle's own modes and sampled entry points agree with its full mode


@pytest.mark.parametrize("window", [0, 7])
def test_band_mode_bitwise_equals_full(oracle_mod, window):
    q, k, v, dO = make_inputs(1, 4, 2, 50, 16, seed=101)
    a = oracle_mod.backward(q, k, v, dO, window, 0.25)
    b = oracle_mod.backward(q, k, v, dO, window, 0.25, band_only=True)
    for n in ("o", "lse", "delta", "dq", "dk", "dv"):
        assert np.array_equal(a[n], b[n]), n


@pytest.mark.parametrize("band", [False, True])
def test_sampled_rows_and_keys_match_full(oracle_mod, band):
    q, k, v, dO = make_inputs(2, 4, 2, 48, 16, seed=111)
    window = 9
    full = oracle_mod.backward(q, k, v, dO, window, 0.25)
    rows = [0, 5, 31, 47]
    r = oracle_mod.rows(q, k, v, dO, window, 0.25, 1, 3, rows, band_only=band)
    for n in ("o", "dq"):
        assert np.array_equal(r[n], full[n][1, 3, rows]), n
    for n in ("lse", "delta"):
        assert np.array_equal(r[n], full[n][1, 3, rows]), n
    keys = [0, 7, 40, 47]
    kr = oracle_mod.key_rows(q, k, v, dO, window, 0.25, 1, 1, keys, band_only=band)
    for n in ("dk", "dv"):
        assert np.array_equal(kr[n], full[n][1, 1, keys]), n


# ---------------------------------------------------------------------------
# queries that are a suffix of the keys (qL < kL) and non-causal windows
# ("Lab 028 lab detail: Off NVIDIA, you fix the platform yourself", "What I
# changed, in plain terms" items 3-6: diag_off = kL - qL, windows "causal and
# not", dK/dV of keys no query reaches)


def _torch_reference_ex(q, k, v, dO, window, scale, causal):
    """Independent path for Lq <= Lk, causal or not: torch fp64 masked softmax
    + matmul + autograd, with the mask written out from the rule here."""
    q = q.double().clone().requires_grad_(True)
    k = k.double().clone().requires_grad_(True)
    v = v.double().clone().requires_grad_(True)
    B, Hq, Lq, D = q.shape
    Lk = k.shape[2]
    G = Hq // k.shape[1]
    kr = k.repeat_interleave(G, dim=1)
    vr = v.repeat_interleave(G, dim=1)
    s = scale * torch.matmul(q, kr.transpose(-1, -2))
    a = torch.arange(Lq).view(Lq, 1) + (Lk - Lq)  # the query's position among the keys
    j = torch.arange(Lk).view(1, Lk)
    if causal:
        keep = j <= a
        if window > 0:
            keep = keep & (a - j < window)
    else:
        keep = torch.ones((Lq, Lk), dtype=torch.bool) if window == 0 else (a - j).abs() < window
    s = s.masked_fill(~keep, float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.matmul(p, vr)
    lse = torch.logsumexp(s, dim=-1)
    (o * dO.double()).sum().backward()
    return dict(o=o.detach(), lse=lse.detach(), dq=q.grad, dk=k.grad, dv=v.grad)


def _suffix_inputs(B, Hq, Hkv, Lq, Lk, D, seed):
    q, k, v, dO = make_inputs(B, Hq, Hkv, Lk, D, seed=seed)
    return q[:, :, Lk - Lq:].contiguous(), k, v, dO[:, :, Lk - Lq:].contiguous()


def test_suffix_mask_matches_pages_rule(oracle_mod):
    """With V = identity (D = kL), o_i is row i of P; its zero pattern is the mask."""
    lines = [l.split() for l in open(os.path.join(GOLD, "suffix_mask_q3_k8_w3.txt")) if l.strip() and not l.startswith("#")]
    window = int(lines[0][1])
    tables, cur = {}, None
    for t in lines[1:]:
        if t[0] == "causal":
            cur = int(t[1])
            tables[cur] = []
        else:
            tables[cur].append([int(x) for x in t])
    Lq, Lk = len(tables[1]), len(tables[1][0])
    q = _rand64((1, 1, Lq, Lk), 41)
    k = _rand64((1, 1, Lk, Lk), 42)
    v = torch.eye(Lk, dtype=torch.float64).view(1, 1, Lk, Lk).contiguous()
    for causal, mask in tables.items():
        o, _ = oracle_mod.forward(q, k, v, window, 0.3, causal=bool(causal))
        np.testing.assert_array_equal((o[0, 0] > 0).astype(int), np.array(mask), err_msg=f"causal={causal}")


@pytest.mark.parametrize(
    "B,Hq,Hkv,Lq,Lk,D,window,causal",
    [(1, 2, 1, 9, 40, 8, 0, True), (2, 4, 2, 17, 33, 8, 5, True), (1, 2, 2, 1, 30, 16, 7, True),
     (1, 4, 2, 20, 20, 8, 6, False), (1, 2, 1, 13, 41, 8, 0, False), (2, 2, 1, 11, 37, 4, 9, False),
     (1, 6, 2, 25, 64, 12, 100, False), (1, 3, 1, 5, 50, 8, 3, True)],
)
def test_suffix_and_noncausal_match_torch_autograd(oracle_mod, B, Hq, Hkv, Lq, Lk, D, window, causal):
    q, k, v, dO = _suffix_inputs(B, Hq, Hkv, Lq, Lk, D, seed=300 + Lq + Lk + window)
    scale = 1.0 / math.sqrt(D)
    r = oracle_mod.backward(q, k, v, dO, window, scale, causal=causal)
    ref = _torch_reference_ex(q, k, v, dO, window, scale, causal)
    for n in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[n], ref[n].numpy(), rtol=1e-10, atol=1e-12, err_msg=n)


def test_noncausal_without_window_is_torch_sdpa(oracle_mod):
    """Non-causal, window 0: plain softmax attention over every key, which is
    torch's own scaled_dot_product_attention with no mask."""
    B, Hq, Hkv, Lq, Lk, D = 1, 4, 2, 12, 29, 8
    q, k, v, dO = _suffix_inputs(B, Hq, Hkv, Lq, Lk, D, seed=51)
    scale = 0.31
    o, _ = oracle_mod.forward(q, k, v, 0, scale, causal=False)
    G = Hq // Hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double().repeat_interleave(G, 1), v.double().repeat_interleave(G, 1), scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("window,causal", [(0, True), (6, True), (0, False), (6, False)])
def test_suffix_equals_rows_of_full_problem(oracle_mod, window, causal):
    """Queries that are the last Lq of Lk positions give the same rows as the
    self-attention problem over all Lk positions; with dO zero on the first
    Lk - Lq rows, dK and dV agree too (those rows contribute exact zeros)."""
    B, Hq, Hkv, Lq, Lk, D = 1, 4, 2, 11, 30, 8
    qf, k, v, dOf = make_inputs(B, Hq, Hkv, Lk, D, seed=61)
    dOf[:, :, :Lk - Lq] = 0
    off = Lk - Lq
    full = oracle_mod.backward(qf, k, v, dOf, window, 0.4, causal=causal)
    suf = oracle_mod.backward(qf[:, :, off:].contiguous(), k, v, dOf[:, :, off:].contiguous(), window, 0.4,
                              causal=causal)
    for n in ("o", "lse", "dq"):
        np.testing.assert_array_equal(suf[n], full[n][:, :, off:], err_msg=n)
    np.testing.assert_allclose(suf["dk"], full["dk"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(suf["dv"], full["dv"], rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("causal", [True, False])
def test_keys_no_query_reaches_get_exact_zero_gradient(oracle_mod, causal):
    """With a window and qL < kL, keys more than window - 1 positions behind
    the first query's diagonal are seen by no query: dK = dV = 0 exactly
    ("What I changed, in plain terms" item 5(b))."""
    B, Hq, Hkv, Lq, Lk, D, W = 1, 2, 1, 4, 40, 8, 5
    q, k, v, dO = _suffix_inputs(B, Hq, Hkv, Lq, Lk, D, seed=71)
    r = oracle_mod.backward(q, k, v, dO, W, 0.35, causal=causal)
    first = (Lk - Lq) - W + 1  # smallest key the first query sees
    assert np.all(r["dk"][:, :, :first] == 0.0) and np.all(r["dv"][:, :, :first] == 0.0)
    assert np.any(r["dv"][:, :, first] != 0.0)


@pytest.mark.parametrize("window,causal", [(4, True), (0, False), (3, False)])
def test_suffix_finite_differences(oracle_mod, window, causal):
    B, Hq, Hkv, Lq, Lk, D = 1, 2, 1, 6, 15, 5
    q = _rand64((B, Hq, Lq, D), 81)
    k = _rand64((B, Hkv, Lk, D), 82)
    v = _rand64((B, Hkv, Lk, D), 83)
    dO = _rand64((B, Hq, Lq, D), 84)
    scale = 0.5
    r = oracle_mod.backward(q, k, v, dO, window, scale, causal=causal)

    def loss(qq, kk, vv):
        o, _ = oracle_mod.forward(qq, kk, vv, window, scale, causal=causal)
        return float((o * dO.numpy()).sum())

    rng = np.random.default_rng(9)
    eps = 1e-6
    for name, grad in (("q", r["dq"]), ("k", r["dk"]), ("v", r["dv"])):
        base = {"q": q, "k": k, "v": v}
        t = base[name]
        for _ in range(10):
            idx = tuple(int(rng.integers(0, s)) for s in t.shape)
            plus = t.clone()
            plus[idx] += eps
            minus = t.clone()
            minus[idx] -= eps
            args_p = dict(base, **{name: plus})
            args_m = dict(base, **{name: minus})
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("causal", [True, False])
def test_suffix_sampled_rows_and_keys_match_full(oracle_mod, causal):
    B, Hq, Hkv, Lq, Lk, D, W = 1, 4, 2, 19, 45, 8, 7
    q, k, v, dO = _suffix_inputs(B, Hq, Hkv, Lq, Lk, D, seed=91)
    full = oracle_mod.backward(q, k, v, dO, W, 0.3, causal=causal)
    rows = [0, 5, Lq - 1]
    r = oracle_mod.rows(q, k, v, dO, W, 0.3, 0, 3, rows, band_only=True, causal=causal)
    np.testing.assert_array_equal(r["o"], full["o"][0, 3, rows])
    np.testing.assert_array_equal(r["dq"], full["dq"][0, 3, rows])
    keys = [0, Lk - Lq - W, Lk - Lq - W + 1, 30, Lk - 1]
    kr = oracle_mod.key_rows(q, k, v, dO, W, 0.3, 0, 1, keys, band_only=True, causal=causal)
    np.testing.assert_allclose(kr["dk"], full["dk"][0, 1, keys], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(kr["dv"], full["dv"][0, 1, keys], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("causal", [True, False])
def test_suffix_band_mode_bitwise_equals_full(oracle_mod, causal):
    q, k, v, dO = _suffix_inputs(1, 2, 1, 21, 52, 8, seed=95)
    a = oracle_mod.backward(q, k, v, dO, 9, 0.3, band_only=False, causal=causal)
    b = oracle_mod.backward(q, k, v, dO, 9, 0.3, band_only=True, causal=causal)
    for n in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


# ---------------------------------------------------------------------------
# shared prompt prefix: one pass over [prompt; chosen; rejected] with the
# block-sparse mask "causal AND NOT rejected->chosen" and a window on logical
# positions ("Training -- design (ORPO, flash-CCE head, prefix sharing,
# segmented backward)", section 5.4 "Shared prompt-prefix forward")


def test_prefix_mask_matches_hand_table(oracle_mod):
    """With V = identity (D = L), o_i is row i of P; its zero pattern is the mask."""
    lines = [l.split() for l in open(os.path.join(GOLD, "prefix_mask_p3_c2_r3.txt")) if l.strip() and not l.startswith("#")]
    P, Rc = int(lines[0][1]), int(lines[1][1])
    tables, cur = {}, None
    for t in lines[2:]:
        if t[0] == "window":
            cur = int(t[1])
            tables[cur] = []
        else:
            tables[cur].append([int(x) for x in t])
    L = len(tables[0])
    q = _rand64((1, 1, L, L), 141)
    k = _rand64((1, 1, L, L), 142)
    v = torch.eye(L, dtype=torch.float64).view(1, 1, L, L).contiguous()
    for window, mask in tables.items():
        for band in (False, True):
            o, _ = oracle_mod.forward(q, k, v, window, 0.3, band_only=band, prefix=(P, Rc))
            np.testing.assert_array_equal((o[0, 0] > 0).astype(int), np.array(mask), err_msg=f"window={window}")
            np.testing.assert_allclose(o[0, 0].sum(-1), 1.0, atol=1e-14)


def _two_forward(oracle_mod, q, k, v, dO, window, scale, P, Rc):
    """The pages' reference for the shared prefix: two plain causal passes,
    [prompt; chosen] and [prompt; rejected] (the rejected response placed
    right after the prompt, where its logical positions put it), assembled
    into the outputs of the single pass.  In the second pass the prompt rows'
    cotangents are zero, so its dK / dV holds only the rejected rows' share
    (the prompt rows are counted once, in the first pass)."""
    L = q.shape[2]
    chosen = slice(0, P + Rc)
    rej = list(range(P)) + list(range(P + Rc, L))
    a = oracle_mod.backward(q[:, :, chosen], k[:, :, chosen], v[:, :, chosen], dO[:, :, chosen], window, scale,
                            band_only=True)
    dOb = dO[:, :, rej].clone()
    dOb[:, :, :P] = 0
    b = oracle_mod.backward(q[:, :, rej].contiguous(), k[:, :, rej].contiguous(), v[:, :, rej].contiguous(),
                            dOb.contiguous(), window, scale, band_only=True)
    out = {}
    for n in ("o", "lse", "dq"):
        full = np.concatenate([a[n], b[n][:, :, P:]], axis=2)
        out[n] = full
    for n in ("dk", "dv"):
        x = np.zeros((q.shape[0], k.shape[1], L, q.shape[3]))
        x[:, :, :P + Rc] = a[n]
        x[:, :, :P] += b[n][:, :, :P]
        x[:, :, P + Rc:] = b[n][:, :, P:]
        out[n] = x
    return out


@pytest.mark.parametrize("P,Rc,Rr,window,G", [(5, 4, 6, 0, 1), (9, 3, 7, 4, 2), (6, 7, 5, 3, 2), (0, 4, 5, 3, 1),
                                              (12, 2, 9, 6, 1), (7, 5, 4, 100, 2)])
def test_prefix_equals_two_forward_construction(oracle_mod, P, Rc, Rr, window, G):
    """One pass with the shared-prefix mask gives what two plain passes give
    ([prompt; chosen] and [prompt; rejected]), the prompt's key gradients
    being the sum over both; the pages report this construction exact for
    the forward."""
    B, Hkv, D = 1, 2, 8
    L = P + Rc + Rr
    q, k, v, dO = make_inputs(B, G * Hkv, Hkv, L, D, seed=150 + L + window)
    scale = 1.0 / math.sqrt(D)
    r = oracle_mod.backward(q, k, v, dO, window, scale, band_only=True, prefix=(P, Rc))
    ref = _two_forward(oracle_mod, q, k, v, dO, window, scale, P, Rc)
    for n in ("o", "lse", "dq"):
        np.testing.assert_array_equal(r[n], ref[n], err_msg=n)
    for n in ("dk", "dv"):
        np.testing.assert_allclose(r[n], ref[n], rtol=1e-12, atol=1e-14, err_msg=n)


@pytest.mark.parametrize("window", [0, 4])
def test_prefix_finite_differences(oracle_mod, window):
    B, Hq, Hkv, D, P, Rc, Rr = 1, 2, 1, 5, 4, 3, 5
    L = P + Rc + Rr
    q = _rand64((B, Hq, L, D), 161)
    k = _rand64((B, Hkv, L, D), 162)
    v = _rand64((B, Hkv, L, D), 163)
    dO = _rand64((B, Hq, L, D), 164)
    scale = 0.5
    r = oracle_mod.backward(q, k, v, dO, window, scale, prefix=(P, Rc))

    def loss(qq, kk, vv):
        o, _ = oracle_mod.forward(qq, kk, vv, window, scale, prefix=(P, Rc))
        return float((o * dO.numpy()).sum())

    rng = np.random.default_rng(17)
    eps = 1e-6
    for name, grad in (("q", r["dq"]), ("k", r["dk"]), ("v", r["dv"])):
        base = {"q": q, "k": k, "v": v}
        t = base[name]
        for _ in range(12):
            idx = tuple(int(rng.integers(0, s)) for s in t.shape)
            plus = t.clone()
            plus[idx] += eps
            minus = t.clone()
            minus[idx] -= eps
            args_p = dict(base, **{name: plus})
            args_m = dict(base, **{name: minus})
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("window", [0, 5])
def test_prefix_degenerate_plans_are_plain_causal(oracle_mod, window):
    """No chosen response (Rc = 0), or no rejected one (P + Rc = L): the mask
    is the plain causal window, bit for bit."""
    q, k, v, dO = make_inputs(1, 4, 2, 23, 8, seed=171)
    plain = oracle_mod.backward(q, k, v, dO, window, 0.3)
    for plan in ((9, 0), (0, 0), (15, 8), (23, 0)):
        r = oracle_mod.backward(q, k, v, dO, window, 0.3, prefix=plan)
        for n in ("o", "lse", "dq", "dk", "dv"):
            np.testing.assert_array_equal(r[n], plain[n], err_msg=(plan, n))


@pytest.mark.parametrize("window", [0, 6])
def test_prefix_band_mode_and_sampled_rows_keys(oracle_mod, window):
    """Band mode is bitwise equal to full mode under the plan, and the row /
    key samplers reproduce the full result (key samples that mix prompt,
    chosen and rejected keys need every row that sees any of them)."""
    P, Rc, Rr = 11, 6, 9
    L = P + Rc + Rr
    q, k, v, dO = make_inputs(1, 4, 2, L, 8, seed=181)
    a = oracle_mod.backward(q, k, v, dO, window, 0.3, band_only=False, prefix=(P, Rc))
    b = oracle_mod.backward(q, k, v, dO, window, 0.3, band_only=True, prefix=(P, Rc))
    for n in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)
    rows = [0, P - 1, P, P + Rc - 1, P + Rc, L - 1]
    r = oracle_mod.rows(q, k, v, dO, window, 0.3, 0, 3, rows, band_only=True, prefix=(P, Rc))
    np.testing.assert_array_equal(r["o"], a["o"][0, 3, rows])
    np.testing.assert_array_equal(r["dq"], a["dq"][0, 3, rows])
    for keys in ([0, P - 1, P + Rc + 2], [P + Rc, L - 1, 2], [P, P + 1]):
        kr = oracle_mod.key_rows(q, k, v, dO, window, 0.3, 0, 1, keys, band_only=True, prefix=(P, Rc))
        np.testing.assert_allclose(kr["dk"], a["dk"][0, 1, keys], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(kr["dv"], a["dv"][0, 1, keys], rtol=1e-13, atol=1e-15)


def test_prefix_chosen_keys_get_no_gradient_from_rejected_rows(oracle_mod):
    """dO nonzero only on the rejected rows: the chosen keys' dK and dV are
    exactly zero (no rejected row sees them), and so is dq on every other
    row."""
    P, Rc, Rr = 6, 5, 7
    L = P + Rc + Rr
    q, k, v, dO = make_inputs(1, 2, 1, L, 8, seed=191)
    dO[:, :, :P + Rc] = 0
    r = oracle_mod.backward(q, k, v, dO, 0, 0.3, prefix=(P, Rc))
    assert np.all(r["dk"][:, :, P:P + Rc] == 0.0) and np.all(r["dv"][:, :, P:P + Rc] == 0.0)
    assert np.all(r["dq"][:, :, :P + Rc] == 0.0)
    assert np.any(r["dk"][:, :, :P] != 0.0) and np.any(r["dv"][:, :, P + Rc:] != 0.0)


# ---------------------------------------------------------------------------
# attention sinks: one logit per query head in every row's softmax normaliser
# (the backward primitive's "sinks" parameter, "Lab 028 lab detail: Off
# NVIDIA, you fix the platform yourself", "What I changed, in plain terms"
# item 2; the reading is stated in the oracle's header)


def _torch_reference_sinks(q, k, v, dO, window, scale, causal, sinks):
    """Independent path: the sink as one extra logit column of a torch fp64
    softmax (its probability dropped before P V), differentiated by autograd
    with respect to q, k, v and the sinks."""
    q = q.double().clone().requires_grad_(True)
    k = k.double().clone().requires_grad_(True)
    v = v.double().clone().requires_grad_(True)
    c = torch.as_tensor(sinks, dtype=torch.float64).clone().requires_grad_(True)
    B, Hq, Lq, D = q.shape
    Lk = k.shape[2]
    G = Hq // k.shape[1]
    kr = k.repeat_interleave(G, dim=1)
    vr = v.repeat_interleave(G, dim=1)
    s = scale * torch.matmul(q, kr.transpose(-1, -2))
    a = torch.arange(Lq).view(Lq, 1) + (Lk - Lq)
    j = torch.arange(Lk).view(1, Lk)
    if causal:
        keep = j <= a
        if window > 0:
            keep = keep & (a - j < window)
    else:
        keep = torch.ones((Lq, Lk), dtype=torch.bool) if window == 0 else (a - j).abs() < window
    s = s.masked_fill(~keep, float("-inf"))
    col = c.view(1, Hq, 1, 1).expand(B, Hq, Lq, 1)
    aug = torch.cat([s, col], dim=-1)
    p = torch.softmax(aug, dim=-1)[..., :Lk]
    o = torch.matmul(p, vr)
    lse = torch.logsumexp(aug, dim=-1)
    (o * dO.double()).sum().backward()
    return dict(o=o.detach(), lse=lse.detach(), dq=q.grad, dk=k.grad, dv=v.grad, dsinks=c.grad)


def test_sinks_of_minus_infinity_are_no_sinks(oracle_mod):
    q, k, v, dO = make_inputs(1, 4, 2, 40, 16, seed=71)
    plain = oracle_mod.backward(q, k, v, dO, 8, 0.25)
    sunk = oracle_mod.backward(q, k, v, dO, 8, 0.25, sinks=[-math.inf] * 4)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert np.array_equal(plain[n], sunk[n]), n
    assert np.array_equal(sunk["dsinks"], np.zeros(4))


def test_sinks_single_key_closed_form(oracle_mod):
    # row 0 of a causal layer sees only key 0: o = v0 e^s / (e^s + e^c)
    q = _rand64((1, 1, 3, 4), 1)
    k = _rand64((1, 1, 3, 4), 2)
    v = _rand64((1, 1, 3, 4), 3)
    c = 0.7
    o, lse = oracle_mod.forward(q, k, v, 0, 0.5, sinks=[c])
    s = 0.5 * float((q[0, 0, 0] * k[0, 0, 0]).sum())
    w = math.exp(s) / (math.exp(s) + math.exp(c))
    assert np.allclose(o[0, 0, 0], w * v[0, 0, 0].numpy(), rtol=1e-13, atol=1e-15)
    assert abs(lse[0, 0, 0] - math.log(math.exp(s) + math.exp(c))) < 1e-13


@pytest.mark.parametrize("Lq,Lk,window,causal", [(24, 24, 0, True), (24, 24, 7, True), (10, 24, 6, True),
                                                  (16, 16, 5, False)])
def test_sinks_match_torch_autograd(oracle_mod, Lq, Lk, window, causal):
    q, k, v, dO = _suffix_inputs(2, 4, 2, Lq, Lk, 16, seed=72)
    sinks = [0.5, -1.25, 2.0, -0.25]
    got = oracle_mod.backward(q, k, v, dO, window, 0.3, causal=causal, sinks=sinks)
    ref = _torch_reference_sinks(q, k, v, dO, window, 0.3, causal, sinks)
    for n in ("o", "lse", "dq", "dk", "dv", "dsinks"):
        assert np.allclose(got[n], ref[n].numpy(), rtol=1e-10, atol=1e-12), n


def test_sinks_gradient_finite_differences(oracle_mod):
    q, k, v, dO = make_inputs(1, 2, 1, 20, 8, seed=73)
    dOd = dO.double().numpy()
    sinks = np.array([0.4, -0.8])
    got = oracle_mod.backward(q, k, v, dO, 6, 0.35, sinks=sinks)
    eps = 1e-6
    for h in range(2):
        up, dn = sinks.copy(), sinks.copy()
        up[h] += eps
        dn[h] -= eps
        lo = (oracle_mod.forward(q, k, v, 6, 0.35, sinks=up)[0] * dOd).sum()
        hi = (oracle_mod.forward(q, k, v, 6, 0.35, sinks=dn)[0] * dOd).sum()
        fd = (lo - hi) / (2 * eps)
        assert abs(fd - got["dsinks"][h]) < 1e-7 * max(1.0, abs(fd)), (h, fd, got["dsinks"][h])
