"""swa_attn_bwd_noalloc: the backward for callers that cannot allocate.

Some callers of this library cannot give it a workspace: their device memory
is owned by a host framework's allocator, or they sit behind a fixed plugin
signature with no workspace argument.  swa_attn_bwd_noalloc serves them by
keeping its scratch in a fixed array built into the library.  These tests
call it through the C ABI and check that its output matches swa_attn_bwd's
(the existing entry point, which takes a caller workspace) within the parity
tolerance used everywhere else, and against the fp64 oracle, on two calls in
a row with different cotangents -- the second call finds the scratch as the
first call left it.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from helpers import assert_close
from sliding_window_attention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _run_noalloc(lib, q, k, v, o, lse, dO, window, scale):
    B, Hq, L, D = q.shape
    Hkv = k.shape[1]
    dq = torch.full((B, Hq, L, D), float("nan"), device=q.device)
    dk = torch.full((B, Hkv, L, D), float("nan"), device=q.device)
    dv = torch.full((B, Hkv, L, D), float("nan"), device=q.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.swa_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                  _ptr(dv), B, Hq, Hkv, L, D, window, ctypes.c_float(scale), stream)
    assert rc == 0, lib.swa_attn_strerror(rc).decode()
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("B,Hq,Hkv,L,D,window", [(1, 4, 2, 333, 64, 50), (2, 8, 2, 1029, 128, 0)])
def test_noalloc_matches_workspace_backward_twice(B, Hq, Hkv, L, D, window):
    """Two calls in a row with different cotangents (dO, then 3 dO): the
    second call's Delta differs from what the first left in the scratch, and
    its result must still match swa_attn_bwd on its own inputs."""
    import sliding_window_attention_gb300 as swa

    lib = swa.load()
    scale = D ** -0.5
    q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, L, D, seed=4242 + L))
    o, lse = swa.forward(q, k, v, window, scale)
    for call, g in enumerate((dO, (dO.float() * 3).to(torch.bfloat16))):
        ref = swa.backward(q, k, v, o, lse, g, window, scale)
        torch.cuda.synchronize()
        got = _run_noalloc(lib, q, k, v, o, lse, g, window, scale)
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a).all(), (call, name)
            assert_close(f"{name} (call {call})", a.cpu().numpy(), r.cpu().numpy())
    assert swa.swa_attn_get_status() == 0


@pytest.mark.parametrize("B,Hq,Hkv,L,D,window", [(1, 4, 2, 300, 256, 64), (1, 2, 1, 257, 512, 0)])
def test_noalloc_matches_oracle_at_wide_heads(oracle_mod, B, Hq, Hkv, L, D, window):
    """Head dims 256 and 512 (the widest per-thread accumulators of its
    kernels) against the fp64 oracle, two calls in a row with different
    cotangents."""
    import sliding_window_attention_gb300 as swa

    lib = swa.load()
    scale = D ** -0.5
    q, k, v, dO = make_inputs(B, Hq, Hkv, L, D, seed=4343 + L)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = swa.forward(qd, kd, vd, window, scale)
    for call, g in enumerate((dO, (dO.float() * -0.5).to(torch.bfloat16))):
        ref = oracle_mod.backward(q, k, v, g, window, scale, band_only=True)
        got = _run_noalloc(lib, qd, kd, vd, o, lse, g.cuda(), window, scale)
        for name, a in zip(("dq", "dk", "dv"), got):
            assert_close(f"{name} (call {call})", a.cpu().numpy(), ref[name])
    assert swa.swa_attn_get_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import sliding_window_attention_gb300 as swa

    lib = swa.load()
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    P = _ptr(t)
    # B * Hq * L = 1 * 64 * 40000 = 2,560,000 rows > 2,097,152
    rc = lib.swa_attn_bwd_noalloc(P, P, P, P, P, P, P, P, P, 1, 64, 8, 40000, 128, 0, ctypes.c_float(0.1), None)
    assert rc == -13
    assert "swa_attn_bwd_noalloc" in lib.swa_attn_strerror(rc).decode()
