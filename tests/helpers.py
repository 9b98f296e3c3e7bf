"""Shared test helpers: the parity bar and GPU invocation through the C ABI."""
from __future__ import annotations

import numpy as np

# Parity bar against the fp64 oracle (bf16 inputs, fp32 accumulation):
# max |gpu - oracle| <= 2e-2 and ||gpu - oracle||_F / ||oracle||_F <= 1e-2 on
# o, dq, dk, dv; |lse_gpu - lse_oracle| <= 1e-3.
MAX_ABS = 2e-2
REL_FRO = 1e-2
LSE_ABS = 1e-3


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff)) / nref if nref > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(name, got, ref, max_abs=MAX_ABS, rel_fro=REL_FRO):
    ma, rf = errors(got, ref)
    assert ma <= max_abs and rf <= rel_fro, f"{name}: max_abs={ma:.3e} (<= {max_abs}) rel_fro={rf:.3e} (<= {rel_fro})"
    return ma, rf


def assert_lse_close(got, ref, tol=LSE_ABS):
    ma, _ = errors(got, ref)
    assert ma <= tol, f"lse: max_abs={ma:.3e} (<= {tol})"
    return ma


def gpu_fwd_bwd(q, k, v, dO, window, scale, device="cuda:0", causal=True, prefix=None):
    """Run forward and backward through the C ABI; return CPU fp32 tensors.
    prefix=(prompt_len, chosen_len) selects the shared-prefix entry points."""
    import torch

    import sliding_window_attention_gb300 as swa

    qd, kd, vd, gd = (t.to(device) for t in (q, k, v, dO))
    o, lse = swa.forward(qd, kd, vd, window, scale, causal=causal, prefix=prefix)
    dq, dk, dv = swa.backward(qd, kd, vd, o, lse, gd, window, scale, causal=causal, prefix=prefix)
    torch.cuda.synchronize()
    status = swa.swa_attn_get_status()
    assert status == 0, f"device status {status}"
    return {n: t.cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
