"""ctypes wrapper around swa_oracle.c (fp64 CPU oracle).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this module.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

What the C file computes is the plain definition of masked softmax attention
and its closed-form backward; the passages it follows are listed in its
header.  This wrapper only builds the shared object, converts inputs to the
C calling convention and allocates the fp64 outputs.

Inputs may be torch tensors (bf16 or float64, CPU) or numpy arrays (uint16
holding bf16 bit patterns, or float64): q and dO shaped [B, Hq, Lq, D], k and
v [B, Hkv, Lk, D] with Lq <= Lk.  The queries are the last Lq positions of
the key sequence (Lq = Lk is self-attention).  ``causal=False`` selects the
non-causal band |i + Lk - Lq - j| < window (no mask at all for window 0).

``prefix=(P, Rc)`` selects the shared-prefix mask over one sequence
[prompt (P rows); chosen response (Rc rows); rejected response (the rest)]:
causal self-attention in which rejected rows do not see chosen keys and the
window is measured on logical positions (the rejected response restarts at
position P).  It needs Lq = Lk and causal.

``sinks`` (forward and backward): one sink logit per query head (Hq values),
an extra term of every row's softmax normaliser that carries no value; the
backward then also returns ``dsinks``.  Not combined with ``prefix``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libswa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile swa_oracle.c into oracle/_build/libswa_oracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: the pragmas are ignored and the oracle runs on one core
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            L, I, D, P = ctypes.c_long, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.swa_oracle_fwd_ex.argtypes = [P, P, P, I, L, L, L, L, L, L, L, I, D, I, P, P]
            lib.swa_oracle_bwd_ex.argtypes = [P, P, P, P, I, L, L, L, L, L, L, L, I, D, I, P, P, P, P, P, P, P]
            lib.swa_oracle_rows_ex.argtypes = [P, P, P, P, I, L, L, L, L, L, L, L, I, D, I, L, L, P, L, P, P, P, P]
            lib.swa_oracle_key_rows_ex.argtypes = [P, P, P, P, I, L, L, L, L, L, L, L, I, D, I, L, L, P, L, P, P]
            # shared-prefix plan: (B, Hq, Hkv, L, D, W, P, Rc) instead of (B, Hq, Hkv, Lq, Lk, D, W, causal)
            lib.swa_oracle_fwd_px.argtypes = [P, P, P, I, L, L, L, L, L, L, L, L, D, I, P, P]
            lib.swa_oracle_bwd_px.argtypes = [P, P, P, P, I, L, L, L, L, L, L, L, L, D, I, P, P, P, P, P, P, P]
            lib.swa_oracle_rows_px.argtypes = [P, P, P, P, I, L, L, L, L, L, L, L, L, D, I, L, L, P, L, P, P, P, P]
            lib.swa_oracle_key_rows_px.argtypes = [P, P, P, P, I, L, L, L, L, L, L, L, L, D, I, L, L, P, L, P, P]
            # attention sinks: the sink logits [Hq] (fp64) after v (after dO for the backward)
            lib.swa_oracle_fwd_sk.argtypes = [P, P, P, P, I, L, L, L, L, L, L, L, I, D, P, P]
            lib.swa_oracle_bwd_sk.argtypes = [P, P, P, P, P, I, L, L, L, L, L, L, L, I, D, P, P, P, P, P, P, P, P]
            for f in (lib.swa_oracle_fwd_ex, lib.swa_oracle_bwd_ex, lib.swa_oracle_rows_ex,
                      lib.swa_oracle_key_rows_ex, lib.swa_oracle_fwd_px, lib.swa_oracle_bwd_px,
                      lib.swa_oracle_rows_px, lib.swa_oracle_key_rows_px, lib.swa_oracle_fwd_sk,
                      lib.swa_oracle_bwd_sk):
                f.restype = ctypes.c_int
            lib.swa_oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().swa_oracle_num_threads())


def _as_array(x):
    """Return (contiguous numpy array, is_f64) for a bf16 / fp64 tensor or array."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), 0
            if x.dtype == torch.float64:
                return x.numpy(), 1
            raise TypeError(f"oracle inputs must be bf16 or float64, got {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, 0
    if x.dtype == np.float64:
        return x, 1
    raise TypeError(f"oracle inputs must be uint16 (bf16 bits) or float64, got {x.dtype}")


def _prep(q, k, v, dO=None):
    arrs = [_as_array(t) for t in (q, k, v) + ((dO,) if dO is not None else ())]
    kinds = {a[1] for a in arrs}
    if len(kinds) != 1:
        raise TypeError("q, k, v (and dO) must share one element type")
    B, Hq, Lq, D = arrs[0][0].shape
    Bk, Hkv, Lk, Dk = arrs[1][0].shape
    if (Bk, Dk) != (B, D) or Lk < Lq or arrs[2][0].shape != arrs[1][0].shape:
        raise ValueError("k and v must be [B, Hkv, Lk, D] matching q's B and D, with Lk >= Lq")
    if dO is not None and arrs[3][0].shape != arrs[0][0].shape:
        raise ValueError("dO must have q's shape")
    return [a[0] for a in arrs], kinds.pop(), (B, Hq, Hkv, Lq, Lk, D)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _plan(prefix, causal, Lq, Lk):
    """(P, Rc) of a shared-prefix plan, checked, or None."""
    if prefix is None:
        return None
    P, Rc = (int(x) for x in prefix)
    if not causal or Lq != Lk or P < 0 or Rc < 0 or P + Rc > Lk:
        raise ValueError("a shared-prefix plan needs causal self-attention and 0 <= P, Rc with P + Rc <= L")
    return P, Rc


def _sinks(sinks, Hq, prefix):
    """The sink logits as a contiguous fp64 [Hq] array, checked, or None."""
    if sinks is None:
        return None
    if prefix is not None:
        raise ValueError("sinks are not combined with a shared-prefix plan")
    try:
        import torch

        if isinstance(sinks, torch.Tensor):
            sinks = sinks.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(sinks, dtype=np.float64).reshape(-1))
    if a.size != Hq:
        raise ValueError(f"sinks needs one value per query head ({Hq}), got {a.size}")
    return a


def forward(q, k, v, window: int, scale: float, band_only: bool = False, causal: bool = True, prefix=None,
            sinks=None):
    """Return (o [B,Hq,Lq,D], lse [B,Hq,Lq]) in fp64."""
    arrs, f64, (B, Hq, Hkv, Lq, Lk, D) = _prep(q, k, v)
    plan = _plan(prefix, causal, Lq, Lk)
    sk = _sinks(sinks, Hq, prefix)
    o = np.empty((B, Hq, Lq, D), np.float64)
    lse = np.empty((B, Hq, Lq), np.float64)
    if sk is not None:
        rc = _load().swa_oracle_fwd_sk(*map(_ptr, arrs), _ptr(sk), f64, B, Hq, Hkv, Lq, Lk, D, int(window),
                                       int(bool(causal)), float(scale), _ptr(o), _ptr(lse))
    elif plan:
        rc = _load().swa_oracle_fwd_px(*map(_ptr, arrs), f64, B, Hq, Hkv, Lk, D, int(window), *plan, float(scale),
                                       int(band_only), _ptr(o), _ptr(lse))
    else:
        rc = _load().swa_oracle_fwd_ex(*map(_ptr, arrs), f64, B, Hq, Hkv, Lq, Lk, D, int(window),
                                       int(bool(causal)), float(scale), int(band_only), _ptr(o), _ptr(lse))
    if rc:
        raise RuntimeError(f"swa_oracle_fwd failed ({rc})")
    return o, lse


def backward(q, k, v, dO, window: int, scale: float, band_only: bool = False, causal: bool = True, prefix=None,
             sinks=None):
    """Return dict with o, lse, delta, dq, dk, dv (fp64) and delta_gap (and dsinks [Hq] with sinks)."""
    arrs, f64, (B, Hq, Hkv, Lq, Lk, D) = _prep(q, k, v, dO)
    plan = _plan(prefix, causal, Lq, Lk)
    sk = _sinks(sinks, Hq, prefix)
    out = dict(
        o=np.empty((B, Hq, Lq, D)), lse=np.empty((B, Hq, Lq)), delta=np.empty((B, Hq, Lq)),
        dq=np.empty((B, Hq, Lq, D)), dk=np.empty((B, Hkv, Lk, D)), dv=np.empty((B, Hkv, Lk, D)),
    )
    gap = ctypes.c_double(0.0)
    outs = [_ptr(out[n]) for n in ("o", "lse", "delta", "dq", "dk", "dv")]
    if sk is not None:
        out["dsinks"] = np.empty(Hq)
        a = list(map(_ptr, arrs))
        rc = _load().swa_oracle_bwd_sk(*a[:4], _ptr(sk), f64, B, Hq, Hkv, Lq, Lk, D, int(window),
                                       int(bool(causal)), float(scale), *outs, _ptr(out["dsinks"]), ctypes.byref(gap))
    elif plan:
        rc = _load().swa_oracle_bwd_px(*map(_ptr, arrs), f64, B, Hq, Hkv, Lk, D, int(window), *plan, float(scale),
                                       int(band_only), *outs, ctypes.byref(gap))
    else:
        rc = _load().swa_oracle_bwd_ex(*map(_ptr, arrs), f64, B, Hq, Hkv, Lq, Lk, D, int(window),
                                       int(bool(causal)), float(scale), int(band_only), *outs, ctypes.byref(gap))
    if rc:
        raise RuntimeError(f"swa_oracle_bwd failed ({rc})")
    out["delta_gap"] = gap.value
    return out


def rows(q, k, v, dO, window: int, scale: float, b: int, h: int, row_ids, band_only: bool = False,
         causal: bool = True, prefix=None):
    """Selected query rows of head (b, h): dict o [n,D], lse [n], and with dO also delta [n], dq [n,D]."""
    arrs, f64, (B, Hq, Hkv, Lq, Lk, D) = _prep(q, k, v, dO)
    plan = _plan(prefix, causal, Lq, Lk)
    ids = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64))
    n = ids.size
    out = dict(o=np.empty((n, D)), lse=np.empty(n), delta=np.empty(n), dq=np.empty((n, D)))
    dptr = _ptr(arrs[3]) if dO is not None else None
    qkv = (_ptr(arrs[0]), _ptr(arrs[1]), _ptr(arrs[2]), dptr, f64)
    tail = (float(scale), int(band_only), int(b), int(h), _ptr(ids), n, _ptr(out["o"]), _ptr(out["lse"]),
            _ptr(out["delta"]), _ptr(out["dq"]))
    if plan:
        rc = _load().swa_oracle_rows_px(*qkv, B, Hq, Hkv, Lk, D, int(window), *plan, *tail)
    else:
        rc = _load().swa_oracle_rows_ex(*qkv, B, Hq, Hkv, Lq, Lk, D, int(window), int(bool(causal)), *tail)
    if rc:
        raise RuntimeError(f"swa_oracle_rows failed ({rc})")
    if dO is None:
        del out["delta"], out["dq"]
    return out


def key_rows(q, k, v, dO, window: int, scale: float, b: int, kvh: int, key_ids, band_only: bool = False,
             causal: bool = True, prefix=None):
    """Selected key rows of kv head (b, kvh): dict dk [n,D], dv [n,D]."""
    arrs, f64, (B, Hq, Hkv, Lq, Lk, D) = _prep(q, k, v, dO)
    plan = _plan(prefix, causal, Lq, Lk)
    ids = np.ascontiguousarray(np.asarray(key_ids, dtype=np.int64))
    n = ids.size
    out = dict(dk=np.empty((n, D)), dv=np.empty((n, D)))
    tail = (float(scale), int(band_only), int(b), int(kvh), _ptr(ids), n, _ptr(out["dk"]), _ptr(out["dv"]))
    if plan:
        rc = _load().swa_oracle_key_rows_px(*map(_ptr, arrs), f64, B, Hq, Hkv, Lk, D, int(window), *plan, *tail)
    else:
        rc = _load().swa_oracle_key_rows_ex(*map(_ptr, arrs), f64, B, Hq, Hkv, Lq, Lk, D, int(window),
                                            int(bool(causal)), *tail)
    if rc:
        raise RuntimeError(f"swa_oracle_key_rows failed ({rc})")
    return out
