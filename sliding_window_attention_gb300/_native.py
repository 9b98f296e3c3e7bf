"""Thin ctypes binding of libswa_attn.so (include/swa_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  There is no CPU fallback; if the library is
missing or was not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(_PKG, "libswa_attn.so")

# names declared in include/swa_attn.h
EXPORTED = (
    "swa_attn_fwd_workspace_bytes",
    "swa_attn_fwd",
    "swa_attn_bwd_workspace_bytes",
    "swa_attn_bwd",
    "swa_attn_get_status",
    "swa_attn_strerror",
    "swa_attn_version",
    "swa_attn_profile_begin",
    "swa_attn_profile_end",
    "swa_attn_bwd_noalloc",
    "swa_attn_selftest_timeout",
    "swa_attn_fwd_workspace_bytes_ex",
    "swa_attn_bwd_workspace_bytes_ex",
    "swa_attn_fwd_ex",
    "swa_attn_bwd_ex",
    "swa_attn_fwd_workspace_bytes_prefix",
    "swa_attn_bwd_workspace_bytes_prefix",
    "swa_attn_fwd_prefix",
    "swa_attn_bwd_prefix",
    "swa_attn_add_rows_f32",
    "swa_attn_fwd_sinks",
    "swa_attn_bwd_sinks",
)

_lock = threading.Lock()
_lib = None


class SwaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or SO_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} not found: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        I, Z, P, F = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
        shape = [I, I, I, I, I, I]
        lib.swa_attn_fwd_workspace_bytes.argtypes = shape
        lib.swa_attn_fwd_workspace_bytes.restype = Z
        lib.swa_attn_bwd_workspace_bytes.argtypes = shape
        lib.swa_attn_bwd_workspace_bytes.restype = Z
        lib.swa_attn_fwd.argtypes = [P, P, P, P, P] + shape + [F, P, Z, P]
        lib.swa_attn_fwd.restype = I
        lib.swa_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P] + shape + [F, P, Z, P]
        lib.swa_attn_bwd.restype = I
        lib.swa_attn_get_status.argtypes = [P]
        lib.swa_attn_get_status.restype = I
        lib.swa_attn_strerror.argtypes = [I]
        lib.swa_attn_strerror.restype = ctypes.c_char_p
        lib.swa_attn_version.argtypes = []
        lib.swa_attn_version.restype = I
        lib.swa_attn_profile_begin.argtypes = []
        lib.swa_attn_profile_begin.restype = I
        lib.swa_attn_profile_end.argtypes = [P, I, ctypes.POINTER(I)]
        lib.swa_attn_profile_end.restype = I
        lib.swa_attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P] + shape + [F, P]
        lib.swa_attn_bwd_noalloc.restype = I
        lib.swa_attn_selftest_timeout.argtypes = [P]
        lib.swa_attn_selftest_timeout.restype = I
        shape_ex = [I, I, I, I, I, I, I, I]  # B, Hq, Hkv, Lq, Lk, D, window, causal
        lib.swa_attn_fwd_workspace_bytes_ex.argtypes = shape_ex
        lib.swa_attn_fwd_workspace_bytes_ex.restype = Z
        lib.swa_attn_bwd_workspace_bytes_ex.argtypes = shape_ex
        lib.swa_attn_bwd_workspace_bytes_ex.restype = Z
        lib.swa_attn_fwd_ex.argtypes = [P, P, P, P, P] + shape_ex + [F, P, Z, P]
        lib.swa_attn_fwd_ex.restype = I
        lib.swa_attn_bwd_ex.argtypes = [P, P, P, P, P, P, P, P, P] + shape_ex + [F, P, Z, P]
        lib.swa_attn_bwd_ex.restype = I
        shape_px = [I, I, I, I, I, I, I, I]  # B, Hq, Hkv, L, D, window, prompt_len, chosen_len
        lib.swa_attn_fwd_workspace_bytes_prefix.argtypes = shape_px
        lib.swa_attn_fwd_workspace_bytes_prefix.restype = Z
        lib.swa_attn_bwd_workspace_bytes_prefix.argtypes = shape_px
        lib.swa_attn_bwd_workspace_bytes_prefix.restype = Z
        lib.swa_attn_fwd_prefix.argtypes = [P, P, P, P, P] + shape_px + [F, P, Z, P]
        lib.swa_attn_fwd_prefix.restype = I
        lib.swa_attn_bwd_prefix.argtypes = [P, P, P, P, P, P, P, P, P] + shape_px + [F, P, Z, P]
        lib.swa_attn_bwd_prefix.restype = I
        lib.swa_attn_add_rows_f32.argtypes = [P, P, I, I, I, I, I, P]
        lib.swa_attn_add_rows_f32.restype = I
        # attention sinks: the sink logits after v; the backward adds dsinks after dv
        lib.swa_attn_fwd_sinks.argtypes = [P, P, P, P, P, P] + shape_ex + [F, P, Z, P]
        lib.swa_attn_fwd_sinks.restype = I
        lib.swa_attn_bwd_sinks.argtypes = [P, P, P, P, P, P, P, P, P, P, P] + shape_ex + [F, P, Z, P]
        lib.swa_attn_bwd_sinks.restype = I
        _lib = lib
        return lib


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_longlong), ("total_ms", ctypes.c_double)]


def profile_begin() -> None:
    rc = load().swa_attn_profile_begin()
    if rc:
        raise SwaError(rc, "swa_attn_profile_begin")


def profile_end(max_entries: int = 32) -> dict:
    """Return {kernel name: (launches, total_ms)} recorded since profile_begin()."""
    buf = (KernelTime * max_entries)()
    n = ctypes.c_int(0)
    rc = load().swa_attn_profile_end(buf, max_entries, ctypes.byref(n))
    if rc:
        raise SwaError(rc, "swa_attn_profile_end")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n.value)}


def strerror(code: int) -> str:
    return load().swa_attn_strerror(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dims(q, k, D=None):
    B, Hq, L, D_ = q.shape
    Hkv = k.shape[1]
    return B, Hq, Hkv, L, D_


def fwd_workspace_bytes(B, Hq, Hkv, L, D, window) -> int:
    return int(load().swa_attn_fwd_workspace_bytes(B, Hq, Hkv, L, D, window))


def bwd_workspace_bytes(B, Hq, Hkv, L, D, window) -> int:
    return int(load().swa_attn_bwd_workspace_bytes(B, Hq, Hkv, L, D, window))


def fwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, causal=True) -> int:
    return int(load().swa_attn_fwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, int(bool(causal))))


def bwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, causal=True) -> int:
    return int(load().swa_attn_bwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, int(bool(causal))))


def _dims_ex(q, k):
    B, Hq, Lq, D = q.shape
    return B, Hq, k.shape[1], Lq, k.shape[2], D


def swa_attn_fwd_ex(q, k, v, o, lse, window: int, causal: bool, scale: float, workspace=None, stream=None) -> None:
    """Forward through the C ABI for q [B,Hq,Lq,D] and k, v [B,Hkv,Lk,D]
    (Lq <= Lk; the queries are the last Lq key positions); o fp32
    [B,Hq,Lq,D] and lse fp32 [B,Hq,Lq] are caller-allocated outputs."""
    B, Hq, Hkv, Lq, Lk, D = _dims_ex(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Lq, Lk, D, int(window),
                                int(bool(causal)), float(scale), _ptr(workspace), nbytes, _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_fwd_ex")


def swa_attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, window: int, causal: bool, scale: float, workspace=None,
                    stream=None) -> None:
    """Backward through the C ABI for q, dO [B,Hq,Lq,D] and k, v [B,Hkv,Lk,D];
    dq, dk, dv are caller-allocated fp32 outputs."""
    B, Hq, Hkv, Lq, Lk, D = _dims_ex(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, Hq, Hkv, Lq, Lk, D, int(window), int(bool(causal)), float(scale),
                                _ptr(workspace), nbytes, _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_bwd_ex")


def swa_attn_fwd_sinks(q, k, v, sinks, o, lse, window: int, causal: bool, scale: float, workspace=None,
                       stream=None) -> None:
    """swa_attn_fwd_ex with one sink logit per query head (sinks fp32 [Hq],
    CUDA; see include/swa_attn.h)."""
    B, Hq, Hkv, Lq, Lk, D = _dims_ex(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_fwd_sinks(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(o), _ptr(lse), B, Hq, Hkv, Lq, Lk,
                                   D, int(window), int(bool(causal)), float(scale), _ptr(workspace), nbytes,
                                   _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_fwd_sinks")


def swa_attn_bwd_sinks(q, k, v, sinks, o, lse, dO, dq, dk, dv, dsinks, window: int, causal: bool, scale: float,
                       workspace=None, stream=None) -> None:
    """Backward of swa_attn_fwd_sinks; dq, dk, dv and dsinks (fp32 [Hq]) are
    caller-allocated outputs."""
    B, Hq, Hkv, Lq, Lk, D = _dims_ex(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_bwd_sinks(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                   _ptr(dk), _ptr(dv), _ptr(dsinks), B, Hq, Hkv, Lq, Lk, D, int(window),
                                   int(bool(causal)), float(scale), _ptr(workspace), nbytes, _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_bwd_sinks")


def fwd_workspace_bytes_prefix(B, Hq, Hkv, L, D, window, prompt_len, chosen_len) -> int:
    return int(load().swa_attn_fwd_workspace_bytes_prefix(B, Hq, Hkv, L, D, window, prompt_len, chosen_len))


def bwd_workspace_bytes_prefix(B, Hq, Hkv, L, D, window, prompt_len, chosen_len) -> int:
    return int(load().swa_attn_bwd_workspace_bytes_prefix(B, Hq, Hkv, L, D, window, prompt_len, chosen_len))


def swa_attn_fwd_prefix(q, k, v, o, lse, window: int, prompt_len: int, chosen_len: int, scale: float,
                        workspace=None, stream=None) -> None:
    """Forward over [prompt; chosen; rejected] with the shared-prefix mask
    (see include/swa_attn.h); q, k, v bf16 [B,H,L,D]; o, lse fp32 outputs."""
    B, Hq, Hkv, L, D = _dims(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_fwd_prefix(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, L, D, int(window),
                                    int(prompt_len), int(chosen_len), float(scale), _ptr(workspace), nbytes,
                                    _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_fwd_prefix")


def swa_attn_bwd_prefix(q, k, v, o, lse, dO, dq, dk, dv, window: int, prompt_len: int, chosen_len: int,
                        scale: float, workspace=None, stream=None) -> None:
    """Backward of swa_attn_fwd_prefix; dq, dk, dv are caller-allocated fp32 outputs."""
    B, Hq, Hkv, L, D = _dims(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_bwd_prefix(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                    _ptr(dv), B, Hq, Hkv, L, D, int(window), int(prompt_len), int(chosen_len),
                                    float(scale), _ptr(workspace), nbytes, _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_bwd_prefix")


def swa_attn_add_rows_f32(dst, src, row0: int, stream=None) -> None:
    """dst[:, :, row0 : row0 + n] += src through the C ABI, for fp32 CUDA
    tensors dst [B, H, dst_rows, D] and src [B, H, n, D] (contiguous)."""
    B, H, dst_rows, D = dst.shape
    n = src.shape[2]
    if tuple(src.shape) != (B, H, n, D) or not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("src must be a contiguous [B, H, n, D] block of dst's heads")
    rc = load().swa_attn_add_rows_f32(_ptr(dst), _ptr(src), B * H, dst_rows, int(row0), n, D, _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_add_rows_f32")


def swa_attn_fwd(q, k, v, o, lse, window: int, scale: float, workspace=None, stream=None) -> None:
    """Forward through the C ABI.  q,k,v: bf16 CUDA tensors [B,H,L,D]; o fp32
    [B,Hq,L,D] and lse fp32 [B,Hq,L] are caller-allocated outputs."""
    B, Hq, Hkv, L, D = _dims(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, L, D, int(window),
                             float(scale), _ptr(workspace), nbytes, _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_fwd")


def swa_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, window: int, scale: float, workspace=None, stream=None) -> None:
    """Backward through the C ABI; dq, dk, dv are caller-allocated fp32 outputs."""
    B, Hq, Hkv, L, D = _dims(q, k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().swa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                             _ptr(dv), B, Hq, Hkv, L, D, int(window), float(scale), _ptr(workspace), nbytes,
                             _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_bwd")


def swa_attn_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, window: int, scale: float, stream=None) -> None:
    """Backward without a workspace (fixed built-in scratch; see include/swa_attn.h)."""
    B, Hq, Hkv, L, D = _dims(q, k)
    rc = load().swa_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                     _ptr(dv), B, Hq, Hkv, L, D, int(window), float(scale), _stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_bwd_noalloc")


def swa_attn_selftest_timeout(stream=None) -> None:
    """Launch the device-side timeout self-test (see include/swa_attn.h)."""
    rc = load().swa_attn_selftest_timeout(_stream_ptr(stream))
    if rc:
        raise SwaError(rc, "swa_attn_selftest_timeout")


def swa_attn_get_status(stream=None) -> int:
    return int(load().swa_attn_get_status(_stream_ptr(stream)))


# ---------------------------------------------------------------------------
# convenience wrappers: allocate outputs / workspace with torch, call the ABI


def _workspace(nbytes, device):
    import torch

    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def forward(q, k, v, window: int, scale: float, stream=None, causal: bool = True, prefix=None, sinks=None):
    """Return (o fp32, lse fp32) for bf16 CUDA tensors q [B,Hq,Lq,D], k/v
    [B,Hkv,Lk,D] (Lq <= Lk; Lq = Lk and causal is self-attention).
    prefix=(prompt_len, chosen_len): the shared-prefix mask over one
    [prompt; chosen; rejected] sequence (self-attention, causal).
    sinks: fp32 CUDA tensor [Hq], one sink logit per query head."""
    import torch

    B, Hq, Hkv, Lq, Lk, D = _dims_ex(q, k)
    o = torch.empty((B, Hq, Lq, D), dtype=torch.float32, device=q.device)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    if sinks is not None:
        if prefix is not None:
            raise ValueError("sinks are not combined with a shared-prefix plan")
        ws = _workspace(fwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, causal), q.device)
        swa_attn_fwd_sinks(q, k, v, sinks, o, lse, window, causal, scale, ws, stream)
    elif prefix is not None:
        ws = _workspace(fwd_workspace_bytes_prefix(B, Hq, Hkv, Lk, D, window, *prefix), q.device)
        swa_attn_fwd_prefix(q, k, v, o, lse, window, prefix[0], prefix[1], scale, ws, stream)
    elif Lq == Lk and causal:
        ws = _workspace(fwd_workspace_bytes(B, Hq, Hkv, Lk, D, window), q.device)
        swa_attn_fwd(q, k, v, o, lse, window, scale, ws, stream)
    else:
        ws = _workspace(fwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, causal), q.device)
        swa_attn_fwd_ex(q, k, v, o, lse, window, causal, scale, ws, stream)
    return o, lse


def backward(q, k, v, o, lse, dO, window: int, scale: float, stream=None, causal: bool = True, prefix=None,
             sinks=None):
    """Return (dq, dk, dv) fp32, and dsinks [Hq] too when sinks are given."""
    import torch

    B, Hq, Hkv, Lq, Lk, D = _dims_ex(q, k)
    dq = torch.empty((B, Hq, Lq, D), dtype=torch.float32, device=q.device)
    dk = torch.empty((B, Hkv, Lk, D), dtype=torch.float32, device=q.device)
    dv = torch.empty((B, Hkv, Lk, D), dtype=torch.float32, device=q.device)
    if sinks is not None:
        if prefix is not None:
            raise ValueError("sinks are not combined with a shared-prefix plan")
        dsinks = torch.empty((Hq,), dtype=torch.float32, device=q.device)
        ws = _workspace(bwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, causal), q.device)
        swa_attn_bwd_sinks(q, k, v, sinks, o, lse, dO, dq, dk, dv, dsinks, window, causal, scale, ws, stream)
        return dq, dk, dv, dsinks
    if prefix is not None:
        ws = _workspace(bwd_workspace_bytes_prefix(B, Hq, Hkv, Lk, D, window, *prefix), q.device)
        swa_attn_bwd_prefix(q, k, v, o, lse, dO, dq, dk, dv, window, prefix[0], prefix[1], scale, ws, stream)
    elif Lq == Lk and causal:
        ws = _workspace(bwd_workspace_bytes(B, Hq, Hkv, Lk, D, window), q.device)
        swa_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, window, scale, ws, stream)
    else:
        ws = _workspace(bwd_workspace_bytes_ex(B, Hq, Hkv, Lq, Lk, D, window, causal), q.device)
        swa_attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, window, causal, scale, ws, stream)
    return dq, dk, dv
