"""Host-only checks of the C-ABI library: it loads without a GPU, exports every
symbol include/swa_attn.h declares, and rejects bad arguments before any CUDA
call (so these run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swa_attn.h")


@pytest.fixture(scope="module")
def lib():
    from sliding_window_attention_gb300 import build as b
    from sliding_window_attention_gb300 import _native

    b.build()
    return _native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swa_attn_\w+)\s*\(", text)))


def declared_codes():
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (SWA_\w+) (-?\d+)", open(HEADER).read())}


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n
    from sliding_window_attention_gb300 import _native

    assert sorted(_native.EXPORTED) == names


def test_strerror_covers_every_code(lib):
    for name, code in declared_codes().items():
        s = lib.swa_attn_strerror(code).decode()
        assert s and s != "unknown error code", name
    assert lib.swa_attn_strerror(12345).decode() == "unknown error code"
    assert lib.swa_attn_version() >= 100


def test_workspace_sizes(lib):
    # backward: at least one fp32 Delta per query row, O(L*D) at most
    for (B, Hq, Hkv, L, D, W) in [(1, 2, 1, 256, 64, 64), (1, 32, 16, 30553, 256, 1024), (1, 32, 4, 16384, 512, 0)]:
        nb = lib.swa_attn_bwd_workspace_bytes(B, Hq, Hkv, L, D, W)
        assert nb >= B * Hq * L * 4
        assert nb <= 8 * B * Hq * L * D + (1 << 20)
        assert nb % 256 == 0
        nf = lib.swa_attn_fwd_workspace_bytes(B, Hq, Hkv, L, D, W)
        assert nf <= 8 * B * Hq * L * D + (1 << 20)
        assert nf % 256 == 0


def test_forward_workspace_is_the_v_copy_and_the_work_counter(lib):
    # tensor-core forward (not a decode shape): an fp16 copy of v, rounded up
    # to 256 bytes, then 256 bytes for the persistent head-dim-512 launch's
    # work counter
    for (B, Hq, Hkv, L, D, W) in [(1, 32, 4, 16384, 512, 0), (1, 32, 16, 8192, 256, 1024), (2, 8, 2, 1000, 128, 0),
                                  (1, 2, 1, 300, 512, 129)]:
        v16 = -(-B * Hkv * L * D * 2 // 256) * 256
        assert lib.swa_attn_fwd_workspace_bytes(B, Hq, Hkv, L, D, W) == v16 + 256


def _fwd(lib, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, Hq=2, Hkv=1, L=16, D=64, W=0, scale=0.125,
         ws=None, wsb=0):
    P = ctypes.c_void_p
    return lib.swa_attn_fwd(P(q), P(k), P(v), P(o), P(lse), B, Hq, Hkv, L, D, W, ctypes.c_float(scale), P(ws), wsb,
                            None)


def _bwd(lib, ptrs=None, B=1, Hq=2, Hkv=1, L=16, D=64, W=0, scale=0.125, ws=0x10000, wsb=1 << 20):
    P = ctypes.c_void_p
    ptrs = ptrs or [0x1000 * (i + 1) for i in range(9)]
    return lib.swa_attn_bwd(*(P(p) for p in ptrs), B, Hq, Hkv, L, D, W, ctypes.c_float(scale), P(ws), wsb, None)


def test_argument_errors_are_reported_before_any_cuda_call(lib):
    c = declared_codes()
    assert _fwd(lib, q=0) == c["SWA_ERR_NULL_POINTER"]
    assert _fwd(lib, B=0) == c["SWA_ERR_BAD_SHAPE"]
    assert _fwd(lib, L=0) == c["SWA_ERR_BAD_SHAPE"]
    assert _fwd(lib, Hq=3, Hkv=2) == c["SWA_ERR_BAD_GROUPS"]
    assert _fwd(lib, D=96) == c["SWA_ERR_BAD_HEAD_DIM"]
    assert _fwd(lib, W=-1) == c["SWA_ERR_BAD_WINDOW"]
    assert _fwd(lib, scale=float("nan")) == c["SWA_ERR_BAD_SCALE"]
    assert _fwd(lib, scale=float("inf")) == c["SWA_ERR_BAD_SCALE"]
    assert _fwd(lib, q=0x1008) == c["SWA_ERR_MISALIGNED"]
    assert _fwd(lib, Hq=70000, Hkv=1) == c["SWA_ERR_TOO_LARGE"]
    ptrs = [0x1000 * (i + 1) for i in range(9)]
    for idx in range(9):
        bad = list(ptrs)
        bad[idx] = 0
        assert _bwd(lib, bad) == c["SWA_ERR_NULL_POINTER"], idx
        bad[idx] = ptrs[idx] + 4
        assert _bwd(lib, bad) == c["SWA_ERR_MISALIGNED"], idx
    assert _bwd(lib, ws=0x10010) == c["SWA_ERR_MISALIGNED"]
    assert _bwd(lib, wsb=16) == c["SWA_ERR_WORKSPACE"]
    assert _bwd(lib, ws=0) == c["SWA_ERR_WORKSPACE"]
    assert _bwd(lib, D=32) == c["SWA_ERR_BAD_HEAD_DIM"]


def test_suffix_entry_points_check_arguments(lib):
    c = declared_codes()
    P = ctypes.c_void_p

    def fwd_ex(Lq=16, Lk=32, D=64, W=0, causal=1, q=0x1000, ws=None, wsb=0):
        return lib.swa_attn_fwd_ex(P(q), P(0x2000), P(0x3000), P(0x4000), P(0x5000), 1, 2, 1, Lq, Lk, D, W, causal,
                                   ctypes.c_float(0.125), P(ws), wsb, None)

    assert fwd_ex(Lq=33, Lk=32) == c["SWA_ERR_BAD_SHAPE"]  # queries must be a suffix of the keys
    assert fwd_ex(Lq=0) == c["SWA_ERR_BAD_SHAPE"]
    assert fwd_ex(D=80) == c["SWA_ERR_BAD_HEAD_DIM"]
    assert fwd_ex(W=-2, causal=0) == c["SWA_ERR_BAD_WINDOW"]
    assert fwd_ex(q=0) == c["SWA_ERR_NULL_POINTER"]
    assert fwd_ex(wsb=0, ws=None) == c["SWA_ERR_WORKSPACE"]
    ptrs = [0x1000 * (i + 1) for i in range(9)]
    rc = lib.swa_attn_bwd_ex(*(P(p) for p in ptrs), 1, 2, 1, 40, 20, 64, 0, 1, ctypes.c_float(0.1), P(0x10000),
                             1 << 20, None)
    assert rc == c["SWA_ERR_BAD_SHAPE"]
    # workspace grows with Lq for the query-side copies and with Lk for the key side
    a = lib.swa_attn_bwd_workspace_bytes_ex(1, 8, 2, 100, 4000, 128, 256, 1)
    b = lib.swa_attn_bwd_workspace_bytes_ex(1, 8, 2, 4000, 4000, 128, 256, 1)
    assert 0 < a < b and a % 256 == 0
    assert lib.swa_attn_bwd_workspace_bytes_ex(1, 8, 2, 4000, 4000, 128, 256, 1) == \
        lib.swa_attn_bwd_workspace_bytes(1, 8, 2, 4000, 128, 256)
    assert lib.swa_attn_fwd_workspace_bytes_ex(1, 8, 2, 5, 3, 128, 0, 1) == 0


def test_prefix_entry_points_check_arguments(lib):
    """The shared-prefix entry points reject plans out of range before any
    CUDA call, and size their workspaces like the plain calls (the decode
    kernel does not take a plan, so tiny shapes size the tensor-core path)."""
    c = declared_codes()
    P = ctypes.c_void_p

    def fwd_px(L=64, D=64, W=0, prompt=20, chosen=10, q=0x1000):
        return lib.swa_attn_fwd_prefix(P(q), P(0x2000), P(0x3000), P(0x4000), P(0x5000), 1, 2, 1, L, D, W, prompt,
                                       chosen, ctypes.c_float(0.125), P(0x10000), 1 << 20, None)

    assert fwd_px(prompt=-1) == c["SWA_ERR_BAD_PLAN"]
    assert fwd_px(chosen=-3) == c["SWA_ERR_BAD_PLAN"]
    assert fwd_px(prompt=40, chosen=25) == c["SWA_ERR_BAD_PLAN"]  # prompt + chosen > L
    assert fwd_px(q=0) == c["SWA_ERR_NULL_POINTER"]
    assert fwd_px(D=96) == c["SWA_ERR_BAD_HEAD_DIM"]
    assert "prompt_len" in lib.swa_attn_strerror(c["SWA_ERR_BAD_PLAN"]).decode()
    ptrs = [0x1000 * (i + 1) for i in range(9)]
    rc = lib.swa_attn_bwd_prefix(*(P(p) for p in ptrs), 1, 2, 1, 64, 64, 0, 60, 5, ctypes.c_float(0.1),
                                 P(0x10000), 1 << 20, None)
    assert rc == c["SWA_ERR_BAD_PLAN"]
    assert lib.swa_attn_bwd_workspace_bytes_prefix(1, 8, 2, 4000, 128, 256, 3000, 400) == \
        lib.swa_attn_bwd_workspace_bytes(1, 8, 2, 4000, 128, 256)
    assert lib.swa_attn_fwd_workspace_bytes_prefix(1, 8, 2, 4000, 128, 256, 3000, 400) == \
        lib.swa_attn_fwd_workspace_bytes(1, 8, 2, 4000, 128, 256)
    assert lib.swa_attn_fwd_workspace_bytes_prefix(1, 8, 2, 100, 128, 0, 90, 20) == 0
    # two query rows per kv head: the plain call takes the decode kernel, the
    # plan the tensor-core path with its fp16 copy of v
    assert lib.swa_attn_fwd_workspace_bytes_prefix(1, 2, 1, 8, 64, 0, 3, 2) >= 8 * 64 * 2


def test_sink_entry_points_check_arguments_before_any_cuda_call(lib):
    c = declared_codes()
    P, F = ctypes.c_void_p, ctypes.c_float
    # fwd: q, k, v, sinks, o, lse, B, Hq, Hkv, Lq, Lk, D, window, causal, scale, ws, bytes, stream
    def fwd(sinks=0x7000, D=64, Lq=16, Lk=16):
        return lib.swa_attn_fwd_sinks(P(0x1000), P(0x2000), P(0x3000), P(sinks), P(0x4000), P(0x5000), 1, 2, 1, Lq,
                                      Lk, D, 0, 1, F(0.125), P(0x10000), 1 << 20, None)

    # bwd: q, k, v, sinks, o, lse, dO, dq, dk, dv, dsinks, B, Hq, Hkv, Lq, Lk, D, window, causal, scale, ...
    def bwd(sinks=0x7000, dsinks=0x8000, D=64):
        return lib.swa_attn_bwd_sinks(*(P(0x1000 * (i + 1)) for i in range(3)), P(sinks),
                                      *(P(0x1000 * (i + 4)) for i in range(6)), P(dsinks), 1, 2, 1, 16, 16, D, 0, 1,
                                      F(0.125), P(0x10000), 1 << 20, None)

    assert fwd(sinks=0) == c["SWA_ERR_NULL_POINTER"]
    assert fwd(sinks=0x7002) == c["SWA_ERR_MISALIGNED"]
    assert fwd(D=96) == c["SWA_ERR_BAD_HEAD_DIM"]
    assert fwd(Lq=32, Lk=16) == c["SWA_ERR_BAD_SHAPE"]
    assert bwd(sinks=0) == c["SWA_ERR_NULL_POINTER"]
    assert bwd(dsinks=0) == c["SWA_ERR_NULL_POINTER"]
    assert bwd(dsinks=0x8002) == c["SWA_ERR_MISALIGNED"]
    assert bwd(D=96) == c["SWA_ERR_BAD_HEAD_DIM"]
