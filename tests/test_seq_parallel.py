"""Sequence-sharded attention with a halo exchange.

On CPU: world sizes 2 and 3 as gloo processes; each rank's attention is the
fp64 oracle (injected by the test), so what is checked is the host logic --
halo planning, the exchange in both directions, the concatenation and the
return of halo key gradients -- against the oracle on the whole sequence.
On one GPU: ranks as threads of one process calling the library's kernels,
against the unsharded library call and the oracle.
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

from helpers import assert_close, assert_lse_close  # noqa: E402
from sliding_window_attention_gb300 import seq_parallel as sp  # noqa: E402
from sliding_window_attention_gb300.inputs import make_inputs  # noqa: E402


def test_halo_plan():
    lens = [5, 3, 4, 6]
    # window 3: two positions before each chunk, from the ranks that own them
    assert sp.halo_pieces(lens, 3, 0) == []
    assert sp.halo_pieces(lens, 3, 1) == [(0, 3, 2)]
    assert sp.halo_pieces(lens, 3, 2) == [(1, 1, 2)]
    # window 6: five positions, spanning two earlier chunks
    assert sp.halo_pieces(lens, 6, 2) == [(0, 3, 2), (1, 0, 3)]
    # no window: every earlier position
    assert sp.halo_pieces(lens, 0, 3) == [(0, 0, 5), (1, 0, 3), (2, 0, 4)]
    assert sp.halo_rows(lens, 100, 3) == 12


class OracleOps:
    """Per-rank steps on the fp64 oracle (test infrastructure)."""

    @staticmethod
    def forward(q, k, v, window, scale):
        import oracle

        o, lse = oracle.forward(q, k, v, window, scale, band_only=True, causal=True)
        return torch.from_numpy(o), torch.from_numpy(lse)

    @staticmethod
    def backward(q, k, v, o, lse, dO, window, scale):
        import oracle

        r = oracle.backward(q, k, v, dO, window, scale, band_only=True, causal=True)
        return tuple(torch.from_numpy(r[n]) for n in ("dq", "dk", "dv"))

    @staticmethod
    def add_rows(dst, src, row0):
        dst[:, :, row0:row0 + src.shape[2]] += src

    @staticmethod
    def cat_rows(parts):
        return torch.cat(parts, dim=2).contiguous()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _chunks(t, lens):
    out, s = [], 0
    for n in lens:
        out.append(t[:, :, s:s + n].contiguous())
        s += n
    return out


def _gloo_worker(rank, world, port, lens, window, out_q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import oracle

    oracle.build()
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        L = sum(lens)
        q, k, v, dO = (t.double() for t in make_inputs(1, 4, 2, L, 8, seed=77))
        x = sp.DistExchange()
        qs, ks, vs, gs = (_chunks(t, lens)[rank] for t in (q, k, v, dO))
        o, lse, ctx = sp.sharded_forward(qs, ks, vs, window, 0.35, lens, x, ops=OracleOps)
        dq, dk, dv = sp.sharded_backward(ctx, gs, x, ops=OracleOps)
        out_q.put((rank, o.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("lens,window", [([40, 30], 9), ([20, 25, 31], 30), ([26, 17, 30], 0), ([15, 15, 15], 1)])
def test_gloo_ranks_match_the_whole_sequence(oracle_mod, lens, window):
    world = len(lens)
    ctx = mp.get_context("spawn")
    q_ = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_worker, args=(r, world, port, lens, window, q_)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q_.get(timeout=300) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    L = sum(lens)
    q, k, v, dO = make_inputs(1, 4, 2, L, 8, seed=77)
    ref = oracle_mod.backward(q, k, v, dO, window, 0.35, band_only=True)
    for i, n in enumerate(("o", "lse", "dq", "dk", "dv")):
        got = np.concatenate([r[1 + i] for r in res], axis=2)
        np.testing.assert_allclose(got, ref[n], rtol=1e-10, atol=1e-12, err_msg=n)


@pytest.mark.gpu
@pytest.mark.parametrize("lens,window,D", [([700, 650], 200, 128), ([300, 260, 400], 500, 64),
                                           ([512, 384, 640, 257], 0, 128), ([600, 500], 129, 256),
                                           ([300, 300], 100, 512)])
def test_thread_ranks_on_one_gpu(oracle_mod, lens, window, D):
    import sliding_window_attention_gb300 as swa

    L, scale = sum(lens), 1.0 / math.sqrt(D)
    q, k, v, dO = make_inputs(1, 4, 2, L, D, seed=88 + L)
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, dO))
    parts = [_chunks(t, lens) for t in (qd, kd, vd, gd)]

    def rank_fn(r, x):
        o, lse, ctx = sp.sharded_forward(parts[0][r], parts[1][r], parts[2][r], window, scale, lens, x)
        dq, dk, dv = sp.sharded_backward(ctx, parts[3][r], x)
        torch.cuda.synchronize()
        return o, lse, dq, dk, dv

    res = sp.run_threads(len(lens), rank_fn)
    assert swa.swa_attn_get_status() == 0
    got = [torch.cat([r[i] for r in res], dim=2).cpu() for i in range(5)]
    o, lse = swa.forward(qd, kd, vd, window, scale)
    whole = (o, lse) + swa.backward(qd, kd, vd, o, lse, gd, window, scale)
    ref = oracle_mod.backward(q, k, v, dO, window, scale, band_only=True)
    for i, n in enumerate(("o", "lse", "dq", "dk", "dv")):
        if n == "lse":
            assert_lse_close(got[i].numpy(), ref[n])
        else:
            assert_close(n, got[i].numpy(), ref[n])
        # against the unsharded call: the same arithmetic, tiles cut at other places
        assert_close(f"{n} vs unsharded", got[i].numpy(), whole[i].cpu().numpy(), max_abs=2e-3, rel_fro=1e-3)
