"""Sequence-sharded (context-parallel) causal / sliding-window attention with
one halo exchange.

A sequence of L tokens is split into contiguous chunks, one per rank: rank r
holds rows [s_r, s_r + C_r) of q, k, v and dO (every head).  The queries of
chunk r see keys of earlier chunks only within their causal window, so
before the forward each rank receives its halo -- the keys and values of the
W - 1 positions before its chunk (all earlier positions when the window is
0) -- from the ranks that own them, and runs its queries as the last C_r rows
of [halo; own keys] through the suffix-query entry points of the library
(the band structure of "Lab 028 lab detail: Off NVIDIA, you fix the platform
yourself", "What I changed, in plain terms" items 3-4, and its diag_off =
kL - qL).  The backward of that call returns dK / dV rows for the halo keys
as well; they go back to the owners, which add them into their own rows
with the library's add kernel.  The pages do not describe the sharding
itself; it follows from the band structure.

The arithmetic runs in the library's kernels; this module only plans the
halo, moves tensors between ranks and concatenates the halo with the local
keys.  The exchange is an object with `rank`, `world` and
`exchange(sends, recv_specs)`; `DistExchange` implements it with
torch.distributed point-to-point operations (NCCL between GPUs, gloo on
CPU).  `ThreadExchange` runs several ranks as threads of one process (each
thread calls the library on its own chunk and the threads meet on the host
to swap tensors), which lets one GPU check the sharded result against the
unsharded one; no kernel of one rank waits for another rank.
"""
from __future__ import annotations

import threading
from dataclasses import dataclass, field


def chunk_starts(lens):
    """First row of every chunk."""
    out, s = [], 0
    for n in lens:
        out.append(s)
        s += n
    return out


def halo_pieces(lens, window: int, r: int):
    """The halo of rank r as pieces (owner rank, first row in the owner's
    chunk, rows), in sequence order: the min(window - 1, s_r) positions
    before the chunk for a window, every earlier position for window 0."""
    starts = chunk_starts(lens)
    s = starts[r]
    h = s if window <= 0 else min(window - 1, s)
    lo = s - h
    pieces = []
    for p in range(r):
        a, b = max(lo, starts[p]), min(s, starts[p] + lens[p])
        if a < b:
            pieces.append((p, a - starts[p], b - a))
    return pieces


def halo_rows(lens, window: int, r: int) -> int:
    return sum(n for _, _, n in halo_pieces(lens, window, r))


@dataclass
class ShardCtx:
    """What the backward of a sharded forward needs."""
    q: object
    k_ext: object
    v_ext: object
    o: object
    lse: object
    halo: int
    pieces: list
    window: int
    scale: float
    lens: list = field(default_factory=list)


class GpuOps:
    """The per-rank steps on this library's kernels (C ABI)."""

    @staticmethod
    def forward(q, k, v, window, scale):
        from . import _native

        return _native.forward(q, k, v, window, scale, causal=True)

    @staticmethod
    def backward(q, k, v, o, lse, dO, window, scale):
        from . import _native

        return _native.backward(q, k, v, o, lse, dO, window, scale, causal=True)

    @staticmethod
    def add_rows(dst, src, row0):
        from . import _native

        _native.swa_attn_add_rows_f32(dst, src, row0)

    @staticmethod
    def cat_rows(parts):
        import torch

        return torch.cat(parts, dim=2).contiguous()


def _senders_to(lens, window, r):
    """(receiving rank t, first row in r's chunk, rows) for every halo piece
    of a later rank that rank r owns."""
    out = []
    for t in range(r + 1, len(lens)):
        for p, row0, n in halo_pieces(lens, window, t):
            if p == r:
                out.append((t, row0, n))
    return out


def sharded_forward(q, k, v, window: int, scale: float, lens, xchg, ops=GpuOps):
    """Forward of this rank's chunk: q [B, Hq, C_r, D], k and v
    [B, Hkv, C_r, D] (bf16), `lens` every rank's chunk length.  Returns
    (o, lse, ctx) for the chunk's rows; ctx feeds sharded_backward."""
    r = xchg.rank
    sends = {}
    for t, row0, n in _senders_to(lens, window, r):
        sends.setdefault(t, []).extend([k[:, :, row0:row0 + n].contiguous(), v[:, :, row0:row0 + n].contiguous()])
    pieces = halo_pieces(lens, window, r)
    B, Hkv, _, D = k.shape
    specs = {}
    for p, _, n in pieces:
        specs.setdefault(p, []).extend([((B, Hkv, n, D), k.dtype)] * 2)
    recv = xchg.exchange(sends, specs)
    halo = sum(n for _, _, n in pieces)
    if halo:
        ks, vs, used = [], [], {}
        for p, _, n in pieces:  # pieces of one owner arrive in sequence order
            i = used.get(p, 0)
            ks.append(recv[p][i])
            vs.append(recv[p][i + 1])
            used[p] = i + 2
        k_ext, v_ext = ops.cat_rows(ks + [k]), ops.cat_rows(vs + [v])
    else:
        k_ext, v_ext = k, v
    o, lse = ops.forward(q, k_ext, v_ext, window, scale)
    return o, lse, ShardCtx(q, k_ext, v_ext, o, lse, halo, pieces, window, scale, list(lens))


def sharded_backward(ctx: ShardCtx, dO, xchg, ops=GpuOps):
    """Backward of this rank's chunk: returns (dq, dk, dv) for its rows, with
    every later rank's halo contributions to its keys added in."""
    r = xchg.rank
    dq, dk_ext, dv_ext = ops.backward(ctx.q, ctx.k_ext, ctx.v_ext, ctx.o, ctx.lse, dO, ctx.window, ctx.scale)
    h = ctx.halo
    dk = dk_ext[:, :, h:].contiguous() if h else dk_ext
    dv = dv_ext[:, :, h:].contiguous() if h else dv_ext
    sends, off = {}, 0
    for p, _, n in ctx.pieces:
        sends.setdefault(p, []).extend([dk_ext[:, :, off:off + n].contiguous(), dv_ext[:, :, off:off + n].contiguous()])
        off += n
    B, Hkv, _, D = dk.shape
    back = _senders_to(ctx.lens, ctx.window, r)
    specs = {}
    for t, _, n in back:
        specs.setdefault(t, []).extend([((B, Hkv, n, D), dk.dtype)] * 2)
    recv = xchg.exchange(sends, specs)
    used = {}
    for t, row0, n in back:
        i = used.get(t, 0)
        ops.add_rows(dk, recv[t][i], row0)
        ops.add_rows(dv, recv[t][i + 1], row0)
        used[t] = i + 2
    return dq, dk, dv


class DistExchange:
    """Point-to-point exchange over torch.distributed: every rank posts its
    sends and receives at once (batch_isend_irecv), in a fixed order per
    pair of ranks."""

    def __init__(self, group=None, device=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.device = device

    def exchange(self, sends, recv_specs):
        import torch

        d = self.dist
        ops, out = [], {}
        for peer in sorted(set(sends) | set(recv_specs)):
            gpeer = d.get_global_rank(self.group, peer) if self.group is not None else peer
            # the lower rank sends first, so both sides list their operations in the same order
            first_send = self.rank < peer
            recvs = [torch.empty(shape, dtype=dt, device=self.device) for shape, dt in recv_specs.get(peer, [])]
            out[peer] = recvs
            s_ops = [d.P2POp(d.isend, t, gpeer, self.group) for t in sends.get(peer, [])]
            r_ops = [d.P2POp(d.irecv, t, gpeer, self.group) for t in recvs]
            ops.extend(s_ops + r_ops if first_send else r_ops + s_ops)
        if ops:
            for req in d.batch_isend_irecv(ops):
                req.wait()
        return out


class ThreadExchange:
    """Ranks as threads of one process (see the module docstring): the
    threads meet at a barrier, each posts its sends, and each collects what
    the others posted for it.  Device work is finished before a tensor
    changes hands."""

    class _Shared:
        def __init__(self, world):
            self.world = world
            self.barrier = threading.Barrier(world)
            self.box = {}

    def __init__(self, shared, rank):
        self.shared = shared
        self.rank = rank
        self.world = shared.world

    @classmethod
    def group(cls, world):
        shared = cls._Shared(world)
        return [cls(shared, r) for r in range(world)]

    def exchange(self, sends, recv_specs):
        import torch

        if torch.cuda.is_available():
            torch.cuda.synchronize()
        sh = self.shared
        for peer, ts in sends.items():
            sh.box[(self.rank, peer)] = list(ts)
        sh.barrier.wait()
        out = {}
        for peer, specs in recv_specs.items():
            got = sh.box[(peer, self.rank)]
            if [tuple(t.shape) for t in got] != [tuple(s) for s, _ in specs]:
                raise RuntimeError("halo exchange: received shapes do not match the plan")
            out[peer] = got
        sh.barrier.wait()
        for peer in sends:
            sh.box.pop((self.rank, peer), None)
        return out


def run_threads(world, fn):
    """Run fn(rank, exchange) on `world` threads; return their results in rank
    order (re-raises the first failure)."""
    xs = ThreadExchange.group(world)
    results, errors = [None] * world, []

    def body(r):
        try:
            results[r] = fn(r, xs[r])
        except BaseException as e:  # noqa: BLE001 - reported to the caller below
            errors.append(e)
            xs[r].shared.barrier.abort()

    threads = [threading.Thread(target=body, args=(r,)) for r in range(world)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]
    return results
