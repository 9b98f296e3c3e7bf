"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: only shapes and random-number
recipes.  It is the one piece the CUDA path's tests and the oracle share.

Recipe (all on the CPU, so both sides see identical bf16 values):
  gen = torch.Generator().manual_seed(seed)
  q, k, v, dO drawn in that order with torch.randn(shape, float32, gen)
  dO multiplied by `do_scale` in fp32
  with outliers: per (b, kv head), round(frac * L) distinct key rows drawn
    without replacement (torch.randperm with the same generator, after dO),
    multiplied by `outlier_mult` in fp32
  finally every tensor is rounded to bf16 (round-to-nearest-even).

The five named workloads are shaped like the pages' Gemma-style sliding and
global layers: the sliding layers use D=256, 16 kv heads, 32 query heads and
a 1,024-token window; the global layers D=512 with 4 kv heads ("Lab 028 lab
detail", "Starting point"), and the long step is 30,553 tokens ("Model
step").  Peaky softmax rows (scores in the 20s on real activations, "fp32
gradient truth", layer-level table) are imitated by scaling 1% of the key
rows by 8.

Two more workloads exercise the band variants the same page's parity sweep
covers ("Gradient parity": qL < kL, windows causal and not): the sliding
layer with its queries a suffix of the keys, and a non-causal window.  A
suffix workload draws the full-length tensors with the recipe above and keeps
the last Lq rows of q and dO.  The decode workload is one generation step
(Lq = 1, forward only) of a batch of 8 over a 16,384-token cache of the
global layer.

The shared-prefix workload is the sliding layer over one preference pair
laid out as [prompt (6,144 tokens); chosen response (1,024); rejected
response (1,024)], the single-pass layout of "Training -- design (ORPO,
flash-CCE head, prefix sharing, segmented backward)", section 5.4, with the
window on logical positions.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    D: int
    window: int
    do_scale: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 8.0
    seed: int = 0
    Lq: int = 0          # query rows (the last Lq of the L key positions); 0 means L
    causal: bool = True
    fwd_only: bool = False  # a decode step: the forward alone
    prompt_len: int = 0  # shared-prefix plan [prompt; chosen; rejected] when chosen_len > 0
    chosen_len: int = 0

    @property
    def prefix(self):
        """(prompt_len, chosen_len) of a shared-prefix plan, or None."""
        return (self.prompt_len, self.chosen_len) if self.chosen_len > 0 else None

    @property
    def q_rows(self) -> int:
        return self.Lq or self.L

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def pairs(self) -> int:
        """In-band (query, key) pairs over all batches and query heads."""
        if self.prefix:
            return self.B * self.Hq * band_pairs_prefix(self.L, self.window, *self.prefix)
        if self.q_rows == self.L and self.causal:
            return self.B * self.Hq * band_pairs(self.L, self.window)
        return self.B * self.Hq * band_pairs_ex(self.q_rows, self.L, self.window, self.causal)

    def fwd_flops(self) -> int:
        return 4 * self.D * self.pairs()

    def bwd_flops(self) -> int:
        return 10 * self.D * self.pairs()


def band_pairs(L: int, window: int) -> int:
    """Number of (i, j) with j <= i and (window == 0 or i - j < window)."""
    if window <= 0 or window >= L:
        return L * (L + 1) // 2
    w = window
    # rows 0..w-1 see i+1 keys, the remaining rows see w keys
    return w * (w + 1) // 2 + (L - w) * w


def band_pairs_ex(Lq: int, Lk: int, window: int, causal: bool) -> int:
    """In-band pairs when query i sits at key position a = i + Lk - Lq:
    causal keeps j <= a (and a - j < window), non-causal |a - j| < window
    (window 0: every key)."""
    w = window if 0 < window < Lk else 0
    total = 0
    for i in range(Lq):
        a = i + Lk - Lq
        lo = max(0, a - w + 1) if w else 0
        hi = a if causal else (min(Lk - 1, a + w - 1) if w else Lk - 1)
        total += hi - lo + 1
    return total


def band_pairs_prefix(L: int, window: int, P: int, Rc: int) -> int:
    """In-band pairs of one [prompt (P); chosen (Rc); rejected (L - P - Rc)]
    sequence under the shared-prefix mask: rows before the rejected response
    see the plain causal window; a rejected row i (logical position i - Rc)
    sees the prompt keys within the window of its logical position and the
    keys of its own response within the window."""
    w = window if 0 < window < L else 0
    R = P + Rc
    total = band_pairs(R, w) if R > 0 else 0
    for i in range(R, L):
        a = i - Rc
        lo = max(0, a - w + 1) if w else 0
        total += max(0, P - lo)                      # prompt keys [lo, P - 1]
        total += i - (max(R, i - w + 1) if w else R) + 1  # own response keys
    return total


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_l256_d64_w64", 1, 2, 1, 256, 64, 64, seed=20260001),
        Workload("causal_gqa_l8192_d128", 1, 8, 4, 8192, 128, 0, seed=20260002),
        Workload("sliding_l8192_d256_w1024", 1, 32, 16, 8192, 256, 1024, do_scale=0.1, seed=20260003),
        Workload("global_l16384_d512", 1, 32, 4, 16384, 512, 0, do_scale=0.1, seed=20260004),
        Workload("ragged_l30553_d256_w1024_outliers", 1, 32, 16, 30553, 256, 1024,
                 outlier_frac=0.01, seed=20260005),
        Workload("suffix_q2048_k8192_d256_w1024", 1, 32, 16, 8192, 256, 1024, do_scale=0.1, seed=20260006,
                 Lq=2048),
        Workload("noncausal_l8192_d128_w512", 1, 8, 4, 8192, 128, 512, seed=20260007, causal=False),
        Workload("decode_b8_q1_k16384_d512", 8, 32, 4, 16384, 512, 0, seed=20260008, Lq=1, fwd_only=True),
        Workload("prefix_p6144_c1024_r1024_d256_w1024", 1, 32, 16, 8192, 256, 1024, do_scale=0.1, seed=20260009,
                 prompt_len=6144, chosen_len=1024),
    ]
}


def make_inputs(B, Hq, Hkv, L, D, seed, do_scale=1.0, outlier_frac=0.0, outlier_mult=8.0):
    """Return (q, k, v, dO) as contiguous CPU bf16 tensors [B, H, L, D]."""
    gen = torch.Generator().manual_seed(int(seed))
    q = torch.randn((B, Hq, L, D), dtype=torch.float32, generator=gen)
    k = torch.randn((B, Hkv, L, D), dtype=torch.float32, generator=gen)
    v = torch.randn((B, Hkv, L, D), dtype=torch.float32, generator=gen)
    dO = torch.randn((B, Hq, L, D), dtype=torch.float32, generator=gen)
    if do_scale != 1.0:
        dO.mul_(do_scale)
    if outlier_frac > 0.0:
        n = int(round(outlier_frac * L))
        for b in range(B):
            for h in range(Hkv):
                idx = torch.randperm(L, generator=gen)[:n]
                k[b, h, idx, :] *= outlier_mult
    return tuple(t.to(torch.bfloat16).contiguous() for t in (q, k, v, dO))


def workload_inputs(w: Workload):
    q, k, v, dO = make_inputs(w.B, w.Hq, w.Hkv, w.L, w.D, w.seed, w.do_scale, w.outlier_frac, w.outlier_mult)
    if w.q_rows < w.L:
        q, dO = (t[:, :, w.L - w.q_rows:].contiguous() for t in (q, dO))
    return q, k, v, dO
