"""Seeded synthetic workloads for block-sparse spatio-temporal attention.

This module holds shapes, mask windows, seeds and random-number draws only --
none of the method's arithmetic -- so that the fp64 oracle side and the CUDA
side can be fed the very same bf16 bytes without sharing any other code.

Shapes follow the blog "Accelerating Spatio-Temporal Attention for Video
Diffusion on TPUs": 75,600 tokens, 10 heads, head dimension 128, bf16
(section "Implementing sparse attention on TPUs"), and 302K tokens at 1440p
(section "End-to-end results and takeaways").  The pages do not print the
frame/height/width split or the mask windows; the values below are this
library's choices (21 x 45 x 80 latent patches for 75.6K tokens, frame window
3, raster window 612; 21 x 90 x 160 and raster window 2450 at 1440p).

Recipe: one CPU ``torch.Generator`` per workload seeded with its index; Q, then
K, then V are drawn i.i.d. N(0, 1) in fp32 with shape [H][N][d] in frame-major
(F,H,W) token order and rounded to bf16 (round-to-nearest-even).  Per-head
routing flags (1 = temporal) come from ``randperm(H)`` of a generator seeded
with index + 100: the heads listed first (half of them) are temporal.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                 # seed of Q/K/V draws
    H: int                     # heads
    F: int                     # latent frames
    Hs: int                    # latent height
    Ws: int                    # latent width
    d: int                     # head dimension
    wf: int                    # spatial heads: |f_k - f_q| <= wf
    ws: int                    # temporal heads: |s_k - s_q| <= ws (raster index)
    flags: tuple = field(default=())   # explicit per-head flags; empty -> seeded
    n_temporal: int = 0        # number of temporal heads when flags are seeded
    BQ: int = 128
    BKV: int = 128
    rounding: tuple = (0,)     # mask modes exercised: 0 exact, 1 tile-aligned
    temporal_permuted: tuple = (1,)

    @property
    def S(self) -> int:
        return self.Hs * self.Ws

    @property
    def N(self) -> int:
        return self.F * self.S

    def head_flags(self) -> list:
        if self.flags:
            return [int(x) for x in self.flags]
        g = torch.Generator().manual_seed(self.index + 100)
        order = torch.randperm(self.H, generator=g).tolist()
        fl = [0] * self.H
        for h in order[: self.n_temporal]:
            fl[h] = 1
        return fl


TINY = Workload("tiny_256tok_1h_d64", 0, H=1, F=4, Hs=8, Ws=8, d=64, wf=1, ws=0,
                flags=(0,), BQ=64, BKV=64, rounding=(0, 1))
SMALL = Workload("small_3072tok_2h_d128", 1, H=2, F=8, Hs=16, Ws=24, d=128, wf=2, ws=40,
                 flags=(0, 1), rounding=(0, 1), temporal_permuted=(1, 0))
SPATIAL_75K = Workload("spatial_75600tok_10h_d128", 2, H=10, F=21, Hs=45, Ws=80, d=128, wf=3, ws=612,
                       flags=(0,) * 10, rounding=(0, 1))
MIXED_75K = Workload("mixed_75600tok_10h_d128", 3, H=10, F=21, Hs=45, Ws=80, d=128, wf=3, ws=612,
                     n_temporal=5, rounding=(0,), temporal_permuted=(1, 0))
P1440_302K = Workload("p1440_302400tok_10h_d128", 4, H=10, F=21, Hs=90, Ws=160, d=128, wf=3, ws=2450,
                      n_temporal=5, rounding=(1,))

ALL = [TINY, SMALL, SPATIAL_75K, MIXED_75K, P1440_302K]
BY_NAME = {w.name: w for w in ALL}


def qkv(w: Workload, H: int | None = None, N: int | None = None, d: int | None = None, seed: int | None = None):
    """Seeded bf16 Q, K, V of shape [H][N][d] on the CPU, (F,H,W) token order."""
    H = w.H if H is None else H
    N = w.N if N is None else N
    d = w.d if d is None else d
    g = torch.Generator().manual_seed(w.index if seed is None else seed)
    out = []
    for _ in range(3):
        x = torch.randn(H, N, d, generator=g, dtype=torch.float32)
        out.append(x.to(torch.bfloat16))
        del x
    return tuple(out)


def bf16_bits(x: torch.Tensor):
    """The uint16 bit pattern of a CPU bf16 tensor, as a numpy array (no copy of values)."""
    return x.contiguous().view(torch.int16).numpy().view("uint16")


def sample_rows(N: int, count: int, seed: int, BQ: int = 128) -> list:
    """Seeded, stratified query rows: both ends, tile edges near the ragged tail, and random rows."""
    g = torch.Generator().manual_seed(seed + 1000)
    fixed = {0, 1, N - 1, N - 2, (N // BQ) * BQ - 1 if N > BQ else 0, min(N - 1, (N // BQ) * BQ)}
    rnd = torch.randint(0, N, (max(0, count - len(fixed)),), generator=g).tolist()
    return sorted(set(int(r) for r in list(fixed) + rnd if 0 <= r < N))


def qkv_device(w: Workload, device, seed: int | None = None):
    """Seeded bf16 Q, K, V [H][N][d] drawn directly on a CUDA device (CUDA
    generator seeded with the workload index): used where the CPU draw of the
    full-size tensors would dominate a run.  Values differ from ``qkv`` but are
    equally seeded and reproducible on a given device type."""
    g = torch.Generator(device=device).manual_seed(w.index if seed is None else seed)
    out = []
    for _ in range(3):
        out.append(torch.randn(w.H, w.N, w.d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16))
    return tuple(out)
