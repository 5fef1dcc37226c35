"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds the workload shapes and the random-number recipe only. It
does none of the attention arithmetic: the CUDA path and the CPU oracle both
take their inputs from here and nothing else is shared between them.

Shapes follow the video-token counts of "Training a Large Video Model on a
Single Machine in a Day": a clip is cut into N = (T/t)(H/h)(W/w) cubes
(§3, "Video Transformer"), e.g. 16 frames of 224x224 with 2x16x16 tubelets give
8x14x14 = 1568 tokens (§5.5). The long-visual cross-attention shape is the one
the LV-XAttn poster (ICML 2025, Abstract) describes: a short query block
against a very long key/value block.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws, in the
order q, k, v, dO, one float32 N(0, 1) tensor each, rounded to bfloat16. The
ViT-L workload doubles K after rounding (exact in bf16) to sharpen the softmax.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    d: int
    seed: int
    k_mult: float = 1.0
    n_chunks: int = 1        # split-KV chunks for the cross-attention forward

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def heads(self) -> int:
        return self.B * self.H

    def fwd_flops(self) -> float:
        """QK^T and PV: 2 * 2 * Lq * Lk * d per head."""
        return 4.0 * self.B * self.H * self.Lq * self.Lk * self.d

    def bwd_flops(self) -> float:
        """Recomputed QK^T plus dP, dV, dK, dQ: 5 * 2 * Lq * Lk * d per head."""
        return 10.0 * self.B * self.H * self.Lq * self.Lk * self.d

    def describe(self) -> str:
        s = f"B{self.B} H{self.H} Lq{self.Lq} Lk{self.Lk} d{self.d}"
        if self.k_mult != 1.0:
            s += f" Kx{self.k_mult:g}"
        if self.n_chunks > 1:
            s += f" split{self.n_chunks}"
        return s


# The five workloads: a tiny self-attention case, two ViT video self-attention
# cases at 1568 tokens, the long-visual cross-attention case split into 8 KV
# chunks, and a 128-frame long-video self-attention case (64x14x14 = 12544).
TINY = Workload("tiny", 1, 1, 98, 98, 64, seed=0)
VIT_B = Workload("vit_b", 32, 12, 1568, 1568, 64, seed=1)
VIT_L = Workload("vit_l", 16, 16, 1568, 1568, 64, seed=2, k_mult=2.0)
CROSS = Workload("cross", 2, 32, 512, 36864, 128, seed=3, n_chunks=8)
LONG_VIDEO = Workload("long_video", 2, 16, 12544, 12544, 64, seed=4)

ALL = {w.name: w for w in (TINY, VIT_B, VIT_L, CROSS, LONG_VIDEO)}

# Factorised space-time attention of the ViT-L clip (16 clips of 8 x 14 x 14
# tubelets, 16 heads, d = 64), as in divided space-time video transformers:
# temporal attention runs over the 8 tubelet-frames of each of the 196 spatial
# positions, (b*h*w, t, d); spatial attention over the 196 patches of each of
# the 8 tubelet-frames, (b*t, h*w, d) (the layouts of the NeMo video page's
# Table 2).
TEMPORAL = Workload("temporal", 16 * 196, 16, 8, 8, 64, seed=6)
SPATIAL = Workload("spatial", 16 * 8, 16, 196, 196, 64, seed=7)


def chunk_bounds(Lk: int, n_chunks: int) -> list[tuple[int, int]]:
    """Contiguous, nearly equal KV ranges [k0, k1) covering [0, Lk)."""
    bounds = []
    for c in range(n_chunks):
        k0 = (Lk * c) // n_chunks
        k1 = (Lk * (c + 1)) // n_chunks
        bounds.append((k0, k1))
    return bounds


def make_inputs(w: Workload, seed: int | None = None, *, B: int | None = None,
                H: int | None = None, Lq: int | None = None, Lk: int | None = None,
                d: int | None = None):
    """Return (q, k, v, do) as contiguous CPU bf16 tensors [B, H, L, d].

    Keyword overrides let tests reuse a workload's recipe at other sizes.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    Lq = w.Lq if Lq is None else Lq
    Lk = w.Lk if Lk is None else Lk
    d = w.d if d is None else d
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    q = torch.randn((B, H, Lq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, H, Lk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, H, Lk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    do = torch.randn((B, H, Lq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    if w.k_mult != 1.0:
        k = (k * w.k_mult).to(torch.bfloat16)
    return q, k, v, do


@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    """Packed sequences of mixed lengths ("sequence packing" of images and
    videos of different sizes, NeMo video foundation-model page, "Efficient
    multimodal dataloading"): lengths are drawn from ``lengths`` (token counts
    of a 224x224 image, 16x16 patches = 196, and of 2/4/8 tubelet-frames of it)
    until ``total`` tokens are packed; the last sequence takes the remainder.
    Self-attention within each sequence: cu_q = cu_k."""
    name: str
    H: int
    d: int
    total: int
    lengths: tuple
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def seqlens(self) -> list[int]:
        g = torch.Generator().manual_seed(self.seed)
        out, used = [], 0
        while True:
            n = self.lengths[int(torch.randint(len(self.lengths), (1,), generator=g))]
            if used + n > self.total:
                break
            out.append(n)
            used += n
        if used < self.total:
            out.append(self.total - used)
        return out

    def cu_seqlens(self) -> list[int]:
        cu = [0]
        for n in self.seqlens():
            cu.append(cu[-1] + n)
        return cu

    def fwd_flops(self) -> float:
        return sum(4.0 * self.H * n * n * self.d for n in self.seqlens())

    def bwd_flops(self) -> float:
        return sum(10.0 * self.H * n * n * self.d for n in self.seqlens())

    def describe(self) -> str:
        return f"packed T{self.total} ({len(self.seqlens())} seqs of {self.lengths}) H{self.H} d{self.d}"


# The ViT-L batch's token count (16 x 1568) packed as a mix of images and clips.
VARLEN_MIX = VarlenWorkload("varlen_mix", H=16, d=64, total=16 * 1568,
                            lengths=(196, 392, 784, 1568), seed=5)


def make_varlen_inputs(Tq: int, Tk: int, H: int, d: int, seed: int, device=None):
    """Return (q, k, v, do) as contiguous bf16 token-major tensors (q, do
    [Tq, H, d]; k, v [Tk, H, d]), drawn as in make_inputs: on the CPU, or, with
    ``device``, directly there (other values; for timing runs)."""
    g = torch.Generator(device=device or "cpu").manual_seed(seed)

    def draw(shape):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)

    q, k, v, do = draw((Tq, H, d)), draw((Tk, H, d)), draw((Tk, H, d)), draw((Tq, H, d))
    return q, k, v, do


def make_inputs_device(w: Workload, device, seed: int | None = None):
    """Same distribution drawn directly on a device (for the large timed runs).

    The values differ from make_inputs (different generator); use this only
    where the check is a sampled or property-based one that draws its own
    oracle inputs from the very tensors used.
    """
    g = torch.Generator(device=device).manual_seed(w.seed if seed is None else seed)
    shp_q = (w.B, w.H, w.Lq, w.d)
    shp_k = (w.B, w.H, w.Lk, w.d)
    q = torch.randn(shp_q, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(shp_k, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(shp_k, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    do = torch.randn(shp_q, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    if w.k_mult != 1.0:
        k = (k * w.k_mult).to(torch.bfloat16)
    return q, k, v, do
