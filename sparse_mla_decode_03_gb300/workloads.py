"""Seeded synthetic inputs for sparse MLA decode.

This module only *produces* inputs: query vectors, packed FP8 KV-cache rows and
top-k index lists.  It contains none of the decode arithmetic (no dequantisation,
no scores, no softmax); both the CUDA path and the CPU oracle consume the bytes it
writes.

KV-cache row (584 bytes, one per cached token), as described on "The Power-of-Two
Trap: Debugging a Triton MMA Kernel on Blackwell GPUs", sections "3. The Scale
Indexing Complication" and "Input Knowledge Required" (7 groups of 64 FP8 columns,
one UE8M0 scale byte per group, one padding byte, then the bf16 rope part):

    bytes [  0, 448)  448 x FP8 e4m3 "nope" values
    bytes [448, 455)  7 x UE8M0 group scales, value 2**(byte - 127), group = col // 64
    byte   455        padding (never used as a scale)
    bytes [456, 584)  64 x bf16 "rope" values, little endian

Writing a row quantises x ~ N(0, 1) per 64-column group with the scale
2**ceil(log2(amax / 448)), so every quantised magnitude is <= 448 (the largest
finite e4m3 value), and rounds x / scale to e4m3 with round-to-nearest-even.

Workloads follow the five benchmark shapes of the project (one decode token per
sequence):

    c1  B=1,  H=64, 4096 rows/seq,   k=128,  uniform unique indices
    c2  B=4,  H=64, 16384 rows/seq,  k=512,  uniform unique indices
    c3  B=32, H=64, 65536 rows/seq,  k=2048, 1024 from the last 4096 positions
                                              + 1024 uniform over the rest, shuffled
    c4  B=96, H=16, 131072 rows/seq, k=2048, uniform unique indices
    c5  B=64, H=64, ragged lengths U[1024, 262144], k=2048, min(2048, L) valid
                                              picks, the tail padded with -1; 1 % of
                                              nope values scaled x50
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

ROW_BYTES = 584
NOPE = 448
ROPE = 64
QK_DIM = 512
GROUP = 64
N_GROUPS = 7
SCALE_OFF = 448
PAD_OFF = 455
ROPE_OFF = 456
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    topk: int
    rows_per_seq: int            # 0 for ragged
    index_law: str               # "uniform" | "recent_half" | "ragged"
    outlier_frac: float = 0.0
    outlier_mult: float = 50.0
    ragged_lo: int = 1024
    ragged_hi: int = 262144
    seed: int = 0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(QK_DIM)


WORKLOADS = {
    "c1": Workload("c1_b1_h64_k128", 1, 64, 128, 4096, "uniform", seed=1001),
    "c2": Workload("c2_b4_h64_k512", 4, 64, 512, 16384, "uniform", seed=1002),
    "c3": Workload("c3_b32_h64_k2048", 32, 64, 2048, 65536, "recent_half", seed=1003),
    "c4": Workload("c4_b96_h16_k2048", 96, 16, 2048, 131072, "uniform", seed=1004),
    "c5": Workload("c5_b64_h64_k2048_ragged", 64, 64, 2048, 0, "ragged",
                   outlier_frac=0.01, seed=1005),
}


def seq_lengths(w: Workload) -> np.ndarray:
    """Cached tokens per sequence (int64 [B])."""
    if w.index_law == "ragged":
        rng = np.random.default_rng(w.seed * 7 + 1)
        return rng.integers(w.ragged_lo, w.ragged_hi + 1, size=w.batch, dtype=np.int64)
    return np.full(w.batch, w.rows_per_seq, dtype=np.int64)


def seq_bases(lengths: np.ndarray) -> np.ndarray:
    """First row of each sequence in the contiguous row pool."""
    return np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)


def make_indices(w: Workload, lengths: np.ndarray, variant: int = 0) -> np.ndarray:
    """Flat row ids int32 [B, topk]; -1 marks a masked slot.

    ``variant`` selects an independent draw (used to rotate index sets so that a
    benchmark loop does not re-read the same rows from L2)."""
    rng = np.random.default_rng([w.seed, 17, variant])
    bases = seq_bases(lengths)
    out = np.full((w.batch, w.topk), -1, dtype=np.int64)
    for b in range(w.batch):
        L = int(lengths[b])
        if w.index_law == "uniform":
            pos = rng.choice(L, size=w.topk, replace=False)
        elif w.index_law == "recent_half":
            recent = min(4096, L)
            half = w.topk // 2
            a = L - recent + rng.choice(recent, size=half, replace=False)
            rest = rng.choice(L - recent, size=w.topk - half, replace=False)
            pos = rng.permutation(np.concatenate([a, rest]))
        elif w.index_law == "ragged":
            n = min(w.topk, L)
            pos = np.full(w.topk, -1, dtype=np.int64)
            pos[:n] = rng.choice(L, size=n, replace=False)
        else:
            raise ValueError(w.index_law)
        row = np.where(pos >= 0, pos + bases[b], -1)
        out[b] = row
    assert out.max() < np.iinfo(np.int32).max
    return out.astype(np.int32)


def _quantise_block(x: torch.Tensor, pad_byte: int) -> torch.Tensor:
    """x: float32 [n, 448] -> uint8 [n, 448 + 8] (FP8 bytes, 7 scale bytes, pad)."""
    n = x.shape[0]
    g = x.view(n, N_GROUPS, GROUP)
    amax = g.abs().amax(dim=2)                                   # [n, 7]
    mant, ex = torch.frexp(amax / E4M3_MAX)
    e = torch.where(mant > 0.5, ex, ex - 1)                      # ceil(log2(amax/448))
    sbyte = torch.clamp(e + 127, 1, 254)
    sbyte = torch.where(amax == 0, torch.full_like(sbyte, 127), sbyte)
    q = torch.ldexp(g, (127 - sbyte).to(torch.float32).unsqueeze(2))
    fp8 = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, NOPE)
    tail = torch.full((n, 8), pad_byte, dtype=torch.uint8, device=x.device)
    tail[:, :N_GROUPS] = sbyte.to(torch.uint8)
    return torch.cat([fp8, tail], dim=1)


def make_cache(w: Workload, lengths: np.ndarray, device="cpu", pad_byte: int = 0,
               chunk: int = 1 << 20, gen_seed: Optional[int] = None) -> torch.Tensor:
    """Packed KV cache uint8 [sum(lengths), 584] on ``device``."""
    total = int(lengths.sum())
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed if gen_seed is None else gen_seed)
    cache = torch.empty((total, ROW_BYTES), dtype=torch.uint8, device=dev)
    for r0 in range(0, total, chunk):
        n = min(chunk, total - r0)
        x = torch.randn((n, NOPE), generator=gen, device=dev, dtype=torch.float32)
        if w.outlier_frac > 0:
            sel = torch.rand((n, NOPE), generator=gen, device=dev) < w.outlier_frac
            x = torch.where(sel, x * w.outlier_mult, x)
        rope = torch.randn((n, ROPE), generator=gen, device=dev, dtype=torch.float32)
        cache[r0:r0 + n, :ROPE_OFF] = _quantise_block(x, pad_byte)
        cache[r0:r0 + n, ROPE_OFF:] = rope.to(torch.bfloat16).view(torch.uint8).view(n, 2 * ROPE)
    return cache


def make_q(w: Workload, device="cpu", gen_seed: Optional[int] = None) -> torch.Tensor:
    """Query bf16 [B, H, 512] = 448 nope | 64 rope, entries ~ N(0, 1)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed((w.seed if gen_seed is None else gen_seed) + 500)
    q = torch.randn((w.batch, w.heads, QK_DIM), generator=gen, device=dev, dtype=torch.float32)
    return q.to(torch.bfloat16)


def compact_rows(kv: torch.Tensor, indices: np.ndarray):
    """Host copy of only the referenced rows, with indices remapped into it.

    Returns (rows uint8 [U, 584] numpy, remapped int64 [B, k] with -1 kept)."""
    idx = np.asarray(indices, dtype=np.int64)
    valid = idx >= 0
    uniq, inv = np.unique(idx[valid], return_inverse=True)
    rows = kv[torch.as_tensor(uniq, device=kv.device)].cpu().numpy()
    remap = np.full(idx.shape, -1, dtype=np.int64)
    remap[valid] = inv
    return rows, remap


def bf16_bits(q: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) of a bf16 tensor, as numpy on the host."""
    return q.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gathered_kv_bytes(indices: np.ndarray) -> int:
    """Bytes of KV rows one decode call must read (584 per valid index)."""
    return int((np.asarray(indices) >= 0).sum()) * ROW_BYTES


def algorithmic_bytes(w: Workload, indices: np.ndarray) -> int:
    """Minimum HBM bytes of one call: gathered rows + q + out + lse + indices."""
    B, H, k = w.batch, w.heads, w.topk
    return (gathered_kv_bytes(indices) + B * H * QK_DIM * 2 + B * H * NOPE * 2
            + B * H * 4 + B * k * 4)


def algorithmic_flops(w: Workload, indices: np.ndarray) -> int:
    """2 * H * (512 + 448) multiply-adds per valid (query, row) pair."""
    valid = int((np.asarray(indices) >= 0).sum())
    return 2 * w.heads * valid * (QK_DIM + NOPE)

