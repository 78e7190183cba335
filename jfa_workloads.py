"""Seeded synthetic jagged-attention workloads.

This module only draws inputs: sequence lengths, offsets and N(0,1) bf16
values.  It holds none of the attention arithmetic, so both the CUDA path and
the fp64 oracle can read the same bytes from it without sharing any method
code.

The pages measure on production jagged shapes ("Optimizing Jagged Flash
Attention with TLX", Performance: broadcast dense Q against jagged K/V, and
equal-length dense shapes) that are not public.  The five workloads below are
synthetic stand-ins with the named length distributions.

Recipe (one seed per workload, k = 1..5 in the order below):
* lengths: numpy.random.default_rng(k)
* values: a CPU torch.Generator seeded with k draws float32 N(0,1) for q, k,
  v, dout in that order, each rounded to bf16 (round to nearest even)
* offsets: exclusive prefix sum of the lengths, int32
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    H: int
    D: int
    causal: bool
    broadcast_q: bool
    q_len: int  # dense Q length in broadcast mode, 0 otherwise
    lengths_desc: str
    extra: dict = field(default_factory=dict)
    Hkv: int = 0  # K/V heads (GQA); 0: as many as query heads
    window: tuple = (-1, -1)  # (left, right) band of a sliding window; -1: unbounded


WORKLOADS = {
    "tiny_self": Workload("tiny_self", 1, 4, 2, 64, False, False, 0,
                          "uniform int [1, 64]"),
    "jagged_self": Workload("jagged_self", 2, 64, 8, 128, False, False, 0,
                            "uniform int [16, 2048]"),
    "broadcast_q": Workload("broadcast_q", 3, 512, 4, 128, False, True, 256,
                            "log-normal, median 512, sigma 0.8, clipped [1, 4096]"),
    "causal_self": Workload("causal_self", 4, 32, 16, 128, True, False, 0,
                            "uniform int [256, 8192]"),
    "skewed_broadcast_q": Workload("skewed_broadcast_q", 5, 4096, 2, 64, False, True, 64,
                                   "geometric mean 200 clipped [1, 8192], 1% forced to 8192"),
}
ORDER = ["tiny_self", "jagged_self", "broadcast_q", "causal_self", "skewed_broadcast_q"]

# The GQA and sliding-window variants ("Optimizing Jagged Flash Attention with
# TLX", sections 3 and 4 name both as supported), measured on the lengths and
# values of two workloads above (same seeds): four query heads per K/V head on
# jagged_self, a 1024-key causal band on causal_self.
VARIANTS = {
    "jagged_self_gqa4": dict(base="jagged_self", Hkv=2),
    "causal_self_window1024": dict(base="causal_self", window=(1024, -1)),
}


def variant(name: str) -> Workload:
    import dataclasses
    v = dict(VARIANTS[name])
    return dataclasses.replace(WORKLOADS[v.pop("base")], **v)


def sample_lengths(w: Workload, B: int | None = None) -> np.ndarray:
    """Sequence lengths of workload `w` (optionally with a different B)."""
    B = w.B if B is None else B
    rng = np.random.default_rng(w.seed)
    if w.name == "tiny_self":
        L = rng.integers(1, 64, size=B, endpoint=True)
    elif w.name == "jagged_self":
        L = rng.integers(16, 2048, size=B, endpoint=True)
    elif w.name == "broadcast_q":
        z = rng.standard_normal(B)
        L = np.clip(np.round(np.exp(math.log(512.0) + 0.8 * z)), 1, 4096)
    elif w.name == "causal_self":
        L = rng.integers(256, 8192, size=B, endpoint=True)
    elif w.name == "skewed_broadcast_q":
        L = np.clip(rng.geometric(1.0 / 200.0, size=B), 1, 8192)
        n_long = max(1, int(round(0.01 * B)))
        L[rng.choice(B, size=n_long, replace=False)] = 8192
    else:
        raise KeyError(w.name)
    return L.astype(np.int64)


def offsets_from_lengths(lengths) -> np.ndarray:
    L = np.asarray(lengths, dtype=np.int64)
    off = np.zeros(L.size + 1, dtype=np.int64)
    np.cumsum(L, out=off[1:])
    if off[-1] >= 2 ** 31:
        raise ValueError("total token count exceeds int32 offsets")
    return off.astype(np.int32)


def draw_values(seed: int, shapes):
    """bf16 CPU tensors drawn as float32 N(0,1) in the given order."""
    import torch
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(s, generator=g, dtype=torch.float32).to(torch.bfloat16)
            for s in shapes]


def make_inputs(w: Workload, lengths=None, seed=None):
    """Host (CPU) inputs of workload `w`: dict with q, k, v, dout (bf16 torch
    CPU tensors), offsets (int32 numpy), lengths, and the shape scalars."""
    L = sample_lengths(w) if lengths is None else np.asarray(lengths, dtype=np.int64)
    off = offsets_from_lengths(L)
    T = int(off[-1])
    B = L.size
    H, D = w.H, w.D
    Hkv = w.Hkv or H
    if w.broadcast_q:
        shapes = [(w.q_len, H, D), (T, Hkv, D), (T, Hkv, D), (B, w.q_len, H, D)]
    else:
        shapes = [(T, H, D), (T, Hkv, D), (T, Hkv, D), (T, H, D)]
    q, k, v, do = draw_values(w.seed if seed is None else seed, shapes)
    return dict(q=q, k=k, v=v, dout=do, offsets=off, lengths=L, B=B, H=H, Hkv=Hkv, D=D,
                T=T, causal=w.causal, broadcast_q=w.broadcast_q, q_len=w.q_len,
                window=tuple(w.window), max_len=int(L.max()) if L.size else 0,
                scale=1.0 / math.sqrt(D))


def pairs(lengths, causal=False, q_len=0, broadcast_q=False, window=(-1, -1)) -> int:
    """Number of (query, key) pairs attended: the useful-work count.  A
    window (left, right) keeps keys [i - left, i + right] of query i."""
    L = np.asarray(lengths, dtype=np.int64)
    if broadcast_q:
        return int(q_len * L.sum())
    wl, wr = window
    if causal:
        wr = 0
    if wl < 0 and wr < 0:
        return int((L * L).sum())
    if wl < 0 and wr == 0:
        return int((L * (L + 1) // 2).sum())
    total = 0
    for n in L.tolist():
        i = np.arange(n, dtype=np.int64)
        lo = np.maximum(0, i - wl) if wl >= 0 else np.zeros_like(i)
        hi = np.minimum(n - 1, i + wr) if wr >= 0 else np.full_like(i, n - 1)
        total += int((hi - lo + 1).sum())
    return total


def random_block_lists(lengths, H, max_len, seed, p_keep=0.5, p_empty=0.0, q_len=0):
    """Seeded random block lists in the layout of the block-sparse forward:
    blocks int32 [B, H, nqb, kcap] (ascending K-block indices, -1 after the
    count) and counts int32 [B, H, nqb], nqb = ceil(max_len / 256) (with
    q_len > 0, broadcast-Q: ceil(q_len / 256)), kcap = ceil(max_len / 128).
    Each K block of the sequence is kept with probability p_keep (at least
    one unless the list is drawn empty, with probability p_empty); Q blocks
    past a sequence, and every Q block of a sequence without keys, get count
    0."""
    rng = np.random.default_rng(seed)
    L = np.asarray(lengths, dtype=np.int64)
    nqb, kcap = -(-(q_len if q_len > 0 else max_len) // 256), -(-max_len // 128)
    blocks = np.full((L.size, H, nqb, kcap), -1, dtype=np.int32)
    counts = np.zeros((L.size, H, nqb), dtype=np.int32)
    for b, n in enumerate(L.tolist()):
        nk = -(-n // 128)
        if nk == 0:
            continue
        for h in range(H):
            for i in range(nqb if q_len > 0 else -(-n // 256)):
                if rng.random() < p_empty:
                    continue
                keep = np.flatnonzero(rng.random(nk) < p_keep)
                if keep.size == 0:
                    keep = np.array([rng.integers(0, nk)])
                blocks[b, h, i, :keep.size] = keep
                counts[b, h, i] = keep.size
    return blocks, counts
