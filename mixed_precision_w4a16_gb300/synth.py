"""Seeded synthetic inputs for the W4A16 linear layer.

This module only draws random numbers; it holds none of the method's
arithmetic (no dequantisation, no packing, no products).  Both the CUDA path
and the CPU oracle are fed from here, so that they see the same bytes.

Value distributions follow the layer shapes the MARLIN paper benchmarks
("MARLIN: Mixed-Precision Auto-Regressive Parallel Inference on LLMs",
Section 3.4 and Figure 1): activations ~ N(0, 1) rounded to FP16, 4-bit codes
uniform on {0..15}, FP16 scales uniform on [0.002, 0.02].  numpy's FP16 cast
rounds to nearest-even.

Generators: ``numpy.random.Generator(PCG64(SeedSequence([seed, stream])))``
with stream 0 for activations and stream 1 for weights, so one layer's
weights stay the same while the batch size M is swept.
"""
from __future__ import annotations

import numpy as np

__all__ = ["make_weights", "make_fp16_weights", "make_raw_weights", "make_activations", "make_layer",
           "make_expert_rows", "make_moe_layer", "make_weights_24", "effective_group"]


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def effective_group(K: int, groupsize: int) -> int:
    """Group size G along K; -1 (or K) selects one scale per column."""
    return K if groupsize in (-1, K) else int(groupsize)


def make_weights(K: int, N: int, groupsize: int, seed: int):
    """Codes ``q`` uint8[K][N] uniform on 0..15 and scales ``s`` float16[K/G][N]
    uniform on [0.002, 0.02]."""
    G = effective_group(K, groupsize)
    if G <= 0 or K % G:
        raise ValueError("K must be a positive multiple of the group size")
    rng = _rng(seed, 1)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s = rng.uniform(0.002, 0.02, size=(K // G, N)).astype(np.float16)
    return q, s


def make_fp16_weights(K: int, N: int, groupsize: int, seed: int, signed_scales: bool = False):
    """Unquantised weights ``w`` float16[K][N] ~ N(0, 0.05) and scales ``s``
    float16[K/G][N] uniform on [0.01, 0.03] (optionally with random signs), the
    inputs of quantise-and-repack: w / s is mostly inside the 4-bit range, with
    some values beyond it on either side."""
    G = effective_group(K, groupsize)
    if G <= 0 or K % G:
        raise ValueError("K must be a positive multiple of the group size")
    rng = _rng(seed, 2)
    w = (rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.05)).astype(np.float16)
    s = rng.uniform(0.01, 0.03, size=(K // G, N))
    if signed_scales:
        s = s * rng.choice(np.array([-1.0, 1.0]), size=s.shape)
    return w, s.astype(np.float16)


def make_raw_weights(K: int, N: int, seed: int) -> np.ndarray:
    """Unquantised weights float16[K][N] ~ N(0, 0.05) for the scale-finding step,
    with some columns of other shapes: every 16th column (from 1) all positive,
    (from 2) all negative, (from 3) scaled by 1e-4 (FP16 subnormal steps),
    (from 4) scaled by 300, and the first rows of column 5 all zero (a zero
    range in its first group)."""
    rng = _rng(seed, 3)
    w = rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.05)
    w[:, 1::16] = np.abs(w[:, 1::16]) + np.float32(0.01)
    w[:, 2::16] = -np.abs(w[:, 2::16]) - np.float32(0.02)
    w[:, 3::16] *= np.float32(1e-4)
    w[:, 4::16] *= np.float32(300.0)
    if N > 5:
        w[: min(K, 128), 5] = 0.0
    return w.astype(np.float16)


def make_activations(M: int, K: int, seed: int) -> np.ndarray:
    """Activations ``A`` float16[M][K] drawn from N(0, 1)."""
    rng = _rng(seed, 0)
    return rng.standard_normal((M, K), dtype=np.float32).astype(np.float16)


def make_layer(M: int, K: int, N: int, groupsize: int, seed: int):
    """A, q, s of one layer from one seed (weights and activations on separate streams)."""
    q, s = make_weights(K, N, groupsize, seed)
    return {"A": make_activations(M, K, seed), "q": q, "s": s,
            "G": effective_group(K, groupsize)}


def make_expert_rows(tokens: int, topk: int, E: int, seed: int, skew: float = 0.0) -> np.ndarray:
    """Rows per expert of a top-k routed batch, int64[E] summing to tokens * topk:
    each token picks topk distinct experts with probabilities proportional to
    (rank + 1) ** -skew over a random ranking of the experts (skew 0: uniform;
    larger: a few hot experts, many cold or empty ones)."""
    if topk > E:
        raise ValueError("topk must not exceed the number of experts")
    rng = _rng(seed, 4)
    p = (np.arange(E) + 1.0) ** -float(skew)
    p = p[rng.permutation(E)]
    p /= p.sum()
    counts = np.zeros(E, dtype=np.int64)
    for _ in range(tokens):
        counts[rng.choice(E, size=topk, replace=False, p=p)] += 1
    return counts


def make_moe_layer(tokens: int, topk: int, E: int, K: int, N: int, groupsize: int, seed: int, skew: float = 0.0,
                   counts=None):
    """An expert-grouped layer: offsets int32[E+1] (rows of expert e are offsets[e] ..
    offsets[e+1] - 1), activations A float16[M][K] with M = sum of the counts (rows
    already sorted by expert), and per-expert codes q uint8[E][K][N] and scales
    s float16[E][K/G][N] (expert e drawn from seed * 1000 + e)."""
    if counts is None:
        counts = make_expert_rows(tokens, topk, E, seed, skew)
    counts = np.asarray(counts, dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1])
    qs = [make_weights(K, N, groupsize, seed * 1000 + e) for e in range(E)]
    return {"offsets": offsets, "A": make_activations(M, K, seed), "q": np.stack([x[0] for x in qs]),
            "s": np.stack([x[1] for x in qs]), "G": effective_group(K, groupsize)}


def make_weights_24(K: int, N: int, groupsize: int, seed: int):
    """2:4-sparse codes: in every group of four consecutive rows of a column two
    positions (one of the six pairs, uniform) hold codes uniform on 0..15 and
    the other two hold 8 (a zero weight); scales as ``make_weights``.  Returns
    dense q uint8[K][N] and s float16[K/G][N]."""
    G = effective_group(K, groupsize)
    if G <= 0 or K % G or K % 4:
        raise ValueError("K must be a positive multiple of the group size and of 4")
    rng = _rng(seed, 5)
    pairs = np.array([(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)])
    choice = pairs[rng.integers(0, 6, size=(K // 4, N))]          # [K/4][N][2]
    vals = rng.integers(0, 16, size=(K // 4, N, 2), dtype=np.uint8)
    q = np.full((K // 4, 4, N), 8, dtype=np.uint8)
    gi, ni = np.meshgrid(np.arange(K // 4), np.arange(N), indexing="ij")
    for j in range(2):
        q[gi, choice[:, :, j], ni] = vals[:, :, j]
    s = rng.uniform(0.002, 0.02, size=(K // G, N)).astype(np.float16)
    return q.reshape(K, N), s
