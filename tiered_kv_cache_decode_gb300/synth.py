"""Seeded synthetic workloads for the tiered KV-cache decode path.

This module only draws inputs: keys, values, queries, initial window scores,
score drift factors and tier draws. It holds none of the cache's arithmetic
(no quantiser, no attention, no routing), so that the CPU oracle and the CUDA
path can both be fed from it without sharing any of the method.

Recipe (the same on CPU and GPU; every function takes a ``device``):

* Random bits: splitmix64 used as a counter-based generator. Element ``i`` of
  a stream with key ``k`` is ``mix64(k + (i + 1) * GAMMA)``; stream keys are
  derived from the seed and a tuple of integer tags by repeated ``mix64``.
* Uniforms: the top 53 bits of a draw times 2**-53, in [0, 1).
* Normals: Box-Muller, cosine branch only; normal ``i`` uses uniforms ``2i``
  and ``2i + 1``. Rounded float64 -> float32 -> bfloat16, each step
  round-to-nearest-even.
* Student-t with 3 degrees of freedom: ``z / sqrt((z1^2 + z2^2 + z3^2) / 3)``.
* Outlier channels, "tiny" mode: 4 head_dim channels (seeded draw without
  replacement) of K are scaled by 8 for every KV head and token.
  "heavy" mode: round(0.01 * Hkv * d) of the Hkv*d (head, channel) pairs per
  layer, drawn separately for K and for V, carry Student-t(3) values instead of
  N(0, 1).
* Window scores: Zipf(1.1) over a seeded permutation of ranks 1..W,
  ``S_w = r_w^-1.1 / H_{W,1.1}``.
* Drift factors at a routing event: ``exp(0.5 * z_w)``.
* Tier draws: a seeded Fisher-Yates permutation of the windows; the first
  ``n_fp`` become full precision, the next ``n_q`` INT2, the rest evicted.

The K/V of token position ``p`` is a pure function of (seed, layer, p), so a
prefill of L tokens followed by appends yields the same stream as a longer
prefill.
"""
from __future__ import annotations

import math

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# stream tags
TAG_K, TAG_V, TAG_Q, TAG_OUTLIER, TAG_SCORE, TAG_DRIFT, TAG_TIER, TAG_TINY = range(1, 9)

TIER_FP, TIER_Q, TIER_E = 0, 1, 2


def _s64(x: int) -> int:
    """Reinterpret an unsigned 64-bit integer as signed (torch int64)."""
    x &= MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def mix64(z: int) -> int:
    """splitmix64 finaliser on a Python integer."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, *tags: int) -> int:
    k = mix64(seed + GAMMA)
    for t in tags:
        k = mix64(k ^ mix64((t + 1) * GAMMA))
    return k


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def bits(key: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """Draws start..start+n-1 of stream ``key`` as int64 bit patterns."""
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    z = i * _s64(GAMMA) + _s64(key)
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def uniforms(key: int, start: int, n: int, device="cpu") -> torch.Tensor:
    b = bits(key, start, n, device)
    return _lsr(b, 11).to(torch.float64) * (2.0 ** -53)


def normals(key: int, start: int, n: int, device="cpu") -> torch.Tensor:
    u = uniforms(key, 2 * start, 2 * n, device).view(n, 2)
    r = torch.sqrt(-2.0 * torch.log1p(-u[:, 0]))
    return r * torch.cos((2.0 * math.pi) * u[:, 1])


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float32).to(torch.bfloat16)


def student_t3(key: int, start: int, n: int, device="cpu") -> torch.Tensor:
    z = normals(key, 4 * start, 4 * n, device).view(n, 4)
    chi2 = (z[:, 1:] ** 2).sum(dim=1)
    return z[:, 0] / torch.sqrt(chi2 / 3.0)


def choose_without_replacement(key: int, population: int, k: int) -> list[int]:
    """Seeded partial Fisher-Yates: k distinct indices of range(population)."""
    u = uniforms(key, 0, k).tolist()
    perm = list(range(population))
    for i in range(k):
        j = i + int(u[i] * (population - i))
        perm[i], perm[j] = perm[j], perm[i]
    return perm[:k]


def permutation(key: int, n: int) -> list[int]:
    return choose_without_replacement(key, n, n)


def outlier_pairs(seed: int, layer: int, kv: int, Hkv: int, d: int) -> list[int]:
    """Flattened (head * d + channel) indices with heavy-tailed values."""
    n = int(round(0.01 * Hkv * d))
    return sorted(choose_without_replacement(stream_key(seed, TAG_OUTLIER, layer, kv), Hkv * d, n))


def tiny_outlier_channels(seed: int, d: int) -> list[int]:
    return sorted(choose_without_replacement(stream_key(seed, TAG_TINY), d, 4))


def kv_tokens(seed: int, layer: int, B: int, pos0: int, n: int, Hkv: int, d: int,
              outliers: str = "heavy", device="cpu"):
    """K, V of positions [pos0, pos0 + n) as bf16 tensors [B][n][Hkv][d].

    Element (b, p, h, c) is draw number ((b * 2^40) + p) * Hkv * d + h * d + c of
    the layer's K (or V) stream, so it does not depend on how the context is
    split between prefill and appends.
    """
    out = []
    per_tok = Hkv * d
    for kv, tag in ((0, TAG_K), (1, TAG_V)):
        key = stream_key(seed, tag, layer)
        vals = torch.empty(B, n, per_tok, dtype=torch.float64, device=device)
        for b in range(B):
            start = ((b << 40) + pos0) * per_tok
            vals[b] = normals(key, start, n * per_tok, device).view(n, per_tok)
        if outliers == "heavy":
            pairs = outlier_pairs(seed, layer, kv, Hkv, d)
            if pairs:
                okey = stream_key(seed, tag, layer, 7)
                idx = torch.tensor(pairs, dtype=torch.int64, device=device)
                for b in range(B):
                    start = ((b << 40) + pos0) * len(pairs)
                    t = student_t3(okey, start, n * len(pairs), device).view(n, len(pairs))
                    vals[b][:, idx] = t
        elif outliers == "tiny":
            if kv == 0:
                ch = tiny_outlier_channels(seed, d)
                v4 = vals.view(B, n, Hkv, d)
                v4[..., ch] *= 8.0
        elif outliers != "none":
            raise ValueError(outliers)
        out.append(to_bf16(vals.view(B, n, Hkv, d)))
    return out[0], out[1]


def queries(seed: int, layer: int, step: int, B: int, Hq: int, d: int, device="cpu") -> torch.Tensor:
    """A fresh N(0, 1) bf16 query [B][Hq][d] for every (layer, step)."""
    key = stream_key(seed, TAG_Q, layer, step)
    return to_bf16(normals(key, 0, B * Hq * d, device).view(B, Hq, d))


def zipf_scores(seed: int, layer: int, B: int, W: int, device="cpu") -> torch.Tensor:
    """Initial cumulative scores [B][W] (float32), Zipf(1.1) over a seeded rank permutation."""
    h = sum(r ** -1.1 for r in range(1, W + 1))
    rows = []
    for b in range(B):
        perm = permutation(stream_key(seed, TAG_SCORE, layer, b), W)
        ranks = torch.tensor(perm, dtype=torch.float64) + 1.0
        rows.append((ranks ** -1.1) / h)
    return torch.stack(rows).to(torch.float32).to(device)


def drift_factors(seed: int, layer: int, event: int, B: int, W: int, device="cpu") -> torch.Tensor:
    """Multiplicative score drift exp(0.5 z) [B][W] (float32) for one routing event."""
    key = stream_key(seed, TAG_DRIFT, layer, event)
    z = normals(key, 0, B * W, device).view(B, W)
    return torch.exp(0.5 * z).to(torch.float32)


def drawn_tiers(seed: int, layer: int, B: int, W: int, n_fp: int, n_q: int) -> torch.Tensor:
    """Tiers [B][W] uint8 from a seeded Fisher-Yates permutation of the windows."""
    t = torch.full((B, W), TIER_E, dtype=torch.uint8)
    for b in range(B):
        perm = permutation(stream_key(seed, TAG_TIER, layer, b), W)
        for i, w in enumerate(perm):
            t[b, w] = TIER_FP if i < n_fp else (TIER_Q if i < n_fp + n_q else TIER_E)
    return t


# Workloads with the shapes of the pages' models (Llama-3.1-8B, Qwen2.5-7B,
# Mistral-7B) and budgets (5-20 % of the full cache).
WORKLOADS = {
    "tiny": dict(B=1, layers=1, Hq=8, Hkv=2, d=128, L=2048, w=32, beta=1.0, rho=0.5,
                 outliers="tiny", tiers=(16, 32, 16)),
    "llama8b_b1_32k_20pct": dict(B=1, layers=32, Hq=32, Hkv=8, d=128, L=32768, w=64,
                                 beta=0.20, rho=0.5, outliers="heavy"),
    "llama8b_b8_32k_5pct": dict(B=8, layers=32, Hq=32, Hkv=8, d=128, L=32768, w=64,
                                beta=0.05, rho=0.5, outliers="heavy", route_every=64),
    "qwen7b_b16_16k_10pct": dict(B=16, layers=28, Hq=28, Hkv=4, d=128, L=16384, w=64,
                                 beta=0.10, rho=0.5, outliers="heavy", steps=256, route_every=64),
}


def mistral_sweep():
    """The Mistral-7B-shaped sweep points (batch 4): context x window x budget."""
    for L in (8192, 32768, 131072):
        for w in (32, 64, 128):
            for beta in (0.05, 0.10, 0.20):
                yield dict(B=4, layers=32, Hq=32, Hkv=8, d=128, L=L, w=w, beta=beta,
                           rho=0.5, outliers="heavy")
