"""The counting the GPU planner uses for the mixed-width allocation, restated
on the CPU and checked against oracle.rd_mixed_widths (the sorted greedy).

The planner does not sort the upgrades. It groups the candidates by chain
class (never quantised; ledger width 2, 4, 8), keeps rank order within a
class, and forms one list per (class, step) whose gains do not rise. An
upgrade is taken iff its gain is positive and the cost of every upgrade
ordered before it (gain higher; on a tie a lower step, then a higher rank),
plus its own, fits the room left by the open window. Each list is counted by
a binary search. This file states that procedure over float64 gains compared
through their orderable bit patterns, as the kernel compares them, and
requires the same widths as the greedy on random and tie-heavy inputs.
"""
import struct

import numpy as np
import pytest

import oracle as O


def _orderable(x: float) -> int:
    u = struct.unpack("<Q", struct.pack("<d", x))[0]
    return (~u & (2 ** 64 - 1)) if u >> 63 else (u | (1 << 63))


def _steps(ci, max_p):
    return 2 + (max_p >= 2) + (max_p >= 4) if ci == 0 else 2


def _width(ci, idx, max_p):
    if idx == 0:
        return 0
    if ci != 0:
        return (2 << (ci - 1)) if idx == 1 else 16
    return (2 << (idx - 1)) if idx < _steps(0, max_p) else 16


def merge_rank_widths(S, classes, L, w, Hkv, beta, max_p, d=128):
    cost = lambda b: O.width_cost(w, Hkv, d, b)
    room = O.budget_bytes(L, Hkv, d, beta) - cost(16)
    lists = [[j for j in range(len(S)) if classes[j] == c] for c in range(4)]
    types = []   # (class, step, cost, gains as orderable keys along the class list)
    for c in range(4):
        for i in range(_steps(c, max_p)):
            a, b = _width(c, i, max_p), _width(c, i + 1, max_p)
            k = (2.0 ** -a - 2.0 ** -b) / (cost(b) - cost(a))
            types.append((c, i, cost(b) - cost(a), [_orderable(k * float(S[j])) for j in lists[c]]))
    take = []
    for c, i, cc, G in types:
        taken = 0
        for q, g in enumerate(G):
            if g <= 1 << 63:          # gain <= 0
                continue
            j = lists[c][q]
            prefix = cc
            for c2, i2, cc2, G2 in types:
                lo, hi = 0, len(G2)
                while lo < hi:
                    mid = (lo + hi) // 2
                    g2 = G2[mid]
                    before = g2 > g or (g2 == g and (i2 < i or (i2 == i and lists[c2][mid] < j)))
                    lo, hi = (mid + 1, hi) if before else (lo, mid)
                prefix += lo * cc2
            taken += prefix <= room
        take.append(taken)
    first, t = {}, 0
    for c in range(4):
        first[c] = t
        t += _steps(c, max_p)
    out, pos = [], [0, 0, 0, 0]
    for j in range(len(S)):
        c = classes[j]
        q = pos[c]
        pos[c] += 1
        st = 0
        while st < _steps(c, max_p) and q < take[first[c] + st]:
            st += 1
        out.append(_width(c, st, max_p))
    return out


@pytest.mark.parametrize("kind", ["pareto", "uniform", "levels"])
def test_merge_rank_counting_is_the_sorted_greedy(kind):
    rng = np.random.default_rng({"pareto": 1, "uniform": 2, "levels": 3}[kind])
    checked = 0
    for _ in range(60):
        Hkv, w = int(rng.choice([1, 2, 8])), int(rng.choice([16, 32, 64]))
        L = int(rng.integers(200, 2000))
        W = -(-L // w)
        beta = float(rng.uniform(max(0.02, 1.3 * w / L), 0.8))
        max_p = int(rng.choice([1, 2, 4]))
        n = W - 1
        if kind == "pareto":
            S = sorted((rng.pareto(1.2, n) * rng.uniform(0.1, 10)).astype(np.float32).astype(float), reverse=True)
        elif kind == "uniform":
            S = [1.0] * n
        else:
            S = sorted(rng.choice([0.0, 0.5, 1.0, 2.0], n).astype(float), reverse=True)
        allowed = [0, 1] + ([2] if max_p >= 2 else []) + ([3] if max_p >= 4 else [])
        classes = [int(rng.choice(allowed)) if rng.random() < 0.4 else 0 for _ in range(n)]
        free = [0] + [x for x in (2, 4, 8) if x <= 2 * max_p] + [16]
        chains = [free if c == 0 else [0, 2 << (c - 1), 16] for c in classes]
        if O.budget_bytes(L, Hkv, 128, beta) < O.width_cost(w, Hkv, 128, 16):
            continue
        want = O.rd_mixed_widths(S, chains, L, w, Hkv, 128, beta)
        assert merge_rank_widths(S, classes, L, w, Hkv, beta, max_p) == want, (Hkv, w, L, beta, max_p)
        checked += 1
    assert checked > 40
