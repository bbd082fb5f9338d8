"""Pins of the oracle's K-channel half of the rate-distortion allocation
("Technische Samenvatting: RDKV", 2.1 and 2.2 Fase 1 and 3): the channel
weights against their closed form and an element-by-element loop, the group
widths against hand-worked cases and against brute force over every width
assignment on small inputs, and the route against the mixed-width route it
reduces to, plus the invariance a dropped group implies."""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_channel_weights_closed_form_for_constant_columns():
    rng = np.random.default_rng(3)
    B, n, nq, Hkv, G, d = 2, 7, 5, 2, 3, 64
    a = rng.normal(size=(B, Hkv, d))
    c = rng.normal(size=(B, Hkv, d))
    k = np.broadcast_to(a[:, None], (B, n, Hkv, d))
    q = np.broadcast_to(np.repeat(c, G, axis=1)[:, None], (B, nq, Hkv * G, d))
    want = np.abs(a) * math.sqrt(n) * np.abs(c) * math.sqrt(nq * G) / math.sqrt(d)
    assert np.allclose(O.k_channel_weights(q, k, Hkv), want, rtol=1e-12, atol=0)


def test_channel_weights_by_an_element_loop():
    rng = np.random.default_rng(4)
    B, n, nq, Hkv, G, d = 1, 4, 3, 2, 2, 32
    k = rng.normal(size=(B, n, Hkv, d))
    q = rng.normal(size=(B, nq, Hkv * G, d))
    got = O.k_channel_weights(q, k, Hkv)
    for h in range(Hkv):
        for ch in range(d):
            sq = sum(q[0, t, h * G + j, ch] ** 2 for t in range(nq) for j in range(G))
            sk = sum(k[0, t, h, ch] ** 2 for t in range(n))
            assert abs(got[0, h, ch] - math.sqrt(sq) * math.sqrt(sk) / math.sqrt(d)) < 1e-12


def _golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "k_channel_widths.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        head, wts, widths = [p.split() for p in line.split("|")]
        rows.append((int(head[0]), int(head[1]), int(head[2]), [float(x) for x in wts], [int(x) for x in widths]))
    return rows


def _weights(Hkv, group_w):
    w = np.zeros((Hkv, 128), np.float32)
    for u, W in enumerate(group_w):
        h, g = divmod(u, 4)
        w[h, g * 32:(g + 1) * 32] = np.float32(W / 32)
    return w


@pytest.mark.parametrize("row", _golden())
def test_channel_widths_hand_worked(row):
    Hkv, n_tok, budget, gw, want = row
    got = O.k_channel_widths(_weights(Hkv, gw), n_tok, budget)
    assert got.reshape(-1).tolist() == want


def _cost(widths, n_tok):
    return n_tok * sum(O.k_group_cost(b) for b in widths)


def _distortion(widths, W):
    return sum(Wg * 2.0 ** -b for Wg, b in zip(W, widths))


@pytest.mark.parametrize("seed", range(12))
def test_channel_widths_are_optimal_at_their_own_cost(seed):
    """The steps are whole and taken in falling gain per byte along convex
    chains, so no assignment that costs at most as much distorts less."""
    rng = np.random.default_rng(100 + seed)
    Hkv = 1 + seed % 2
    n_tok = int(rng.integers(1, 5))
    w = rng.exponential(size=(Hkv, 128)).astype(np.float32)
    if seed % 3 == 0:
        w[:, 96:] = 0   # a group of no weight stays at width 0
    W = [sum(float(x) for x in w[h, g * 32:(g + 1) * 32]) for h in range(Hkv) for g in range(4)]
    lo, hi = _cost([0] * 4 * Hkv, n_tok), _cost([8] * 4 * Hkv, n_tok)
    budget = int(rng.integers(lo, hi + 1))
    got = O.k_channel_widths(w, n_tok, budget).reshape(-1).tolist()
    c_got = _cost(got, n_tok)
    assert c_got <= budget
    d_got = _distortion(got, W)
    best = min(_distortion(a, W) for a in itertools.product(O.K_WIDTHS, repeat=4 * Hkv)
               if _cost(a, n_tok) <= c_got)
    assert d_got <= best * (1 + 1e-12) + 1e-15
    if seed % 3 == 0:
        assert all(got[h * 4 + 3] == 0 for h in range(Hkv))


def _layer(seed, B=1, Hq=8, Hkv=2, w=16, L=256):
    rng = np.random.default_rng(seed)
    k = O.bf16_round(rng.normal(size=(B, L, Hkv, 128)).astype(np.float32))
    v = O.bf16_round(rng.normal(size=(B, L, Hkv, 128)).astype(np.float32))
    c = O.OracleCache(B, Hq, Hkv, 128, w, beta=0.3, rho=0.5)
    c.append(k, v)
    S = rng.exponential(size=(B, c.W))
    return c, S, rng


def test_route_rd_kv_with_equal_channel_weights_is_the_int2_route():
    """Equal channel weights and widths up to 2: every quantised window's K
    budget is exactly its INT2 K, so every group takes width 2 and the route
    is route_rd_mixed's, codes, tiers and outputs alike."""
    a, S, rng = _layer(1)
    b, _, _ = _layer(1)
    wts = np.ones((a.B, a.Hkv, 128), np.float32)
    O.route_rd_kv(a, wts, scores_override=S, max_bits=2)
    O.route_rd_mixed(b, scores_override=S, max_bits=2)
    assert (a.kch == 2).all()
    assert np.array_equal(a.tiers(), b.tiers())
    for wa, wb in zip(a.win[0], b.win[0]):
        assert (wa.ledger is None) == (wb.ledger is None)
        if wa.ledger is not None:
            for x, y in zip(wa.ledger, wb.ledger):
                assert np.array_equal(x, y)
    q = O.bf16_round(rng.normal(size=(a.B, a.Hq, 128)).astype(np.float32))
    oa, ma = a.decode(q, accumulate=False)
    ob, mb = b.decode(q, accumulate=False)
    assert np.array_equal(oa, ob) and np.array_equal(ma, mb)


def test_a_dropped_k_group_takes_no_part_in_the_logits():
    """Channels of a group at width 0 are zero in every quantised window: the
    decode does not change when the queries change on those channels only
    (the open window, in full precision, is emptied of them too, so that it
    does not see them either)."""
    c, S, rng = _layer(2)
    wts = rng.exponential(size=(c.B, c.Hkv, 128)).astype(np.float32)
    wts[:, :, 64:96] = 0
    O.route_rd_kv(c, wts, scores_override=S, max_bits=8)
    assert (c.kch[:, :, 2] == 0).all()
    quantised = [wi for wi, win in enumerate(c.win[0]) if win.tier in O.BITS_OF_TIER]
    assert quantised
    for wi in quantised:
        kk, _ = c.window_kv(0, wi, 0)
        assert not kk[:, 64:96].any()
    for win in c.win[0]:
        if win.tier == O.TIER_FP:
            win.k[:, :, 64:96] = 0
    q = O.bf16_round(rng.normal(size=(c.B, c.Hq, 128)).astype(np.float32))
    q2 = q.copy()
    q2[:, :, 64:96] = O.bf16_round(rng.normal(size=q2[:, :, 64:96].shape).astype(np.float32))
    o1, m1 = c.decode(q, accumulate=False)
    o2, m2 = c.decode(q2, accumulate=False)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(m1, m2, rtol=0, atol=1e-12)


def test_route_rd_kv_budget_and_state_rules():
    c, S, rng = _layer(3)
    wts = rng.exponential(size=(c.B, c.Hkv, 128)).astype(np.float32)
    O.route_rd_kv(c, wts, scores_override=S, max_bits=8)
    # the K groups spend no more than the K halves the windows had at their widths
    bits = [O.BITS_OF_TIER[win.tier] for win in c.win[0] if win.tier in O.BITS_OF_TIER]
    n_tok = len(bits) * c.w
    k_budget = sum(O.width_cost(c.w, c.Hkv, c.d, b) // 2 for b in bits)
    assert n_tok * sum(O.k_group_cost(int(b)) for b in c.kch[0].reshape(-1)) <= k_budget
    with pytest.raises(O.StateError):
        O.route_rd_kv(c, wts, scores_override=S)
    with pytest.raises(O.StateError):
        c.route(scores_override=S)
    d, S2, _ = _layer(4)
    O.route_rd_mixed(d, scores_override=S2)
    with pytest.raises(O.StateError):
        O.route_rd_kv(d, wts, scores_override=S2)
