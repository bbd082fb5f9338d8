"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

This is how the pins in test_oracle_pins.py are shown to be sensitive: a
dropped term, a wrong rounding, a flipped tie rule or a wrong softmax
denominator must make at least one of them fail.
"""
import math

import numpy as np
import oracle as O
from oracle import qevict_oracle as QO
import test_oracle_pins as P


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, Exception):
        return True
    return False


def test_dropping_fp16_rounding_of_min_is_caught(monkeypatch):
    orig = QO.half_round

    def no_round_min(x):
        # plant: skip rounding (keeps float32) for the minimum only is hard to
        # isolate, so round through bf16 instead of fp16 for everything
        return orig(O.bf16_round(np.asarray(x, np.float32)))

    monkeypatch.setattr(QO, "half_round", no_round_min)
    groups = P._parse_golden_groups()
    assert any(_fails(P.test_quantizer_hand_derived_groups, *g) for g in groups) or \
        _fails(P.test_half_round_matches_torch_conversion)


def test_round_half_away_instead_of_even_is_caught(monkeypatch):
    monkeypatch.setattr(QO.np, "rint", lambda x: np.floor(np.asarray(x) + 0.5))
    groups = P._parse_golden_groups()
    assert any(_fails(P.test_quantizer_hand_derived_groups, *g) for g in groups)


def test_missing_score_scale_is_caught(monkeypatch):
    def bad(q, keys, values):
        s = np.asarray(keys, np.float64) @ np.asarray(q, np.float64)   # no 1/sqrt(d)
        s = s - s.max()
        e = np.exp(s)
        p = e / e.sum()
        return p @ np.asarray(values, np.float64), p
    monkeypatch.setattr(QO, "softmax_attention", bad)
    assert _fails(P.test_all_full_precision_equals_dense_sdpa)


def test_evicted_tokens_in_denominator_is_caught(monkeypatch):
    orig = QO.OracleCache.window_kv

    def keep_evicted(self, b, wi, kvh):
        win = self.win[b][wi]
        if win.tier == O.TIER_E:
            # plant: an evicted window still contributes zero keys to the softmax
            n = self.w
            return np.zeros((n, self.d)), np.zeros((n, self.d))
        return orig(self, b, wi, kvh)
    monkeypatch.setattr(QO.OracleCache, "window_kv", keep_evicted)
    # _evict drops the data, so keep it around for the planted variant
    monkeypatch.setattr(QO.OracleCache, "_evict", lambda self, b, wi: setattr(self.win[b][wi], "tier", O.TIER_E))
    assert _fails(P.test_masses_evicted_zero_and_single_window)


def test_tie_break_to_higher_index_is_caught(monkeypatch):
    def bad_route(S, tiers, L, w, Hkv, d, beta, rho):
        W = -(-L // w)
        tiers = np.asarray(tiers, np.uint8)
        cand = [i for i in range(W) if tiers[i] != O.TIER_E]
        if not cand:
            return tiers.copy()
        n_fp, n_q = O.route_counts(len(cand), L, w, Hkv, d, beta, rho)
        order = sorted(cand, key=lambda i: (i != W - 1, -float(S[i]), -i))   # plant
        new = tiers.copy()
        for r, i in enumerate(order):
            new[i] = O.TIER_FP if r < n_fp else (O.TIER_Q if r < n_fp + n_q else O.TIER_E)
        return new
    monkeypatch.setattr(O, "route_tiers", bad_route)
    assert any(_fails(P.test_route_matches_brute_force, s) for s in range(40))


def test_budget_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(QO, "fp_budget_windows",
                        lambda Bt, c_fp, rho: int(math.ceil((rho * Bt) / c_fp)))
    rows = P._golden_counts()
    assert any(_fails(P.test_route_counts_hand_derived, r) for r in rows)


def test_promote_without_bf16_rounding_is_caught(monkeypatch):
    bad = lambda c, s, m: QO.dequant_exact(c, s, m).astype(np.float32)   # plant: no bf16 step
    monkeypatch.setattr(QO, "dequant_promote", bad)
    monkeypatch.setattr(O, "dequant_promote", bad)
    assert _fails(P.test_promote_dequant_single_rounding)
