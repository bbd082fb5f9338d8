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


# ---- the 4- and 8-bit widths and the allocation over {0, 2, 4, 8, 16}

def _mixed_widths_variant(k_of, stop):
    """oracle.rd_mixed_widths with the per-byte gain factor and the stop rule
    replaced (for planting mistakes)."""
    def fn(S_ranked, chains, L, w, Hkv, d, beta):
        c_fp = O.width_cost(w, Hkv, d, 16)
        Bt = O.budget_bytes(L, Hkv, d, beta)
        ups = []
        for r, (s, ch) in enumerate(zip(S_ranked, chains)):
            for i in range(len(ch) - 1):
                a, b = ch[i], ch[i + 1]
                cost = O.width_cost(w, Hkv, d, b) - O.width_cost(w, Hkv, d, a)
                ups.append((k_of(a, b, cost) * float(s), i, r, cost))
        ups.sort(key=lambda u: (-u[0], u[1], u[2]))
        used, steps = c_fp, [0] * len(chains)
        for gain, i, r, cost in ups:
            if gain <= 0.0:
                break
            if used + cost > Bt:
                if stop:
                    break
                continue
            if steps[r] != i:
                continue
            used += cost
            steps[r] += 1
        return [ch[st] for ch, st in zip(chains, steps)]
    return fn


def _patch_both(monkeypatch, name, fn):
    monkeypatch.setattr(QO, name, fn)
    monkeypatch.setattr(O, name, fn)


def _quantiser_variant(levels_of):
    """oracle.quantize_groups (finite inputs) with the level count replaced."""
    def fn(x, bits=2):
        x = np.asarray(x, np.float32)
        levels = levels_of(bits)
        mn, mx = x.min(axis=-1), x.max(axis=-1)
        mn16 = QO.half_round(mn)
        s16 = QO.half_round(((mx - mn).astype(np.float32) / np.float32(levels)).astype(np.float32))
        s, m = s16.astype(np.float32), mn16.astype(np.float32)
        den = np.where(s == 0, np.float32(1), s)
        q = np.rint(((x - m[..., None]).astype(np.float32) / den[..., None]).astype(np.float32))
        codes = np.clip(np.where(s[..., None] == 0, 0, q), 0, levels).astype(np.uint8)
        return codes, s16, mn16, np.zeros(mn.shape, bool)
    return fn


def test_mutant_harnesses_pass_without_a_plant(monkeypatch):
    """Control: the re-implementations the plants below start from pass the pins."""
    _patch_both(monkeypatch, "quantize_groups", _quantiser_variant(lambda b: (1 << b) - 1))
    P.test_wide_quantiser_exact_grid_and_nearest_level(4)
    P.test_wide_quantiser_exact_grid_and_nearest_level(8)
    _patch_both(monkeypatch, "rd_mixed_widths",
                _mixed_widths_variant(lambda a, b, c: (2.0 ** -a - 2.0 ** -b) / c, True))
    P.test_rd_mixed_is_a_lagrangian_solution()
    P.test_rd_mixed_hand_derived()
    P.test_rd_mixed_route_keeps_ledger_widths_and_is_lagrangian()


def test_wide_quantiser_with_2_to_the_b_levels_is_caught(monkeypatch):
    # plant: 2^b levels instead of 2^b - 1
    _patch_both(monkeypatch, "quantize_groups", _quantiser_variant(lambda b: 1 << b))
    assert _fails(P.test_wide_quantiser_exact_grid_and_nearest_level, 4)
    assert _fails(P.test_wide_quantiser_exact_grid_and_nearest_level, 8)


def test_mixed_gain_without_the_upper_width_term_is_caught(monkeypatch):
    # plant: the distortion removed by a -> b taken as 2^-a (the 2^-b left in is dropped)
    _patch_both(monkeypatch, "rd_mixed_widths", _mixed_widths_variant(lambda a, b, c: 2.0 ** -a / c, True))
    assert _fails(P.test_rd_mixed_is_a_lagrangian_solution)


def test_mixed_greedy_that_skips_instead_of_stopping_is_caught(monkeypatch):
    # plant: an upgrade that does not fit is skipped and later, cheaper ones still taken
    _patch_both(monkeypatch, "rd_mixed_widths",
                _mixed_widths_variant(lambda a, b, c: (2.0 ** -a - 2.0 ** -b) / c, False))
    assert _fails(P.test_rd_mixed_is_a_lagrangian_solution)


def test_mixed_route_ignoring_ledger_widths_is_caught(monkeypatch):
    orig = QO.rd_mixed_widths

    def free_chains(S_ranked, chains, L, w, Hkv, d, beta):
        # plant: every window gets the chain of a window never quantised
        return orig(S_ranked, [[0, 2, 4, 8, 16]] * len(chains), L, w, Hkv, d, beta)
    _patch_both(monkeypatch, "rd_mixed_widths", free_chains)
    assert _fails(P.test_rd_mixed_route_keeps_ledger_widths_and_is_lagrangian)


def test_width_cost_without_meta_is_caught(monkeypatch):
    # plant: the fp16 scale and minimum of each group left out of a quantised window's bytes
    bad = lambda w, Hkv, d, bits: 0 if bits == 0 else (w * Hkv * d * 4 if bits == 16 else w * Hkv * 2 * (d * bits // 8))
    _patch_both(monkeypatch, "width_cost", bad)
    assert _fails(P.test_rd_mixed_hand_derived)
