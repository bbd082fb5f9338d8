"""Routing diagnostics of the CUDA path against the oracle, through the C ABI.

Tier-move counts (FP / INT2 tier sizes before and after, kept, promoted,
demoted, evicted) are integers and must match the oracle's bit for bit after
every kind of move. Future missed mass is fp32 on the GPU against the fp64
oracle, within the attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_decode, close, make_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def check_counts(cache, layer, ref, what):
    got = cache.tier_move_counts(layer).numpy()
    assert np.array_equal(got, ref.last_counts.astype(np.int32)), (what, got, ref.last_counts)
    return got


def test_counts_are_zero_before_the_first_move():
    cache = binding.TieredCache(2, 2, 8, 2, 32, 512)
    k, v = synth.kv_tokens(20, 0, 2, 0, 100, 2, 128, "heavy", device="cuda")
    cache.append(0, k, v)
    assert not cache.tier_move_counts(0).any()
    assert not cache.tier_move_counts(1).any()


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [(2, 32, 8, 64, 4096, 0.2), (3, 28, 4, 32, 1500, 0.1),
                                                (1, 8, 2, 16, 777, 0.3)])
def test_counts_after_each_kind_of_move(B, Hq, Hkv, w, L, beta):
    W = -(-L // w)
    scores = synth.zipf_scores(21, 0, B, W)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, scores=[scores], seed=21,
                              fp_capacity=W, ledger_capacity=W)
    c = check_counts(cache, 0, ref, "prefill with scores")
    assert (c[:, 0] == W).all() and (c[:, 7] > 0).all()   # everything starts full precision; some are evicted
    # routing events on fresh scores: windows move both ways between the visible tiers
    for event in range(3):
        sc = synth.zipf_scores(22 + event, 0, B, W)
        cache.route(0, scores_override=sc.cuda())
        ref.route(scores_override=sc.numpy())
        c = check_counts(cache, 0, ref, f"route {event}")
    # explicit tiers: demote every other full-precision window, evict one INT2 window
    t = ref.tiers().copy()
    for b in range(B):
        fp = np.flatnonzero(t[b, :-1] == O.TIER_FP)
        t[b, fp[::2]] = O.TIER_Q
        q = np.flatnonzero(ref.tiers()[b] == O.TIER_Q)
        if q.size:
            t[b, q[0]] = O.TIER_E
    cache.set_tiers(0, torch.from_numpy(t).cuda())
    ref.set_tiers(t)
    check_counts(cache, 0, ref, "set tiers")
    # listed promotions and demotions
    t = ref.tiers()
    pairs_p = [[b, int(wi)] for b in range(B) for wi in np.flatnonzero(t[b] == O.TIER_Q)[:3]]
    cache.promote(0, torch.tensor(pairs_p, dtype=torch.int32).cuda())
    ref.promote(pairs_p)
    c = check_counts(cache, 0, ref, "promote")
    assert c[:, 5].sum() == len(pairs_p)
    t = ref.tiers()
    pairs_d = [[b, int(wi)] for b in range(B) for wi in np.flatnonzero(t[b, :-1] == O.TIER_FP)[:2]]
    cache.demote(0, torch.tensor(pairs_d, dtype=torch.int32).cuda())
    ref.demote(pairs_d)
    c = check_counts(cache, 0, ref, "demote")
    assert c[:, 6].sum() == len(pairs_d)
    assert cache.status() == 0, cache.last_error()


def test_counts_of_a_failed_move_stay():
    """A set_tiers that asks to bring back an evicted window stops with STATE and
    leaves the previous move's counts."""
    B, Hq, Hkv, w, L = 1, 8, 2, 32, 640
    W = L // w
    tiers = synth.drawn_tiers(23, 0, B, W, 5, 8)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, tiers=[tiers], fp_capacity=W, ledger_capacity=W, seed=23)
    before = check_counts(cache, 0, ref, "prefill with tiers")
    t = ref.tiers().copy()
    e = np.flatnonzero(t[0] == O.TIER_E)
    assert e.size
    t[0, e[0]] = O.TIER_FP
    cache.set_tiers(0, torch.from_numpy(t).cuda())
    assert binding.STATUS[cache.status()] == "STATE"
    cache.clear_status()
    assert np.array_equal(cache.tier_move_counts(0).numpy(), before)


def fmm_case(B, Hq, Hkv, w, L, beta, seed, appended=0):
    W = -(-L // w)
    scores = synth.zipf_scores(seed, 0, B, W)
    maxc = L + appended
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, scores=[scores], seed=seed, max_context=maxc)
    k, _ = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy")
    keys = [k]
    for i in range(appended):
        kn, vn = synth.kv_tokens(seed, 0, B, L + i, 1, Hkv, 128)
        cache.append(0, kn.cuda(), vn.cuda())
        ref.append(kn.float().numpy(), vn.float().numpy())
        keys.append(kn)
    k_full = torch.cat(keys, dim=1)
    q = synth.queries(seed, 0, 0, B, Hq, 128)
    got = cache.future_missed_mass(0, q.cuda(), k_full.cuda())
    torch.cuda.synchronize()
    assert cache.status() == 0, cache.last_error()
    want = O.future_missed_mass(ref, q.float().numpy(), k_full.float().numpy())
    close(got.cpu().numpy(), want, "future missed mass")
    # the measurement shares the decode scratch: decoding after it is unaffected
    check_decode(cache, 0, ref, synth.queries(seed, 0, 1, B, Hq, 128))
    return got.cpu().numpy(), want


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [(2, 8, 2, 32, 1000, 0.1), (3, 28, 4, 64, 3000, 0.05),
                                                (1, 32, 8, 16, 777, 0.2), (2, 8, 8, 64, 4096, 0.1)])
def test_future_missed_mass_matches_oracle(B, Hq, Hkv, w, L, beta):
    got, want = fmm_case(B, Hq, Hkv, w, L, beta, seed=24)
    assert (want > 0).any()


def test_future_missed_mass_full_size_llama_b1_32k_20pct():
    got, want = fmm_case(1, 32, 8, 64, 32768, 0.2, seed=0)
    assert (want > 0).all()


def test_future_missed_mass_after_appends_and_without_evictions():
    fmm_case(2, 16, 4, 32, 900, 0.15, seed=25, appended=37)
    got, want = fmm_case(1, 8, 2, 32, 500, 1.0, seed=26)   # a budget that keeps everything
    assert not want.any() and not got.any()


def test_future_missed_mass_rejects_a_wrong_length():
    cache, _ = make_pair(1, 8, 2, 32, 300, beta=0.3, scores=[synth.zipf_scores(27, 0, 1, 10)], seed=27)
    k, _ = synth.kv_tokens(27, 0, 1, 0, 299, 2, 128, "heavy", device="cuda")
    q = synth.queries(27, 0, 0, 1, 8, 128).cuda()
    with pytest.raises(binding.QevictError) as e:
        cache.future_missed_mass(0, q, k)
    assert e.value.name == "INVALID_ARG"


def test_future_missed_mass_single_window_cache():
    """max_context below one window: one window per sequence, nothing evicted."""
    B, Hq, Hkv, w, L = 8, 8, 2, 32, 20
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, tiers=[torch.zeros(B, 1, dtype=torch.uint8)], seed=28)
    k, _ = synth.kv_tokens(28, 0, B, 0, L, Hkv, 128, "heavy")
    q = synth.queries(28, 0, 0, B, Hq, 128)
    got = cache.future_missed_mass(0, q.cuda(), k.cuda())
    torch.cuda.synchronize()
    assert cache.status() == 0, cache.last_error()
    want = O.future_missed_mass(ref, q.float().numpy(), k.float().numpy())
    assert not want.any() and not got.cpu().numpy().any()
    check_decode(cache, 0, ref, q)
