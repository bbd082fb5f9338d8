"""Rate-distortion routing on the GPU against oracle.route_rd.

The tier counts come from the allocation (float64 per-byte gains on both
sides), the windows from the score rank: tiers, slot tables, stored bf16,
ledger entries and tier-move counts bit for bit; the decode after each event
within the attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_decode, check_state, close, make_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [(1, 32, 8, 64, 4096, 0.2), (2, 28, 4, 32, 3000, 0.1),
                                                (3, 8, 2, 16, 777, 0.3), (2, 8, 2, 64, 8192, 0.05)])
def test_rd_route_matches_oracle(B, Hq, Hkv, w, L, beta):
    W = -(-L // w)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, seed=60, tiers=[torch.zeros(B, W, dtype=torch.uint8)],
                              fp_capacity=W, ledger_capacity=W)
    scores = synth.zipf_scores(60, 0, B, W)
    cache.route_rd(0, scores_override=scores.cuda())
    O.route_rd(ref, scores_override=scores.numpy())
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    # like the score route, the override becomes the stored scores (checked before the decode adds to them)
    assert np.array_equal(cache.scores(0).cpu().numpy(), scores.numpy())
    check_decode(cache, 0, ref, synth.queries(60, 0, 0, B, Hq, 128))


def test_rd_route_uniform_scores_hand_count():
    """All weights equal at the 32K Llama-8B layer, 20 %: every window to INT2
    first, then six upgrades to full precision fit (tests/golden/rd_counts.txt)."""
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 64, 32768, 0.2
    W = L // w
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, seed=0, tiers=[torch.zeros(B, W, dtype=torch.uint8)],
                              fp_capacity=W, ledger_capacity=W)
    ones = torch.ones(B, W)
    cache.route_rd(0, scores_override=ones.cuda())
    O.route_rd(ref, scores_override=ones.numpy())
    t = cache.tables(0)[0].numpy()
    assert ((t == 0).sum(), (t == 1).sum(), (t == 2).sum()) == (7, 505, 0)
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(0, 0, 0, B, Hq, 128))


def test_rd_route_full_size_zipf():
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 64, 32768, 0.2
    W = L // w
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, seed=0, tiers=[torch.zeros(B, W, dtype=torch.uint8)],
                              fp_capacity=W, ledger_capacity=W)
    scores = synth.zipf_scores(0, 0, B, W)
    cache.route_rd(0, scores_override=scores.cuda())
    O.route_rd(ref, scores_override=scores.numpy())
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(0, 0, 0, B, Hq, 128))


def test_rd_routes_between_decode_steps_teacher_forced():
    B, Hq, Hkv, w, L0, beta = 2, 16, 4, 32, 1024, 0.2
    steps, every = 96, 32
    W0 = L0 // w
    Wmax = -(-(L0 + steps) // w)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L0, beta=beta, seed=61, max_context=L0 + steps,
                              scores=[synth.zipf_scores(61, 0, B, W0)], fp_capacity=Wmax, ledger_capacity=Wmax)
    for step in range(steps):
        kn, vn = synth.kv_tokens(61, 0, B, L0 + step, 1, Hkv, 128)
        cache.append(0, kn.cuda(), vn.cuda())
        ref.append(kn.float().numpy(), vn.float().numpy())
        check_decode(cache, 0, ref, synth.queries(61, 0, step, B, Hq, 128))
        if step % every == every - 1:
            gs = cache.scores(0).cpu().numpy()
            close(gs, np.stack(ref.S), "cumulative scores")
            drift = synth.drift_factors(61, 0, step, B, cache.num_windows(0))
            cache.route_rd(0, score_mult=drift.cuda())
            O.route_rd(ref, scores_override=np.asarray(cache.scores(0).cpu().numpy(), np.float64))
            check_state(cache, 0, ref)
            assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    assert cache.status() == 0, cache.last_error()
