"""The rate-distortion route over all widths (0, 2, 4, 8, 16 bits) on the GPU
against oracle.route_rd_mixed.

The widths come from the Lagrangian greedy over every window's chain of
upgrades (float64 gains per byte on both sides); tiers, slot tables, stored
bf16, ledger entries of every width and tier-move counts must match bit for
bit, the decode after each event within the attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_decode, check_state, close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def make_wide(B, Hq, Hkv, w, L, bits, beta, seed, tiers=None, scores=None, max_context=None):
    """Both caches prefilled with the same tokens (all full precision unless tiers are given)."""
    maxc = max_context or L
    Wmax = -(-maxc // w)
    W = -(-L // w)
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, maxc, budget_frac=beta, max_ledger_bits=bits,
                                fp_capacity=Wmax, ledger_capacity=Wmax)
    ref = O.OracleCache(B, Hq, Hkv, 128, w, beta=beta)
    k, v = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy")
    t = np.zeros((B, W), np.uint8) if tiers is None else tiers
    cache.prefill(0, k.cuda(), v.cuda(), tiers=torch.from_numpy(t).cuda())
    ref.prefill(k.float().numpy(), v.float().numpy(), tiers=t)
    assert cache.status() == 0, cache.last_error()
    return cache, ref


def route_both(cache, ref, scores, bits):
    cache.route_rd_mixed(0, scores_override=scores.cuda())
    # max_ledger_bits 0 means INT2 only, as 2 does
    O.route_rd_mixed(ref, scores_override=scores.numpy(), max_bits=max(bits, 2))
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta,bits", [(1, 32, 8, 64, 4096, 0.2, 8), (2, 28, 4, 32, 3000, 0.1, 8),
                                                     (3, 8, 2, 16, 777, 0.3, 4), (2, 8, 2, 64, 8192, 0.05, 8),
                                                     (2, 16, 4, 32, 2048, 0.15, 0)])
def test_rd_mixed_route_matches_oracle(B, Hq, Hkv, w, L, beta, bits):
    W = -(-L // w)
    cache, ref = make_wide(B, Hq, Hkv, w, L, bits, beta, seed=70)
    scores = synth.zipf_scores(70, 0, B, W)
    route_both(cache, ref, scores, bits)
    assert np.array_equal(cache.scores(0).cpu().numpy(), scores.numpy())
    t = ref.tiers()
    if bits >= 4:
        assert (t == O.TIER_Q4).any(), "the allocation should use INT4 here"
    check_decode(cache, 0, ref, synth.queries(70, 0, 0, B, Hq, 128))


def test_rd_mixed_uniform_scores_hand_count():
    """All weights equal at the 32K Llama-8B layer, 20 %: 1 bf16, 44 INT4 and 467
    INT2 windows (tests/golden/rd_counts.txt, the MIXED line)."""
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 64, 32768, 0.2
    W = L // w
    cache, ref = make_wide(B, Hq, Hkv, w, L, 8, beta, seed=0)
    route_both(cache, ref, torch.ones(B, W), 8)
    t = cache.tables(0)[0].numpy()
    counts = [(t == x).sum() for x in (O.TIER_FP, O.TIER_Q8, O.TIER_Q4, O.TIER_Q, O.TIER_E)]
    assert counts == [1, 0, 44, 467, 0]
    check_decode(cache, 0, ref, synth.queries(0, 0, 0, B, Hq, 128))


def test_rd_mixed_full_size_zipf_llama_b1_32k_20pct():
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 64, 32768, 0.2
    W = L // w
    cache, ref = make_wide(B, Hq, Hkv, w, L, 8, beta, seed=0)
    route_both(cache, ref, synth.zipf_scores(0, 0, B, W), 8)
    t = ref.tiers()
    assert all((t == x).any() for x in (O.TIER_FP, O.TIER_Q4, O.TIER_Q))
    check_decode(cache, 0, ref, synth.queries(0, 0, 0, B, Hq, 128))


def test_rd_mixed_keeps_ledger_widths():
    """Windows promoted from INT2, INT4 and INT8 keep their ledger: their only
    options are evicted, that width, or full precision."""
    B, Hq, Hkv, w, L, beta = 2, 8, 2, 32, 1280, 0.3
    W = L // w
    rng = np.random.default_rng(71)
    t0 = rng.choice([O.TIER_FP, O.TIER_Q, O.TIER_Q4, O.TIER_Q8], size=(B, W)).astype(np.uint8)
    t0[:, -1] = O.TIER_FP
    cache, ref = make_wide(B, Hq, Hkv, w, L, 8, beta, seed=71, tiers=t0)
    t1 = np.where(t0 == O.TIER_E, O.TIER_E, O.TIER_FP).astype(np.uint8)   # promote all: the ledgers stay
    cache.set_tiers(0, torch.from_numpy(t1).cuda())
    ref.set_tiers(t1)
    check_state(cache, 0, ref)
    route_both(cache, ref, synth.zipf_scores(71, 0, B, W), 8)
    t2 = ref.tiers()
    width = {O.TIER_Q: 2, O.TIER_Q4: 4, O.TIER_Q8: 8}
    for b in range(B):
        for wi in range(W - 1):
            if t0[b, wi] in width and t2[b, wi] in width:
                assert width[t2[b, wi]] == width[t0[b, wi]], (b, wi)
    assert cache.stats()["ledger_reuses"] == ref.stats["ledger_reuses"] > 0
    check_decode(cache, 0, ref, synth.queries(71, 0, 0, B, Hq, 128))


def test_rd_mixed_on_an_int2_cache_is_route_rd():
    B, Hq, Hkv, w, L, beta = 2, 16, 4, 32, 4096, 0.1
    W = L // w
    scores = synth.zipf_scores(72, 0, B, W).cuda()
    k, v = synth.kv_tokens(72, 0, B, 0, L, Hkv, 128, "heavy", device="cuda")
    tables = []
    for mixed in (False, True):
        c = binding.TieredCache(B, 1, Hq, Hkv, w, L, budget_frac=beta, fp_capacity=W, ledger_capacity=W)
        c.prefill(0, k, v, tiers=torch.zeros(B, W, dtype=torch.uint8).cuda())
        (c.route_rd_mixed if mixed else c.route_rd)(0, scores_override=scores)
        assert c.status() == 0, c.last_error()
        tables.append([x.clone() for x in c.tables(0)])
    for x, y in zip(*tables):
        assert torch.equal(x, y)


def test_rd_mixed_max_windows():
    """4096 windows of one sequence (the planner's maximum), widths up to INT8."""
    B, Hq, Hkv, w, L, beta = 1, 8, 1, 16, 65536, 0.15
    W = L // w
    cache, ref = make_wide(B, Hq, Hkv, w, L, 8, beta, seed=73)
    route_both(cache, ref, synth.zipf_scores(73, 0, B, W), 8)
    check_decode(cache, 0, ref, synth.queries(73, 0, 0, B, Hq, 128))


def test_rd_mixed_routes_between_fused_steps_teacher_forced():
    B, Hq, Hkv, w, L0, beta = 2, 16, 4, 32, 1024, 0.2
    steps, every = 96, 32
    W0 = L0 // w
    cache, ref = make_wide(B, Hq, Hkv, w, L0, 8, beta, seed=74, max_context=L0 + steps)
    route_both(cache, ref, synth.zipf_scores(74, 0, B, W0), 8)
    for step in range(steps):
        kn, vn = synth.kv_tokens(74, 0, B, L0 + step, 1, Hkv, 128)
        q = synth.queries(74, 0, step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].cuda(), vn[:, 0].cuda())
        torch.cuda.synchronize()
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        close(out.cpu().numpy(), ro, f"output, step {step}")
        close(mass.cpu().numpy(), rm, f"mass, step {step}")
        if step % every == every - 1:
            close(cache.scores(0).cpu().numpy(), np.stack(ref.S), "cumulative scores")
            drift = synth.drift_factors(74, 0, step, B, cache.num_windows(0))
            cache.route_rd_mixed(0, score_mult=drift.cuda())
            O.route_rd_mixed(ref, scores_override=np.asarray(cache.scores(0).cpu().numpy(), np.float64), max_bits=8)
            check_state(cache, 0, ref)
            assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    assert cache.status() == 0, cache.last_error()
    s = cache.stats()
    for key in ("demotions", "promotions", "evictions", "ledger_writes", "ledger_reuses"):
        assert s[key] == ref.stats[key], key


def test_rd_mixed_per_head_cache():
    B, Hq, Hkv, w, L, beta = 2, 16, 4, 32, 2048, 0.15
    W = L // w
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, L, budget_frac=beta, per_head=True, max_ledger_bits=4,
                                fp_capacity=W, ledger_capacity=W)
    ref = O.per_head_cache(B, Hq, Hkv, 128, w, beta=beta)
    k, v = synth.kv_tokens(75, 0, B, 0, L, Hkv, 128, "heavy")
    zeros = np.zeros((B * Hkv, W), np.uint8)
    cache.prefill(0, k.cuda(), v.cuda(), tiers=torch.from_numpy(zeros).cuda())
    ref.prefill(O.to_units(k.float().numpy()), O.to_units(v.float().numpy()), tiers=zeros)
    route_both(cache, ref, synth.zipf_scores(75, 0, B * Hkv, W), 4)
    q = synth.queries(75, 0, 0, B, Hq, 128)
    out, mass = cache.decode(0, q.cuda(), accumulate=False)
    torch.cuda.synchronize()
    ro, rm = ref.decode(O.queries_to_units(q.float().numpy(), Hkv), accumulate=False)
    close(out.cpu().numpy(), ro.reshape(B, Hq, 128), "attention output")
    close(mass.cpu().numpy(), rm.reshape(B, Hq, -1), "window mass")


def test_rd_mixed_errors_leave_the_tables():
    """A non-finite score among the candidates sets DEVICE and moves nothing; a
    budget that cannot hold the open window is BUDGET on the host."""
    B, Hq, Hkv, w, L = 1, 8, 2, 32, 256
    W = L // w
    cache, ref = make_wide(B, Hq, Hkv, w, L, 8, 0.5, seed=76)
    before = [x.clone() for x in cache.tables(0)]
    bad = torch.full((B, W), 0.1)
    bad[0, 2] = float("inf")
    cache.route_rd_mixed(0, scores_override=bad.cuda())
    assert binding.STATUS[cache.status()] == "DEVICE"
    cache.clear_status()
    for x, y in zip(before, cache.tables(0)):
        assert torch.equal(x, y)
    small = binding.TieredCache(1, 1, 8, 2, 32, 64, budget_frac=0.05, max_ledger_bits=8)
    small.append(0, *[x.cuda() for x in synth.kv_tokens(0, 0, 1, 0, 64, 2, 128)])
    with pytest.raises(binding.QevictError) as ei:
        small.route_rd_mixed(0)
    assert ei.value.name == "BUDGET"


@pytest.mark.parametrize("w,bits", [(128, 8), (128, 4), (16, 8)])
def test_rd_mixed_window_sizes(w, bits):
    B, Hq, Hkv, L, beta = 2, 16, 4, 4096 + 40, 0.12
    W = -(-L // w)
    cache, ref = make_wide(B, Hq, Hkv, w, L, bits, beta, seed=77 + w)
    route_both(cache, ref, synth.zipf_scores(77, w, B, W), bits)
    check_decode(cache, 0, ref, synth.queries(77, 0, 0, B, Hq, 128))


def test_rd_mixed_second_event_moves_between_widths():
    """Two events on different scores: windows quantised by the first keep their
    width, are promoted back to bf16 or evicted by the second; the ledger is
    reused, never rewritten."""
    B, Hq, Hkv, w, L, beta = 2, 16, 4, 32, 3072, 0.15
    W = L // w
    cache, ref = make_wide(B, Hq, Hkv, w, L, 8, beta, seed=78)
    route_both(cache, ref, synth.zipf_scores(78, 0, B, W), 8)
    first = ref.tiers().copy()
    route_both(cache, ref, synth.zipf_scores(79, 0, B, W), 8)
    second = ref.tiers()
    width = {O.TIER_Q: 2, O.TIER_Q4: 4, O.TIER_Q8: 8}
    moved = 0
    for b in range(B):
        for wi in range(W):
            if first[b, wi] in width and second[b, wi] in width:
                assert width[first[b, wi]] == width[second[b, wi]]
            moved += first[b, wi] != second[b, wi]
    assert moved > 0
    assert np.all(cache.tables(0)[3].numpy() <= 1), "a ledger entry was written twice"
    check_decode(cache, 0, ref, synth.queries(78, 0, 0, B, Hq, 128))


@pytest.mark.parametrize("mixed", [False, True])
def test_rate_distortion_routes_on_an_all_evicted_layer_move_nothing(mixed):
    """Every window evicted, the last one full: there is no candidate, so both
    rate-distortion routes leave every table as it is and count no move."""
    B, Hq, Hkv, w, L = 2, 8, 2, 16, 96
    W = L // w
    bits = 8 if mixed else 0     # the INT2 rate-distortion route wants an INT2-only cache
    cache, ref = make_wide(B, Hq, Hkv, w, L, bits, 0.5, seed=23, tiers=np.full((B, W), O.TIER_E, np.uint8))
    scores = synth.zipf_scores(23, 0, B, W)
    if mixed:
        route_both(cache, ref, scores, bits)
    else:
        cache.route_rd(0, scores_override=scores.cuda())
        O.route_rd(ref, scores_override=scores.numpy())
        assert cache.status() == 0, cache.last_error()
        check_state(cache, 0, ref)
    assert np.all(cache.tables(0)[0].numpy() == O.TIER_E)
    assert not cache.tier_move_counts(0).numpy().any()
    assert not ref.last_counts.any()
