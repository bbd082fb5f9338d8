"""Per-KV-head tiers: the CUDA path against the oracle's per-head cache.

With per-head tiers every (sequence, KV head) pair is a unit with its own
windows, scores, tiers and budget. The oracle builds the same units from the
same seeded tokens (oracle.per_head_cache, oracle.to_units); tables, stored
bf16 and INT2 ledger entries must match bit for bit, attention outputs,
masses and scores within the attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_state, close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def make_ph(B, Hq, Hkv, w, L, beta=1.0, seed=0, scores=None, tiers=None, max_context=None, **kw):
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, max_context or L, budget_frac=beta, per_head=True, **kw)
    ref = O.per_head_cache(B, Hq, Hkv, 128, w, beta=beta)
    k, v = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy")
    cache.prefill(0, k.cuda(), v.cuda(), scores=None if scores is None else scores.cuda(),
                  tiers=None if tiers is None else tiers.cuda())
    ref.prefill(O.to_units(k.float().numpy()), O.to_units(v.float().numpy()),
                scores=None if scores is None else scores.numpy(), tiers=None if tiers is None else tiers.numpy())
    return cache, ref, k


def check_decode_ph(cache, ref, q, accumulate=True):
    B, Hq = q.shape[0], q.shape[1]
    out, mass = cache.decode(0, q.cuda(), accumulate=accumulate)
    torch.cuda.synchronize()
    ro, rm = ref.decode(O.queries_to_units(q.float().numpy(), cache.Hkv), accumulate=accumulate)
    close(out.cpu().numpy(), ro.reshape(B, Hq, 128), "attention output")
    close(mass.cpu().numpy(), rm.reshape(B, Hq, -1), "window mass")
    assert cache.status() == 0, cache.last_error()
    return out


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [(1, 32, 8, 64, 4096, 0.2), (2, 28, 4, 64, 3000, 0.1),
                                                (3, 8, 2, 16, 777, 0.3), (2, 8, 8, 32, 1000, 0.05)])
def test_per_head_routing_quantises_and_attends(B, Hq, Hkv, w, L, beta):
    W = -(-L // w)
    scores = synth.zipf_scores(30, 0, B * Hkv, W)
    cache, ref, _ = make_ph(B, Hq, Hkv, w, L, beta=beta, seed=30, scores=scores)
    t = ref.tiers()
    assert (t == O.TIER_Q).any() and (t == O.TIER_E).any()
    # heads of one sequence keep different windows
    assert any(not np.array_equal(t[b * Hkv], t[b * Hkv + 1]) for b in range(B))
    check_state(cache, 0, ref)
    for step in range(2):
        check_decode_ph(cache, ref, synth.queries(30, 0, step, B, Hq, 128))
    close(cache.scores(0).cpu().numpy(), ref.scores(), "cumulative scores per unit")
    s = cache.stats()
    for key in ("demotions", "promotions", "evictions", "ledger_writes", "ledger_reuses"):
        assert s[key] == ref.stats[key], key


def test_per_head_equal_scores_match_the_shared_cache():
    """Every head ranked on its sequence's scores: the per-head cache keeps the
    shared cache's windows and gives its outputs (both on the GPU)."""
    B, Hq, Hkv, w, L, beta = 2, 32, 8, 64, 4096, 0.25
    W = L // w
    scores = synth.zipf_scores(31, 0, B, W)
    k, v = synth.kv_tokens(31, 0, B, 0, L, Hkv, 128, "heavy", device="cuda")
    shared = binding.TieredCache(B, 1, Hq, Hkv, w, L, budget_frac=beta)
    shared.prefill(0, k, v, scores=scores.cuda())
    ph = binding.TieredCache(B, 1, Hq, Hkv, w, L, budget_frac=beta, per_head=True)
    ph.prefill(0, k, v, scores=scores.repeat_interleave(Hkv, dim=0).cuda())
    assert torch.equal(ph.tables(0)[0], shared.tables(0)[0].repeat_interleave(Hkv, dim=0))
    q = synth.queries(31, 0, 0, B, Hq, 128).cuda()
    o1, m1 = shared.decode(0, q, accumulate=False)
    o2, m2 = ph.decode(0, q, accumulate=False)
    torch.cuda.synchronize()
    close(o2.cpu().numpy(), o1.cpu().numpy(), "output, per-head vs shared", max_abs=1e-5, rel_l2=1e-5)
    close(m2.cpu().numpy(), m1.cpu().numpy(), "mass, per-head vs shared", max_abs=1e-5, rel_l2=1e-5)


def test_per_head_multistep_fused_steps_and_routes_teacher_forced():
    """Fused decode steps (append + attend + score) and routing events with
    drift; at each event the oracle routes on the GPU's scores."""
    B, Hq, Hkv, w, L0, beta = 2, 16, 4, 32, 1024, 0.25
    steps, every = 96, 32
    W0 = L0 // w
    scores = synth.zipf_scores(32, 0, B * Hkv, W0)
    cache, ref, _ = make_ph(B, Hq, Hkv, w, L0, beta=beta, seed=32, scores=scores, max_context=L0 + steps)
    check_state(cache, 0, ref)
    for step in range(steps):
        kn, vn = synth.kv_tokens(32, 0, B, L0 + step, 1, Hkv, 128)
        q = synth.queries(32, 0, step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].cuda(), vn[:, 0].cuda())
        torch.cuda.synchronize()
        ref.append(O.to_units(kn.float().numpy()), O.to_units(vn.float().numpy()))
        ro, rm = ref.decode(O.queries_to_units(q.float().numpy(), Hkv))
        close(out.cpu().numpy(), ro.reshape(B, Hq, 128), f"output, step {step}")
        close(mass.cpu().numpy(), rm.reshape(B, Hq, -1), f"mass, step {step}")
        if step % every == every - 1:
            gs = cache.scores(0).cpu().numpy()
            close(gs, ref.scores(), "cumulative scores")
            drift = synth.drift_factors(32, 0, step, B * Hkv, cache.num_windows(0))
            cache.route(0, score_mult=drift.cuda())
            ref.route(scores_override=np.asarray(cache.scores(0).cpu().numpy(), np.float64))
            check_state(cache, 0, ref)
            assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    assert cache.status() == 0, cache.last_error()
    assert cache.stats()["promotions"] > 0


def test_per_head_full_size_llama_b1_32k_20pct():
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 64, 32768, 0.2
    W = L // w
    scores = synth.zipf_scores(0, 0, B * Hkv, W)
    cache, ref, _ = make_ph(B, Hq, Hkv, w, L, beta=beta, seed=0, scores=scores)
    t = ref.tiers()
    # the shared mode's counts, per head
    assert all(((r == 0).sum(), (r == 1).sum(), (r == 2).sum()) == (51, 274, 187) for r in t)
    check_state(cache, 0, ref)
    check_decode_ph(cache, ref, synth.queries(0, 0, 0, B, Hq, 128))


def test_per_head_demote_promote_set_tiers_and_diagnostics():
    B, Hq, Hkv, w, L = 2, 8, 2, 32, 640
    W = L // w
    tiers = torch.stack([synth.drawn_tiers(33, u, 1, W, 6, 8)[0] for u in range(B * Hkv)])
    cache, ref, k = make_ph(B, Hq, Hkv, w, L, seed=33, tiers=tiers, fp_capacity=W, ledger_capacity=W)
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    t = ref.tiers()
    pairs = [[u, int(np.flatnonzero(t[u] == O.TIER_Q)[0])] for u in range(B * Hkv)]
    cache.promote(0, torch.tensor(pairs, dtype=torch.int32).cuda())
    ref.promote(pairs)
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    cache.demote(0, torch.tensor(pairs, dtype=torch.int32).cuda())
    ref.demote(pairs)
    check_state(cache, 0, ref)
    q = synth.queries(33, 0, 0, B, Hq, 128)
    check_decode_ph(cache, ref, q, accumulate=False)
    got = cache.future_missed_mass(0, q.cuda(), k.cuda())
    torch.cuda.synchronize()
    want = O.future_missed_mass(ref, O.queries_to_units(q.float().numpy(), Hkv), O.to_units(k.float().numpy()))
    close(got.cpu().numpy(), want.reshape(B, Hq), "future missed mass per head")
    assert cache.status() == 0, cache.last_error()


def test_per_head_full_size_batched_llama_b8_32k_5pct():
    """Batch 8 of the Llama-8B shape at 5 %, per-head tiers: 64 units of 512 windows."""
    B, Hq, Hkv, w, L, beta = 8, 32, 8, 64, 32768, 0.05
    W = L // w
    scores = synth.zipf_scores(34, 0, B * Hkv, W)
    cache, ref, _ = make_ph(B, Hq, Hkv, w, L, beta=beta, seed=34, scores=scores)
    t = ref.tiers()
    assert all(((r == 0).sum(), (r == 1).sum(), (r == 2).sum()) == (12, 72, 428) for r in t)
    check_state(cache, 0, ref)
    for step in range(2):
        check_decode_ph(cache, ref, synth.queries(34, 0, step, B, Hq, 128))


def test_per_head_rate_distortion_route():
    B, Hq, Hkv, w, L, beta = 2, 16, 4, 32, 2048, 0.15
    W = L // w
    cache, ref, _ = make_ph(B, Hq, Hkv, w, L, beta=beta, seed=35, tiers=torch.zeros(B * Hkv, W, dtype=torch.uint8),
                            fp_capacity=W, ledger_capacity=W)
    scores = synth.zipf_scores(35, 0, B * Hkv, W)
    cache.route_rd(0, scores_override=scores.cuda())
    O.route_rd(ref, scores_override=scores.numpy())
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    check_decode_ph(cache, ref, synth.queries(35, 0, 0, B, Hq, 128))
