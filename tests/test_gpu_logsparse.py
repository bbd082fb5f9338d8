"""The log-sparse positional router on the GPU against oracle.route_logsparse.

Tiers, slot tables, stored bf16, ledger entries and tier-move counts bit for
bit; the decode after each event within the attention tolerance. As windows
age their log-sparse rank changes (a window can move to a region where it
joins in an earlier round), so repeated events promote windows back from
INT2 and exercise the write-once ledger.
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


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta,R", [(1, 32, 8, 64, 4096, 0.2, 2), (2, 28, 4, 32, 3000, 0.1, 4),
                                                  (3, 8, 2, 16, 777, 0.3, 1), (2, 8, 2, 64, 8192, 0.05, 2)])
def test_logsparse_route_matches_oracle(B, Hq, Hkv, w, L, beta, R):
    W = -(-L // w)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, seed=50, tiers=[torch.zeros(B, W, dtype=torch.uint8)],
                              fp_capacity=W, ledger_capacity=W)
    for step in range(2):
        check_decode(cache, 0, ref, synth.queries(50, 0, step, B, Hq, 128))   # scores the route must ignore
    scores_before = cache.scores(0).cpu().numpy()
    cache.route_logsparse(0, recent=R)
    O.route_logsparse(ref, recent=R)
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    assert np.array_equal(cache.scores(0).cpu().numpy(), scores_before)
    t = ref.tiers()
    assert (t == O.TIER_Q).any() and (t == O.TIER_E).any()
    check_decode(cache, 0, ref, synth.queries(50, 0, 2, B, Hq, 128))


def test_logsparse_route_per_head_cache():
    B, Hq, Hkv, w, L, beta, R = 2, 16, 4, 32, 2048, 0.15, 2
    W = L // w
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, L, budget_frac=beta, per_head=True)
    ref = O.per_head_cache(B, Hq, Hkv, 128, w, beta=beta)
    k, v = synth.kv_tokens(51, 0, B, 0, L, Hkv, 128, "heavy")
    scores = synth.zipf_scores(51, 0, B * Hkv, W)
    cache.prefill(0, k.cuda(), v.cuda(), scores=scores.cuda())
    ref.prefill(O.to_units(k.float().numpy()), O.to_units(v.float().numpy()), scores=scores.numpy())
    cache.route_logsparse(0, recent=R)
    O.route_logsparse(ref, recent=R)
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    q = synth.queries(51, 0, 0, B, Hq, 128)
    out, mass = cache.decode(0, q.cuda(), accumulate=False)
    torch.cuda.synchronize()
    ro, rm = ref.decode(O.queries_to_units(q.float().numpy(), Hkv), accumulate=False)
    close(out.cpu().numpy(), ro.reshape(B, Hq, 128), "attention output")
    close(mass.cpu().numpy(), rm.reshape(B, Hq, -1), "window mass")


def test_logsparse_routes_between_fused_steps_promote_and_reuse_the_ledger():
    B, Hq, Hkv, w, L0, beta, R = 2, 8, 2, 16, 512, 0.25, 2
    steps, every = 160, 16
    W0 = L0 // w
    Wmax = -(-(L0 + steps) // w)
    # pools for every window: the prefill starts with all of them in full precision
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L0, beta=beta, seed=52, max_context=L0 + steps,
                              tiers=[torch.zeros(B, W0, dtype=torch.uint8)], fp_capacity=Wmax, ledger_capacity=Wmax)
    cache.route_logsparse(0, recent=R)
    O.route_logsparse(ref, recent=R)
    check_state(cache, 0, ref)
    for step in range(steps):
        kn, vn = synth.kv_tokens(52, 0, B, L0 + step, 1, Hkv, 128)
        q = synth.queries(52, 0, step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].cuda(), vn[:, 0].cuda())
        torch.cuda.synchronize()
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        close(out.cpu().numpy(), ro, f"output, step {step}")
        close(mass.cpu().numpy(), rm, f"mass, step {step}")
        if step % every == every - 1:
            cache.route_logsparse(0, recent=R)
            O.route_logsparse(ref, recent=R)
            check_state(cache, 0, ref)
            assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    assert cache.status() == 0, cache.last_error()
    s = cache.stats()
    assert s["promotions"] > 0 and s["ledger_reuses"] > 0
    for key in ("demotions", "promotions", "evictions", "ledger_writes", "ledger_reuses"):
        assert s[key] == ref.stats[key], key


def test_logsparse_full_size_llama_b1_32k_20pct():
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 64, 32768, 0.2
    W = L // w
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, seed=0, tiers=[torch.zeros(B, W, dtype=torch.uint8)],
                              fp_capacity=W, ledger_capacity=W)
    cache.route_logsparse(0, recent=2)
    O.route_logsparse(ref, recent=2)
    t = ref.tiers()
    assert ((t == 0).sum(), (t == 1).sum(), (t == 2).sum()) == (51, 274, 187)
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(0, 0, 0, B, Hq, 128))


def test_logsparse_rejects_a_bad_recent_count():
    cache, _ = make_pair(1, 8, 2, 32, 256, beta=0.5, tiers=[torch.zeros(1, 8, dtype=torch.uint8)])
    with pytest.raises(binding.QevictError) as e:
        cache.route_logsparse(0, recent=0)
    assert e.value.name == "INVALID_ARG"
