"""One routing event over all layers (and KV heads) under one budget per
sequence: the CUDA path against oracle.route_global.

Tiers, slot tables, stored bf16, ledger entries and tier-move counts must
match bit for bit in every layer; the decode after the event within the
attention tolerance. The second event of each test routes on the scores the
GPU accumulated while decoding, given to the oracle as they are (teacher
forcing), after they are checked against the oracle's own.
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


def build_pair(B, NL, Hq, Hkv, w, lengths, beta, per_head, seed):
    maxc = max(lengths)
    W = -(-maxc // w)
    cache = binding.TieredCache(B, NL, Hq, Hkv, w, maxc, budget_frac=beta, per_head=per_head,
                                fp_capacity=W, ledger_capacity=W)
    units = B * Hkv if per_head else B
    refs = []
    for l, L in enumerate(lengths):
        k, v = synth.kv_tokens(seed, l, B, 0, L, Hkv, 128, "heavy")
        tiers = torch.zeros(units, -(-L // w), dtype=torch.uint8)
        cache.prefill(l, k.cuda(), v.cuda(), tiers=tiers.cuda())
        if per_head:
            ref = O.per_head_cache(B, Hq, Hkv, 128, w, beta=beta)
            ref.prefill(O.to_units(k.float().numpy()), O.to_units(v.float().numpy()), tiers=tiers.numpy())
        else:
            ref = O.OracleCache(B, Hq, Hkv, 128, w, beta=beta)
            ref.prefill(k.float().numpy(), v.float().numpy(), tiers=tiers.numpy())
        refs.append(ref)
    return cache, refs, units


def decode_all(cache, refs, B, Hq, Hkv, per_head, seed, step):
    for l, ref in enumerate(refs):
        q = synth.queries(seed, l, step, B, Hq, 128)
        out, mass = cache.decode(l, q.cuda())
        torch.cuda.synchronize()
        qr = O.queries_to_units(q.float().numpy(), Hkv) if per_head else q.float().numpy()
        ro, rm = ref.decode(qr)
        close(out.cpu().numpy(), ro.reshape(B, Hq, 128), f"output, layer {l}")
        close(mass.cpu().numpy(), rm.reshape(B, Hq, -1), f"mass, layer {l}")


def check_all(cache, refs):
    for l, ref in enumerate(refs):
        check_state(cache, l, ref)
        assert np.array_equal(cache.tier_move_counts(l).numpy(), ref.last_counts.astype(np.int32)), l


@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("B,NL,Hq,Hkv,w,lengths,beta", [
    (2, 3, 8, 2, 32, (1024, 1024, 1024), 0.2),
    (1, 4, 32, 8, 64, (4096, 4096, 4096, 4096), 0.1),
    (3, 3, 28, 4, 16, (700, 512, 333), 0.25),          # layers of different lengths
])
def test_global_route_matches_oracle(B, NL, Hq, Hkv, w, lengths, beta, per_head):
    seed = 40
    cache, refs, units = build_pair(B, NL, Hq, Hkv, w, lengths, beta, per_head, seed)
    hs = Hkv if per_head else 1
    # event 1: seeded scores, scaled per layer so the layers' shares differ
    ov = [synth.zipf_scores(seed, l, units, -(-L // w)) * (1.0 + 0.5 * l) for l, L in enumerate(lengths)]
    cache.route_global([t.cuda() for t in ov])
    O.route_global(refs, hs=hs, scores_override=[t.numpy() for t in ov])
    assert cache.status() == 0, cache.last_error()
    check_all(cache, refs)
    kept = [(ref.tiers() != O.TIER_E).sum() for ref in refs]
    assert (np.concatenate([r.tiers().ravel() for r in refs]) == O.TIER_E).any()
    # decode steps accumulate scores; event 2 routes on the GPU's scores
    for step in range(2):
        decode_all(cache, refs, B, Hq, Hkv, per_head, seed, step)
    for l, ref in enumerate(refs):
        gs = cache.scores(l).cpu().numpy()
        close(gs, ref.scores(), f"cumulative scores, layer {l}")
        ref.S = [gs[u].astype(np.float64) for u in range(units)]
    cache.route_global()
    O.route_global(refs, hs=hs)
    assert cache.status() == 0, cache.last_error()
    check_all(cache, refs)
    decode_all(cache, refs, B, Hq, Hkv, per_head, seed, 2)
    s = cache.stats()
    for key in ("demotions", "promotions", "evictions", "ledger_writes", "ledger_reuses"):
        assert s[key] == sum(r.stats[key] for r in refs), key
    assert len(set(kept)) > 1 or NL == 1   # the one budget moved between layers


def test_global_route_budget_rejected_on_host():
    cache = binding.TieredCache(1, 4, 8, 2, 32, 64, budget_frac=0.05)
    for l in range(4):
        cache.append(l, *[x.cuda() for x in synth.kv_tokens(41, l, 1, 0, 64, 2, 128)])
    with pytest.raises(binding.QevictError) as e:
        cache.route_global()
    assert e.value.name == "BUDGET"
    assert cache.status() == 0
