"""INT4 and INT8 tiers (the wider widths of the rate-distortion option) on the
GPU against the oracle: quantisation into bit planes, the ledger width fixed
at the first quantisation, promotion from any width, and the tables, all bit
for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_state

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def mixed_tiers(seed, B, W, allowed):
    rng = np.random.default_rng(seed)
    t = rng.choice(allowed, size=(B, W)).astype(np.uint8)
    t[:, -1] = O.TIER_FP
    return t


def make_wide(B, Hq, Hkv, w, L, bits, tiers, seed):
    W = -(-L // w)
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, L, max_ledger_bits=bits, fp_capacity=W, ledger_capacity=W)
    ref = O.OracleCache(B, Hq, Hkv, 128, w)
    k, v = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy")
    cache.prefill(0, k.cuda(), v.cuda(), tiers=torch.from_numpy(tiers).cuda())
    ref.prefill(k.float().numpy(), v.float().numpy(), tiers=tiers)
    assert cache.status() == 0, cache.last_error()
    return cache, ref


@pytest.mark.parametrize("B,Hq,Hkv,w,L,bits", [(2, 8, 2, 32, 640, 8), (1, 32, 8, 64, 4096, 8), (3, 28, 4, 16, 777, 4)])
def test_wide_prefill_and_moves_bit_exact(B, Hq, Hkv, w, L, bits):
    W = -(-L // w)
    allowed = [O.TIER_FP, O.TIER_Q, O.TIER_Q4, O.TIER_E] + ([O.TIER_Q8] if bits == 8 else [])
    tiers = mixed_tiers(40 + bits, B, W, allowed)
    cache, ref = make_wide(B, Hq, Hkv, w, L, bits, tiers, seed=40 + bits)
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    # promote every quantised window, then quantise the full-precision ones that have no
    # ledger at a random width and send the promoted ones back to theirs (ledger reuse)
    t = ref.tiers()
    t1 = np.where(np.isin(t, [O.TIER_Q, O.TIER_Q4, O.TIER_Q8]), O.TIER_FP, t).astype(np.uint8)
    cache.set_tiers(0, torch.from_numpy(t1).cuda())
    ref.set_tiers(t1)
    check_state(cache, 0, ref)
    rng = np.random.default_rng(50 + bits)
    t2 = t1.copy()
    for b in range(B):
        for wi in range(W - 1):
            if t1[b, wi] != O.TIER_FP:
                continue
            win = ref.win[b][wi]
            if win.ledger is not None:
                t2[b, wi] = {2: O.TIER_Q, 4: O.TIER_Q4, 8: O.TIER_Q8}[win.ledger_bits]
            else:
                t2[b, wi] = rng.choice(allowed[:3] + allowed[4:])
    cache.set_tiers(0, torch.from_numpy(t2).cuda())
    ref.set_tiers(t2)
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
    s = cache.stats()
    for key in ("demotions", "promotions", "evictions", "ledger_writes", "ledger_reuses"):
        assert s[key] == ref.stats[key], key


def test_wide_width_rules_on_the_device():
    B, Hq, Hkv, w, L = 1, 8, 2, 32, 256
    tiers = np.array([[O.TIER_Q4, O.TIER_Q8, O.TIER_FP, O.TIER_Q, 0, 0, 0, 0]], np.uint8)
    cache, ref = make_wide(B, Hq, Hkv, w, L, 8, tiers, seed=60)
    # a quantised window cannot change width directly
    bad = tiers.copy()
    bad[0, 0] = O.TIER_Q8
    cache.set_tiers(0, torch.from_numpy(bad).cuda())
    assert binding.STATUS[cache.status()] == "STATE"
    cache.clear_status()
    check_state(cache, 0, ref)   # nothing moved
    # after a promotion the ledger keeps its width: INT2 for an INT4 window is refused
    t = tiers.copy()
    t[0, 0] = O.TIER_FP
    cache.set_tiers(0, torch.from_numpy(t).cuda())
    ref.set_tiers(t)
    t2 = t.copy()
    t2[0, 0] = O.TIER_Q
    cache.set_tiers(0, torch.from_numpy(t2).cuda())
    assert binding.STATUS[cache.status()] == "STATE"
    cache.clear_status()
    check_state(cache, 0, ref)
    # INT8 is refused by a cache that allows INT4 only
    small = binding.TieredCache(1, 1, 8, 2, 32, 256, max_ledger_bits=4, fp_capacity=8, ledger_capacity=8)
    k, v = synth.kv_tokens(61, 0, 1, 0, 256, 2, 128)
    small.prefill(0, k.cuda(), v.cuda(), tiers=torch.from_numpy(tiers).cuda())
    assert binding.STATUS[small.status()] == "STATE"


def test_wide_cache_rejects_the_int2_routes():
    cache = binding.TieredCache(1, 1, 8, 2, 32, 256, max_ledger_bits=4)
    k, v = synth.kv_tokens(62, 0, 1, 0, 256, 2, 128)
    cache.prefill(0, k.cuda(), v.cuda(), tiers=torch.zeros(1, 8, dtype=torch.uint8).cuda())
    for call in (lambda: cache.route(0), lambda: cache.route_rd(0), lambda: cache.route_logsparse(0),
                 lambda: cache.route_global()):
        with pytest.raises(binding.QevictError) as e:
            call()
        assert e.value.name == "INVALID_ARG"


@pytest.mark.parametrize("B,Hq,Hkv,w,L,bits", [(2, 8, 2, 32, 640, 8), (1, 32, 8, 64, 4096, 8), (3, 28, 4, 16, 777, 4),
                                               (1, 32, 8, 64, 32768, 8)])
def test_wide_decode_matches_oracle(B, Hq, Hkv, w, L, bits):
    from parity_util import check_decode
    W = -(-L // w)
    allowed = [O.TIER_FP, O.TIER_Q, O.TIER_Q4, O.TIER_E] + ([O.TIER_Q8] if bits == 8 else [])
    tiers = mixed_tiers(70 + bits, B, W, allowed)
    cache, ref = make_wide(B, Hq, Hkv, w, L, bits, tiers, seed=70 + bits)
    for step in range(2):
        check_decode(cache, 0, ref, synth.queries(70, 0, step, B, Hq, 128))


def test_wide_decode_steps_append_into_a_mixed_cache():
    B, Hq, Hkv, w, L0, steps = 2, 16, 4, 32, 512, 40
    W0 = L0 // w
    tiers = mixed_tiers(80, B, W0, [O.TIER_FP, O.TIER_Q, O.TIER_Q4, O.TIER_Q8, O.TIER_E])
    Wmax = -(-(L0 + steps) // w)
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, L0 + steps, max_ledger_bits=8, fp_capacity=Wmax,
                                ledger_capacity=Wmax)
    ref = O.OracleCache(B, Hq, Hkv, 128, w)
    k, v = synth.kv_tokens(80, 0, B, 0, L0, Hkv, 128, "heavy")
    cache.prefill(0, k.cuda(), v.cuda(), tiers=torch.from_numpy(tiers).cuda())
    ref.prefill(k.float().numpy(), v.float().numpy(), tiers=tiers)
    from parity_util import close
    for step in range(steps):
        kn, vn = synth.kv_tokens(80, 0, B, L0 + step, 1, Hkv, 128)
        q = synth.queries(80, 0, step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].cuda(), vn[:, 0].cuda())
        torch.cuda.synchronize()
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        close(out.cpu().numpy(), ro, f"output, step {step}")
        close(mass.cpu().numpy(), rm, f"mass, step {step}")
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)


def test_wide_cache_with_int2_windows_decodes_like_an_int2_cache():
    """A cache that allows INT4 / INT8 but holds INT2 windows only decodes as an
    INT2-only cache does. The two instantiations claim quantised tiles in
    chunks of different sizes, so their fp32 sums run in another order: both
    must meet the oracle, and each other, within the attention tolerance."""
    from parity_util import close
    B, Hq, Hkv, w, L = 1, 32, 8, 64, 4096
    W = L // w
    tiers = mixed_tiers(90, B, W, [O.TIER_FP, O.TIER_Q, O.TIER_E])
    k, v = synth.kv_tokens(90, 0, B, 0, L, Hkv, 128, "heavy", device="cuda")
    q = synth.queries(90, 0, 0, B, Hq, 128)
    ref = O.OracleCache(B, Hq, Hkv, 128, w)
    ref.prefill(k.float().cpu().numpy(), v.float().cpu().numpy(), tiers=tiers)
    ro, rm = ref.decode(q.float().numpy(), accumulate=False)
    outs = []
    for bits in (0, 8):
        c = binding.TieredCache(B, 1, Hq, Hkv, w, L, max_ledger_bits=bits, fp_capacity=W, ledger_capacity=W)
        c.prefill(0, k, v, tiers=torch.from_numpy(tiers).cuda())
        o, m = c.decode(0, q.cuda(), accumulate=False)
        torch.cuda.synchronize()
        assert c.status() == 0, c.last_error()
        close(o.cpu().numpy(), ro, f"output, max_ledger_bits {bits}")
        close(m.cpu().numpy(), rm, f"mass, max_ledger_bits {bits}")
        outs.append((o.cpu().numpy(), m.cpu().numpy()))
    close(outs[1][0], outs[0][0], "output, wide against INT2-only")
    close(outs[1][1], outs[0][1], "mass, wide against INT2-only")
