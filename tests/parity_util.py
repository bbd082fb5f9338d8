"""Helpers shared by the GPU parity tests: build both sides from the same seeded
inputs and compare the CUDA cache's state and outputs with the oracle's."""
import numpy as np
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth

# Attention outputs and window scores: the tolerance the target states
# (fp32 accumulation over bf16 inputs, against the fp64 oracle).
MAX_ABS = 2e-3
REL_L2 = 1e-3


def close(gpu, ref, what, max_abs=MAX_ABS, rel_l2=REL_L2):
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r).max() if g.size else 0.0
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g - r)
    assert err <= max_abs and rel <= rel_l2, f"{what}: max|d|={err:.3e} relL2={rel:.3e}"
    return err, rel


def make_pair(B, Hq, Hkv, w, L, layers=1, beta=1.0, rho=0.5, max_context=None, seed=0,
              outliers="heavy", scores=None, tiers=None, fp_capacity=0, ledger_capacity=0, fp_slack=0):
    """A CUDA cache and an oracle cache prefilled with the same seeded tokens."""
    d = 128
    maxc = max_context or L
    cache = binding.TieredCache(B, layers, Hq, Hkv, w, maxc, budget_frac=beta, fp_share=rho,
                                fp_capacity=fp_capacity, ledger_capacity=ledger_capacity, fp_slack=fp_slack)
    refs = []
    for layer in range(layers):
        k, v = synth.kv_tokens(seed, layer, B, 0, L, Hkv, d, outliers)
        ref = O.OracleCache(B, Hq, Hkv, d, w, beta=beta, rho=rho)
        sc = scores[layer] if scores is not None else None
        tr = tiers[layer] if tiers is not None else None
        cache.prefill(layer, k.cuda(), v.cuda(), scores=None if sc is None else sc.cuda(),
                      tiers=None if tr is None else tr.cuda())
        ref.prefill(k.float().numpy(), v.float().numpy(), scores=None if sc is None else sc.numpy(),
                    tiers=None if tr is None else tr.numpy())
        refs.append(ref)
    return cache, refs


def check_state(cache, layer, ref):
    """Tiers, ledger entries, ledger write counts and stored bf16 are bit-exact."""
    tier, fps, lgs, lw = cache.tables(layer)
    rt = ref.tiers()
    assert np.array_equal(tier.numpy(), rt), "tiers differ"
    lbits = cache.ledger_bits(layer).numpy()
    for b in range(ref.B):
        for wi, win in enumerate(ref.win[b]):
            assert int(lw[b, wi]) == win.ledger_writes, ("ledger writes", b, wi)
            if win.tier == O.TIER_E:
                continue
            has_ledger = int(lgs[b, wi]) >= 0
            assert has_ledger == (win.ledger is not None), ("ledger presence", b, wi)
            if win.tier == O.TIER_FP:
                data = cache.fp_window(layer, int(fps[b, wi])).float().numpy()
                n = win.ntok
                assert np.array_equal(data[:, 0, :n], win.k[:, :n]), ("FP K", b, wi)
                assert np.array_equal(data[:, 1, :n], win.v[:, :n]), ("FP V", b, wi)
            if win.ledger is not None:
                assert int(lbits[b, wi]) == win.ledger_bits, ("ledger width", b, wi)
                codes, scale, mn = cache.ledger_window(layer, int(lgs[b, wi]), win.ledger_bits)
                ck, sk, mk, cv, sv, mv = win.ledger
                assert np.array_equal(codes[:, 0].numpy(), ck), ("K codes", b, wi)
                assert np.array_equal(codes[:, 1].numpy(), cv), ("V codes", b, wi)
                assert np.array_equal(scale[:, 0].numpy().view(np.uint16), sk.view(np.uint16)), ("K scale", b, wi)
                assert np.array_equal(mn[:, 0].numpy().view(np.uint16), mk.view(np.uint16)), ("K min", b, wi)
                assert np.array_equal(scale[:, 1].numpy().view(np.uint16), sv.view(np.uint16)), ("V scale", b, wi)
                assert np.array_equal(mn[:, 1].numpy().view(np.uint16), mv.view(np.uint16)), ("V min", b, wi)


def check_decode(cache, layer, ref, q, accumulate=True):
    out, mass = cache.decode(layer, q.cuda(), accumulate=accumulate)
    torch.cuda.synchronize()
    ro, rm = ref.decode(q.float().numpy(), accumulate=accumulate)
    close(out.cpu().numpy(), ro, "attention output")
    close(mass.cpu().numpy(), rm, "window mass")
    assert cache.status() == 0, cache.last_error()
    return out, mass, ro, rm


def stats_of(ref):
    return dict(ref.stats)


def check_stats(cache, refs):
    s = cache.stats()
    tot = {k: sum(r.stats[k] for r in refs) for k in refs[0].stats}
    for k in tot:
        assert s[k] == tot[k], (k, s[k], tot[k])
