"""A seeded sweep of shapes against the oracle: batch 1-3, 1-8 KV heads, GQA
groups of 1-8 query heads, windows of 16-128 tokens, lengths with ragged last
windows, budgets from 5 % to 60 % and full-precision shares from a quarter to
three quarters. Each case prefills with routing on seeded scores, decodes,
runs fused steps (append + decode + scores, the open window crossing a window
boundary), routes on the GPU's accumulated scores (teacher forced, as in the
multistep test) and decodes again. Bit-exact: tiers, stored bf16, ledger codes
and meta, write counts, transition statistics; outputs, masses and scores
within the attention tolerance. A second sweep does the same through the
wide kernel: caches that allow INT4 and INT8, mixed-width routing events on
seeded scores, fused steps, and a second event on the accumulated scores."""
import os

import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_decode, check_state, check_stats, close, make_pair

pytestmark = pytest.mark.gpu

# more cases on request (the seeds continue the same sequences)
N_CASES = int(os.environ.get("QEVICT_SWEEP_CASES", "32"))
N_WIDE = int(os.environ.get("QEVICT_SWEEP_WIDE", "16"))


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def draw_case(i):
    rng = np.random.default_rng(5000 + i)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.integers(1, 9))
    B = int(rng.integers(1, 4))
    w = int(rng.choice([16, 32, 64, 128]))
    beta = float(rng.choice([0.05, 0.1, 0.2, 0.35, 0.6]))
    rho = float(rng.choice([0.25, 0.5, 0.75]))
    # long enough that the budget holds the open window (beta L >= w), and a ragged tail
    lo = int(np.ceil(w / beta)) + w
    L = int(rng.integers(lo, max(lo + 1, 2600)))
    if L % w == 0:
        L += int(rng.integers(1, w))
    steps = int(rng.integers(w // 2, w + 8))   # enough appends to cross into a new window sometimes
    return B, G * Hkv, Hkv, w, L, beta, rho, steps


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_prefill_steps_route_decode(i):
    B, Hq, Hkv, w, L, beta, rho, steps = draw_case(i)
    seed = 300 + i
    W = -(-L // w)
    scores = synth.zipf_scores(seed, 0, B, W)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, rho=rho, scores=[scores], max_context=L + steps,
                              seed=seed)
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(seed, 0, 0, B, Hq, 128))
    for step in range(steps):
        kn, vn = synth.kv_tokens(seed, 0, B, L + step, 1, Hkv, 128, "heavy")
        q = synth.queries(seed, 0, 1 + step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].cuda(), vn[:, 0].cuda())
        torch.cuda.synchronize()
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        if step % 8 == 0 or step == steps - 1:
            close(out.cpu().numpy(), ro, f"output after {step + 1} fused steps")
            close(mass.cpu().numpy(), rm, f"mass after {step + 1} fused steps")
    assert cache.status() == 0, cache.last_error()
    cache.refresh_lengths()
    check_state(cache, 0, ref)
    # a routing event on the accumulated scores, the oracle fed the GPU's scores
    gs = cache.scores(0).cpu().numpy()
    close(gs, np.stack(ref.S), "cumulative scores")
    cache.route(0)
    ref.route(scores_override=np.asarray(gs, np.float64))
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    check_stats(cache, [ref])
    check_decode(cache, 0, ref, synth.queries(seed, 0, 10_000, B, Hq, 128))


def draw_wide(i):
    rng = np.random.default_rng(7000 + i)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.integers(1, 9))
    B = int(rng.integers(1, 4))
    w = int(rng.choice([16, 32, 64, 128]))
    beta = float(rng.choice([0.05, 0.1, 0.2, 0.35]))
    bits = int(rng.choice([4, 8]))
    lo = int(np.ceil(w / beta)) + w
    L = int(rng.integers(lo, max(lo + 1, 2600)))
    if L % w == 0:
        L += int(rng.integers(1, w))
    steps = int(rng.integers(w // 2, w + 8))
    return B, G * Hkv, Hkv, w, L, beta, bits, steps


@pytest.mark.parametrize("i", range(N_WIDE))
def test_random_shape_mixed_widths(i):
    B, Hq, Hkv, w, L, beta, bits, steps = draw_wide(i)
    seed = 700 + i
    maxc = L + steps
    Wmax, W = -(-maxc // w), -(-L // w)
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, maxc, budget_frac=beta, max_ledger_bits=bits,
                                fp_capacity=Wmax, ledger_capacity=Wmax)
    ref = O.OracleCache(B, Hq, Hkv, 128, w, beta=beta)
    k, v = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy")
    t0 = np.zeros((B, W), np.uint8)
    cache.prefill(0, k.cuda(), v.cuda(), tiers=torch.from_numpy(t0).cuda())
    ref.prefill(k.float().numpy(), v.float().numpy(), tiers=t0)
    scores = synth.zipf_scores(seed, 0, B, W)
    cache.route_rd_mixed(0, scores_override=scores.cuda())
    O.route_rd_mixed(ref, scores_override=scores.numpy(), max_bits=bits)
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(seed, 0, 0, B, Hq, 128))
    for step in range(steps):
        kn, vn = synth.kv_tokens(seed, 0, B, L + step, 1, Hkv, 128, "heavy")
        q = synth.queries(seed, 0, 1 + step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].cuda(), vn[:, 0].cuda())
        torch.cuda.synchronize()
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        if step % 8 == 0 or step == steps - 1:
            close(out.cpu().numpy(), ro, f"output after {step + 1} fused steps")
            close(mass.cpu().numpy(), rm, f"mass after {step + 1} fused steps")
    assert cache.status() == 0, cache.last_error()
    cache.refresh_lengths()
    check_state(cache, 0, ref)
    # a second event on the accumulated scores (the oracle fed the GPU's), windows
    # moving within their ledger widths
    gs = cache.scores(0).cpu().numpy()
    close(gs, np.stack(ref.S), "cumulative scores")
    cache.route_rd_mixed(0, scores_override=torch.from_numpy(gs).cuda())
    O.route_rd_mixed(ref, scores_override=np.asarray(gs, np.float64), max_bits=bits)
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(seed, 0, 10_000, B, Hq, 128))
