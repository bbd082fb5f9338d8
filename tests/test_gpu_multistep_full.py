"""Full-size multi-step parity: the batched workloads through fused decode
steps and routing events with score drift, and the longest-context decodes.

Per step the CUDA cache runs one fused decode step (append, attention, masses,
cumulative scores). The oracle appends the same token every step and decodes
on a sample of the steps (every `sample` steps, and the steps around each
routing event); on every step the cache's score growth must equal the mean
over query heads of the masses it returned. At each routing event the scores
are scaled by seeded drift factors and both sides route; the oracle routes on
the GPU's scores (teacher forcing, because near-ties of fp32 scores could
otherwise flip), and tiers, slot tables, stored bf16 and the ledger must then
match bit for bit (QEvict, "Kernmechanismen": demotion writes the ledger once,
promotion dequantises from it, later demotions reuse it).
"""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_state, check_stats, close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def _pair(B, Hq, Hkv, w, L, beta, seed, max_context):
    """Both caches prefilled with the same seeded tokens and routed once on Zipf scores."""
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, max_context, budget_frac=beta, fp_share=0.5)
    k, v = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy", device="cuda")
    scores = synth.zipf_scores(seed, 0, B, -(-L // w))
    cache.prefill(0, k, v, scores=scores.cuda())
    ref = O.OracleCache(B, Hq, Hkv, 128, w, beta=beta, rho=0.5)
    ref.prefill(k.float().cpu().numpy(), v.float().cpu().numpy(), scores=scores.numpy())
    del k, v
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)
    return cache, ref


@pytest.mark.parametrize("name,steps,sample", [("llama8b_b8_32k_5pct", 128, 16),
                                               ("qwen7b_b16_16k_10pct", 256, 32)])
def test_full_size_steps_with_routing_events(name, steps, sample):
    """Llama-3.1-8B-shaped batch 8 at 32K tokens and a 5 % budget (about 84 %
    of windows evicted), and Qwen2.5-7B-shaped batch 16 (GQA 7:1) at 16K and
    10 %: fused decode steps with a routing event every 64 steps."""
    c = synth.WORKLOADS[name]
    B, Hq, Hkv, w, L0, beta, every = c["B"], c["Hq"], c["Hkv"], c["w"], c["L"], c["beta"], c["route_every"]
    seed = 41
    cache, ref = _pair(B, Hq, Hkv, w, L0, beta, seed, L0 + steps)
    events = 0
    for step in range(steps):
        kn, vn = synth.kv_tokens(seed, 0, B, L0 + step, 1, Hkv, 128, "heavy", device="cuda")
        q = synth.queries(seed, 0, step, B, Hq, 128, device="cuda")
        before = cache.scores(0).cpu().numpy().astype(np.float64)
        out, mass = cache.decode_step(0, q, kn[:, 0].contiguous(), vn[:, 0].contiguous())
        after = cache.scores(0).cpu().numpy().astype(np.float64)
        ref.append(kn.float().cpu().numpy(), vn.float().cpu().numpy())
        assert cache.status() == 0, (step, cache.last_error())
        m = mass.cpu().numpy().astype(np.float64)
        assert m.shape == (B, Hq, ref.W)
        # the score of every window grows by its mass averaged over the query heads
        grown = after.copy()
        grown[:, : before.shape[1]] -= before
        close(grown, m.mean(axis=1), f"score growth, step {step}", max_abs=1e-4, rel_l2=1e-4)
        near_event = step % every in (0, every - 1)
        if step % sample == 0 or near_event or step == steps - 1:
            ro, rm = ref.decode(q.float().cpu().numpy(), accumulate=False)
            close(out.cpu().numpy(), ro, f"output, step {step}")
            close(m, rm, f"mass, step {step}")
        if step % every == every - 1:
            gs = cache.scores(0).cpu().numpy()
            drift = synth.drift_factors(seed, 0, step, B, ref.W)
            cache.route(0, score_mult=drift.cuda())
            routed = cache.scores(0).cpu().numpy()
            assert np.array_equal(routed, gs * drift.numpy())
            ref.route(scores_override=routed.astype(np.float64))
            assert cache.status() == 0, cache.last_error()
            check_state(cache, 0, ref)
            assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))
            events += 1
    assert events == steps // every
    check_stats(cache, [ref])
    s = cache.stats()
    assert s["promotions"] > 0 and s["ledger_reuses"] > 0, s


@pytest.mark.parametrize("w,beta", [(64, 0.05), (64, 0.20), (128, 0.05), (128, 0.20)])
def test_mistral_128k_batch4_decode(w, beta):
    """The 128K-token corners of the Mistral-7B-shaped sweep at batch 4: one
    decode and one fused decode step."""
    B, Hq, Hkv, L = 4, 32, 8, 131072
    seed = 43
    cache, ref = _pair(B, Hq, Hkv, w, L, beta, seed, L + 1)
    t = ref.tiers()
    assert (t == O.TIER_Q).any() and (t == O.TIER_E).any()
    q = synth.queries(seed, 0, 0, B, Hq, 128, device="cuda")
    out, mass = cache.decode(0, q, accumulate=False)
    ro, rm = ref.decode(q.float().cpu().numpy(), accumulate=False)
    close(out.cpu().numpy(), ro, "output")
    close(mass.cpu().numpy(), rm, "mass")
    kn, vn = synth.kv_tokens(seed, 0, B, L, 1, Hkv, 128, "heavy", device="cuda")
    q = synth.queries(seed, 0, 1, B, Hq, 128, device="cuda")
    out, mass = cache.decode_step(0, q, kn[:, 0].contiguous(), vn[:, 0].contiguous(), accumulate=False)
    ref.append(kn.float().cpu().numpy(), vn.float().cpu().numpy())
    ro, rm = ref.decode(q.float().cpu().numpy(), accumulate=False)
    close(out.cpu().numpy(), ro, "fused step output")
    close(mass.cpu().numpy(), rm, "fused step mass")
    assert cache.status() == 0, cache.last_error()
