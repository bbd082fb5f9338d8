"""The static-scratch decode entry point against qevict_decode_attention.

qevict_decode_attention_static_scratch runs the same decode kernel with its
per-call scratch in a library-owned device array. Two calls in a row must give
what the regular entry point gives, within the attention tolerance, and must
leave nothing behind that a later call could read as its own. The file is
named to be collected last, so it also runs after the other GPU tests have
used the library in the same process; it passes alone as well (the first call
in the process does the per-device set-up).
"""
import pytest
import torch

from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import close

pytestmark = pytest.mark.gpu

STATIC_BYTES = 4 * 1024 * 1024


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def _routed_cache(B, Hq, Hkv, w, L, beta, seed):
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, L, budget_frac=beta, fp_share=0.5)
    k, v = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy", device="cuda")
    W = -(-L // w)
    cache.prefill(0, k, v, scores=synth.zipf_scores(seed, 0, B, W).cuda())
    return cache


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [(1, 32, 8, 64, 32768, 0.2), (2, 28, 4, 64, 3000, 0.1),
                                                (3, 8, 2, 16, 777, 0.3)])
def test_static_scratch_matches_decode_attention(B, Hq, Hkv, w, L, beta):
    cache = _routed_cache(B, Hq, Hkv, w, L, beta, seed=11)
    W = cache.num_windows(0)
    for step in range(2):
        q = synth.queries(11, 0, step, B, Hq, 128).cuda()
        ref_out, ref_mass = cache.decode(0, q, accumulate=False)
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        mass = torch.full((B, Hq, W), float("nan"), dtype=torch.float32, device="cuda")
        before = cache.scores(0)
        cache.decode_static_scratch(0, q, out, mass, accumulate=True)
        after = cache.scores(0)
        torch.cuda.synchronize()
        assert cache.status() == 0, cache.last_error()
        close(out.cpu().numpy(), ref_out.cpu().numpy(), f"output, call {step}")
        close(mass.cpu().numpy(), ref_mass.cpu().numpy(), f"mass, call {step}")
        # accumulate: every window's score grows by its mass averaged over the query heads
        close((after - before).cpu().numpy(), ref_mass.mean(dim=1).cpu().numpy(), f"score growth, call {step}")


def test_static_scratch_without_mass():
    cache = _routed_cache(1, 32, 8, 64, 4096, 0.2, seed=12)
    q = synth.queries(12, 0, 0, 1, 32, 128).cuda()
    ref_out, _ = cache.decode(0, q, want_mass=False, accumulate=False)
    out = torch.empty(1, 32, 128, dtype=torch.float32, device="cuda")
    for _ in range(2):
        cache.decode_static_scratch(0, q, out, None, accumulate=False)
        torch.cuda.synchronize()
        close(out.cpu().numpy(), ref_out.cpu().numpy(), "output without mass")


def test_static_scratch_rejects_a_cache_that_needs_more():
    # 128 (sequence, KV head) pairs x 2048 records (one per slot of 1024 full-precision and
    # 1024 ledger slots of 16-token windows) x 4 query heads x 8 B is 8 MiB
    cache = binding.TieredCache(16, 1, 32, 8, 16, 16384, budget_frac=0.05, fp_share=0.5, fp_capacity=1024,
                                ledger_capacity=1024)
    k, v = synth.kv_tokens(13, 0, 16, 0, 100, 8, 128, "heavy", device="cuda")
    cache.append(0, k, v)
    q = synth.queries(13, 0, 0, 16, 32, 128).cuda()
    out = torch.empty(16, 32, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.QevictError) as e:
        cache.decode_static_scratch(0, q, out)
    assert e.value.name == "INVALID_ARG"
    assert str(STATIC_BYTES) in str(e.value)
    # nothing was enqueued: the regular entry point still serves this cache
    cache.decode(0, q, out=out, want_mass=False, accumulate=False)
    torch.cuda.synchronize()
    assert cache.status() == 0
    assert torch.isfinite(out).all()


def test_static_scratch_across_cache_shapes():
    """Caches of different (sequences x KV heads) one after another on one
    stream: the array's counters, records and partials sit at shape-dependent
    offsets, so a call must not take what a call on another cache left there."""
    caches = {shape: _routed_cache(*shape, seed=14) for shape in [(1, 32, 8, 64, 4096, 0.2),
                                                                   (8, 32, 8, 64, 2048, 0.2)]}
    order = [(1, 32, 8, 64, 4096, 0.2), (8, 32, 8, 64, 2048, 0.2), (1, 32, 8, 64, 4096, 0.2),
             (8, 32, 8, 64, 2048, 0.2)]
    for i, shape in enumerate(order):
        cache = caches[shape]
        B, Hq = shape[0], shape[1]
        q = synth.queries(14, 0, i, B, Hq, 128).cuda()
        ref_out, ref_mass = cache.decode(0, q, accumulate=False)
        for call in range(2):
            out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
            mass = torch.full_like(ref_mass, float("nan"))
            cache.decode_static_scratch(0, q, out, mass, accumulate=False)
            torch.cuda.synchronize()
            assert cache.status() == 0, cache.last_error()
            close(out.cpu().numpy(), ref_out.cpu().numpy(), f"output, cache {shape}, call {call}")
            close(mass.cpu().numpy(), ref_mass.cpu().numpy(), f"mass, cache {shape}, call {call}")
