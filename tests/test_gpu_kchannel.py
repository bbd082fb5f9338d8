"""RDKV's K-channel half on the GPU against the oracle: the channel weights
(fp32 sums against float64, within tolerance), then, fed the same float32
weights, the window widths, the K group widths, tiers, slot tables and every
ledger entry (K groups at their own widths, V at the window's) bit for bit,
and the decode of such a layer, before and after appends, within the
attention tolerance. Also the state rules: the widths are set with the
layer's first quantisation and the layer takes no further tier moves."""
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


def make_kch(B, Hq, Hkv, w, L, beta, seed, max_context=None):
    maxc = max_context or L
    Wmax = -(-maxc // w)
    W = -(-L // w)
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, maxc, budget_frac=beta, max_ledger_bits=8,
                                fp_capacity=Wmax, ledger_capacity=Wmax)
    ref = O.OracleCache(B, Hq, Hkv, 128, w, beta=beta)
    k, v = synth.kv_tokens(seed, 0, B, 0, L, Hkv, 128, "heavy")
    t = np.zeros((B, W), np.uint8)
    cache.prefill(0, k.cuda(), v.cuda(), tiers=torch.from_numpy(t).cuda())
    ref.prefill(k.float().numpy(), v.float().numpy(), tiers=t)
    assert cache.status() == 0, cache.last_error()
    # queries observed over the prefill (the last 64 positions' worth)
    q_obs = torch.stack([synth.queries(seed, 0, 1000 + i, B, Hq, 128) for i in range(64)], dim=1)
    return cache, ref, k, q_obs


def weights_both(cache, k, q_obs):
    wg = cache.k_channel_weights(0, q_obs.cuda(), k.cuda())
    torch.cuda.synchronize()
    wo = O.k_channel_weights(q_obs.float().numpy(), k.float().numpy(), cache.Hkv)
    got = wg.cpu().numpy().astype(np.float64)
    assert np.allclose(got, wo, rtol=2e-5, atol=0), np.abs(got / wo - 1).max()
    return wg


def route_kv_both(cache, ref, wg, scores):
    cache.route_rd_kv(0, wg, scores_override=scores.cuda())
    O.route_rd_kv(ref, wg.cpu().numpy(), scores_override=scores.numpy(), max_bits=8)
    assert cache.status() == 0, cache.last_error()
    assert np.array_equal(cache.k_group_bits(0).numpy().astype(np.int64), ref.kch)
    check_state(cache, 0, ref)
    assert np.array_equal(cache.tier_move_counts(0).numpy(), ref.last_counts.astype(np.int32))


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [(1, 32, 8, 64, 4096, 0.2), (2, 28, 4, 32, 3000, 0.1),
                                               (3, 8, 2, 16, 777, 0.3), (2, 8, 2, 64, 8192, 0.05),
                                               (2, 16, 4, 32, 2048, 0.4)])
def test_k_channel_route_and_decode_match_oracle(B, Hq, Hkv, w, L, beta):
    W = -(-L // w)
    cache, ref, k, q_obs = make_kch(B, Hq, Hkv, w, L, beta, seed=90)
    wg = weights_both(cache, k, q_obs)
    route_kv_both(cache, ref, wg, synth.zipf_scores(90, 0, B, W))
    widths = cache.k_group_bits(0).numpy()
    assert len(set(widths.reshape(-1).tolist())) > 1   # the groups do differ
    for step in range(2):
        check_decode(cache, 0, ref, synth.queries(90, 0, step, B, Hq, 128))


def test_k_channel_layer_decodes_after_appends():
    B, Hq, Hkv, w, L = 2, 16, 4, 32, 1000
    W = -(-L // w)
    cache, ref, k, q_obs = make_kch(B, Hq, Hkv, w, L, 0.2, seed=91, max_context=L + 80)
    wg = weights_both(cache, k, q_obs)
    route_kv_both(cache, ref, wg, synth.zipf_scores(91, 0, B, W))
    for step in range(70):
        kn, vn = synth.kv_tokens(91, 0, B, L + step, 1, Hkv, 128, "heavy")
        q = synth.queries(91, 0, 10 + step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].cuda(), vn[:, 0].cuda())
        torch.cuda.synchronize()
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        if step % 10 == 0 or step == 69:
            close(out.cpu().numpy(), ro, f"output after {step + 1} appends")
            close(mass.cpu().numpy(), rm, f"mass after {step + 1} appends")
    assert cache.status() == 0, cache.last_error()
    cache.refresh_lengths()
    check_state(cache, 0, ref)


def test_k_channel_full_size_llama_32k():
    B, Hq, Hkv, w, L = 1, 32, 8, 64, 32768
    W = L // w
    cache, ref, k, q_obs = make_kch(B, Hq, Hkv, w, L, 0.2, seed=92)
    wg = weights_both(cache, k, q_obs)
    route_kv_both(cache, ref, wg, synth.zipf_scores(92, 0, B, W))
    check_decode(cache, 0, ref, synth.queries(92, 0, 0, B, Hq, 128))


def test_k_channel_state_rules():
    B, Hq, Hkv, w, L = 1, 8, 2, 16, 512
    W = L // w
    cache, ref, k, q_obs = make_kch(B, Hq, Hkv, w, L, 0.3, seed=93)
    wg = cache.k_channel_weights(0, q_obs.cuda(), k.cuda())
    scores = synth.zipf_scores(93, 0, B, W).cuda()
    cache.route_rd_kv(0, wg, scores_override=scores)
    assert cache.status() == 0, cache.last_error()
    for call in (lambda: cache.route_rd_kv(0, wg, scores_override=scores),
                 lambda: cache.route_rd_mixed(0, scores_override=scores),
                 lambda: cache.set_tiers(0, torch.zeros(B, W, dtype=torch.uint8, device="cuda"))):
        with pytest.raises(binding.QevictError) as e:
            call()
        assert e.value.code == 4   # STATE
    # a layer quantised before: the device refuses (STATE in the status word)
    other, _, k2, q2 = make_kch(B, Hq, Hkv, w, L, 0.3, seed=94)
    other.route_rd_mixed(0, scores_override=scores)
    assert other.status() == 0, other.last_error()
    other.route_rd_kv(0, other.k_channel_weights(0, q2.cuda(), k2.cuda()), scores_override=scores)
    assert binding.STATUS[other.status()] == "STATE"
    # keys that do not start on a 16-byte boundary (the kernel reads rows in 16-byte pieces)
    kk = torch.empty(k.numel() + 8, dtype=k.dtype, device="cuda")[1:1 + k.numel()].view(k.shape)
    kk.copy_(k.cuda())
    with pytest.raises(binding.QevictError) as e:
        cache.k_channel_weights(0, q_obs.cuda(), kk)
    assert e.value.code == 1   # INVALID_ARG
    # caches that cannot hold K-channel tiles
    int2 = binding.TieredCache(B, 1, Hq, Hkv, w, L, budget_frac=0.3)
    with pytest.raises(binding.QevictError) as e:
        int2.route_rd_kv(0, wg, scores_override=scores)
    assert e.value.code == 1   # INVALID_ARG
