"""The headline workload in the launch configuration bench.py times: the
Llama-3.1-8B-shaped cache (32 query / 8 KV heads, 32768 tokens, 64-token
windows, 20 % budget), non-cooperative grids with programmatic dependent
launch between layers, fused decode steps (append + decode + scores) captured
in one CUDA graph over the layers and replayed. Every layer's output after
every replay is checked against the oracle, and the tables, stored windows
and cumulative scores after the last."""
import numpy as np
import pytest
import torch

from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_state, close, make_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def test_headline_shape_graph_of_fused_steps_non_cooperative_with_overlap():
    B, Hq, Hkv, w, L0, beta, NL, steps = 1, 32, 8, 64, 32768, 0.2, 2, 3
    W = L0 // w
    seed = 11
    scores = [synth.zipf_scores(seed, l, B, W) for l in range(NL)]
    cache, refs = make_pair(B, Hq, Hkv, w, L0, layers=NL, beta=beta, scores=scores, max_context=L0 + steps,
                            seed=seed)
    cache.set_launch_overlap(True)
    cache.set_cooperative_launch(False)
    kbuf = [torch.empty(B, Hkv, 128, dtype=torch.bfloat16, device="cuda") for _ in range(NL)]
    vbuf = [torch.empty_like(kbuf[0]) for _ in range(NL)]
    qbuf = [torch.empty(B, Hq, 128, dtype=torch.bfloat16, device="cuda") for _ in range(NL)]
    out = [torch.empty(B, Hq, 128, dtype=torch.float32, device="cuda") for _ in range(NL)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for l in range(NL):
                cache.decode_step(l, qbuf[l], kbuf[l], vbuf[l], out=out[l], want_mass=False, accumulate=True,
                                  stream=s)
    torch.cuda.synchronize()
    for step in range(steps):
        for l in range(NL):
            kn, vn = synth.kv_tokens(seed, l, B, L0 + step, 1, Hkv, 128)
            kbuf[l].copy_(kn[:, 0])
            vbuf[l].copy_(vn[:, 0])
            qbuf[l].copy_(synth.queries(seed, l, step, B, Hq, 128))
        g.replay()
        torch.cuda.synchronize()
        for l in range(NL):
            kn, vn = synth.kv_tokens(seed, l, B, L0 + step, 1, Hkv, 128)
            refs[l].append(kn.float().numpy(), vn.float().numpy())
            ro, _ = refs[l].decode(synth.queries(seed, l, step, B, Hq, 128).float().numpy())
            close(out[l].cpu().numpy(), ro, f"replay {step} layer {l}")
    assert cache.status() == 0, cache.last_error()
    cache.refresh_lengths()
    for l in range(NL):
        assert cache.length(l) == L0 + steps
        close(cache.scores(l).cpu().numpy(), np.stack(refs[l].S), f"scores of layer {l}")
        check_state(cache, l, refs[l])


def test_mixed_width_shape_graph_of_decodes_non_cooperative_with_overlap():
    """The bench's mixed-width leg in its launch configuration: two 32K layers
    routed over widths {0, 2, 4, 8, 16}, decodes with score accumulation in one
    CUDA graph, replayed; outputs after each replay against the oracle."""
    import oracle as O
    B, Hq, Hkv, w, L0, beta, NL, reps = 1, 32, 8, 64, 32768, 0.2, 2, 2
    W = L0 // w
    seed = 12
    cache = binding.TieredCache(B, NL, Hq, Hkv, w, L0, budget_frac=beta, max_ledger_bits=8, fp_capacity=W,
                                ledger_capacity=W)
    cache.set_launch_overlap(True)
    cache.set_cooperative_launch(False)
    refs = []
    t0 = np.zeros((B, W), np.uint8)
    for l in range(NL):
        k, v = synth.kv_tokens(seed, l, B, 0, L0, Hkv, 128)
        cache.prefill(l, k.cuda(), v.cuda(), tiers=torch.from_numpy(t0).cuda())
        ref = O.OracleCache(B, Hq, Hkv, 128, w, beta=beta)
        ref.prefill(k.float().numpy(), v.float().numpy(), tiers=t0)
        sc = synth.zipf_scores(seed, l, B, W)
        cache.route_rd_mixed(l, scores_override=sc.cuda())
        O.route_rd_mixed(ref, scores_override=sc.numpy(), max_bits=8)
        refs.append(ref)
    assert cache.status() == 0, cache.last_error()
    assert any((r.tiers() == O.TIER_Q4).any() for r in refs)
    q = [synth.queries(seed, l, 0, B, Hq, 128).cuda() for l in range(NL)]
    out = [torch.empty(B, Hq, 128, dtype=torch.float32, device="cuda") for _ in range(NL)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for l in range(NL):
                cache.decode(l, q[l], out=out[l], want_mass=False, accumulate=True, stream=s)
    torch.cuda.synchronize()
    for r in range(reps):
        g.replay()
        torch.cuda.synchronize()
        for l in range(NL):
            ro, _ = refs[l].decode(q[l].cpu().float().numpy())
            close(out[l].cpu().numpy(), ro, f"replay {r} layer {l}")
    assert cache.status() == 0, cache.last_error()
    for l in range(NL):
        close(cache.scores(l).cpu().numpy(), np.stack(refs[l].S), f"scores of layer {l}")
        check_state(cache, l, refs[l])
