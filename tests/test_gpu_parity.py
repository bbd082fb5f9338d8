"""CUDA path against the CPU oracle, through the C ABI, on the same seeded inputs.

Bit-exact: tiers, stored bf16 windows, INT2 codes, fp16 scale/min, ledger
write counts, transition statistics. Within max|d| <= 2e-3 and relative L2 <=
1e-3: attention outputs, window masses, cumulative scores.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import check_decode, check_state, check_stats, close, make_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def test_tiny_decode_step_drawn_tiers():
    """Batch 1, 8/2 heads, 2048 tokens in 64 windows of 32, 16 FP / 32 INT2 / 16 evicted."""
    W = 64
    tiers = synth.drawn_tiers(0, 0, 1, W, 16, 32)
    cache, (ref,) = make_pair(1, 8, 2, 32, 2048, outliers="tiny", tiers=[tiers],
                              fp_capacity=W, ledger_capacity=W)
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(0, 0, 0, 1, 8, 128))
    check_stats(cache, [ref])


@pytest.mark.parametrize("B,Hq,Hkv,w,L", [(1, 8, 2, 32, 1000), (2, 32, 8, 64, 777), (3, 28, 4, 16, 333),
                                           (1, 4, 4, 128, 129), (2, 8, 1, 64, 1)])
def test_all_full_precision_matches_oracle(B, Hq, Hkv, w, L):
    W = -(-L // w)
    tiers = torch.zeros(B, W, dtype=torch.uint8)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, tiers=[tiers], fp_capacity=W, ledger_capacity=1)
    check_state(cache, 0, ref)
    for step in range(2):
        check_decode(cache, 0, ref, synth.queries(1, 0, step, B, Hq, 128))


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [(1, 32, 8, 64, 4096, 0.2), (2, 28, 4, 64, 3000, 0.1),
                                                (4, 32, 8, 32, 2048, 0.05), (1, 8, 2, 128, 5000, 0.2)])
def test_prefill_routing_quantises_and_attends(B, Hq, Hkv, w, L, beta):
    W = -(-L // w)
    scores = synth.zipf_scores(3, 0, B, W)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, scores=[scores])
    check_state(cache, 0, ref)
    t = ref.tiers()
    assert (t == O.TIER_Q).any() and (t == O.TIER_E).any()
    check_decode(cache, 0, ref, synth.queries(3, 0, 0, B, Hq, 128))
    check_stats(cache, [ref])


def test_quantiser_edge_groups_bit_exact():
    """Constant groups, exact grids, tiny (fp16-subnormal) values and heavy outliers."""
    B, Hkv, w, L = 1, 2, 16, 64
    k, v = synth.kv_tokens(5, 0, B, 0, L, Hkv, 128, "heavy")
    k = k.clone()
    v = v.clone()
    k[0, 0:16, 0, :32] = 0.75                          # constant group
    k[0, 0:16, 1, 32:64] = torch.tensor([-1, -0.5, 0, 0.5] * 8, dtype=torch.bfloat16)   # exact grid
    v[0, 16:32, 0, :] = (v[0, 16:32, 0, :].float() * 1e-5 + 1e-5).to(torch.bfloat16)  # subnormal range
    v[0, 32:48, 1, 64:96] = (v[0, 32:48, 1, 64:96].float() * 300).to(torch.bfloat16)   # wide range
    k[0, 16:32, 1, 96:128] = (k[0, 16:32, 1, 96:128].float() * 30).to(torch.bfloat16)    # wide keys
    k[0, 32:48, 0, 0:32] = (k[0, 32:48, 0, 0:32].float() * 300).to(torch.bfloat16)       # very wide keys
    tiers = torch.tensor([[1, 1, 1, 0]], dtype=torch.uint8)
    cache = binding.TieredCache(B, 1, 4, Hkv, w, L, fp_capacity=4, ledger_capacity=4)
    cache.prefill(0, k.cuda(), v.cuda(), tiers=tiers.cuda())
    ref = O.OracleCache(B, 4, Hkv, 128, w)
    ref.prefill(k.float().numpy(), v.float().numpy(), tiers=tiers.numpy())
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(5, 0, 0, B, 4, 128))


def test_quantiser_flags_nonfinite_and_fp16_overflow_on_the_gpu():
    """Groups holding +inf or -inf, a range whose step passes fp16 and a
    minimum below -65504: the quantiser sets DEVICE in the status word and
    stores each such group as zero codes with a zero scale and minimum. Every
    other group is quantised exactly as the oracle quantises it."""
    B, Hkv, w, L = 1, 2, 16, 64
    k, v = synth.kv_tokens(15, 0, B, 0, L, Hkv, 128, "heavy")
    k = k.clone()
    v = v.clone()
    k[0, 3, 0, 5] = float("inf")          # window 0, KV head 0, token 3, group 0
    v[0, 7, 1, 40] = -float("inf")        # window 0, KV head 1, token 7, group 1
    v[0, 9, 0, 70] = 3e5                  # window 0, group 2: (max - min) / 3 passes 65504
    k[0, 2, 1, 96:128] = -7e4             # window 0, group 3: the minimum passes -65504
    k[0, 20, 1, 64] = float("inf")        # window 1, KV head 1, token 4, group 2
    tiers = torch.tensor([[1, 1, 0, 0]], dtype=torch.uint8)
    cache = binding.TieredCache(B, 1, 4, Hkv, w, L, fp_capacity=4, ledger_capacity=4)
    cache.prefill(0, k.cuda(), v.cuda(), tiers=tiers.cuda())
    torch.cuda.synchronize()
    assert binding.STATUS[cache.status()] == "DEVICE"
    tier, _, lgs, _ = cache.tables(0)
    assert tier[0].tolist() == [1, 1, 0, 0]
    n_bad = 0
    for wi in range(2):
        codes, scale, mn = cache.ledger_window(0, int(lgs[0, wi]), 2)
        for kv, x in enumerate((k, v)):
            xs = x[0, wi * w:(wi + 1) * w].float().numpy().transpose(1, 0, 2)    # [Hkv][w][d]
            ec, es, em, bad = O.quantize_groups(xs.reshape(Hkv, w, 4, 32))
            ec = np.where(bad[..., None], 0, ec).reshape(Hkv, w, 128)
            es = np.where(bad, np.float16(0), es)
            em = np.where(bad, np.float16(0), em)
            n_bad += int(bad.sum())
            assert np.array_equal(codes[:, kv].numpy(), ec), ("codes", wi, kv)
            assert np.array_equal(scale[:, kv].numpy().view(np.uint16), es.view(np.uint16)), ("scale", wi, kv)
            assert np.array_equal(mn[:, kv].numpy().view(np.uint16), em.view(np.uint16)), ("min", wi, kv)
    assert n_bad == 5
    cache.clear_status()
    assert cache.status() == 0


def test_ledger_write_once_through_cycles():
    B, Hq, Hkv, w, L = 2, 8, 2, 32, 320
    W = L // w
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, tiers=[torch.zeros(B, W, dtype=torch.uint8)],
                              fp_capacity=W, ledger_capacity=W)
    pairs = torch.tensor([[0, 1], [1, 3], [0, 4], [1, 0]], dtype=torch.int32)
    for cycle in range(3):
        cache.demote(0, pairs.cuda())
        ref.demote(pairs.tolist())
        check_state(cache, 0, ref)
        check_decode(cache, 0, ref, synth.queries(6, 0, cycle, B, Hq, 128), accumulate=False)
        cache.promote(0, pairs.cuda())
        ref.promote(pairs.tolist())
        check_state(cache, 0, ref)
    check_stats(cache, [ref])
    s = cache.stats()
    assert s["ledger_writes"] == 4 and s["ledger_reuses"] == 8


def test_multistep_appends_decodes_routes_teacher_forced():
    """Appends, decode steps with score accumulation and routing events with drift.
    At each routing event the oracle routes on the GPU's scores (teacher forcing)
    after the GPU scores are checked against the oracle's."""
    B, Hq, Hkv, w, L0, beta = 2, 32, 8, 64, 2048, 0.25
    steps, every = 160, 32
    W0 = L0 // w
    scores = synth.zipf_scores(7, 0, B, W0)
    maxc = L0 + steps
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L0, beta=beta, scores=[scores], max_context=maxc, seed=7)
    check_state(cache, 0, ref)
    for step in range(steps):
        kn, vn = synth.kv_tokens(7, 0, B, L0 + step, 1, Hkv, 128)
        cache.append(0, kn.cuda(), vn.cuda())
        ref.append(kn.float().numpy(), vn.float().numpy())
        check_decode(cache, 0, ref, synth.queries(7, 0, step, B, Hq, 128))
        if step % every == every - 1:
            gs = cache.scores(0).cpu().numpy()
            close(gs, np.stack(ref.S), "cumulative scores")
            drift = synth.drift_factors(7, 0, step, B, cache.num_windows(0))
            cache.route(0, score_mult=drift.cuda())
            forced = (gs.astype(np.float32) * drift.numpy()).astype(np.float64)
            ref.route(scores_override=np.asarray(cache.scores(0).cpu().numpy(), np.float64))
            # the GPU scores after the event are its pre-event scores times the drift
            assert np.array_equal(cache.scores(0).cpu().numpy().astype(np.float64), forced)
            check_state(cache, 0, ref)
    check_stats(cache, [ref])
    assert cache.stats()["promotions"] > 0


def test_full_size_llama_b1_32k_20pct_one_layer():
    """The full-size Llama-3.1-8B-shaped layer: 32/8 heads, 32768 tokens, 64-token windows, 20 %."""
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 64, 32768, 0.2
    W = L // w
    scores = synth.zipf_scores(0, 0, B, W)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, scores=[scores])
    t = ref.tiers()
    assert ((t == 0).sum(), (t == 1).sum(), (t == 2).sum()) == (51, 274, 187)
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(0, 0, 0, B, Hq, 128))


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [
    (8, 32, 8, 64, 32768, 0.05),    # Llama-8B-shaped batch 8: 64 (sequence, KV head) pairs, 2 splits each
    (16, 28, 4, 64, 16384, 0.10),   # Qwen-7B-shaped batch 16: G = 7, 64 pairs
    (4, 32, 8, 32, 8192, 0.20),     # a Mistral-7B-shaped sweep point: 32-token windows
])
def test_full_size_batched_workloads_one_layer(B, Hq, Hkv, w, L, beta):
    """One full-size layer of the batched workloads, decoded twice (the second
    decode follows the first on the same scratch, so stale records from the
    first must not be taken for the second's)."""
    W = L // w
    scores = synth.zipf_scores(5, 0, B, W)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, scores=[scores], seed=5)
    t = ref.tiers()
    assert (t == O.TIER_Q).any() and (t == O.TIER_E).any()
    check_state(cache, 0, ref)
    for step in range(2):
        check_decode(cache, 0, ref, synth.queries(5, 0, step, B, Hq, 128))


@pytest.mark.parametrize("B,Hq,Hkv,w,L,beta", [
    (2, 64, 8, 48, 3000, 0.2),     # G = 8, windows of 3 units
    (1, 8, 8, 80, 2000, 0.3),      # G = 1, windows of 5 units
    (3, 12, 4, 112, 1500, 0.25),   # G = 3, windows of 7 units
    (2, 20, 4, 96, 2500, 0.15),    # G = 5, windows of 6 units
])
def test_uneven_windows_and_group_sizes(B, Hq, Hkv, w, L, beta):
    """Window sizes whose unit count is not a power of two, and group sizes
    from 1 to 8, through routing, decode and a fused decode step."""
    W = -(-L // w)
    scores = synth.zipf_scores(9, 0, B, W)
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, scores=[scores], max_context=L + 8, seed=9)
    t = ref.tiers()
    assert (t == O.TIER_Q).any()
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(9, 0, 0, B, Hq, 128))
    k, v = synth.kv_tokens(9, 0, B, L, 1, Hkv, 128, "heavy")
    q = synth.queries(9, 0, 1, B, Hq, 128)
    out, mass = cache.decode_step(0, q.cuda(), k[:, 0].cuda(), v[:, 0].cuda())
    torch.cuda.synchronize()
    ref.append(k.float().numpy(), v.float().numpy())
    ro, rm = ref.decode(q.float().numpy())
    close(out.cpu().numpy(), ro, "decode step output")
    close(mass.cpu().numpy(), rm, "decode step mass")
    assert cache.status() == 0, cache.last_error()


def test_layers_route_concurrently_on_separate_streams():
    """Routing events of different layers share no state: routed side by side
    on their own streams they give exactly the sequential result."""
    B, Hq, Hkv, w, L, layers = 2, 16, 4, 64, 2048, 4
    W = L // w
    scores = [synth.zipf_scores(7, l, B, W) for l in range(layers)]
    cache, refs = make_pair(B, Hq, Hkv, w, L, layers=layers, beta=0.5, scores=scores)
    new_scores = [synth.zipf_scores(8, l, B, W) for l in range(layers)]
    streams = [torch.cuda.Stream() for _ in range(layers)]
    torch.cuda.synchronize()
    for l in range(layers):
        with torch.cuda.stream(streams[l]):
            cache.route(l, scores_override=new_scores[l].cuda(), stream=streams[l])
    torch.cuda.synchronize()
    assert cache.status() == 0, cache.last_error()
    for l in range(layers):
        refs[l].route(scores_override=new_scores[l].numpy())
        check_state(cache, l, refs[l])
        check_decode(cache, l, refs[l], synth.queries(8, l, 0, B, Hq, 128))
    check_stats(cache, refs)


def test_device_errors_set_status_without_faulting():
    B, Hq, Hkv, w, L = 1, 8, 2, 32, 100
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, tiers=[torch.zeros(B, 4, dtype=torch.uint8)],
                              fp_capacity=6, ledger_capacity=1)
    # demoting the partially filled last window is illegal
    cache.demote(0, torch.tensor([[0, 3]], dtype=torch.int32).cuda())
    assert binding.STATUS[cache.status()] == "STATE"
    cache.clear_status()
    # two first demotions with a single ledger slot: the second runs out of capacity
    cache.demote(0, torch.tensor([[0, 0], [0, 1]], dtype=torch.int32).cuda())
    assert binding.STATUS[cache.status()] == "CAPACITY"
    cache.clear_status()
    # evicted windows cannot come back
    cache.set_tiers(0, torch.tensor([[2, 1, 0, 0]], dtype=torch.uint8).cuda())
    assert cache.status() == 0
    cache.set_tiers(0, torch.tensor([[0, 1, 0, 0]], dtype=torch.uint8).cuda())
    assert binding.STATUS[cache.status()] == "STATE"
    cache.clear_status()
    # a non-finite score among the candidates
    bad = torch.tensor([[1.0, float("nan"), 0.5, 0.1]]).cuda()
    cache.route(0, scores_override=bad)
    assert binding.STATUS[cache.status()] == "DEVICE"
    cache.clear_status()
    # host-side: budget too small for the open window
    small = binding.TieredCache(1, 1, 8, 2, 32, 64, budget_frac=0.05)
    small.append(0, *[x.cuda() for x in synth.kv_tokens(0, 0, 1, 0, 64, 2, 128)])
    with pytest.raises(binding.QevictError) as ei:
        small.route(0)
    assert ei.value.name == "BUDGET"


def test_decode_step_fused_append_matches_oracle_over_layers():
    """decode_step (append one token + attention, one launch) on 3 interleaved layers,
    so consecutive launches touch different layers (the programmatic-launch path);
    windows open along the way and a routing event runs in between."""
    B, Hq, Hkv, w, L0, beta, NL = 2, 28, 4, 32, 1000, 0.3, 3
    W0 = -(-L0 // w)
    steps = 70
    scores = [synth.zipf_scores(11, l, B, W0) for l in range(NL)]
    cache, refs = make_pair(B, Hq, Hkv, w, L0, layers=NL, beta=beta, scores=scores, max_context=L0 + steps,
                            seed=11)
    for step in range(steps):
        for l in range(NL):
            kn, vn = synth.kv_tokens(11, l, B, L0 + step, 1, Hkv, 128)
            q = synth.queries(11, l, step, B, Hq, 128)
            out, mass = cache.decode_step(l, q.cuda(), kn[:, 0].contiguous().cuda(), vn[:, 0].contiguous().cuda())
            refs[l].append(kn.float().numpy(), vn.float().numpy())
            ro, rm = refs[l].decode(q.float().numpy())
            torch.cuda.synchronize()
            close(out.cpu().numpy(), ro, f"out layer {l} step {step}")
            close(mass.cpu().numpy(), rm, f"mass layer {l} step {step}")
        if step == 40:
            for l in range(NL):
                cache.route(l)
                refs[l].route(scores_override=np.asarray(cache.scores(l).cpu().numpy(), np.float64))
            assert cache.status() == 0, cache.last_error()
            for l in range(NL):
                check_state(cache, l, refs[l])
    assert cache.status() == 0, cache.last_error()
    for l in range(NL):
        close(cache.scores(l).cpu().numpy(), np.stack(refs[l].S), f"scores layer {l}")
        check_state(cache, l, refs[l])
    check_stats(cache, refs)


def test_decode_step_on_empty_layer_and_window_edges():
    B, Hq, Hkv, w = 1, 8, 2, 16
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, 64, budget_frac=1.0, fp_capacity=8, ledger_capacity=2)
    ref = O.OracleCache(B, Hq, Hkv, 128, w)
    for step in range(40):     # from an empty layer across two window boundaries
        kn, vn = synth.kv_tokens(13, 0, B, step, 1, Hkv, 128)
        q = synth.queries(13, 0, step, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].contiguous().cuda(), vn[:, 0].contiguous().cuda())
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        torch.cuda.synchronize()
        close(out.cpu().numpy(), ro, f"out step {step}")
        close(mass.cpu().numpy(), rm, f"mass step {step}")
    assert cache.status() == 0, cache.last_error()
    check_state(cache, 0, ref)


def test_graph_replay_advances_device_length():
    """A CUDA graph of fused decode steps over two layers, replayed N times, equals N eager steps."""
    B, Hq, Hkv, w, L0, NL = 1, 8, 2, 32, 200, 2
    W = -(-L0 // w)
    steps = 40
    cache, refs = make_pair(B, Hq, Hkv, w, L0, layers=NL, tiers=[torch.zeros(B, W, dtype=torch.uint8)] * NL,
                            max_context=L0 + steps + 1, fp_capacity=16, ledger_capacity=4)
    kbuf = [torch.empty(B, Hkv, 128, dtype=torch.bfloat16, device="cuda") for _ in range(NL)]
    vbuf = [torch.empty_like(kbuf[0]) for _ in range(NL)]
    qbuf = [torch.empty(B, Hq, 128, dtype=torch.bfloat16, device="cuda") for _ in range(NL)]
    out = [torch.empty(B, Hq, 128, dtype=torch.float32, device="cuda") for _ in range(NL)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    cache.set_launch_overlap(True)   # layer 1's decode follows layer 0's decode kernel in the graph
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for l in range(NL):
                cache.decode_step(l, qbuf[l], kbuf[l], vbuf[l], out=out[l], want_mass=False, stream=s)
    torch.cuda.synchronize()
    for step in range(steps):
        for l in range(NL):
            kn, vn = synth.kv_tokens(9, l, B, L0 + step, 1, Hkv, 128)
            q = synth.queries(9, l, step, B, Hq, 128)
            kbuf[l].copy_(kn[:, 0])
            vbuf[l].copy_(vn[:, 0])
            qbuf[l].copy_(q)
        g.replay()
        torch.cuda.synchronize()
        for l in range(NL):
            kn, vn = synth.kv_tokens(9, l, B, L0 + step, 1, Hkv, 128)
            q = synth.queries(9, l, step, B, Hq, 128)
            refs[l].append(kn.float().numpy(), vn.float().numpy())
            ro, _ = refs[l].decode(q.float().numpy())
            close(out[l].cpu().numpy(), ro, f"graph step {step} layer {l}")
    cache.refresh_lengths()
    assert cache.length(0) == L0 + steps
    assert cache.status() == 0
    for l in range(NL):
        close(cache.scores(l).cpu().numpy(), np.stack(refs[l].S), "scores after graph replays")
        check_state(cache, l, refs[l])


@pytest.mark.parametrize("L", [1000, 1001, 1015, 1017])
def test_stale_rows_of_open_window_never_reach_the_output(L):
    """The slot of a partially filled window keeps whatever its rows held before.
    Poison the whole full-precision pool with NaN first: attention must still
    equal the oracle's over the tokens that exist."""
    B, Hq, Hkv, w = 2, 16, 4, 16
    W = -(-L // w)
    cache = binding.TieredCache(B, 1, Hq, Hkv, w, L + 40, fp_capacity=W + 8, ledger_capacity=W)
    v = cache.view(0)
    pool = binding.device_tensor(v.fp_pool, (B * v.fp_capacity * v.fp_slot_bytes // 2,), "<i2")
    pool.fill_(-1)                                         # 0xFFFF: a bf16 NaN in every row
    torch.cuda.synchronize()
    k, vv = synth.kv_tokens(17, 0, B, 0, L, Hkv, 128)
    tiers = torch.zeros(B, W, dtype=torch.uint8)
    tiers[:, : W // 3] = 1
    cache.prefill(0, k.cuda(), vv.cuda(), tiers=tiers.cuda())
    ref = O.OracleCache(B, Hq, Hkv, 128, w)
    ref.prefill(k.float().numpy(), vv.float().numpy(), tiers=tiers.numpy())
    check_decode(cache, 0, ref, synth.queries(17, 0, 0, B, Hq, 128))
    for step in range(20):
        kn, vn = synth.kv_tokens(17, 0, B, L + step, 1, Hkv, 128)
        q = synth.queries(17, 0, step + 1, B, Hq, 128)
        out, mass = cache.decode_step(0, q.cuda(), kn[:, 0].contiguous().cuda(), vn[:, 0].contiguous().cuda())
        ref.append(kn.float().numpy(), vn.float().numpy())
        ro, rm = ref.decode(q.float().numpy())
        torch.cuda.synchronize()
        close(out.cpu().numpy(), ro, f"out step {step}")
        close(mass.cpu().numpy(), rm, f"mass step {step}")
    assert cache.status() == 0


def test_max_windows_128k_context_every_router():
    """The largest table a sequence can have: 131,072 tokens in 32-token
    windows (4,096 windows, the size the plan kernel sorts and the 12 age bits
    of the log-sparse rank), Mistral-7B-shaped heads, 10 % budget. Score,
    log-sparse and rate-distortion routes over all of it."""
    B, Hq, Hkv, w, L, beta = 1, 32, 8, 32, 131072, 0.1
    W = L // w
    cache, (ref,) = make_pair(B, Hq, Hkv, w, L, beta=beta, scores=[synth.zipf_scores(70, 0, B, W)], seed=70,
                              fp_capacity=W, ledger_capacity=W)
    t = ref.tiers()
    assert t.shape[1] == 4096 and (t == O.TIER_Q).any() and (t == O.TIER_E).any()
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(70, 0, 0, B, Hq, 128))
    sc = synth.zipf_scores(71, 0, B, W)
    cache.route(0, scores_override=sc.cuda())
    ref.route(scores_override=sc.numpy())
    check_state(cache, 0, ref)
    cache.route_logsparse(0, recent=2)
    O.route_logsparse(ref, recent=2)
    check_state(cache, 0, ref)
    sc = synth.zipf_scores(72, 0, B, W)
    cache.route_rd(0, scores_override=sc.cuda())
    O.route_rd(ref, scores_override=sc.numpy())
    check_state(cache, 0, ref)
    check_decode(cache, 0, ref, synth.queries(70, 0, 1, B, Hq, 128))
    check_stats(cache, [ref])
