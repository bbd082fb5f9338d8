"""Splits with more claims than the descriptor table holds (1024 per split in
shared memory; later claims are computed when they are taken) and more
windows than the tail has mass threads (128; later windows are taken in
turn). That needs one split per (sequence, KV head), i.e. at least 152
pairs, and over 1024 kept windows per sequence: 152 sequences of one KV head
and one query head, 1500 windows of 16 tokens, 30 % of the bytes kept.

Sequences are independent (each has its own budget, tiers and scores), so
the oracle checks three of them, fed exactly the GPU's inputs for those
sequences. Bit-exact: tiers, stored bf16, ledger codes and meta; outputs and
masses within the attention tolerance."""
import numpy as np
import pytest
import torch

import oracle as O
from tiered_kv_cache_decode_gb300 import binding, synth
from parity_util import close

pytestmark = pytest.mark.gpu

B, HQ, HKV, W_TOK, N_WIN, BETA = 152, 1, 1, 16, 1500, 0.3
L = W_TOK * N_WIN
PICK = [0, 77, 151]


@pytest.fixture(autouse=True, scope="module")
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_decode_gb300 import build
    build.build()
    binding.load()


def sub_state(cache, ref, rows):
    """Tiers and stored windows of the picked sequences against the oracle."""
    tier, fps, lgs, lw = cache.tables(0)
    lbits = cache.ledger_bits(0).numpy()
    for j, b in enumerate(rows):
        assert np.array_equal(tier[b].numpy(), ref.tiers()[j]), ("tiers", b)
        for wi, win in enumerate(ref.win[j]):
            if win.tier == O.TIER_E:
                continue
            if win.tier == O.TIER_FP:
                data = cache.fp_window(0, int(fps[b, wi])).float().numpy()
                assert np.array_equal(data[:, 0, :win.ntok], win.k[:, :win.ntok]), ("FP K", b, wi)
                assert np.array_equal(data[:, 1, :win.ntok], win.v[:, :win.ntok]), ("FP V", b, wi)
            if win.ledger is not None:
                codes, scale, mn = cache.ledger_window(0, int(lgs[b, wi]), int(lbits[b, wi]))
                ck, sk, mk, cv, sv, mv = win.ledger
                assert np.array_equal(codes[:, 0].numpy(), ck), ("K codes", b, wi)
                assert np.array_equal(codes[:, 1].numpy(), cv), ("V codes", b, wi)
                assert np.array_equal(scale[:, 0].numpy().view(np.uint16), sk.view(np.uint16)), ("K scale", b, wi)
                assert np.array_equal(mn[:, 0].numpy().view(np.uint16), mk.view(np.uint16)), ("K min", b, wi)
                assert np.array_equal(scale[:, 1].numpy().view(np.uint16), sv.view(np.uint16)), ("V scale", b, wi)
                assert np.array_equal(mn[:, 1].numpy().view(np.uint16), mv.view(np.uint16)), ("V min", b, wi)


def inputs(seed):
    k, v = synth.kv_tokens(seed, 0, B, 0, L, HKV, 128, "heavy", device="cuda")
    scores = synth.zipf_scores(seed, 0, B, N_WIN)
    return k, v, scores


def decode_both(cache, ref, seed, step):
    q = synth.queries(seed, 0, step, B, HQ, 128)
    out, mass = cache.decode(0, q.cuda())
    torch.cuda.synchronize()
    ro, rm = ref.decode(q[PICK].float().numpy())
    close(out[PICK].cpu().numpy(), ro, "attention output")
    close(mass[PICK].cpu().numpy(), rm, "window mass")
    assert cache.status() == 0, cache.last_error()


def test_int2_split_beyond_descriptor_table():
    seed = 41
    cache = binding.TieredCache(B, 1, HQ, HKV, W_TOK, L, budget_frac=BETA)
    k, v, scores = inputs(seed)
    cache.prefill(0, k, v, scores=scores.cuda())
    ref = O.OracleCache(len(PICK), HQ, HKV, 128, W_TOK, beta=BETA)
    ref.prefill(k[PICK].float().cpu().numpy(), v[PICK].float().cpu().numpy(), scores=scores[PICK].numpy())
    assert cache.status() == 0, cache.last_error()
    kept = (ref.tiers() != O.TIER_E).sum(axis=1)
    assert kept.min() > 1024, kept   # more claims than the table holds, more windows than mass threads
    sub_state(cache, ref, PICK)
    for step in range(2):
        decode_both(cache, ref, seed, step)


def test_wide_split_beyond_descriptor_table():
    seed = 42
    cache = binding.TieredCache(B, 1, HQ, HKV, W_TOK, L, budget_frac=BETA, max_ledger_bits=8,
                                fp_capacity=N_WIN, ledger_capacity=N_WIN)
    k, v, scores = inputs(seed)
    t0 = torch.zeros(B, N_WIN, dtype=torch.uint8)
    cache.prefill(0, k, v, tiers=t0.cuda())
    cache.route_rd_mixed(0, scores_override=scores.cuda())
    ref = O.OracleCache(len(PICK), HQ, HKV, 128, W_TOK, beta=BETA)
    ref.prefill(k[PICK].float().cpu().numpy(), v[PICK].float().cpu().numpy(), tiers=t0[PICK].numpy())
    O.route_rd_mixed(ref, scores_override=scores[PICK].numpy(), max_bits=8)
    assert cache.status() == 0, cache.last_error()
    t = ref.tiers()
    assert (t != O.TIER_E).sum(axis=1).min() > 1024
    assert (t == O.TIER_Q4).any()
    sub_state(cache, ref, PICK)
    for step in range(2):
        decode_both(cache, ref, seed, step)
