"""CPU-side checks of the C ABI: the library builds, loads and exports every
function include/qevict.h declares, and host-side argument checks answer
without touching a GPU."""
import ctypes
import os
import re

import pytest

from tiered_kv_cache_decode_gb300 import binding
from tiered_kv_cache_decode_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return binding.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "qevict.h")).read()
    return sorted(set(re.findall(r"\b(qevict_[a-z_]+)\s*\(", text)))


def test_header_declares_what_binding_exports():
    assert _declared() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_struct_layouts_match_header_sizes():
    # int32 x 10 + double x 2 + int32 x 2 = 64 bytes
    assert ctypes.sizeof(binding.Config) == 64
    assert binding.Config.tier_per_kv_head.offset == 56 and binding.Config.max_ledger_bits.offset == 60
    assert ctypes.sizeof(binding.Stats) == 48
    # 9 int32, padding, 3 int64, 7 pointers, int32 and padding, the K group widths pointer
    assert ctypes.sizeof(binding.View) == 9 * 4 + 4 + 3 * 8 + 7 * 8 + 8 + 8
    assert binding.View.k_group_bits.offset == 128


def _cfg(**kw):
    base = dict(batch=1, num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=128, window=32,
                max_context=2048, fp_capacity=0, ledger_capacity=0, fp_slack=0,
                budget_frac=0.2, fp_share=0.5)
    base.update(kw)
    return binding.Config(**base)


@pytest.mark.parametrize("bad", [dict(head_dim=64), dict(window=24), dict(window=256),
                                 dict(num_q_heads=9), dict(num_q_heads=32, num_kv_heads=2),
                                 dict(budget_frac=0.0), dict(budget_frac=1.5), dict(fp_share=0.0),
                                 dict(batch=0), dict(max_context=0), dict(max_context=4096 * 32 + 1)])
def test_create_rejects_bad_config_on_host(lib, bad):
    h = ctypes.c_void_p()
    rc = lib.qevict_cache_create(ctypes.byref(_cfg(**bad)), None, None, ctypes.byref(h))
    assert rc == 1, (bad, rc)
    assert not h.value
    assert lib.qevict_last_error()


def test_calls_on_null_cache_fail_cleanly(lib):
    assert lib.qevict_decode_attention(None, 0, None, None, None, 0, None) == 1
    assert lib.qevict_route(None, 0, None, None, None) == 1
    assert lib.qevict_length(None, 0) == -1
    assert lib.qevict_cache_destroy(None) == 1


@pytest.mark.parametrize("fail_at", [0, 1, 2, 3])
def test_failing_allocator_reports_oom_and_frees_everything(lib, fail_at):
    """Host-side fault injection: the allocator returns NULL on its n-th call."""
    live, calls = set(), [0]

    def _a(size, stream, ctx):
        i = calls[0]
        calls[0] += 1
        if i == fail_at:
            return None
        p = 0x10000000 + 0x100000 * i
        live.add(p)
        return p

    def _f(ptr, stream, ctx):
        live.remove(ptr)

    al = binding.Allocator(binding.ALLOC_FN(_a), binding.FREE_FN(_f), None)
    h = ctypes.c_void_p()
    rc = lib.qevict_cache_create(ctypes.byref(_cfg(num_layers=4)), ctypes.byref(al), None, ctypes.byref(h))
    assert rc == 2 and not h.value
    assert calls[0] == fail_at + 1
    assert not live


@pytest.mark.parametrize("Hkv,w,maxc,beta,rho", [(8, 64, 32768 + 300, 0.20, 0.5), (8, 64, 32768 + 300, 0.05, 0.5),
                                                 (4, 64, 16640, 0.10, 0.5), (4, 32, 1070, 0.30, 0.5),
                                                 (8, 32, 8192 + 64, 0.05, 0.5), (8, 128, 8192 + 64, 0.05, 0.3),
                                                 (2, 16, 3000, 0.6, 0.8), (8, 64, 131072, 0.2, 0.5)])
def test_pool_capacity_covers_every_routing_event(lib, Hkv, w, maxc, beta, rho):
    """Brute force over every context length: the routed tier counts of the oracle
    never exceed the pools the library sizes for the config."""
    import oracle as O
    cfg = _cfg(num_kv_heads=Hkv, num_q_heads=Hkv * 4, window=w, max_context=maxc, budget_frac=beta,
               fp_share=rho)
    cf, cq, nbytes = binding.pool_capacity(cfg)
    c_fp, c_q = O.window_costs(w, Hkv, 128)
    worst_fp = worst_led = 0
    for L in range(1, maxc + 1):
        if O.budget_bytes(L, Hkv, 128, beta) < c_fp:
            continue
        W = -(-L // w)
        n_fp, n_q = O.route_counts(W, L, w, Hkv, 128, beta, rho)
        worst_fp = max(worst_fp, n_fp)
        worst_led = max(worst_led, n_fp + n_q)
    assert worst_fp + 1 <= cf          # one more for the slot kept for the next window
    assert worst_led <= cq
    assert nbytes == cf * c_fp + cq * c_q


def test_per_head_pools_match_the_shared_pools(lib):
    """With per-head tiers a unit is one (sequence, KV head): its budget and
    window costs are the sequence's divided by Hkv, so it gets the shared
    mode's slot counts and the layer's pool bytes do not change."""
    out = []
    for per_head in (0, 1):
        cf, cq, nb = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        cfg = _cfg(batch=3, num_q_heads=32, num_kv_heads=8, window=64, max_context=32768, budget_frac=0.25,
                   tier_per_kv_head=per_head)
        assert lib.qevict_pool_capacity(ctypes.byref(cfg), ctypes.byref(cf), ctypes.byref(cq), ctypes.byref(nb)) == 0
        out.append((cf.value, cq.value, nb.value))
    assert out[0] == out[1]


def test_per_head_rejects_too_many_units(lib):
    h = ctypes.c_void_p()
    cfg = _cfg(batch=16384, num_q_heads=8, num_kv_heads=8, max_context=64, tier_per_kv_head=1)
    assert lib.qevict_cache_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == 1
    assert b"65535" in lib.qevict_last_error()
