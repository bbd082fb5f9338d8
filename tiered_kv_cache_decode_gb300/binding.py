"""Thin ctypes binding over the C ABI in include/qevict.h (libqevict.so).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the ABI. PyTorch supplies device memory (through the
allocator callbacks, or the caller's tensors) and the current stream. There
is no fallback: if the shared library is missing or a call fails, a Python
exception says so.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqevict.so")

TIER_FP, TIER_Q, TIER_E = 0, 1, 2
HEAD_DIM = 128

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "OUT_OF_MEMORY", 3: "BUDGET", 4: "STATE", 5: "CUDA",
          6: "TIMEOUT", 7: "DEVICE", 8: "CAPACITY"}

# every function the header declares
EXPORTS = ["qevict_pool_capacity", "qevict_cache_create", "qevict_cache_destroy", "qevict_prefill", "qevict_append_kv",
           "qevict_decode_attention", "qevict_decode_step", "qevict_route", "qevict_demote_quantize",
           "qevict_promote_dequantize", "qevict_set_tiers", "qevict_get_scores", "qevict_get_view",
           "qevict_get_status", "qevict_clear_status", "qevict_get_stats", "qevict_set_launch_overlap",
           "qevict_set_wait_limit", "qevict_set_cooperative_launch",
           "qevict_refresh_lengths", "qevict_decode_attention_static_scratch",
           "qevict_get_tier_move_counts", "qevict_future_missed_mass", "qevict_route_global", "qevict_route_logsparse", "qevict_route_rd",
           "qevict_route_rd_mixed", "qevict_k_channel_weights", "qevict_route_rd_kv",
           "qevict_length",
           "qevict_last_error"]


class QevictError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code
        self.name = STATUS.get(code, str(code))


class Config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32),
                ("max_context", ctypes.c_int32), ("fp_capacity", ctypes.c_int32),
                ("ledger_capacity", ctypes.c_int32), ("fp_slack", ctypes.c_int32),
                ("budget_frac", ctypes.c_double), ("fp_share", ctypes.c_double),
                ("tier_per_kv_head", ctypes.c_int32), ("max_ledger_bits", ctypes.c_int32)]


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)


class Allocator(ctypes.Structure):
    _fields_ = [("alloc", ALLOC_FN), ("free", FREE_FN), ("ctx", ctypes.c_void_p)]


class View(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("window", ctypes.c_int32), ("max_windows", ctypes.c_int32),
                ("num_windows", ctypes.c_int32), ("fp_capacity", ctypes.c_int32),
                ("ledger_capacity", ctypes.c_int32), ("length", ctypes.c_int64),
                ("fp_slot_bytes", ctypes.c_int64), ("ledger_slot_bytes", ctypes.c_int64),
                ("tier", ctypes.c_void_p), ("fp_slot", ctypes.c_void_p),
                ("ledger_slot", ctypes.c_void_p), ("ledger_writes", ctypes.c_void_p),
                ("fp_pool", ctypes.c_void_p), ("ledger_pool", ctypes.c_void_p),
                ("ledger_bits", ctypes.c_void_p), ("max_ledger_bits", ctypes.c_int32),
                ("k_group_bits", ctypes.c_void_p)]


class Stats(ctypes.Structure):
    _fields_ = [("demotions", ctypes.c_uint64), ("promotions", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("ledger_writes", ctypes.c_uint64),
                ("ledger_reuses", ctypes.c_uint64), ("device_bytes", ctypes.c_int64)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libqevict.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -m "
                           "tiered_kv_cache_decode_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "qevict_pool_capacity": [ctypes.POINTER(Config), ctypes.POINTER(I32), ctypes.POINTER(I32),
                                 ctypes.POINTER(I64)],
        "qevict_cache_create": [ctypes.POINTER(Config), ctypes.POINTER(Allocator), P, ctypes.POINTER(P)],
        "qevict_cache_destroy": [P],
        "qevict_prefill": [P, I32, P, P, I32, P, P, P],
        "qevict_append_kv": [P, I32, P, P, I32, P],
        "qevict_decode_attention": [P, I32, P, P, P, I32, P],
        "qevict_decode_step": [P, I32, P, P, P, P, P, I32, P],
        "qevict_route": [P, I32, P, P, P],
        "qevict_demote_quantize": [P, I32, P, I32, P],
        "qevict_promote_dequantize": [P, I32, P, I32, P],
        "qevict_set_tiers": [P, I32, P, P],
        "qevict_get_scores": [P, I32, P, P],
        "qevict_get_view": [P, I32, ctypes.POINTER(View)],
        "qevict_get_status": [P, P],
        "qevict_clear_status": [P, P],
        "qevict_get_stats": [P, ctypes.POINTER(Stats), P],
        "qevict_set_launch_overlap": [P, I32],
        "qevict_set_wait_limit": [P, I64],
        "qevict_set_cooperative_launch": [P, I32],
        "qevict_refresh_lengths": [P, P],
        "qevict_decode_attention_static_scratch": [P, I32, P, P, P, I32, P],
        "qevict_get_tier_move_counts": [P, I32, P, P],
        "qevict_route_global": [P, P, P],
        "qevict_route_logsparse": [P, I32, I32, P],
        "qevict_route_rd": [P, I32, P, P, P],
        "qevict_route_rd_mixed": [P, I32, P, P, P],
        "qevict_k_channel_weights": [P, I32, P, I64, P, I64, P, P],
        "qevict_route_rd_kv": [P, I32, P, P, P],
        "qevict_future_missed_mass": [P, I32, P, P, I64, P, P],
        "qevict_length": [P, I32],
        "qevict_last_error": [],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.qevict_length.restype = I64
    lib.qevict_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def pool_capacity(cfg: Config):
    """(fp_capacity, ledger_capacity, pool bytes per layer) a cache with this config gets."""
    lib = load()
    a, b_, n = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
    rc = lib.qevict_pool_capacity(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(b_), ctypes.byref(n))
    if rc != 0:
        raise QevictError(rc, lib.qevict_last_error().decode())
    return a.value, b_.value, n.value


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class _DeviceArray:
    """Exposes a device pointer owned by the cache through __cuda_array_interface__."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def device_tensor(ptr: int, shape, typestr: str) -> torch.Tensor:
    return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")


class TieredCache:
    """A multi-layer tiered KV cache living on the current CUDA device."""

    def __init__(self, batch, num_layers, num_q_heads, num_kv_heads, window, max_context,
                 budget_frac=1.0, fp_share=0.5, fp_capacity=0, ledger_capacity=0, fp_slack=0,
                 head_dim=HEAD_DIM, torch_allocator=True, per_head=False, max_ledger_bits=0):
        """per_head: one tier per (sequence, KV head, window); scores, tiers and
        tier-move counts then have one row per unit b * num_kv_heads + kvh.
        max_ledger_bits 4 or 8 allows the INT4 (and INT8) tiers."""
        self.lib = load()
        self.cfg = Config(batch, num_layers, num_q_heads, num_kv_heads, head_dim, window, max_context,
                          fp_capacity, ledger_capacity, fp_slack, float(budget_frac), float(fp_share),
                          1 if per_head else 0, int(max_ledger_bits))
        self.B, self.Hq, self.Hkv, self.w = batch, num_q_heads, num_kv_heads, window
        self.per_head = bool(per_head)
        self.units = batch * num_kv_heads if per_head else batch
        self.layers = num_layers
        self.device = torch.cuda.current_device()
        self._alloc = None
        if torch_allocator:
            dev = self.device

            def _a(size, stream, ctx):
                try:
                    return torch.cuda.caching_allocator_alloc(int(size), dev, stream or 0)
                except Exception:
                    return None

            def _f(ptr, stream, ctx):
                torch.cuda.caching_allocator_delete(ptr)

            self._alloc = Allocator(ALLOC_FN(_a), FREE_FN(_f), None)
        self.handle = ctypes.c_void_p()
        rc = self.lib.qevict_cache_create(ctypes.byref(self.cfg),
                                          ctypes.byref(self._alloc) if self._alloc else None,
                                          _stream(), ctypes.byref(self.handle))
        self._check(rc)

    # ---- plumbing ----------------------------------------------------------
    def _check(self, rc):
        if rc != 0:
            raise QevictError(rc, self.lib.qevict_last_error().decode())

    def close(self):
        if self.handle:
            self._check(self.lib.qevict_cache_destroy(self.handle))
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_launch_overlap(self, enable=True):
        self._check(self.lib.qevict_set_launch_overlap(self.handle, 1 if enable else 0))

    def set_cooperative_launch(self, enable=True):
        self._check(self.lib.qevict_set_cooperative_launch(self.handle, 1 if enable else 0))

    def set_wait_limit(self, cycles=0):
        self._check(self.lib.qevict_set_wait_limit(self.handle, int(cycles)))

    def refresh_lengths(self, stream=None):
        self._check(self.lib.qevict_refresh_lengths(self.handle, _stream(stream)))

    def length(self, layer=0) -> int:
        return int(self.lib.qevict_length(self.handle, layer))

    def num_windows(self, layer=0) -> int:
        return -(-self.length(layer) // self.w)

    # ---- the path -----------------------------------------------------------
    def prefill(self, layer, k, v, scores=None, tiers=None, stream=None):
        n = k.shape[1]
        self._check(self.lib.qevict_prefill(self.handle, layer, _ptr(k), _ptr(v), n, _ptr(scores),
                                            _ptr(tiers), _stream(stream)))

    def append(self, layer, k, v, stream=None):
        self._check(self.lib.qevict_append_kv(self.handle, layer, _ptr(k), _ptr(v), k.shape[1],
                                              _stream(stream)))

    def decode(self, layer, q, out=None, mass=None, want_mass=True, accumulate=True, stream=None):
        if out is None:
            out = torch.empty(self.B, self.Hq, HEAD_DIM, dtype=torch.float32, device=q.device)
        if mass is None and want_mass:
            mass = torch.empty(self.B, self.Hq, self.num_windows(layer), dtype=torch.float32,
                               device=q.device)
        self._check(self.lib.qevict_decode_attention(self.handle, layer, _ptr(q), _ptr(out), _ptr(mass),
                                                     1 if accumulate else 0, _stream(stream)))
        return out, mass

    def decode_static_scratch(self, layer, q, out, mass=None, accumulate=True, stream=None):
        """decode() on the library's static device scratch; out (and mass, if
        wanted) are caller-owned, so nothing is allocated on this call."""
        self._check(self.lib.qevict_decode_attention_static_scratch(self.handle, layer, _ptr(q), _ptr(out),
                                                                    _ptr(mass), 1 if accumulate else 0,
                                                                    _stream(stream)))
        return out, mass

    def decode_step(self, layer, q, k_new, v_new, out=None, mass=None, want_mass=True, accumulate=True,
                    stream=None):
        """Append one token ([B][Hkv][d] or [B][1][Hkv][d]) and decode, in one launch."""
        if out is None:
            out = torch.empty(self.B, self.Hq, HEAD_DIM, dtype=torch.float32, device=q.device)
        if mass is None and want_mass:
            W = -(-(self.length(layer) + 1) // self.w)
            mass = torch.empty(self.B, self.Hq, W, dtype=torch.float32, device=q.device)
        self._check(self.lib.qevict_decode_step(self.handle, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                                _ptr(mass), 1 if accumulate else 0, _stream(stream)))
        return out, mass

    def route(self, layer, scores_override=None, score_mult=None, stream=None):
        self._check(self.lib.qevict_route(self.handle, layer, _ptr(scores_override), _ptr(score_mult),
                                          _stream(stream)))

    def route_rd(self, layer, scores_override=None, score_mult=None, stream=None):
        """Route a layer with tier counts from the rate-distortion allocation."""
        self._check(self.lib.qevict_route_rd(self.handle, layer, _ptr(scores_override), _ptr(score_mult),
                                             _stream(stream)))

    def route_rd_mixed(self, layer, scores_override=None, score_mult=None, stream=None):
        """Route a layer by the rate-distortion allocation over the widths the
        cache allows (0, 2, 4, 8, 16 bits)."""
        self._check(self.lib.qevict_route_rd_mixed(self.handle, layer, _ptr(scores_override), _ptr(score_mult),
                                                   _stream(stream)))

    def route_logsparse(self, layer, recent=2, stream=None):
        """Route a layer by log-sparse position (the scores are not used)."""
        self._check(self.lib.qevict_route_logsparse(self.handle, layer, recent, _stream(stream)))

    def route_global(self, scores_override=None, stream=None):
        """One routing event over all layers under one budget per sequence;
        scores_override: None or a list (per layer) of None / device [units][W] fp32."""
        arr = None
        if scores_override is not None:
            arr = (ctypes.c_void_p * self.layers)(*[None if t is None else t.data_ptr() for t in scores_override])
        self._check(self.lib.qevict_route_global(self.handle, arr, _stream(stream)))

    def demote(self, layer, pairs, stream=None):
        self._check(self.lib.qevict_demote_quantize(self.handle, layer, _ptr(pairs), pairs.shape[0],
                                                    _stream(stream)))

    def promote(self, layer, pairs, stream=None):
        self._check(self.lib.qevict_promote_dequantize(self.handle, layer, _ptr(pairs), pairs.shape[0],
                                                       _stream(stream)))

    def set_tiers(self, layer, tiers, stream=None):
        self._check(self.lib.qevict_set_tiers(self.handle, layer, _ptr(tiers), _stream(stream)))

    def scores(self, layer, stream=None):
        out = torch.empty(self.units, self.num_windows(layer), dtype=torch.float32, device="cuda")
        self._check(self.lib.qevict_get_scores(self.handle, layer, _ptr(out), _stream(stream)))
        return out

    # ---- diagnostics ----------------------------------------------------------
    def tier_move_counts(self, layer, stream=None):
        """int32 [B][8] counts of the layer's last tier move: FP and INT2 windows
        before, the same after, kept, promoted, demoted, evicted (host tensor)."""
        out = torch.zeros(self.units, 8, dtype=torch.int32)
        self._check(self.lib.qevict_get_tier_move_counts(self.handle, layer, ctypes.c_void_p(out.data_ptr()),
                                                         _stream(stream)))
        return out

    def future_missed_mass(self, layer, q, k_full, out=None, stream=None):
        """fp32 [B][Hq]: attention share of the full keys k_full [B][L][Hkv][d]
        (L = the layer's length) that falls on evicted windows."""
        if out is None:
            out = torch.empty(self.B, self.Hq, dtype=torch.float32, device=q.device)
        self._check(self.lib.qevict_future_missed_mass(self.handle, layer, _ptr(q), _ptr(k_full), k_full.shape[1],
                                                       _ptr(out), _stream(stream)))
        return out

    # ---- inspection ---------------------------------------------------------
    def view(self, layer) -> View:
        v = View()
        self._check(self.lib.qevict_get_view(self.handle, layer, ctypes.byref(v)))
        return v

    def status(self, stream=None) -> int:
        return int(self.lib.qevict_get_status(self.handle, _stream(stream)))

    def last_error(self) -> str:
        return self.lib.qevict_last_error().decode()

    def clear_status(self, stream=None):
        self._check(self.lib.qevict_clear_status(self.handle, _stream(stream)))

    def stats(self, stream=None) -> dict:
        s = Stats()
        self._check(self.lib.qevict_get_stats(self.handle, ctypes.byref(s), _stream(stream)))
        return {f: getattr(s, f) for f, _ in Stats._fields_}

    def tables(self, layer):
        """(tier, fp_slot, ledger_slot, ledger_writes) of the current windows, copied to host."""
        v = self.view(layer)
        W, Wm, B = v.num_windows, v.max_windows, v.batch
        get = lambda p, t: device_tensor(p, (B, Wm), t)[:, :W].cpu()
        return (get(v.tier, "|u1"), get(v.fp_slot, "<i4"), get(v.ledger_slot, "<i4"),
                get(v.ledger_writes, "<i4"))

    def fp_window(self, layer, slot):
        """bf16 [Hkv][2 (K, V)][w][d] content of a full-precision slot (host copy)."""
        v = self.view(layer)
        raw = device_tensor(v.fp_pool + slot * v.fp_slot_bytes, (v.fp_slot_bytes,), "|u1").cpu()
        H = v.num_kv_heads   # KV heads of a unit: 1 with per-head tiers
        x = raw.view(torch.bfloat16).view(H, 2, 2, self.w, 64)     # [kvh][kv][half][token][64]
        return x.permute(0, 1, 3, 2, 4).reshape(H, 2, self.w, HEAD_DIM)

    def ledger_window(self, layer, slot, bits=2, seq=None):
        """Decoded ledger slot of a window quantised to `bits` (2, 4, 8): codes
        uint8 [Hkv][2][w][d], scale/min fp16 [Hkv][2][w][d/32]. On a layer
        routed with K channels, `seq` names the sequence whose K group widths
        the tiles follow."""
        v = self.view(layer)
        raw = device_tensor(v.ledger_pool + slot * v.ledger_slot_bytes, (v.ledger_slot_bytes,), "|u1").cpu()
        if v.k_group_bits:
            kgw = self.k_group_bits(layer)[seq if seq is not None else slot // v.ledger_capacity]
            return decode_kch_slot(raw, v.num_kv_heads, self.w, bits, kgw)
        return decode_ledger_slot(raw, v.num_kv_heads, self.w, bits)

    def k_group_bits(self, layer):
        """uint8 [batch][Hkv][4] K group widths of a layer routed by route_rd_kv (else None)."""
        v = self.view(layer)
        if not v.k_group_bits:
            return None
        return device_tensor(v.k_group_bits, (v.batch, v.num_kv_heads, 4), "|u1").cpu()

    # ---- RDKV's K-channel half -----------------------------------------------
    def k_channel_weights(self, layer, q_obs, k_full, stream=None):
        """fp32 [B][Hkv][d] channel weights from observed queries [B][n_q][Hq][d]
        and keys [B][n][Hkv][d] (bf16, device)."""
        out = torch.empty(self.B, self.Hkv, HEAD_DIM, dtype=torch.float32, device=k_full.device)
        self._check(self.lib.qevict_k_channel_weights(self.handle, layer, _ptr(q_obs), q_obs.shape[1], _ptr(k_full),
                                                      k_full.shape[1], _ptr(out), _stream(stream)))
        return out

    def route_rd_kv(self, layer, weights, scores_override=None, stream=None):
        self._check(self.lib.qevict_route_rd_kv(self.handle, layer, _ptr(weights), _ptr(scores_override),
                                                _stream(stream)))

    def ledger_bits(self, layer):
        """uint8 [units][W]: width of each window's ledger entry (0 none, 2, 4, 8), host copy."""
        v = self.view(layer)
        return device_tensor(v.ledger_bits, (v.batch, v.max_windows), "|u1")[:, :v.num_windows].cpu()


def decode_kch_slot(raw: torch.Tensor, Hkv: int, w: int, bits: int, kgw):
    """Unpack a K-channel ledger slot (see qevict_view.k_group_bits): tiles of
    4608 B; per tile the K groups' planes in turn ([16 tokens][2 words] each),
    the K meta, then the V codes and meta of a `bits` window. Returns what
    decode_ledger_slot returns."""
    d = HEAD_DIM
    nt = w // 16
    P = bits // 2
    raw = raw[:Hkv * nt * 4608].view(Hkv, nt, 4608)
    shifts = torch.arange(16, dtype=torch.int64) * 2
    i = torch.arange(d)
    ch = 16 * ((i >> 1) & 7) + (i >> 4) + 8 * (i & 1)
    kcodes = torch.zeros(Hkv, nt * 16, d, dtype=torch.int64)
    vcodes = torch.zeros(Hkv, nt * 16, d, dtype=torch.int64)
    km = torch.zeros(Hkv, nt * 16, 4, 2, dtype=torch.float16)
    vm = torch.zeros(Hkv, nt * 16, 4, 2, dtype=torch.float16)
    for h in range(Hkv):
        goff = 0
        for g in range(4):
            for p in range(int(kgw[h][g]) // 2):
                kw = raw[h, :, goff + 128 * p:goff + 128 * (p + 1)].contiguous().view(torch.int32).to(torch.int64)
                kc = ((kw & 0xFFFFFFFF).view(nt, 16, 2)[..., None] >> shifts) & 3                # [nt][tok][2][16]
                kcodes[h, :, 32 * g:32 * (g + 1)] |= kc.reshape(nt * 16, 32) << (2 * p)
            goff += 128 * (int(kgw[h][g]) // 2)
        km[h] = raw[h, :, goff:goff + 256].contiguous().view(torch.float16).view(nt * 16, 4, 2)
        for p in range(P):
            v0 = goff + 256 + 512 * p
            vw = raw[h, :, v0:v0 + 512].contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
            vc = (vw[..., None] >> shifts) & 3
            vp = torch.empty(nt, d, 16, dtype=torch.int64)
            vp[:, ch] = vc
            vcodes[h] |= vp.permute(0, 2, 1).reshape(nt * 16, d) << (2 * p)
        v1 = goff + 256 + 512 * P
        vm[h] = raw[h, :, v1:v1 + 256].contiguous().view(torch.float16).view(nt * 16, 4, 2)
    codes = torch.stack([kcodes, vcodes], dim=1).to(torch.uint8)
    meta = torch.stack([km, vm], dim=1)
    return codes, meta[..., 0].clone(), meta[..., 1].clone()


def decode_ledger_slot(raw: torch.Tensor, Hkv: int, w: int, bits: int = 2):
    """Unpack the documented ledger slot layout (see include/qevict.h) on the host.

    A window quantised to `bits` keeps P = bits / 2 two-bit planes, code =
    sum_p 4^p c_p. Returns codes uint8 [Hkv][2 (K, V)][w][d] and scale, min
    fp16 [Hkv][2][w][d/32].
    """
    d = HEAD_DIM
    nt = w // 16
    P = bits // 2
    tb = 1024 * P + 512
    raw = raw[:Hkv * nt * tb].view(Hkv, nt, tb)
    shifts = torch.arange(16, dtype=torch.int64) * 2
    i = torch.arange(d)
    ch = 16 * ((i >> 1) & 7) + (i >> 4) + 8 * (i & 1)                                   # channel of word i
    kcodes = torch.zeros(Hkv, nt * 16, d, dtype=torch.int64)
    vcodes = torch.zeros(Hkv, nt * 16, d, dtype=torch.int64)
    for p in range(P):
        kw = raw[:, :, 512 * p:512 * (p + 1)].contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
        kc = (kw.view(Hkv, nt, 16, 8)[..., None] >> shifts) & 3                         # [Hkv][nt][tok][q][16]
        kcodes |= kc.reshape(Hkv, nt * 16, d) << (2 * p)
        v0 = 512 * P + 256 + 512 * p
        vw = raw[:, :, v0:v0 + 512].contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF   # [Hkv][nt][128]
        vc = (vw[..., None] >> shifts) & 3                                               # [Hkv][nt][word][tok]
        vp = torch.empty(Hkv, nt, d, 16, dtype=torch.int64)
        vp[:, :, ch] = vc
        vcodes |= vp.permute(0, 1, 3, 2).reshape(Hkv, nt * 16, d) << (2 * p)
    codes = torch.stack([kcodes, vcodes], dim=1).to(torch.uint8)
    km = raw[:, :, 512 * P:512 * P + 256].contiguous().view(torch.float16).view(Hkv, nt * 16, 4, 2)
    vm = raw[:, :, 1024 * P + 256:1024 * P + 512].contiguous().view(torch.float16).view(Hkv, nt * 16, 4, 2)
    meta = torch.stack([km, vm], dim=1)
    return codes, meta[..., 0].clone(), meta[..., 1].clone()
