"""The host-side ledger decoder (binding.decode_ledger_slot) against the slot
layout documented in include/qevict.h, on the CPU.

The encoder below is written from the header's description alone: tiles of 16
tokens per KV head; K code word q of a token holds channels 16 q .. 16 q + 15
(channel j at bits 2 (j % 16)); V word i = (g 8 + mt) 2 + h holds channel
16 mt + g + 8 h with token t at bits 2 t; half2 (scale, min) meta per token and
group of 32 channels; a b-bit code is kept as b / 2 two-bit planes,
code = sum_p 4^p c_p, with K planes at 512 p, K meta at 512 P, V planes at
512 P + 256 + 512 p and V meta at 1024 P + 256 of a 1024 P + 512-byte tile.
"""
import numpy as np
import pytest
import torch

from tiered_kv_cache_decode_gb300 import binding

D = 128


def encode_slot(codes, scale, mn, bits):
    """codes uint8 [Hkv][2][w][d]; scale, mn float16 [Hkv][2][w][d/32] -> raw bytes."""
    Hkv, _, w, d = codes.shape
    P, nt = bits // 2, w // 16
    tb = 1024 * P + 512
    raw = np.zeros((Hkv, nt, tb), np.uint8)
    for kvh in range(Hkv):
        for tile in range(nt):
            tok = slice(16 * tile, 16 * tile + 16)
            buf = raw[kvh, tile]
            for p in range(P):
                kpl = (codes[kvh, 0, tok].astype(np.uint32) >> (2 * p)) & 3          # [16 tok][128 ch]
                words = np.zeros((16, 8), np.uint32)
                for j in range(d):
                    words[:, j // 16] |= kpl[:, j] << (2 * (j % 16))
                buf[512 * p:512 * (p + 1)] = words.reshape(-1).view(np.uint8)
                vpl = (codes[kvh, 1, tok].astype(np.uint32) >> (2 * p)) & 3          # [16 tok][128 ch]
                vw = np.zeros(128, np.uint32)
                for g in range(8):
                    for mt in range(8):
                        for h in range(2):
                            ch = 16 * mt + g + 8 * h
                            i = (g * 8 + mt) * 2 + h
                            for t in range(16):
                                vw[i] |= vpl[t, ch] << (2 * t)
                v0 = 512 * P + 256 + 512 * p
                buf[v0:v0 + 512] = vw.view(np.uint8)
            for kv, off in ((0, 512 * P), (1, 1024 * P + 256)):
                meta = np.stack([scale[kvh, kv, tok], mn[kvh, kv, tok]], axis=-1).astype(np.float16)   # [16][4][2]
                buf[off:off + 256] = meta.reshape(-1).view(np.uint8)
    return torch.from_numpy(raw.reshape(-1).copy())


@pytest.mark.parametrize("bits,Hkv,w", [(2, 2, 32), (4, 1, 64), (8, 3, 16)])
def test_ledger_decoder_reads_the_documented_layout(bits, Hkv, w):
    rng = np.random.default_rng(bits * 10 + Hkv)
    codes = rng.integers(0, 1 << bits, size=(Hkv, 2, w, D)).astype(np.uint8)
    scale = rng.standard_normal((Hkv, 2, w, D // 32)).astype(np.float16)
    mn = rng.standard_normal((Hkv, 2, w, D // 32)).astype(np.float16)
    raw = encode_slot(codes, scale, mn, bits)
    got_c, got_s, got_m = binding.decode_ledger_slot(raw, Hkv, w, bits)
    assert np.array_equal(got_c.numpy(), codes)
    assert np.array_equal(got_s.numpy().view(np.uint16), scale.view(np.uint16))
    assert np.array_equal(got_m.numpy().view(np.uint16), mn.view(np.uint16))


def test_single_code_bit_positions():
    """One non-zero 4-bit code: K channel 37 of token 5 = 9 (planes 1 and 2),
    V channel 90 of token 11 = 6 (planes 2 and 1): the bytes the header places
    them in, and nothing else."""
    Hkv, w, bits = 1, 16, 4
    codes = np.zeros((Hkv, 2, w, D), np.uint8)
    codes[0, 0, 5, 37] = 9
    codes[0, 1, 11, 90] = 6
    z = np.zeros((Hkv, 2, w, D // 32), np.float16)
    raw = encode_slot(codes, z, z, bits).numpy()
    nz = np.flatnonzero(raw)
    # K: token 5, word 37 // 16 = 2, field 37 % 16 = 5 -> bits 10-11: plane 0 holds 1, plane 1 holds 2
    k_word = 5 * 8 + 2
    assert raw[4 * k_word + 1] == 1 << 2                     # plane 0, bit 10 = byte 1 bit 2
    assert raw[512 + 4 * k_word + 1] == 2 << 2               # plane 1
    # V: channel 90 = 16 * 5 + 10 -> mt 5, g 2, h 1 -> word (2 * 8 + 5) * 2 + 1 = 43; token 11 -> bits 22-23
    v_word = 43
    v0 = 512 * 2 + 256
    assert raw[v0 + 4 * v_word + 2] == 2 << 6                # plane 0 holds 6 % 4 = 2 at bit 22
    assert raw[v0 + 512 + 4 * v_word + 2] == 1 << 6          # plane 1 holds 6 // 4 = 1
    assert len(nz) == 4
    got, _, _ = binding.decode_ledger_slot(torch.from_numpy(raw), Hkv, w, bits)
    assert np.array_equal(got.numpy(), codes)
