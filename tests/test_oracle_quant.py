"""Pins of the oracle's quantize-and-store and dequantize.

FP8 codes and every dequantized bf16 value are compared with PyTorch's own
float8 / float32 / bfloat16 conversions.  The block formats are checked
against a nearest-value search over the OCP E2M1 table written here in numpy,
plus the defining invariants of each scale rule (the MX shared exponent puts
the block maximum in [4, 8) times the scale; the NVFP4 block scale is the
E4M3 rounding of amax / (6 g)).  Page/slot layout is checked by placing
recognisable rows at known slots.
"""
import math

import numpy as np
import pytest
import torch

import synth
from conftest import read_golden

E2M1_TABLE = np.array([float(v) for _, v in read_golden("e2m1_values.txt")[:8]])  # codes 0..7


def _nearest_e2m1(y):
    """Nearest E2M1 code to each float (ties to the even code), sign copied."""
    y = np.asarray(y, np.float64)
    a = np.minimum(np.abs(y), 6.0)
    d = np.abs(a[:, None] - E2M1_TABLE[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equal distances prefer the even code
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    code = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    return code | np.where(np.signbit(y), 8, 0)


def _small_workload(fmt, B=3, T=(40, 17, 64), seed=5):
    return synth.make_workload(f"t_{fmt}", fmt, Hq=8, Hkv=2, D=64, seq_lens=list(T)[:B], seed=seed)


def _store_all(orc, wl, layer=0):
    c = orc.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    s = wl.scales(layer)
    for b in range(wl.B):
        k, v = wl.kv(layer, b)
        assert c.quantize_store(k, v, wl.slots(b), s) == 0
    return c


def _rows(c, wl, b, which):
    data = c.k_data if which == "k" else c.v_data
    scl = c.k_scales if which == "k" else c.v_scales
    slots = wl.slots(b)
    idx = np.array([[c.row_index(int(s), h) for h in range(wl.Hkv)] for s in slots])
    return data[idx], scl[idx]


@pytest.mark.parametrize("fmt,dtype", [("fp8_e4m3", torch.float8_e4m3fn),
                                       ("fp8_e5m2", torch.float8_e5m2)])
def test_fp8_store_matches_torch(orc, fmt, dtype):
    wl = _small_workload(fmt)
    c = _store_all(orc, wl)
    s = wl.scales()
    for b in range(wl.B):
        k, v = wl.kv(0, b)
        for which, x, sc in (("k", k, s[0]), ("v", v, s[1])):
            xf = torch.from_numpy(synth.bf16_bits_to_float(x))
            ref = (xf / torch.tensor(sc, dtype=torch.float32)).to(dtype).view(torch.uint8).numpy()
            got, _ = _rows(c, wl, b, which)
            assert np.array_equal(got, ref)


def test_fp8_scale_one_default(orc):
    wl = synth.make_workload("t1", "fp8_e4m3", Hq=4, Hkv=2, D=32, seq_lens=[20], scale_mode="one")
    assert np.array_equal(wl.scales(), [1.0, 1.0])
    c = _store_all(orc, wl)
    k, _ = wl.kv(0, 0)
    ref = torch.from_numpy(synth.bf16_bits_to_float(k)).to(torch.float8_e4m3fn).view(torch.uint8)
    got, _ = _rows(c, wl, 0, "k")
    assert np.array_equal(got, ref.numpy())


def test_fp4_block16_scale_rule_and_codes(orc):
    wl = _small_workload("fp4_mx_block16")
    c = _store_all(orc, wl)
    for b in range(wl.B):
        k, v = wl.kv(0, b)
        for which, x in (("k", k), ("v", v)):
            data, scl = _rows(c, wl, b, which)
            xf = synth.bf16_bits_to_float(x).reshape(-1, wl.D // 16, 16)
            E = scl.reshape(-1, wl.D // 16).astype(np.int64) - 127
            amax = np.abs(xf).max(axis=2)
            # MX shared exponent: block max lands in [4, 8) after scaling by 2^-E
            r = amax * np.exp2(-E.astype(np.float64))
            assert np.all(((r >= 4) & (r < 8)) | ((amax == 0) & (E == -127)))
            y = xf.astype(np.float64) * np.exp2(-E.astype(np.float64))[..., None]
            codes = _nearest_e2m1(y.reshape(-1)).reshape(-1, wl.D)
            packed = data.reshape(-1, wl.D // 2)
            assert np.array_equal(packed & 0xF, codes[:, 0::2])      # even d: low nibble
            assert np.array_equal(packed >> 4, codes[:, 1::2])


def test_fp4_block16_degenerate_blocks(orc):
    c = orc.OracleCache("fp4_mx_block16", 1, 32, 16, 1)
    x = np.zeros((3, 1, 32), np.float32)
    x[1, 0, :16] = 1.5 * 2.0 ** -126    # floor(log2) - 2 = -128 clamps to -127: x * 2^127 = 3
    x[2, 0, 16:] = 3.0e38               # near the bf16 maximum
    x[2, 0, 17] = -1.0
    bits = synth.to_bf16_bits(torch.from_numpy(x))
    assert c.quantize_store(bits, bits, np.arange(3), None) == 0
    assert list(c.k_scales[0]) == [0, 0]                       # all-zero row: E = -127
    assert c.k_scales[1, 0] == 0 and (c.k_data[1, :8] == 0x55).all()   # code 0x5 = 3.0
    assert c.k_scales[2, 1] == 127 + 125                       # floor(log2 3e38) = 127 -> E = 125
    assert c.k_data[2, 8] >> 4 == 0x8                          # -1 * 2^-125 rounds to -0


def test_nvfp4_scale_rule_and_codes(orc):
    wl = _small_workload("nvfp4")
    c = _store_all(orc, wl)
    g = wl.scales()
    for b in range(wl.B):
        k, v = wl.kv(0, b)
        for which, x, gs in (("k", k, g[0]), ("v", v, g[1])):
            data, scl = _rows(c, wl, b, which)
            xf = synth.bf16_bits_to_float(x).reshape(-1, wl.D // 16, 16)
            amax = np.abs(xf).max(axis=2)
            gs32 = np.float32(gs)
            ratio = amax / (np.float32(6.0) * gs32)                # fp32 ops
            sc_ref = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(scl.reshape(sc_ref.shape), sc_ref)
            S = torch.from_numpy(sc_ref).view(torch.float8_e4m3fn).float().numpy() * gs32
            y = np.where(S[..., None] == 0, 0, xf / np.where(S == 0, 1, S)[..., None])
            codes = _nearest_e2m1(y.reshape(-1)).reshape(-1, wl.D)
            codes = np.where(np.repeat(S.reshape(-1, wl.D // 16) == 0, 16, axis=1), 0, codes)
            packed = data.reshape(-1, wl.D // 2)
            assert np.array_equal(packed & 0xF, codes[:, 0::2])
            assert np.array_equal(packed >> 4, codes[:, 1::2])
            # the scaled block maximum sits near E2M1_MAX (E4M3 rounding of the scale)
            nz = S > 0
            assert np.all(np.abs(amax[nz] / S[nz] - 6.0) <= 6.0 * 2.0 ** -3)


def _torch_dequant(fmt, data, scl, s):
    """Independent dequantization with PyTorch: bf16(fp32(dec(code) * S))."""
    if fmt in ("fp8_e4m3", "fp8_e5m2"):
        dt = torch.float8_e4m3fn if fmt == "fp8_e4m3" else torch.float8_e5m2
        val = torch.from_numpy(data).view(dt).float()
        S = torch.full_like(val, float(np.float32(s)))
    else:
        nib = np.stack([data & 0xF, data >> 4], axis=-1).reshape(data.shape[0], -1)
        mag = E2M1_TABLE[nib & 7] * np.where(nib & 8, -1.0, 1.0)
        val = torch.from_numpy(mag.astype(np.float32))
        if fmt == "fp4_mx_block16":
            S = torch.from_numpy(scl).view(torch.float8_e8m0fnu).float()
        else:
            S = torch.from_numpy(scl).view(torch.float8_e4m3fn).float() * np.float32(s)
        S = S.repeat_interleave(16, dim=1)
    return (val * S).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", ["bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4"])
def test_dequantize_matches_torch(orc, fmt):
    wl = _small_workload(fmt)
    c = _store_all(orc, wl)
    s = wl.scales()
    for b in range(wl.B):
        slots = wl.slots(b)
        ko, vo, rc = c.dequantize(slots)
        assert rc == 0
        for which, out, sc in (("k", ko, s[0]), ("v", vo, s[1])):
            data, scl = _rows(c, wl, b, which)
            if fmt == "bf16":
                k, v = wl.kv(0, b)
                assert np.array_equal(out, k if which == "k" else v)
                continue
            ref = _torch_dequant(fmt, data.reshape(-1, data.shape[-1]),
                                 scl.reshape(-1, scl.shape[-1]), sc)
            assert np.array_equal(out.reshape(ref.shape), ref)


def test_slot_layout_and_skips(orc):
    H, D, P, NP = 2, 16, 16, 3
    c = orc.OracleCache("bf16", H, D, P, NP)
    n = 4
    x = np.zeros((n, H, D), np.uint16)
    for i in range(n):
        for h in range(H):
            x[i, h, :] = 0x3F80 + 16 * i + h          # distinct bf16 values per (token, head)
    slots = np.array([17, -1, 2 * P + 15, 5], np.int64)  # page 1 off 1, skipped, page 2 off 15, page 0 off 5
    assert c.quantize_store(x, x, slots, None) == 0
    rows = c.k_data.view(np.uint16).reshape(NP, H, P, D)
    assert (rows[1, :, 1, 0] == x[0, :, 0]).all()
    assert (rows[2, :, 15, 0] == x[2, :, 0]).all()
    assert (rows[0, :, 5, 0] == x[3, :, 0]).all()
    assert int((rows != 0).any(axis=-1).sum()) == 3 * H   # nothing else written
    assert c.quantize_store(x, x, np.array([0, 1, NP * P, 2], np.int64), None) == -1
    ko, vo, rc = c.dequantize(np.array([17, -1, NP * P], np.int64))
    assert rc == -1 and (ko[1] == 0).all() and (ko[2] == 0).all() and (ko[0] == x[0]).all()
