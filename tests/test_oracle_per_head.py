"""Pins of the oracle's per-attention-head scales and scale calibration.

"Quantized KV cache" (vLLM features page), Supported schemes: per-attention-head
quantization has one scale per kv head (k/v_scale = [num_kv_heads]); Scale
calibration approaches: scales estimated once from a batch of tokens.

- Per-head FP8 codes of head h are PyTorch's float8 conversion of x_h / s_h
  (fp32 division), head by head.
- Per-head NVFP4 block scales of head h follow the E4M3 rounding of
  amax / (6 g_h), computed with PyTorch.
- Per-head attention equals PyTorch's fp64 SDPA over K/V that PyTorch
  dequantizes with each head's own scale.
- Calibration equals numpy's amax over the finite values divided (float32) by
  the format maximum the pages print (tests/golden/format_constants.txt), and
  places the largest value on the format's largest code.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import read_golden
from test_oracle_quant import E2M1_TABLE

_MAX = {(r[0], r[1]): float(r[2]) for r in read_golden("format_constants.txt")}
CAL_DIV = {"fp8_e4m3": _MAX[("max", "fp8_e4m3")], "fp8_e5m2": _MAX[("max", "fp8_e5m2")],
           "nvfp4": _MAX[("max", "e2m1")] * _MAX[("max", "fp8_e4m3")]}
F8 = {"fp8_e4m3": torch.float8_e4m3fn, "fp8_e5m2": torch.float8_e5m2}
# encoding saturates at the largest finite code (reading R2); PyTorch's float8
# conversion gives NaN beyond it, so the reference clamps first
FMAX = {"fp8_e4m3": _MAX[("max", "fp8_e4m3")], "fp8_e5m2": _MAX[("max", "fp8_e5m2")]}


def _rows(orc, fmt, H=3, D=32, n=21, seed=3, spread=(1.0, 40.0, 0.02)):
    """bf16 rows [n][H][D] whose kv heads have very different magnitudes."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, H, D)).astype(np.float32) * np.array(spread, np.float32)[None, :, None]
    return synth.to_bf16_bits(torch.from_numpy(x))


def _store(orc, fmt, k, v, scales, P=16):
    n, H, D = k.shape
    c = orc.OracleCache(fmt, H, D, P, (n + P - 1) // P)
    assert c.quantize_store(k, v, np.arange(n), scales) == 0
    return c


def _head_rows(c, n, which, h):
    data = c.k_data if which == 0 else c.v_data
    return data[[c.row_index(i, h) for i in range(n)]]


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
def test_per_head_fp8_codes_match_torch(orc, fmt):
    k, v = _rows(orc, fmt, seed=1), _rows(orc, fmt, seed=2)
    scales = np.array([[0.01, 0.5, 3.0e-4], [2.0, 0.07, 1.0 / 3.0]], np.float32)
    c = _store(orc, fmt, k, v, scales)
    n, H, _ = k.shape
    for which, x in ((0, k), (1, v)):
        xf = torch.from_numpy(synth.bf16_bits_to_float(x))
        for h in range(H):
            q = (xf[:, h] / torch.tensor(scales[which, h])).clamp(-FMAX[fmt], FMAX[fmt])  # R2
            ref = q.to(F8[fmt]).view(torch.uint8).numpy()
            assert np.array_equal(_head_rows(c, n, which, h), ref), (which, h)


def test_equal_head_scales_are_the_per_tensor_case(orc):
    k, v = _rows(orc, "fp8_e4m3", seed=4), _rows(orc, "fp8_e4m3", seed=5)
    a = _store(orc, "fp8_e4m3", k, v, [0.25, 0.125])
    b = _store(orc, "fp8_e4m3", k, v, np.array([[0.25] * 3, [0.125] * 3], np.float32))
    assert np.array_equal(a.k_data, b.k_data) and np.array_equal(a.v_data, b.v_data)


def test_per_head_nvfp4_block_scales(orc):
    k, v = _rows(orc, "nvfp4", seed=6), _rows(orc, "nvfp4", seed=7)
    g = np.array([[0.02, 0.001, 1.5e-5], [0.3, 0.004, 0.05]], np.float32)
    c = _store(orc, "nvfp4", k, v, g)
    n, H, D = k.shape
    for which, x in ((0, k), (1, v)):
        scl = c.k_scales if which == 0 else c.v_scales
        xf = synth.bf16_bits_to_float(x).reshape(n, H, D // 16, 16)
        for h in range(H):
            amax = np.abs(xf[:, h]).max(axis=2)
            ratio = amax / (np.float32(6.0) * g[which, h])
            ratio = np.minimum(ratio.astype(np.float32), np.float32(FMAX["fp8_e4m3"]))  # R2
            ref = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            got = scl[[c.row_index(i, h) for i in range(n)]]
            assert np.array_equal(got, ref), (which, h)


def _dequant_torch(fmt, c, n, which, h, s):
    data = _head_rows(c, n, which, h)
    if fmt in F8:
        return torch.from_numpy(data.copy()).view(F8[fmt]).double() * float(s)
    scl = (c.k_scales if which == 0 else c.v_scales)[[c.row_index(i, h) for i in range(n)]]
    nib = np.stack([data & 0xF, data >> 4], axis=-1).reshape(n, -1)
    mag = torch.from_numpy(E2M1_TABLE[nib & 7] * np.where(nib & 8, -1.0, 1.0))
    S = torch.from_numpy(scl.copy()).view(torch.float8_e4m3fn).double() * float(s)
    return mag * S.repeat_interleave(16, dim=1)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_per_head_attention_matches_torch_sdpa(orc, fmt):
    n, H, D, G = 37, 3, 32, 2
    k, v = _rows(orc, fmt, H=H, D=D, n=n, seed=8), _rows(orc, fmt, H=H, D=D, n=n, seed=9)
    scales = np.array([[0.02, 0.3, 0.001], [0.5, 0.004, 0.06]], np.float32)
    c = _store(orc, fmt, k, v, scales)
    q = synth.to_bf16_bits(torch.randn(1, H * G, D, generator=torch.Generator().manual_seed(3)))
    pt = np.arange(c.num_pages, dtype=np.int32)[None]
    out, rc = c.decode_attention(q, pt, np.array([n], np.int32), 0.3)
    assert rc == 0
    qd = torch.from_numpy(q.view(np.int16).copy()).view(torch.bfloat16).double()
    K = torch.stack([_dequant_torch(fmt, c, n, 0, h, scales[0, h]) for h in range(H)])[None]
    V = torch.stack([_dequant_torch(fmt, c, n, 1, h, scales[1, h]) for h in range(H)])[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qd[:, :, None, :], K, V, scale=0.3,
                                                           enable_gqa=True)[0, :, 0, :]
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2", "nvfp4"])
@pytest.mark.parametrize("per_head", [False, True])
def test_calibration_is_amax_over_format_max(orc, fmt, per_head):
    x = _rows(orc, fmt, n=50, seed=10)
    xf = synth.bf16_bits_to_float(x)
    xf_special = xf.copy()
    xf_special[3, 1, 5] = np.inf                  # non-finite values do not count
    xf_special[7, 0, 2] = np.nan
    xs = synth.to_bf16_bits(torch.from_numpy(xf_special))
    got = orc.calibrate_scales(fmt, xs, per_head)
    amax = np.abs(xf).max(axis=(0, 2)) if per_head else np.abs(xf).max(keepdims=True).reshape(1)
    ref = amax.astype(np.float32) / np.float32(CAL_DIV[fmt])
    assert got.dtype == np.float32 and np.array_equal(got, ref)


@pytest.mark.parametrize("fmt,max_code", [("fp8_e4m3", 0x7E), ("fp8_e5m2", 0x7B)])
def test_calibrated_scale_puts_amax_on_the_largest_code(orc, fmt, max_code):
    k = _rows(orc, fmt, n=40, seed=11)
    s = orc.calibrate_scales(fmt, k, per_head=True)
    c = _store(orc, fmt, k, k, np.stack([s, s]))
    n, H, _ = k.shape
    xf = np.abs(synth.bf16_bits_to_float(k))
    for h in range(H):
        rows = _head_rows(c, n, 0, h)
        i, d = np.unravel_index(np.argmax(xf[:, h]), xf[:, h].shape)
        assert rows[i, d] & 0x7F == max_code
        assert ((rows & 0x7F) <= max_code).all()


def test_calibration_degenerate_cases(orc):
    z = np.zeros((4, 2, 16), np.uint16)
    for fmt in ("fp8_e4m3", "nvfp4"):
        assert np.array_equal(orc.calibrate_scales(fmt, z, True), np.ones(2, np.float32))
    x = _rows(orc, "bf16", H=2, D=16, n=4, spread=(1.0, 2.0))
    for fmt in ("bf16", "fp4_mx_block16"):   # no per-tensor scale: 1.0
        assert np.array_equal(orc.calibrate_scales(fmt, x, False), np.ones(1, np.float32))
