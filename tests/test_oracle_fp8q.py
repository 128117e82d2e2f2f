"""Pins of the oracle's FP8-domain attention with a quantized query (reading
R17, "Quantized KV cache" (vLLM), FP8 KV cache overview and Supported schemes).

- The query codes equal PyTorch's float8_e4m3fn cast of q / q_scale (fp32),
  per tensor and per q head, over every finite bf16 value that stays in range;
  values beyond the range saturate to the largest finite code.
- Attention over the quantized query equals PyTorch's fp64
  scaled_dot_product_attention with the query decoded by PyTorch (codes x
  q_scale) and K/V decoded by PyTorch from the oracle's cache bytes.
- A query already on the E4M3 grid (times its scale) is quantized losslessly,
  so the FP8-domain result equals the bf16-query result.
"""
import numpy as np
import pytest
import torch

import synth
from test_oracle_attention import _exact_kv
from test_oracle_quant import _store_all


def _all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_float(bits)
    return bits[np.isfinite(f)]


@pytest.mark.parametrize("scale", [1.0, 0.0078125, 0.37, 3.1e-3, 17.5])
def test_query_codes_match_torch_per_tensor(orc, scale):
    bits = _all_finite_bf16()
    x = synth.bf16_bits_to_float(bits)
    s32 = np.float32(scale)
    keep = np.abs(x / s32) <= 448.0           # torch's cast does not saturate
    q = bits[keep]
    n = (q.shape[0] // 8) * 8
    q = q[:n].reshape(-1, 8, 1)
    got = orc.quantize_query(q, [scale])
    ref = (torch.from_numpy(synth.bf16_bits_to_float(q)) / torch.tensor(s32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_query_codes_saturate_and_keep_sign(orc):
    vals = np.array([1e6, -1e6, 448.0 * 1.01, -0.0, 0.0, 1e-30, -1e-30], np.float32)
    q = synth.to_bf16_bits(torch.from_numpy(vals)).reshape(1, 1, -1)
    got = orc.quantize_query(q, [1.0]).reshape(-1)
    assert list(got) == [0x7E, 0xFE, 0x7E, 0x80, 0x00, 0x00, 0x80]


def test_query_codes_per_head_scales(orc):
    rng = np.random.default_rng(5)
    Hq, D = 6, 32
    scales = np.array([0.01, 0.02, 0.5, 1.0, 2.0, 0.003], np.float32)
    x = rng.standard_normal((3, Hq, D)).astype(np.float32) * 2.0
    q = synth.to_bf16_bits(torch.from_numpy(x))
    got = orc.quantize_query(q, scales)
    xf = torch.from_numpy(synth.bf16_bits_to_float(q))
    # torch's cast does not saturate: clamp to the largest finite value first
    ref = (xf / torch.from_numpy(scales).view(1, Hq, 1)).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(got, ref.numpy())
    # a per-tensor call equals the per-head call with every head at that scale
    assert np.array_equal(orc.quantize_query(q, [0.5]), orc.quantize_query(q, np.full(Hq, 0.5)))


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("per_head", [False, True])
def test_fp8q_attention_matches_torch_sdpa(orc, fmt, per_head):
    wl = synth.make_workload(f"q8_{fmt}", fmt, Hq=8, Hkv=2, D=64, seq_lens=[1, 37, 50, 16], seed=19)
    c = _store_all(orc, wl)
    q = wl.q()
    qs = (np.linspace(0.004, 0.02, wl.Hq).astype(np.float32) if per_head
          else np.array([0.011], np.float32))
    out, rc = c.decode_attention_fp8q(q, qs, wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0
    qf = torch.from_numpy(synth.bf16_bits_to_float(q))
    sq = torch.from_numpy(np.broadcast_to(qs, (wl.Hq,)).copy()).view(1, wl.Hq, 1)
    qhat = (qf / sq).clamp(-448, 448).to(torch.float8_e4m3fn).double() * sq.double()
    for b in range(wl.B):
        K = _exact_kv(fmt, c, wl, b, "k").permute(1, 0, 2)[None]
        V = _exact_kv(fmt, c, wl, b, "v").permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qhat[b][None, :, None, :], K, V, scale=wl.sm_scale, enable_gqa=True)[0, :, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_fp8q_on_grid_query_equals_bf16_query(orc):
    """q = code value x 2^-3 for random E4M3 codes of magnitude <= 8: q / q_scale
    is exactly that E4M3 value, so quantization loses nothing."""
    wl = synth.make_workload("grid", "fp8_e4m3", Hq=8, Hkv=2, D=64, seq_lens=[40, 9], seed=23)
    c = _store_all(orc, wl)
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 0x51, size=(wl.B, wl.Hq, wl.D)).astype(np.uint8)   # |value| <= 8
    codes |= (rng.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float() * 0.125
    q = synth.to_bf16_bits(vals)
    assert np.array_equal(synth.bf16_bits_to_float(q), vals.numpy())   # exact in bf16
    a, rc = c.decode_attention_fp8q(q, [0.125], wl.page_table, wl.seq_lens, wl.sm_scale)
    b, rc2 = c.decode_attention(q, wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0 and rc2 == 0
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
