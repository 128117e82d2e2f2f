"""Pins of the oracle's fp64 decode attention.

- Against PyTorch's scaled_dot_product_attention in float64 (with its own GQA
  head mapping) on K/V that PyTorch dequantizes independently.
- Closed forms: one token returns its value row; identical keys give the mean
  of the values; a dominant logit selects its row; a hand-computed two-token
  case; an empty sequence gives zeros.
"""
import math

import numpy as np
import pytest
import torch

import synth
from test_oracle_quant import E2M1_TABLE, _store_all


def _exact_kv(fmt, c, wl, b, which):
    """fp64 K^ or V^ [T][Hkv][D] decoded with PyTorch from the oracle's stored bytes."""
    data = c.k_data if which == "k" else c.v_data
    scl = c.k_scales if which == "k" else c.v_scales
    s = float(wl.scales()[0 if which == "k" else 1])
    slots = wl.slots(b)
    idx = np.array([[c.row_index(int(t), h) for h in range(wl.Hkv)] for t in slots]).reshape(-1)
    d, sc = data[idx], scl[idx]
    if fmt == "bf16":
        val = torch.from_numpy(d.view(np.int16).copy()).view(torch.bfloat16).double()
    elif fmt in ("fp8_e4m3", "fp8_e5m2"):
        dt = torch.float8_e4m3fn if fmt == "fp8_e4m3" else torch.float8_e5m2
        val = torch.from_numpy(d.copy()).view(dt).double() * s
    else:
        nib = np.stack([d & 0xF, d >> 4], axis=-1).reshape(d.shape[0], -1)
        mag = torch.from_numpy(E2M1_TABLE[nib & 7] * np.where(nib & 8, -1.0, 1.0))
        if fmt == "fp4_mx_block16":
            S = torch.from_numpy(sc.copy()).view(torch.float8_e8m0fnu).double()
        else:
            S = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).double() * s
        val = mag * S.repeat_interleave(16, dim=1)
    return val.reshape(len(slots), wl.Hkv, wl.D)


@pytest.mark.parametrize("fmt", ["bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4"])
def test_attention_matches_torch_sdpa(orc, fmt):
    wl = synth.make_workload(f"a_{fmt}", fmt, Hq=8, Hkv=2, D=64, seq_lens=[1, 37, 50, 16], seed=9)
    c = _store_all(orc, wl)
    q = wl.q()
    out, rc = c.decode_attention(q, wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0
    qd = torch.from_numpy(q.view(np.int16).copy()).view(torch.bfloat16).double()
    for b in range(wl.B):
        K = _exact_kv(fmt, c, wl, b, "k").permute(1, 0, 2)[None]     # [1, Hkv, T, D]
        V = _exact_kv(fmt, c, wl, b, "v").permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qd[b][None, :, None, :], K, V, scale=wl.sm_scale, enable_gqa=True)[0, :, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-12)


def _bf16(x):
    return synth.to_bf16_bits(torch.tensor(x, dtype=torch.float32))


def _single_seq_cache(orc, k, v, P=16):
    T, H, D = k.shape
    npages = max(1, (T + P - 1) // P)
    c = orc.OracleCache("bf16", H, D, P, npages)
    assert c.quantize_store(k, v, np.arange(T, dtype=np.int64), None) == 0
    pt = np.arange(npages, dtype=np.int32)[None]
    return c, pt


def test_closed_forms(orc):
    rng = np.random.default_rng(0)
    D = 16
    # one token: output equals its value row
    k = _bf16(rng.standard_normal((1, 1, D)))
    v = _bf16(rng.standard_normal((1, 1, D)))
    c, pt = _single_seq_cache(orc, k, v)
    q = _bf16(rng.standard_normal((1, 3, D)))
    out, _ = c.decode_attention(q, pt, np.array([1]), 0.3)
    for j in range(3):
        assert np.array_equal(out[0, j], synth.bf16_bits_to_float(v[0, 0]).astype(np.float64))
    # identical keys: uniform weights, output is the mean of the values
    T = 23
    k = np.repeat(_bf16(rng.standard_normal((1, 1, D))), T, axis=0)
    v = _bf16(rng.standard_normal((T, 1, D)))
    c, pt = _single_seq_cache(orc, k, v)
    out, _ = c.decode_attention(q[:, :1], pt, np.array([T]), 0.7)
    mean = synth.bf16_bits_to_float(v[:, 0]).astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(out[0, 0], mean, rtol=1e-13, atol=1e-15)
    # one dominant logit selects its value row
    kf = np.zeros((T, 1, D), np.float32)
    kf[11, 0, 0] = 64.0
    qf = np.zeros((1, 1, D), np.float32)
    qf[0, 0, 0] = 64.0
    c, pt = _single_seq_cache(orc, _bf16(kf), v)
    out, _ = c.decode_attention(_bf16(qf), pt, np.array([T]), 1.0)
    np.testing.assert_allclose(out[0, 0], synth.bf16_bits_to_float(v[11, 0]), rtol=0, atol=1e-300)


def test_two_token_hand_computed(orc):
    D = 16
    k = np.zeros((2, 1, D), np.float32)
    k[1, 0, 0] = 1.0                     # logits: z0 = 0, z1 = 1 (q = e0, scale 1)
    v = np.zeros((2, 1, D), np.float32)
    v[0, 0, 0] = 1.0
    v[1, 0, 1] = 1.0
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 1.0
    c, pt = _single_seq_cache(orc, _bf16(k), _bf16(v))
    out, _ = c.decode_attention(_bf16(q), pt, np.array([2]), 1.0)
    e = math.e
    expect = np.zeros(D)
    expect[0], expect[1] = 1 / (1 + e), e / (1 + e)
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-15, atol=0)


def test_empty_sequence_and_bad_page(orc):
    wl = synth.make_workload("e", "fp8_e4m3", Hq=4, Hkv=2, D=32, seq_lens=[0, 20], seed=3)
    c = _store_all(orc, wl)
    out, rc = c.decode_attention(wl.q(), wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0 and (out[0] == 0).all() and np.isfinite(out[1]).all() and (out[1] != 0).any()
    pt = wl.page_table.copy()
    pt[1, 1] = wl.num_pages + 5
    out, rc = c.decode_attention(wl.q(), pt, wl.seq_lens, wl.sm_scale)
    assert rc == -1 and (out[1] == 0).all()


def test_b_list_selects_sequences(orc):
    wl = synth.make_workload("s", "nvfp4", Hq=4, Hkv=2, D=32, seq_lens=[5, 30, 17], seed=4)
    c = _store_all(orc, wl)
    full, _ = c.decode_attention(wl.q(), wl.page_table, wl.seq_lens, wl.sm_scale)
    part, _ = c.decode_attention(wl.q(), wl.page_table, wl.seq_lens, wl.sm_scale, b_list=[2])
    assert np.array_equal(part[2], full[2]) and (part[:2] == 0).all()


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_extend_attention_matches_torch_causal_sdpa(orc, fmt):
    """A chunk of new query tokens at the end of each sequence: query i sees the
    sequence's tokens up to and including its own position (causal prefill)."""
    wl = synth.make_workload(f"x_{fmt}", fmt, Hq=8, Hkv=2, D=64, seq_lens=[45, 20], seed=13)
    c = _store_all(orc, wl)
    chunk = [5, 3]                                 # newest tokens of each sequence are queries
    q_seq = np.concatenate([np.full(n, b) for b, n in enumerate(chunk)])
    q_len = np.concatenate([np.arange(wl.seq_lens[b] - n, wl.seq_lens[b]) + 1 for b, n in enumerate(chunk)])
    q = synth.to_bf16_bits(torch.randn(len(q_seq), wl.Hq, wl.D, generator=torch.Generator().manual_seed(4)))
    out, rc = c.extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    qd = torch.from_numpy(q.view(np.int16).copy()).view(torch.bfloat16).double()
    i0 = 0
    for b, n in enumerate(chunk):
        T = int(wl.seq_lens[b])
        K = _exact_kv(fmt, c, wl, b, "k").permute(1, 0, 2)[None]      # [1, Hkv, T, D]
        V = _exact_kv(fmt, c, wl, b, "v").permute(1, 0, 2)[None]
        Q = qd[i0:i0 + n].permute(1, 0, 2)[None]                       # [1, Hq, n, D]
        # query j sits at position T - n + j: bottom-right aligned causal mask
        mask = torch.ones(n, T, dtype=torch.bool).tril(diagonal=T - n)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                               scale=wl.sm_scale, enable_gqa=True)
        np.testing.assert_allclose(out[i0:i0 + n], ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
        i0 += n


def test_extend_attention_arbitrary_positions(orc):
    """Queries at arbitrary positions of interleaved sequences: each equals
    PyTorch's SDPA over exactly its own prefix (no mask needed)."""
    fmt = "nvfp4"
    wl = synth.make_workload("xa", fmt, Hq=8, Hkv=2, D=32, seq_lens=[40, 23, 9], seed=17)
    c = _store_all(orc, wl)
    rng = np.random.default_rng(3)
    q_seq = rng.integers(0, wl.B, 12).astype(np.int32)
    q_len = np.array([rng.integers(0, int(wl.seq_lens[b]) + 1) for b in q_seq], np.int32)
    q = synth.to_bf16_bits(torch.randn(12, wl.Hq, wl.D, generator=torch.Generator().manual_seed(8)))
    out, rc = c.extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    qd = torch.from_numpy(q.view(np.int16).copy()).view(torch.bfloat16).double()
    for i, (b, T) in enumerate(zip(q_seq, q_len)):
        if T == 0:
            assert (out[i] == 0).all()
            continue
        K = _exact_kv(fmt, c, wl, int(b), "k")[:T].permute(1, 0, 2)[None]
        V = _exact_kv(fmt, c, wl, int(b), "v")[:T].permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qd[i][None, :, None, :], K, V,
                                                               scale=wl.sm_scale, enable_gqa=True)
        np.testing.assert_allclose(out[i], ref[0, :, 0, :].numpy(), rtol=1e-12, atol=1e-12)
