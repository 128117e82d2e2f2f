"""GPU parity of FP8-domain decode attention ("Quantized KV cache" (vLLM), FP8
KV cache overview and Supported schemes; reading R17): the query quantized to
E4M3 with a per-tensor or per-q-head q_scale, QK^T on FP8 tensor cores over
the query and cache codes.

- Query codes (kvq_quantize_query) are bit-exact against the oracle for every
  bf16 bit pattern under per-tensor scales on both sides of the range where
  the corrected quotient is used, and for per-head scales.
- Attention is compared element by element with the oracle's fp64 attention
  over the dequantized query, with the decode tolerance (relative L2 <= 2e-3
  and abs <= 1e-2 per (sequence, q head), in excess of bf16(ref)'s rounding).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (assert_attention_close, bits_to_cuda, cuda_to_bits, gpu_cache_for,
                      oracle_cache_for, store_layer)

pytestmark = pytest.mark.gpu
FP8 = ["fp8_e4m3", "fp8_e5m2"]


def _gpu_fp8q(c, wl, qs, layer=0):
    q = bits_to_cuda(wl.q(layer))
    pt = torch.from_numpy(wl.page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    out = c.decode_attention_fp8q(layer, q, list(qs), pt, sl, wl.sm_scale)
    torch.cuda.synchronize()
    return synth.bf16_bits_to_float(cuda_to_bits(out)).astype(np.float64)


def _run(kvq, orc, wl, per_head, seqs=None):
    qs = wl.q_scales(0, per_head)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    got = _gpu_fp8q(c, wl, qs)
    assert c.device_error() == 0
    oc = oracle_cache_for(orc, wl, seqs=seqs)
    ref, rc = oc.decode_attention_fp8q(wl.q(0), qs, wl.page_table, wl.seq_lens, wl.sm_scale,
                                       b_list=seqs)
    assert rc == 0
    if seqs is not None:
        got, ref = got[seqs], ref[seqs]
    return got, ref


@pytest.mark.parametrize("scale", [1.0, 0.37, 3.1e-3, 2.5e-27, 1e30])
def test_quantize_query_every_bf16_value(kvq, orc, cuda, scale):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(128, 4, 128)
    codes = torch.empty(bits.shape, dtype=torch.uint8, device="cuda")
    kvq.kvq_quantize_query(bits_to_cuda(bits), [scale], codes)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), orc.quantize_query(bits, [scale]))


def test_quantize_query_per_head(kvq, orc, cuda):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((33, 16, 128)).astype(np.float32) * np.float32(3.0)
    bits = synth.to_bf16_bits(torch.from_numpy(x))
    scales = np.geomspace(1e-3, 5.0, 16).astype(np.float32)
    codes = torch.empty(bits.shape, dtype=torch.uint8, device="cuda")
    kvq.kvq_quantize_query(bits_to_cuda(bits), list(scales), codes)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), orc.quantize_query(bits, scales))


@pytest.mark.parametrize("fmt", FP8)
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (32, 8), (8, 8), (12, 3)])
def test_fp8q_decode_small(kvq, orc, cuda, fmt, per_head, Hq, Hkv):
    wl = synth.make_workload(f"q8s_{fmt}", fmt, Hq=Hq, Hkv=Hkv, seq_lens=[37, 1, 16, 0, 130, 17],
                             seed=60 + Hq)
    got, ref = _run(kvq, orc, wl, per_head)
    assert_attention_close(got, ref, f"fp8q {fmt} Hq={Hq} Hkv={Hkv} per_head={per_head}")
    assert (got[3] == 0).all()


@pytest.mark.parametrize("fmt", FP8)
def test_fp8q_decode_pages_and_whole_stages(kvq, orc, cuda, fmt):
    for P, lens in ((32, [300, 65, 15]), (64, [200] * 8), (16, [49] * 8)):
        wl = synth.make_workload(f"q8p_{fmt}", fmt, Hq=8, Hkv=1, P=P, seq_lens=lens, seed=P)
        got, ref = _run(kvq, orc, wl, per_head=True)
        assert_attention_close(got, ref, f"fp8q {fmt} P={P}")


@pytest.mark.parametrize("fmt", FP8)
def test_fp8q_32k_full_size_sampled(kvq, orc, cuda, fmt):
    """70B layer, 8 x 32K, in the benchmark's launch configuration: every warp
    segment spans several page-id windows; three sequences against the oracle."""
    wl = synth.cfg5_sweep_cell(fmt, 32768, 8)
    got, ref = _run(kvq, orc, wl, per_head=False, seqs=[0, 3, 7])
    assert_attention_close(got, ref, f"fp8q {fmt} 32K x 8 sampled")


def test_fp8q_rejects_other_formats_and_bad_scales(kvq, cuda):
    wl = synth.make_workload("q8bad", "nvfp4", Hq=8, Hkv=2, seq_lens=[20], seed=1)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q = bits_to_cuda(wl.q())
    pt = torch.from_numpy(wl.page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    with pytest.raises(kvq.KVQError) as e:
        c.decode_attention_fp8q(0, q, [0.01], pt, sl, wl.sm_scale)
    assert e.value.code == "KVQ_ERR_UNSUPPORTED"
    wl8 = synth.make_workload("q8bad8", "fp8_e4m3", Hq=8, Hkv=2, seq_lens=[20], seed=1)
    c8 = gpu_cache_for(kvq, wl8)
    store_layer(c8, wl8)
    for qs in ([0.0], [float("nan")], [0.01] * 3, [-1.0]):
        with pytest.raises(kvq.KVQError) as e:
            c8.decode_attention_fp8q(0, q, qs, pt, sl, wl8.sm_scale)
        assert e.value.code == "KVQ_ERR_INVALID_ARG"


def test_fp8q_bad_page_poisons_only_its_sequence(kvq, cuda):
    wl = synth.make_workload("q8pg", "fp8_e4m3", Hq=8, Hkv=2, seq_lens=[40, 40, 40], seed=2)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    pt = wl.page_table.copy()
    pt[1, 1] = wl.num_pages + 3
    q = bits_to_cuda(wl.q())
    out = c.decode_attention_fp8q(0, q, list(wl.q_scales()), torch.from_numpy(pt).cuda(),
                                  torch.from_numpy(wl.seq_lens).cuda(), wl.sm_scale)
    got = synth.bf16_bits_to_float(cuda_to_bits(out))
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_DEVICE_RANGE"]
    assert (got[1] == 0).all() and (got[0] != 0).any() and (got[2] != 0).any()
