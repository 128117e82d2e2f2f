"""GPU parity of quantize-and-store and dequantize against the CPU oracle:
every byte of the data pools and scale planes, and every dequantized bf16
value, must be identical."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (bits_to_cuda, cuda_to_bits, gpu_cache_for, gpu_pools, oracle_cache_for,
                      store_layer)

pytestmark = pytest.mark.gpu
FORMATS = ["bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4"]


def _assert_pools_equal(gpu, orc_cache, fmt):
    ref = [orc_cache.k_data, orc_cache.v_data]
    if fmt in ("fp4_mx_block16", "nvfp4"):
        ref += [orc_cache.k_scales, orc_cache.v_scales]
    names = ["k_data", "v_data", "k_scales", "v_scales"]
    for n, g, r in zip(names, gpu, ref):
        bad = np.argwhere(g != r)
        assert bad.size == 0, f"{fmt} {n}: {len(bad)} bytes differ, first at row/col {bad[0]}"


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("D", [128, 64, 16])
def test_store_bit_exact(kvq, orc, cuda, fmt, D):
    wl = synth.make_workload(f"s_{fmt}", fmt, Hq=8, Hkv=3, D=D, seq_lens=[40, 17, 1, 64, 33],
                             seed=21 + D)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl, chunk=7)            # several calls per sequence, ragged chunks
    torch.cuda.synchronize()
    assert c.device_error() == 0
    _assert_pools_equal(gpu_pools(c, 0), oracle_cache_for(orc, wl), fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_dequantize_bit_exact(kvq, orc, cuda, fmt):
    wl = synth.make_workload(f"d_{fmt}", fmt, Hq=8, Hkv=2, D=128, seq_lens=[50, 16, 3], seed=31)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    oc = oracle_cache_for(orc, wl)
    slots = np.concatenate([wl.slots(b) for b in range(wl.B)] + [np.array([-1], np.int64)])
    k, v = c.dequantize(0, torch.from_numpy(slots).cuda())
    ko, vo, rc = oc.dequantize(slots)
    assert rc == 0
    assert np.array_equal(cuda_to_bits(k), ko) and np.array_equal(cuda_to_bits(v), vo)
    assert c.device_error() == 0


def _special_rows(D):
    x = np.random.default_rng(5).standard_normal((6, 1, D)).astype(np.float32)
    x[0, 0, :8] = [0.0, -0.0, np.inf, -np.inf, 1e38, -1e38, 1e-40, -1e-40]
    x[1, 0, :4] = [np.nan, -np.nan, 3.0e-45, 448.0]
    x[2] = 0.0                                           # all-zero row
    x[3] *= 1e-39                                        # subnormal row
    x[4] *= 1e30
    x[5, 0, ::2] = 1.0e-6
    return synth.to_bf16_bits(torch.from_numpy(x))


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("scale", [1.0, 0.37, 3.0e-3])
def test_fp8_special_values(kvq, orc, cuda, fmt, scale):
    D = 32
    x = _special_rows(D)
    slots = np.arange(x.shape[0], dtype=np.int64)
    c = kvq.KVQCache(fmt, 1, 1, D, 16, 1)
    c.quantize_and_store(0, bits_to_cuda(x), bits_to_cuda(x), torch.from_numpy(slots).cuda(),
                         [scale, scale])
    oc = orc.OracleCache(fmt, 1, D, 16, 1)
    assert oc.quantize_store(x, x, slots, [scale, scale]) == 0
    _assert_pools_equal(gpu_pools(c, 0), oc, fmt)


@pytest.mark.parametrize("fmt", ["fp4_mx_block16", "nvfp4"])
def test_fp4_extreme_finite_values(kvq, orc, cuda, fmt):
    D = 32
    x = _special_rows(D)
    x[0, 0, 2:4] = 0                                     # no infinities for the FP4 formats
    x[1, 0, :2] = 0                                      # no NaN for the FP4 formats
    slots = np.arange(x.shape[0], dtype=np.int64)
    c = kvq.KVQCache(fmt, 1, 1, D, 16, 1)
    g = [1.0e-3, 2.5] if fmt == "nvfp4" else None
    c.quantize_and_store(0, bits_to_cuda(x), bits_to_cuda(x), torch.from_numpy(slots).cuda(), g)
    oc = orc.OracleCache(fmt, 1, D, 16, 1)
    assert oc.quantize_store(x, x, slots, g) == 0
    _assert_pools_equal(gpu_pools(c, 0), oc, fmt)


def test_slot_skip_and_out_of_range(kvq, orc, cuda):
    D = 128
    x = synth.to_bf16_bits(torch.randn(4, 2, D, generator=torch.Generator().manual_seed(3)))
    c = kvq.KVQCache("nvfp4", 1, 2, D, 16, 2)
    slots = np.array([3, -1, 16 * 2 + 5, 20], np.int64)
    c.quantize_and_store(0, bits_to_cuda(x), bits_to_cuda(x), torch.from_numpy(slots).cuda(), [0.01, 0.02])
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_DEVICE_RANGE"]
    assert c.device_error() == 0                          # read-and-clear
    oc = orc.OracleCache("nvfp4", 2, D, 16, 2)
    assert oc.quantize_store(x, x, slots, [0.01, 0.02]) == -1
    _assert_pools_equal(gpu_pools(c, 0), oc, "nvfp4")


def test_scale_rules(kvq, cuda):
    D = 32
    x = bits_to_cuda(synth.to_bf16_bits(torch.randn(2, 1, D)))
    s = torch.tensor([0, 1], dtype=torch.int64, device="cuda")
    c = kvq.KVQCache("fp8_e4m3", 2, 1, D, 16, 1)
    c.quantize_and_store(0, x, x, s, [0.5, 0.25])
    c.quantize_and_store(0, x, x, s, [0.5, 0.25])          # same scales: fine
    with pytest.raises(kvq.KVQError) as e:
        c.quantize_and_store(0, x, x, s, [0.5, 0.3])
    assert e.value.code == "KVQ_ERR_SCALE_MISMATCH"
    c.quantize_and_store(1, x, x, s, None)                  # default scale 1.0
    assert c.layer_scales(1) == (1.0, 1.0) and c.layer_scales(0) == (0.5, 0.25)
    for bad in ([0.0, 1.0], [float("nan"), 1.0], [-1.0, 1.0], [float("inf"), 1.0]):
        with pytest.raises(kvq.KVQError) as e:
            c.quantize_and_store(1, x, x, s, bad)
        assert e.value.code == "KVQ_ERR_INVALID_ARG"
    c.quantize_and_store(0, x, x, s[:0], [0.5, 0.25])       # empty call is a no-op


def test_allocation_failure_is_reported(kvq, cuda, monkeypatch):
    monkeypatch.setenv("KVQ_FAULT", "alloc")
    with pytest.raises(kvq.KVQError) as e:
        kvq.KVQCache("fp8_e4m3", 1, 8, 128, 16, 4)
    assert e.value.code == "KVQ_ERR_OOM"


def test_prefill_16k_fp4_block16_sampled(kvq, orc, cuda):
    """The 70B-layer FP4 block-16 prefill (batch 8 x 16K tokens) stored in one
    call per sequence; two sequences compared byte for byte."""
    wl = synth.cfg3_fp4b16_70b()
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    torch.cuda.synchronize()
    assert c.device_error() == 0
    sample = [0, 5]
    oc = oracle_cache_for(orc, wl, seqs=sample)
    gk, gv, gks, gvs = gpu_pools(c, 0)
    for b in sample:
        rows = np.array([oc.row_index(int(s), h) for s in wl.slots(b) for h in range(wl.Hkv)])
        assert np.array_equal(gk[rows], oc.k_data[rows]) and np.array_equal(gv[rows], oc.v_data[rows])
        assert np.array_equal(gks[rows], oc.k_scales[rows]) and np.array_equal(gvs[rows], oc.v_scales[rows])


def _all_finite_bf16(shuffle_seed=0):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7F80) != 0x7F80
    bits = bits[finite]
    return np.random.default_rng(shuffle_seed).permutation(bits)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("scale", [1.0, 0.37, 3.0, 1.0 / 3.0, 0.0137, 2.0 ** -70, 2.0 ** -90, 1e30])
def test_fp8_store_every_bf16_value(kvq, orc, cuda, fmt, scale):
    """Every finite bf16 input, quantized with per-tensor scales that make the
    fp32 quotient exact, inexact, tiny, huge or overflowing: the kernel's
    division must round exactly like IEEE fp32 division (the oracle's)."""
    D = 64
    bits = _all_finite_bf16(1)
    n = bits.size // D
    x = bits[: n * D].reshape(n, 1, D)
    P = 16
    num_pages = (n + P - 1) // P
    slots = np.arange(n, dtype=np.int64)
    c = kvq.KVQCache(fmt, 1, 1, D, P, num_pages)
    c.quantize_and_store(0, bits_to_cuda(x), bits_to_cuda(x[::-1].copy()), torch.from_numpy(slots).cuda(),
                         [scale, scale * 1.5])
    oc = orc.OracleCache(fmt, 1, D, P, num_pages)
    assert oc.quantize_store(x, x[::-1].copy(), slots, [scale, scale * 1.5]) == 0
    _assert_pools_equal(gpu_pools(c, 0), oc, fmt)


@pytest.mark.parametrize("fmt", ["nvfp4", "fp4_mx_block16"])
@pytest.mark.parametrize("g", [0.0137, 1.0, 3.0e-5, 2.0 ** -85])
def test_fp4_store_every_bf16_value(kvq, orc, cuda, fmt, g):
    """Every finite bf16 input, in 16-element blocks of mixed magnitude: block
    scales and codes must match the oracle byte for byte."""
    D = 128
    bits = _all_finite_bf16(2)
    n = bits.size // D
    x = bits[: n * D].reshape(n, 1, D)
    P = 16
    num_pages = (n + P - 1) // P
    slots = np.arange(n, dtype=np.int64)
    c = kvq.KVQCache(fmt, 1, 1, D, P, num_pages)
    scales = [g, g * 7.0] if fmt == "nvfp4" else None
    c.quantize_and_store(0, bits_to_cuda(x), bits_to_cuda(x[::-1].copy()), torch.from_numpy(slots).cuda(),
                         scales)
    oc = orc.OracleCache(fmt, 1, D, P, num_pages)
    assert oc.quantize_store(x, x[::-1].copy(), slots, scales) == 0
    _assert_pools_equal(gpu_pools(c, 0), oc, fmt)


def _bf16_neighbors(v):
    """bf16 bit patterns of v and of its two bf16 neighbours (v exactly representable)."""
    b = int(np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16)
    return [b - 1, b, b + 1]


@pytest.mark.parametrize("g", [1.0, 1.0 + 2.0 ** -22, 1.0 - 2.0 ** -23, 1.0 + 2.0 ** -20, 1.0 - 2.0 ** -19,
                               0.75 * (1.0 + 2.0 ** -21)])
def test_nvfp4_store_near_decision_points(kvq, orc, cuda, g):
    """Blocks whose quotients x / S fall on, or within a few ulp of, the E2M1
    decision points 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 (and the code values):
    each block holds 6 * 2^k, so its scale code decodes to 2^k and S = 2^k g;
    g = 1 gives exact ties, g = 1 -+ 2^-22.. puts x / S just above / below them.
    Every code must be the correctly rounded quotient's, byte for byte with the
    oracle ("SGLang PR #21954 analysis: NVFP4 KV cache", NVFP4 two-level scaling)."""
    D, P = 128, 16
    pts = [0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0]
    cand = []
    for m in pts:
        for b in _bf16_neighbors(m):
            cand += [b, b | 0x8000]
    rows = []
    for k in (0, -3, 5):
        six = int(np.array([6.0 * 2.0 ** k], dtype=np.float32).view(np.uint32)[0] >> 16)
        sc = [((b & 0x7FFF) + (k << 7)) | (b & 0x8000) for b in cand]  # times 2^k (exponent add)
        blocks = [[six] + sc[i:i + 15] for i in range(0, len(sc), 15)]
        blocks = [bl + [0] * (16 - len(bl)) for bl in blocks]
        flat = [x for bl in blocks for x in bl]
        flat += [0] * (-len(flat) % D)
        rows += [flat[i:i + D] for i in range(0, len(flat), D)]
    x = np.array(rows, dtype=np.uint16).reshape(len(rows), 1, D)
    n = x.shape[0]
    num_pages = (n + P - 1) // P
    slots = np.arange(n, dtype=np.int64)
    scales = [g, 2.0 * g]
    c = kvq.KVQCache("nvfp4", 1, 1, D, P, num_pages)
    c.quantize_and_store(0, bits_to_cuda(x), bits_to_cuda(x[::-1].copy()), torch.from_numpy(slots).cuda(),
                         scales)
    oc = orc.OracleCache("nvfp4", 1, D, P, num_pages)
    assert oc.quantize_store(x, x[::-1].copy(), slots, scales) == 0
    _assert_pools_equal(gpu_pools(c, 0), oc, "nvfp4")
