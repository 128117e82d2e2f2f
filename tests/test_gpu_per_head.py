"""GPU parity of per-attention-head scales and on-device scale calibration
("Quantized KV cache" (vLLM features page): Supported schemes -- one scale per
kv head; Scale calibration approaches -- scales estimated from one batch of
tokens, then fixed).

Stores are compared with the oracle byte for byte, calibrated scales bit for
bit, attention within the decode tolerance (excess over bf16 rounding).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (assert_attention_close, bits_to_cuda, cuda_to_bits, gpu_decode, gpu_pools)

pytestmark = pytest.mark.gpu

HEAD_GAIN = np.array([1.0, 30.0, 0.003, 0.2, 5.0, 1e-4, 70.0, 0.5], np.float32)


def _workload(fmt, seq_lens, Hq=16, Hkv=4, seed=5, P=16):
    return synth.make_workload(f"ph_{fmt}", fmt, Hq=Hq, Hkv=Hkv, P=P, seq_lens=seq_lens, seed=seed)


def _rows(wl, b):
    """K, V bf16 bits of sequence b with very different magnitudes per kv head."""
    k, v = wl.kv_float(0, b)
    g = torch.from_numpy(HEAD_GAIN[: wl.Hkv]).view(1, -1, 1)
    return synth.to_bf16_bits(k * g), synth.to_bf16_bits(v * g.flip(1))


def _all_rows(wl):
    ks, vs = zip(*[_rows(wl, b) for b in range(wl.B)])
    return np.concatenate(ks), np.concatenate(vs)


def _per_head_scales(orc, wl):
    k, v = _all_rows(wl)
    return orc.calibrate_scales(wl.fmt, k, True), orc.calibrate_scales(wl.fmt, v, True)


def _assert_pools_equal(gpu, oc, fmt):
    ref = [oc.k_data, oc.v_data] + ([oc.k_scales, oc.v_scales] if fmt in ("fp4_mx_block16", "nvfp4") else [])
    for name, g, r in zip(["k_data", "v_data", "k_scales", "v_scales"], gpu, ref):
        bad = np.argwhere(g != r)
        assert bad.size == 0, f"{fmt} {name}: {len(bad)} bytes differ, first at {bad[0]}"


def _store_both(kvq, orc, wl, ks, vs, chunk=None):
    c = kvq.KVQCache(wl.fmt, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
    oc = orc.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    for b in range(wl.B):
        k, v = _rows(wl, b)
        T = int(wl.seq_lens[b])
        step = chunk or max(T, 1)
        for t0 in range(0, T, step):
            t1 = min(T, t0 + step)
            c.quantize_and_store_per_head(0, bits_to_cuda(k[t0:t1]), bits_to_cuda(v[t0:t1]),
                                          torch.from_numpy(wl.slots(b, t0, t1)).cuda(), ks, vs)
        assert oc.quantize_store(k, v, wl.slots(b), np.stack([ks, vs])) == 0
    torch.cuda.synchronize()
    assert c.device_error() == 0
    return c, oc


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2", "nvfp4", "fp4_mx_block16", "bf16"])
def test_per_head_store_bit_exact(kvq, orc, cuda, fmt):
    wl = _workload(fmt, [40, 17, 1, 33])
    ks, vs = _per_head_scales(orc, wl)
    c, oc = _store_both(kvq, orc, wl, ks, vs, chunk=7)
    _assert_pools_equal(gpu_pools(c, 0), oc, fmt)
    got_k, got_v = c.layer_head_scales(0)
    if fmt in ("fp8_e4m3", "fp8_e5m2", "nvfp4"):
        assert np.array_equal(np.float32(got_k), ks) and np.array_equal(np.float32(got_v), vs)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_per_head_dequantize_bit_exact(kvq, orc, cuda, fmt):
    wl = _workload(fmt, [30, 9])
    ks, vs = _per_head_scales(orc, wl)
    c, oc = _store_both(kvq, orc, wl, ks, vs)
    slots = np.concatenate([wl.slots(b) for b in range(wl.B)] + [np.array([-1], np.int64)])
    k, v = c.dequantize(0, torch.from_numpy(slots).cuda())
    ko, vo, rc = oc.dequantize(slots)
    assert rc == 0 and np.array_equal(cuda_to_bits(k), ko) and np.array_equal(cuda_to_bits(v), vo)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2", "nvfp4"])
@pytest.mark.parametrize("Hq,Hkv", [(16, 4), (64, 8)])
def test_per_head_decode_matches_oracle(kvq, orc, cuda, fmt, Hq, Hkv):
    wl = _workload(fmt, [300, 65, 0, 130], Hq=Hq, Hkv=Hkv, seed=Hq)
    ks, vs = _per_head_scales(orc, wl)
    c, oc = _store_both(kvq, orc, wl, ks, vs)
    got = gpu_decode(c, wl)
    assert c.device_error() == 0
    ref, rc = oc.decode_attention(wl.q(), wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0
    assert_attention_close(got, ref, f"{fmt} per-head Hq={Hq} Hkv={Hkv}")
    assert (got[2] == 0).all()


def test_uniform_per_head_scales_equal_the_per_tensor_path(kvq, orc, cuda):
    wl = _workload("nvfp4", [50, 20])
    outs = []
    for per_head in (False, True):
        c = kvq.KVQCache("nvfp4", 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
        for b in range(wl.B):
            k, v = _rows(wl, b)
            args = (0, bits_to_cuda(k), bits_to_cuda(v), torch.from_numpy(wl.slots(b)).cuda())
            if per_head:
                c.quantize_and_store_per_head(*args, [0.01] * wl.Hkv, [0.02] * wl.Hkv)
            else:
                c.quantize_and_store(*args, [0.01, 0.02])
        outs.append((gpu_pools(c, 0), gpu_decode(c, wl)))
    for a, b in zip(outs[0][0], outs[1][0]):
        assert np.array_equal(a, b)
    assert np.array_equal(outs[0][1], outs[1][1])


def _nonfinite(x):
    x = x.copy()
    x[0, 0, 3] = 0x7F80   # +inf
    x[1, 1, 5] = 0x7FC0   # NaN
    x[2, 2, 7] = 0xFF80   # -inf
    return x


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2", "nvfp4"])
@pytest.mark.parametrize("per_head", [False, True])
def test_calibration_matches_oracle(kvq, orc, cuda, fmt, per_head):
    wl = _workload(fmt, [70, 33], Hkv=8, Hq=16)
    k, v = _all_rows(wl)
    k, v = _nonfinite(k), _nonfinite(v)
    c = kvq.KVQCache(fmt, 2, wl.Hkv, wl.D, wl.P, wl.num_pages)
    c.calibrate_scales(1, bits_to_cuda(k), bits_to_cuda(v), per_head)
    got_k, got_v = c.layer_head_scales(1)
    ref_k, ref_v = orc.calibrate_scales(fmt, k, per_head), orc.calibrate_scales(fmt, v, per_head)
    n = wl.Hkv if per_head else 1
    assert np.array_equal(np.float32(got_k), np.broadcast_to(ref_k, (wl.Hkv,))[:wl.Hkv]), (got_k, ref_k)
    assert np.array_equal(np.float32(got_v), np.broadcast_to(ref_v, (wl.Hkv,))[:wl.Hkv])
    assert ref_k.shape == (n,)
    if not per_head:
        assert c.layer_scales(1) == (float(ref_k[0]), float(ref_v[0]))


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_calibration_many_tokens_odd_head_count(kvq, orc, cuda, fmt):
    """3 kv heads x 4 blocks per row (12 block columns, not a divisor of a
    CTA's 256 threads) over 40,000 tokens, more than one token per thread of
    the calibration grid: every head's maximum (planted at scattered tokens,
    beside non-finite values) is found."""
    n, H, D = 40000, 3, 64
    g = torch.Generator().manual_seed(17)
    x = [synth.to_bf16_bits(torch.randn(n, H, D, generator=g) * torch.tensor([0.5, 8.0, 0.01]).view(1, H, 1))
         for _ in range(2)]
    for i, (t, h, d) in enumerate([(39999, 0, 63), (12345, 1, 0), (7, 2, 31)]):
        x[0][t, h, d] = 0x4480 + i          # 1024 + i ulps: each head's largest K
        x[1][n - 1 - t, h, d] = 0xC300 + i  # -128 - ...: each head's largest V
    x[0][100, 1, 5] = 0x7F80
    x[1][200, 2, 9] = 0xFFC0
    c = kvq.KVQCache(fmt, 1, H, D, 16, 8)
    c.calibrate_scales(0, bits_to_cuda(x[0]), bits_to_cuda(x[1]), True)
    got_k, got_v = c.layer_head_scales(0)
    ref_k, ref_v = orc.calibrate_scales(fmt, x[0], True), orc.calibrate_scales(fmt, x[1], True)
    assert np.array_equal(np.float32(got_k), ref_k), (got_k, ref_k)
    assert np.array_equal(np.float32(got_v), ref_v), (got_v, ref_v)


def test_calibration_of_zeros_gives_one(kvq, cuda):
    c = kvq.KVQCache("fp8_e4m3", 1, 2, 32, 16, 2)
    z = torch.zeros(5, 2, 32, dtype=torch.bfloat16, device="cuda")
    c.calibrate_scales(0, z, z, True)
    assert c.layer_head_scales(0) == ([1.0, 1.0], [1.0, 1.0])


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_calibrated_layer_store_and_decode(kvq, orc, cuda, fmt):
    """Calibrate on the first sequence's rows on the device, then store every
    sequence with NULL scales: pools match the oracle stored with the oracle's
    calibration of the same rows; attention matches the oracle."""
    wl = _workload(fmt, [120, 64, 31], Hq=16, Hkv=4, seed=21)
    k0, v0 = _rows(wl, 0)
    c = kvq.KVQCache(fmt, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
    c.calibrate_scales(0, bits_to_cuda(k0), bits_to_cuda(v0), True)
    oc = orc.OracleCache(fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    s = np.stack([orc.calibrate_scales(fmt, k0, True), orc.calibrate_scales(fmt, v0, True)])
    for b in range(wl.B):
        k, v = _rows(wl, b)
        c.quantize_and_store(0, bits_to_cuda(k), bits_to_cuda(v), torch.from_numpy(wl.slots(b)).cuda())
        assert oc.quantize_store(k, v, wl.slots(b), s) == 0
    torch.cuda.synchronize()
    assert c.device_error() == 0
    _assert_pools_equal(gpu_pools(c, 0), oc, fmt)
    got = gpu_decode(c, wl)
    ref, rc = oc.decode_attention(wl.q(), wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0
    assert_attention_close(got, ref, f"{fmt} calibrated")


def test_scale_rules_per_head_and_calibrated(kvq, cuda):
    D, H = 32, 2
    x = bits_to_cuda(synth.to_bf16_bits(torch.randn(2, H, D)))
    s = torch.tensor([0, 1], dtype=torch.int64, device="cuda")
    c = kvq.KVQCache("fp8_e4m3", 4, H, D, 16, 1)
    c.quantize_and_store_per_head(0, x, x, s, [0.5, 0.25], [1.0, 2.0])
    c.quantize_and_store_per_head(0, x, x, s, [0.5, 0.25], [1.0, 2.0])     # same: fine
    for call in (lambda: c.quantize_and_store_per_head(0, x, x, s, [0.5, 0.3], [1.0, 2.0]),
                 lambda: c.quantize_and_store(0, x, x, s, [0.5, 1.0]),
                 lambda: c.calibrate_scales(0, x, x, True)):
        with pytest.raises(kvq.KVQError) as e:
            call()
        assert e.value.code == "KVQ_ERR_SCALE_MISMATCH"
    with pytest.raises(kvq.KVQError) as e:
        c.layer_scales(0)                                              # heads differ
    assert e.value.code == "KVQ_ERR_INVALID_ARG"
    assert c.layer_head_scales(0) == ([0.5, 0.25], [1.0, 2.0])
    # per-tensor store on a layer whose per-head scales are all equal
    c.quantize_and_store_per_head(1, x, x, s, [0.5, 0.5], [2.0, 2.0])
    c.quantize_and_store(1, x, x, s, [0.5, 2.0])
    assert c.layer_scales(1) == (0.5, 2.0)
    # calibrated layer: NULL scales only
    c.calibrate_scales(2, x, x, False)
    c.quantize_and_store(2, x, x, s)
    with pytest.raises(kvq.KVQError) as e:
        c.quantize_and_store(2, x, x, s, [1.0, 1.0])
    assert e.value.code == "KVQ_ERR_SCALE_MISMATCH"
    # bad per-head values
    for bad in ([0.0, 1.0], [float("nan"), 1.0], [-1.0, 1.0]):
        with pytest.raises(kvq.KVQError) as e:
            c.quantize_and_store_per_head(3, x, x, s, bad, [1.0, 1.0])
        assert e.value.code == "KVQ_ERR_INVALID_ARG"
    torch.cuda.synchronize()
    assert c.device_error() == 0


def test_per_head_calls_capture_in_a_cuda_graph(kvq, orc, cuda):
    """Calibration, per-head store and decode are stream-ordered with no host
    synchronization: captured once and replayed, they give the eager result."""
    wl = _workload("nvfp4", [48, 20], Hq=16, Hkv=4, seed=8)
    k, v = _all_rows(wl)
    kd, vd = bits_to_cuda(k), bits_to_cuda(v)
    slots = torch.from_numpy(np.concatenate([wl.slots(b) for b in range(wl.B)])).cuda()
    q = bits_to_cuda(wl.q())
    pt = torch.from_numpy(wl.page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()

    def run(c):
        c.calibrate_scales(0, kd, vd, True)
        c.quantize_and_store(0, kd, vd, slots)
        return c.decode_attention(0, q, pt, sl, wl.sm_scale, out=out, workspace=ws)

    eager = kvq.KVQCache("nvfp4", 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
    ws = torch.empty(eager.workspace_size(wl.B, wl.Hq, wl.max_pages), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    ref = cuda_to_bits(run(eager)).copy()
    graphed = kvq.KVQCache("nvfp4", 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
    out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run(graphed)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(cuda_to_bits(out), ref)
    assert graphed.device_error() == 0
