"""GPU parity of decode attention against the oracle's fp64 attention on the
same dequantized K/V.  Tolerance (per sequence and q head): relative L2 error
<= 2e-3 and elementwise abs error <= 1e-2, both counted in excess of the
exact answer's own bf16 rounding -- bf16(ref) is the best any bf16 output can
be, and its rounding alone exceeds 2e-3 relative L2 on some vectors."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (assert_attention_close, bits_to_cuda, gpu_cache_for, gpu_decode,
                      oracle_cache_for, store_layer)

pytestmark = pytest.mark.gpu
FORMATS = ["bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4"]


def _run(kvq, orc, wl, layer=0, seqs=None, **kw):
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl, layer)
    got = gpu_decode(c, wl, layer, **kw)
    assert c.device_error() == 0
    oc = oracle_cache_for(orc, wl, layer, seqs=seqs)
    ref, rc = oc.decode_attention(wl.q(layer), wl.page_table, wl.seq_lens, wl.sm_scale, b_list=seqs)
    assert rc == 0
    if seqs is not None:
        got, ref = got[seqs], ref[seqs]
    return got, ref


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (32, 8), (8, 8), (32, 2), (12, 3)])
def test_decode_small(kvq, orc, cuda, fmt, Hq, Hkv):
    wl = synth.make_workload(f"dec_{fmt}", fmt, Hq=Hq, Hkv=Hkv, seq_lens=[37, 1, 16, 0, 130, 17],
                             seed=40 + Hq)
    got, ref = _run(kvq, orc, wl)
    assert_attention_close(got, ref, f"{fmt} Hq={Hq} Hkv={Hkv}")
    assert (got[3] == 0).all()                            # empty sequence


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("P", [32, 64])
def test_decode_page_sizes(kvq, orc, cuda, fmt, P):
    wl = synth.make_workload(f"p_{fmt}", fmt, Hq=16, Hkv=4, P=P, seq_lens=[300, 65, 15], seed=7 + P)
    got, ref = _run(kvq, orc, wl)
    assert_attention_close(got, ref, f"{fmt} P={P}")


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_decode_many_short_sequences(kvq, orc, cuda, fmt):
    lens = list(np.random.default_rng(1).integers(0, 40, 300))
    wl = synth.make_workload(f"m_{fmt}", fmt, Hq=8, Hkv=2, seq_lens=lens, seed=77)
    got, ref = _run(kvq, orc, wl)
    assert_attention_close(got, ref, f"{fmt} 300 short sequences")


def test_cfg1_e4m3_small(kvq, orc, cuda):
    wl = synth.cfg1_e4m3_small()
    got, ref = _run(kvq, orc, wl)
    assert_attention_close(got, ref, "cfg1")


@pytest.mark.parametrize("fmt", ["fp8_e5m2", "fp8_e4m3"])
@pytest.mark.parametrize("scale_mode", ["amax", "one"])
def test_cfg2_llama8b_stack_sampled_layers(kvq, orc, cuda, fmt, scale_mode):
    wl = synth.cfg2_llama8b_stack(fmt, scale_mode=scale_mode)
    c = gpu_cache_for(kvq, wl)
    for layer in range(wl.layers):
        store_layer(c, wl, layer)
    torch.cuda.synchronize()
    assert c.device_error() == 0
    for layer in (0, 31):
        got = gpu_decode(c, wl, layer)
        oc = oracle_cache_for(orc, wl, layer)
        ref, rc = oc.decode_attention(wl.q(layer), wl.page_table, wl.seq_lens, wl.sm_scale)
        assert rc == 0
        assert_attention_close(got, ref, f"cfg2 {fmt} {scale_mode} layer {layer}")


def test_cfg4_nvfp4_32k_full_size_sampled(kvq, orc, cuda):
    """The benchmark's workload (70B layer, batch 32, ragged 24K-32K) in the
    benchmark's launch configuration; two sequences checked against the oracle."""
    wl = synth.cfg4_nvfp4_70b_32k()
    seqs = [int(np.argmax(wl.seq_lens)), 3]
    got, ref = _run(kvq, orc, wl, seqs=seqs)
    assert_attention_close(got, ref, "cfg4 sampled")


@pytest.mark.parametrize("fmt,B", [("bf16", 8), ("fp8_e4m3", 8), ("fp8_e5m2", 8),
                                   ("fp4_mx_block16", 8), ("fp8_e4m3", 32),
                                   ("fp4_mx_block16", 32)])
def test_32k_full_size_sampled(kvq, orc, cuda, fmt, B):
    """70B layer (Hq 64, Hkv 8) at 32K context, in the launch configuration the
    benchmark times: with 8 sequences every warp worker of the persistent grid
    gets 54 to 108 tiles (215 and more at 32 sequences), so each segment runs
    past several 30-tile page-id windows and long stage chains (and, for FP4
    block-16, long running V reference-exponent chains).  Three sequences, all
    q heads, element by element against the oracle."""
    wl = synth.cfg5_sweep_cell(fmt, 32768, B)
    seqs = [0, B // 2 - 1, B - 1]
    got, ref = _run(kvq, orc, wl, seqs=seqs)
    assert_attention_close(got, ref, f"{fmt} 32K x {B} sampled")


def test_cfg3_fp4_block16_16k_full_size_sampled(kvq, orc, cuda):
    """The FP4 block-16 workload (70B layer, batch 8 at 16K), two sequences."""
    wl = synth.cfg3_fp4b16_70b()
    seqs = [1, 6]
    got, ref = _run(kvq, orc, wl, seqs=seqs)
    assert_attention_close(got, ref, "cfg3 sampled")


def test_decode_bounded_wait_reports_timeout(kvq, cuda, monkeypatch):
    """Failure detection without a fault: with KVQ_FAULT=wait every warp's first
    stage wait targets an mbarrier that is never armed and gives up after a
    short limit.  The kernel stops issuing copies, lets the ones in flight land
    (bounded drain), reports KVQ_ERR_TIMEOUT and zeroes every output it could
    not compute; the next call on the same cache is correct again."""
    wl = synth.make_workload("tmo", "nvfp4", Hq=16, Hkv=2, seq_lens=[700, 300, 0, 64], seed=5)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    good = gpu_decode(c, wl)
    assert c.device_error() == 0
    monkeypatch.setenv("KVQ_FAULT", "wait")
    got = gpu_decode(c, wl)
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_TIMEOUT"]
    assert (got == 0).all()
    monkeypatch.delenv("KVQ_FAULT")
    again = gpu_decode(c, wl)
    assert c.device_error() == 0
    assert np.array_equal(again, good)


def test_decode_bad_page_and_length(kvq, cuda):
    wl = synth.make_workload("bad", "fp8_e4m3", Hq=8, Hkv=2, seq_lens=[40, 40, 40], seed=2)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    pt = wl.page_table.copy()
    pt[1, 1] = wl.num_pages + 3
    got = gpu_decode(c, wl, page_table=pt)
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_DEVICE_RANGE"]
    assert (got[1] == 0).all() and (got[0] != 0).any() and (got[2] != 0).any()
    got = gpu_decode(c, wl, seq_lens=[40, wl.max_pages * wl.P + 1, -1])
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_DEVICE_RANGE"]
    assert (got[1] == 0).all() and (got[2] == 0).all() and (got[0] != 0).any()


def test_decode_deterministic_and_workspace_checks(kvq, cuda):
    wl = synth.make_workload("det", "nvfp4", Hq=16, Hkv=2, seq_lens=[500, 77], seed=12)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    a = gpu_decode(c, wl)
    b = gpu_decode(c, wl)
    assert np.array_equal(a, b)
    q = bits_to_cuda(wl.q())
    pt = torch.from_numpy(wl.page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    n = c.workspace_size(wl.B, wl.Hq, wl.max_pages)
    small = torch.empty(n - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        c.decode_attention(0, q, pt, sl, wl.sm_scale, workspace=small)
    assert e.value.code == "KVQ_ERR_INVALID_ARG"
    with pytest.raises(kvq.KVQError) as e:
        c.workspace_size(1, 17 * 2, 4)                    # group 17 > 16
    cbad = kvq.KVQCache("fp8_e4m3", 1, 2, 64, 16, 4)     # head_dim 64: store only
    with pytest.raises(kvq.KVQError) as e:
        cbad.workspace_size(1, 4, 4)
    assert e.value.code == "KVQ_ERR_UNSUPPORTED"


@pytest.mark.parametrize("spread", [10, 20, 30])
def test_fp4_block16_wide_exponent_spread(kvq, orc, cuda, spread):
    """K and V rows whose 16-element blocks differ by up to 2^spread: inside the
    kernel each K block is held relative to its row's largest block and each V
    block relative to the largest seen so far (f16 subnormals down to 2^-24,
    smaller contributions flush); the result must stay within tolerance."""
    wl = synth.make_workload("spread", "fp4_mx_block16", Hq=16, Hkv=2, seq_lens=[70, 33], seed=spread)
    rng = np.random.default_rng(spread)
    mult = 2.0 ** (-spread * (np.arange(8) % 2)) * 2.0 ** rng.integers(-3, 4, size=8)
    ks, vs = [], []
    for b in range(wl.B):
        k, v = wl.kv_float(0, b)
        k = k * torch.from_numpy(np.repeat(mult, 16)).float()
        v = v * torch.from_numpy(np.repeat(mult[::-1].copy(), 16)).float()
        ks.append(synth.to_bf16_bits(k))
        vs.append(synth.to_bf16_bits(v))
    c = gpu_cache_for(kvq, wl)
    oc = orc.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    for b in range(wl.B):
        c.quantize_and_store(0, bits_to_cuda(ks[b]), bits_to_cuda(vs[b]),
                             torch.from_numpy(wl.slots(b)).cuda(), None)
        assert oc.quantize_store(ks[b], vs[b], wl.slots(b), None) == 0
    got = gpu_decode(c, wl)
    ref, rc = oc.decode_attention(wl.q(), wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0 and c.device_error() == 0
    assert_attention_close(got, ref, f"fp4 block-16 spread 2^{spread}")


@pytest.mark.parametrize("pattern", ["early_large", "late_large", "alternating"])
def test_fp4_block16_token_scale_jumps(kvq, orc, cuda, pattern):
    """Token groups whose magnitudes jump by 2^6 to 2^12 along the sequence: the
    K reference exponent is re-anchored per chunk (up and down) and the V
    running reference is raised mid-segment, while other chunks stay on the
    packed-integer factor path; long sequences so segments span many chunks."""
    T = 2000
    wl = synth.make_workload("jump", "fp4_mx_block16", Hq=16, Hkv=2, seq_lens=[T, 1500], seed=21)
    t = np.arange(T)
    if pattern == "early_large":
        e = np.where(t < 48, 12, 0)
    elif pattern == "late_large":
        e = np.where((t > 1200) & (t < 1260), 12, 0) - np.where((t > 400) & (t < 700), 6, 0)
    else:
        e = ((t // 64) % 3 - 1) * 6
    ks, vs = [], []
    for b in range(wl.B):
        k, v = wl.kv_float(0, b)
        # K jumps down where V jumps up: those tokens keep moderate logits, so
        # every chunk's logits and values carry weight in the output
        m = torch.from_numpy(2.0 ** e[: k.shape[0]]).float().view(-1, 1, 1)
        ks.append(synth.to_bf16_bits(k / m))
        vs.append(synth.to_bf16_bits(v * m))
    c = gpu_cache_for(kvq, wl)
    oc = orc.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    for b in range(wl.B):
        c.quantize_and_store(0, bits_to_cuda(ks[b]), bits_to_cuda(vs[b]),
                             torch.from_numpy(wl.slots(b)).cuda(), None)
        assert oc.quantize_store(ks[b], vs[b], wl.slots(b), None) == 0
    got = gpu_decode(c, wl)
    ref, rc = oc.decode_attention(wl.q(), wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0 and c.device_error() == 0
    assert_attention_close(got, ref, f"fp4 block-16 token jumps {pattern}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("L,P", [(34, 16), (48, 16), (49, 16), (100, 32), (200, 64), (47, 48)])
def test_decode_whole_stages_per_worker(kvq, orc, cuda, fmt, L, P):
    """Eight equal sequences over one kv head: each worker gets whole multi-tile
    stages (page slabs of 1 to 4 tiles, full and partial last tiles)."""
    wl = synth.make_workload(f"w_{fmt}", fmt, Hq=8, Hkv=1, P=P, seq_lens=[L] * 8, seed=L + P)
    got, ref = _run(kvq, orc, wl)
    assert_attention_close(got, ref, f"{fmt} L={L} P={P}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("sm_scale", [-0.0884, 0.0, -1.5])
def test_decode_nonpositive_sm_scale(kvq, orc, cuda, fmt, sm_scale):
    """sm_scale is any finite number: zero gives the mean of V, a negative one
    favours the least similar keys (the kernel folds the sign into the query)."""
    wl = synth.make_workload(f"neg_{fmt}", fmt, Hq=16, Hkv=4, seq_lens=[70, 1, 33, 200], seed=93)
    wl.sm_scale = sm_scale
    got, ref = _run(kvq, orc, wl)
    assert_attention_close(got, ref, f"{fmt} sm_scale={sm_scale}")


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
def test_decode_fp8q_negative_sm_scale(kvq, orc, cuda, fmt):
    """FP8-domain decode with sm_scale < 0 against the oracle's attention over
    the dequantized query."""
    wl = synth.make_workload(f"negq_{fmt}", fmt, Hq=16, Hkv=4, seq_lens=[70, 1, 33, 200], seed=94)
    wl.sm_scale = -0.0884
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    qs = [float(wl.q_scales(0)[0])]
    out = c.decode_attention_fp8q(0, bits_to_cuda(wl.q(0)), qs, torch.from_numpy(wl.page_table).cuda(),
                                  torch.from_numpy(wl.seq_lens).cuda(), wl.sm_scale)
    torch.cuda.synchronize()
    assert c.device_error() == 0
    got = synth.bf16_bits_to_float(
        out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    oc = oracle_cache_for(orc, wl, 0)
    ref, rc = oc.decode_attention_fp8q(wl.q(0), qs, wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0
    assert_attention_close(got, ref, f"{fmt} fp8 query, sm_scale < 0")
