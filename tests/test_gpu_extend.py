"""GPU parity of extend (chunked-prefill) attention over the quantized cache:
query token i of sequence q_seq[i] attends to that sequence's tokens
[0, q_len[i]).  Compared with the oracle's fp64 attention within the decode
tolerance (excess over bf16 rounding)."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (assert_attention_close, bits_to_cuda, cuda_to_bits, gpu_cache_for,
                      oracle_cache_for, store_layer)

pytestmark = pytest.mark.gpu
FORMATS = ["bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4"]


def _queries(wl, chunk, seed):
    """The newest chunk[b] tokens of each sequence b as queries (causal prefill
    of the chunk), plus their bf16 query rows."""
    q_seq = np.concatenate([np.full(n, b, np.int32) for b, n in enumerate(chunk)])
    q_len = np.concatenate([np.arange(int(wl.seq_lens[b]) - n, int(wl.seq_lens[b])) + 1
                            for b, n in enumerate(chunk)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed)
    q = synth.to_bf16_bits(torch.randn(len(q_seq), wl.Hq, wl.D, generator=g))
    return q, q_seq, q_len


def _gpu_extend(c, wl, q, q_seq, q_len):
    out = c.extend_attention(0, bits_to_cuda(q), torch.from_numpy(q_seq).cuda(),
                             torch.from_numpy(q_len).cuda(), torch.from_numpy(wl.page_table).cuda(),
                             wl.sm_scale)
    torch.cuda.synchronize()
    return synth.bf16_bits_to_float(cuda_to_bits(out)).astype(np.float64)


@pytest.mark.parametrize("fmt", FORMATS)
def test_extend_matches_oracle(kvq, orc, cuda, fmt):
    wl = synth.make_workload(f"ext_{fmt}", fmt, Hq=16, Hkv=4, seq_lens=[300, 65, 130, 17], seed=31)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q, q_seq, q_len = _queries(wl, [24, 1, 16, 17], seed=2)
    got = _gpu_extend(c, wl, q, q_seq, q_len)
    assert c.device_error() == 0
    ref, rc = oracle_cache_for(orc, wl).extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    assert_attention_close(got, ref, f"{fmt} extend")


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_extend_70b_shape_random_positions(kvq, orc, cuda, fmt):
    """70B head layout (64 q heads, 8 kv heads); queries at arbitrary positions
    of two long sequences, interleaved."""
    wl = synth.make_workload(f"ext70_{fmt}", fmt, Hq=64, Hkv=8, seq_lens=[2000, 777], seed=7)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    rng = np.random.default_rng(5)
    q_seq = rng.integers(0, 2, 40).astype(np.int32)
    q_len = np.array([rng.integers(1, int(wl.seq_lens[b]) + 1) for b in q_seq], np.int32)
    q = synth.to_bf16_bits(torch.randn(40, wl.Hq, wl.D, generator=torch.Generator().manual_seed(1)))
    got = _gpu_extend(c, wl, q, q_seq, q_len)
    assert c.device_error() == 0
    ref, rc = oracle_cache_for(orc, wl).extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    assert_attention_close(got, ref, f"{fmt} extend 70B")


@pytest.mark.parametrize("fmt", ["nvfp4", "fp4_mx_block16"])
def test_extend_last_token_matches_decode(kvq, orc, cuda, fmt):
    """One query per sequence at its last position is a decode: extend and
    decode agree with the oracle (and with each other) within the tolerance."""
    wl = synth.make_workload(f"ext_dec_{fmt}", fmt, Hq=16, Hkv=2, seq_lens=[500, 77, 0, 33], seed=4)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q = bits_to_cuda(wl.q())
    pt = torch.from_numpy(wl.page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    dec = c.decode_attention(0, q, pt, sl, wl.sm_scale)
    ext = c.extend_attention(0, q, torch.arange(wl.B, dtype=torch.int32, device="cuda"), sl, pt,
                             wl.sm_scale)
    torch.cuda.synchronize()
    assert c.device_error() == 0
    d = synth.bf16_bits_to_float(cuda_to_bits(dec)).astype(np.float64)
    e = synth.bf16_bits_to_float(cuda_to_bits(ext)).astype(np.float64)
    ref, rc = oracle_cache_for(orc, wl).decode_attention(wl.q(), wl.page_table, wl.seq_lens,
                                                         wl.sm_scale)
    assert rc == 0
    assert_attention_close(d, ref, "decode")
    assert_attention_close(e, ref, "extend")
    assert (e[2] == 0).all()


def test_extend_bad_rows_and_lengths(kvq, cuda):
    wl = synth.make_workload("ext_bad", "fp8_e4m3", Hq=8, Hkv=2, seq_lens=[40, 40], seed=2)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q, _, _ = _queries(wl, [2, 2], seed=3)
    q_seq = np.array([0, 5, 1, -1], np.int32)          # rows 5 and -1 do not exist
    q_len = np.array([40, 10, 40, 10], np.int32)
    got = _gpu_extend(c, wl, q, q_seq, q_len)
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_DEVICE_RANGE"]
    assert (got[1] == 0).all() and (got[3] == 0).all()
    assert (got[0] != 0).any() and (got[2] != 0).any()
    q_len = np.array([40, wl.max_pages * wl.P + 1, 40, 3], np.int32)
    got = _gpu_extend(c, wl, q, np.array([0, 1, 1, 0], np.int32), q_len)
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_DEVICE_RANGE"]
    assert (got[1] == 0).all() and (got[3] != 0).any()


@pytest.mark.parametrize("fmt", ["bf16", "fp8_e4m3", "nvfp4"])
@pytest.mark.parametrize("split", [False, True])
def test_extend_bad_page_poisons_only_its_sequence(kvq, orc, cuda, fmt, split):
    """A page id outside the pool in one sequence's page table: that
    sequence's rows are zero and the device error word says
    KVQ_ERR_DEVICE_RANGE; rows of the other sequences (some in the same CTA,
    in other passes) still match the oracle.  With a workspace the context is
    split and the poisoned partials are merged to zeros."""
    wl = synth.make_workload(f"extbad_{fmt}", fmt, Hq=16, Hkv=4, seq_lens=[3000, 2600, 4100], seed=41)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q, q_seq, q_len = _queries(wl, [16, 16, 16], seed=6)
    ref, rc = oracle_cache_for(orc, wl).extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    pt = wl.page_table.copy()
    pt[1, 40] = wl.num_pages + 5   # a page in the middle of sequence 1's context
    ws = None
    if split:
        need = kvq.kvq_extend_workspace_size(c.handle, len(q_seq), wl.Hq, wl.max_pages)
        assert need > 0
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = c.extend_attention(0, bits_to_cuda(q), torch.from_numpy(q_seq).cuda(), torch.from_numpy(q_len).cuda(),
                             torch.from_numpy(pt).cuda(), wl.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    assert c.device_error() == kvq._binding._STATUS_CODES["KVQ_ERR_DEVICE_RANGE"]
    got = synth.bf16_bits_to_float(cuda_to_bits(out)).astype(np.float64)
    bad = q_seq == 1
    assert (got[bad] == 0).all()
    assert_attention_close(got[~bad], ref[~bad], f"{fmt} extend beside a bad page")


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_extend_split_and_unsplit_plans_agree(kvq, orc, cuda, fmt):
    """Long contexts: the fastest plan splits each sequence's context across
    CTAs (partials merged from the workspace); without a workspace the call
    runs unsplit.  Both match the oracle."""
    wl = synth.make_workload(f"exs_{fmt}", fmt, Hq=64, Hkv=8, seq_lens=[3000, 1200, 4100], seed=8)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q, q_seq, q_len = _queries(wl, [16, 5, 16], seed=4)
    need = kvq.kvq_extend_workspace_size(c.handle, len(q_seq), wl.Hq, wl.max_pages)
    assert need > 0
    ref, rc = oracle_cache_for(orc, wl).extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    outs = []
    for ws_bytes in (need, 16):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out = c.extend_attention(0, bits_to_cuda(q), torch.from_numpy(q_seq).cuda(),
                                 torch.from_numpy(q_len).cuda(), torch.from_numpy(wl.page_table).cuda(),
                                 wl.sm_scale, workspace=ws)
        torch.cuda.synchronize()
        assert c.device_error() == 0
        got = synth.bf16_bits_to_float(cuda_to_bits(out)).astype(np.float64)
        assert_attention_close(got, ref, f"{fmt} extend workspace {ws_bytes}")
        outs.append(got)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("sm_scale", [-0.0884, 0.0])
def test_extend_nonpositive_sm_scale(kvq, orc, cuda, fmt, sm_scale):
    """sm_scale is any finite number (zero: the mean of V over the prefix; a
    negative one: the kernel folds the sign into the query)."""
    wl = synth.make_workload(f"extneg_{fmt}", fmt, Hq=16, Hkv=4, seq_lens=[300, 65, 130, 17], seed=32)
    wl.sm_scale = sm_scale
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q, q_seq, q_len = _queries(wl, [24, 1, 16, 17], seed=3)
    got = _gpu_extend(c, wl, q, q_seq, q_len)
    assert c.device_error() == 0
    ref, rc = oracle_cache_for(orc, wl).extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    assert_attention_close(got, ref, f"{fmt} extend sm_scale={sm_scale}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8_e5m2", "nvfp4", "fp4_mx_block16"])
@pytest.mark.parametrize("P", [32, 48])
def test_extend_page_sizes(kvq, orc, cuda, fmt, P):
    """Pages of 32 and 48 tokens: a 64-token chunk spans pages at other
    boundaries (48: not a power of two)."""
    wl = synth.make_workload(f"extP_{fmt}", fmt, Hq=16, Hkv=4, P=P, seq_lens=[300, 65, 130, 17], seed=33 + P)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q, q_seq, q_len = _queries(wl, [24, 1, 16, 17], seed=4)
    got = _gpu_extend(c, wl, q, q_seq, q_len)
    assert c.device_error() == 0
    ref, rc = oracle_cache_for(orc, wl).extend_attention(q, q_seq, q_len, wl.page_table, wl.sm_scale)
    assert rc == 0
    assert_attention_close(got, ref, f"{fmt} extend P={P}")
