"""kvq_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory at call time (an application that must not call
cudaMalloc/cudaFree after start-up, or a plugin whose host framework owns all
device memory).  Its scratch is a static device array inside the library.

The entry point is called through the C ABI and its output is compared with
kvq_decode_attention (caller-provided workspace) on the same inputs, within the
decode tests' tolerance, on two calls in a row (the static scratch keeps the
previous call's contents).  This file is collected last on purpose, and it
passes both alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import bits_to_cuda, cuda_to_bits, gpu_cache_for, store_layer

pytestmark = pytest.mark.gpu


def _rel_abs(a, b):
    num = np.linalg.norm(a - b, axis=-1)
    den = np.linalg.norm(b, axis=-1)
    rel = np.where(den > 0, num / np.where(den > 0, den, 1), num)
    return float(rel.max()), float(np.abs(a - b).max())


@pytest.mark.parametrize("fmt,lens,Hq", [("nvfp4", [3000, 17, 0, 1500], 64),
                                         ("fp8_e4m3", [256, 256], 32)])
def test_noalloc_matches_workspace_entry_point(kvq, cuda, fmt, lens, Hq):
    wl = synth.make_workload(f"na_{fmt}", fmt, Hq=Hq, Hkv=8, seq_lens=lens, seed=99)
    c = gpu_cache_for(kvq, wl)
    store_layer(c, wl)
    q = bits_to_cuda(wl.q())
    pt = torch.from_numpy(wl.page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    ref_out = c.decode_attention(0, q, pt, sl, wl.sm_scale)
    ref = synth.bf16_bits_to_float(cuda_to_bits(ref_out)).astype(np.float64)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        kvq.kvq_decode_attention_noalloc(c.handle, 0, q, pt, sl, wl.sm_scale, out)
        torch.cuda.synchronize()
        assert c.device_error() == 0
        got = synth.bf16_bits_to_float(cuda_to_bits(out)).astype(np.float64)
        assert np.isfinite(got).all(), f"call {call}"
        rel, ab = _rel_abs(got, ref)
        assert rel <= 2e-3 and ab <= 1e-2, f"call {call}: rel {rel:.3e} abs {ab:.3e}"
        assert (got[np.asarray(lens) == 0] == 0).all()


def test_noalloc_rejects_sizes_beyond_its_scratch(kvq, cuda):
    c = kvq.KVQCache("fp8_e4m3", 1, 8, 128, 16, 64)
    limit = 16 << 20
    # 4096 sequences x 8 kv heads need more partial slots than 16 MiB holds
    B, Hq, mp = 4096, 64, 4
    assert kvq.kvq_decode_workspace_size(c.handle, B, Hq, mp) > limit
    q = torch.zeros(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros(B, mp, dtype=torch.int32, device="cuda")
    sl = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_attention_noalloc(c.handle, 0, q, pt, sl, 0.1, out)
    assert e.value.code == "KVQ_ERR_UNSUPPORTED" and "static" in str(e.value)


def test_noalloc_reports_invalid_arguments_as_the_workspace_call_does(kvq, cuda):
    """Bad sizes give KVQ_ERR_INVALID_ARG and an unsupported shape gives
    KVQ_ERR_UNSUPPORTED, exactly as kvq_decode_attention reports them."""
    c = kvq.KVQCache("fp8_e4m3", 1, 8, 128, 16, 64)
    q = torch.zeros(2, 64, 128, dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    sl = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    st = kvq.lib.kvq_decode_attention_noalloc(c.handle, 0, q.data_ptr(), 64, pt.data_ptr(), 4,
                                              sl.data_ptr(), -1, 0.1, out.data_ptr(), None)
    assert kvq._binding._STATUS[st] == "KVQ_ERR_INVALID_ARG"
    st = kvq.lib.kvq_decode_attention_noalloc(c.handle, 0, q.data_ptr(), 8 * 17, pt.data_ptr(), 4,
                                              sl.data_ptr(), 2, 0.1, out.data_ptr(), None)
    assert kvq._binding._STATUS[st] == "KVQ_ERR_UNSUPPORTED"
