"""CPU checks of the benchmark's report helpers: the exact unquantized
attention the quantization error is measured against, the error summary, and
the CPU-baseline record of the oracle."""
import numpy as np

import synth


def test_exact_attention_matches_oracle_on_a_bf16_cache(orc):
    """fp64 attention over the unquantized bf16 rows (plain torch in bench.py)
    equals the oracle's attention over a bf16 cache of the same rows: the bf16
    cache stores the rows unchanged, so both compute the same real numbers."""
    import bench
    wl = synth.make_workload("qe", "bf16", Hq=16, Hkv=4, seq_lens=[70, 1, 33], seed=3)
    ks, vs = wl.kv_all(0)
    q = wl.q(0)
    exact = bench.exact_attention_fp64(wl, ks, vs, [0, 1, 2], q)
    oc = orc.OracleCache("bf16", wl.Hkv, wl.D, wl.P, wl.num_pages)
    for b in range(wl.B):
        assert oc.quantize_store(ks[b], vs[b], wl.slots(b)) == 0
    ref, rc = oc.decode_attention(q, wl.page_table, wl.seq_lens, wl.sm_scale)
    assert rc == 0
    for b in range(wl.B):
        np.testing.assert_allclose(exact[b], ref[b], rtol=0, atol=1e-12)


def test_quant_error_orders_the_formats(orc):
    """On the same rows, the oracle's quantized attention is further from the
    unquantized answer the fewer bits the format keeps: bf16 is exact, E4M3
    (3 mantissa bits) beats E5M2 (2), and the FP4 formats are the furthest."""
    import bench
    wl = synth.make_workload("qe2", "bf16", Hq=16, Hkv=2, seq_lens=[300, 120], seed=9)
    ks, vs = wl.kv_all(0)
    q = wl.q(0)
    exact = bench.exact_attention_fp64(wl, ks, vs, [0, 1], q)
    err = {}
    for f in ("bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4"):
        oc = orc.OracleCache(f, wl.Hkv, wl.D, wl.P, wl.num_pages)
        s = wl.scales_for(f, ks, vs)
        for b in range(wl.B):
            assert oc.quantize_store(ks[b], vs[b], wl.slots(b), s) == 0
        got, rc = oc.decode_attention(q, wl.page_table, wl.seq_lens, wl.sm_scale)
        assert rc == 0
        err[f] = bench.quant_error({b: got[b] for b in (0, 1)}, exact)
        assert err[f]["rows"] == 2 * wl.Hq
    assert err["bf16"]["max_rel_l2"] < 1e-12
    assert 0 < err["fp8_e4m3"]["mean_rel_l2"] < err["fp8_e5m2"]["mean_rel_l2"]
    assert err["fp8_e5m2"]["mean_rel_l2"] < min(err["fp4_mx_block16"]["mean_rel_l2"],
                                               err["nvfp4"]["mean_rel_l2"])


def test_cpu_baseline_record(orc):
    """The oracle timings report all-core and one-thread rates for decode and
    for quantize-and-store, with the core counts used."""
    import bench
    wl = synth.make_workload("cb", "nvfp4", Hq=16, Hkv=2, seq_lens=[200, 64, 100, 90], seed=4)
    ks, vs = wl.kv_all(0)
    rec = bench.cpu_baseline(wl, ks, vs, seed=1003)
    assert rec["kind"] == "oracle" and rec["cores"] == orc.num_threads()
    assert rec["value"] > 0 and rec["single_thread"]["value"] > 0
    assert rec["single_thread"]["cores"] == 1
    assert rec["store"]["value"] > 0 and rec["store"]["single_thread_value"] > 0
