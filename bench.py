#!/usr/bin/env python
"""Decode-step benchmark of the quantized paged KV store on GB300.

One step = quantize-and-store of each sequence's newest token (K and V) into
the paged cache, then fused-dequant split-K GQA decode attention of one query
token per sequence over the whole cache (store + decode + merge kernels).

Workload (default): one Llama-3-70B-shaped layer (64 q heads, 8 kv heads,
head_dim 128), NVFP4 cache, page size 16, batch 32 with ragged context lengths
uniform in [24K, 32K] and random page tables ("32K ctx x 32 seqs").  The
cache (~1.06 GB) is larger than L2 (129 MB), so no L2 flush is needed between
steps.

Prints ONE JSON line on rank 0.  Under torchrun each rank runs its own batch
(weak scaling, no collective on the data path); the timed region is bracketed
by a barrier and the max over ranks is taken.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--format nvfp4|fp8_e4m3|...] [--sweep FILE]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV GB/s and tokens/s at 32K ctx×32 seqs (fp8/fp4) vs HBM peak"
FALLBACK_HBM_GBS = 6800.0   # one earlier GB300 copy-bandwidth measurement
# Bytes per (token, kv head) of K plus V at head_dim 128.
KV_BYTES = {"bf16": 512, "fp8_e4m3": 256, "fp8_e5m2": 256, "fp4_mx_block16": 144, "nvfp4": 144}
DTYPE = {"bf16": "bf16 cache; bf16 mma, f32 accumulate",
         "fp8_e4m3": "e4m3 cache; f16 mma, f32 accumulate",
         "fp8_e5m2": "e5m2 cache; f16 mma, f32 accumulate",
         "fp4_mx_block16": "e2m1+e8m0 cache; f16 mma, f32 accumulate",
         "nvfp4": "e2m1+e4m3 cache; f16 mma, f32 accumulate"}
# dram read+write bytes per decode call on the full-size workload, from an ncu
# capture of the batch-8 case of the same workload scaled by units processed,
# keyed by the hash of the split-kernel sources it was taken on: any change to
# those sources reports null until re-measured.
NCU_TRAFFIC = {("nvfp4", "c4e8e5df00bf1dc9"): 1091647038,
               ("fp4_mx_block16", "c4e8e5df00bf1dc9"): 1093249874}

# steps between timed decode calls inside the timed step loop
DECODE_SAMPLE = 8


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--format", default="nvfp4")
    p.add_argument("--seed", type=int, default=1004)
    p.add_argument("--sweep", default=None, help="also run the format x context x batch sweep, "
                   "one JSON line per cell appended to this file")
    p.add_argument("--sweep-cells", default=None, help="comma-separated fmt:ctx:batch cells of "
                   "the sweep to run (default: all)")
    p.add_argument("--sweep-only", action="store_true", help="run only the --sweep measurement")
    p.add_argument("--store", default=None, help="also time quantize-and-store of the 70B-layer "
                   "16K x 8 prefill in every format, one JSON line per format appended to this file")
    p.add_argument("--store-formats", default=None, help="comma-separated subset for --store")
    p.add_argument("--store-only", action="store_true",
                   help="run only the --store measurement (no decode line)")
    p.add_argument("--next", default=None, help="time the per-head-scale decode, on-device "
                   "calibration and extend attention paths, one JSON line each appended to this file")
    p.add_argument("--quant-error", default=None, help="report the quantization error of every "
                   "format on the specified workloads (sampled sequences, GPU output against fp64 "
                   "attention over the unquantized bf16 K/V), one JSON line each appended to this file")
    p.add_argument("--no-per-format", action="store_true",
                   help="skip the per-format decode timings of the bench workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--batch", type=int, default=32,
                   help="sequences per rank (32 is the specified workload; smaller only for profiling)")
    return p.parse_args(argv)


# ---------------------------------------------------------------- distributed
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, init_method="env://", rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_ms: float, per_rank_bytes: float, device=None):
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    import torch.distributed as dist
    world = dist.get_world_size() if (dist.is_available() and dist.is_initialized()) else 1
    ms = max_over_ranks(per_rank_ms, device)
    return ms, per_rank_bytes * world / (ms * 1e-3) / 1e9


# --------------------------------------------------------------------- helpers
def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBps", "hbm"):
            if k in d:
                return float(d[k]), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def peak_bf16():
    """Measured dense bf16 tensor TFLOP/s (burst) from MEASURED_PEAKS.json, else
    the 1915 TFLOP/s fallback of an earlier GB300 measurement."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError, TypeError):
        return 1915.0, "fallback"


def decode_source_hash():
    h = hashlib.sha256()
    for n in ("kvq_decode.cu", "kvq_decode_args.cuh", "kvq_codecs.cuh"):
        with open(os.path.join(ROOT, "quantized_paged_kv_store_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.out,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    mx.append(float(c[2]))
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def algorithmic_bytes(wl, fmt):
    """KV bytes of every cached token + Q + O of one decode call."""
    kv = int(wl.seq_lens.astype("int64").sum()) * wl.Hkv * KV_BYTES[fmt]
    qo = 2 * wl.B * wl.Hq * wl.D * 2
    return kv + qo


def store_bytes(wl, fmt):
    """bf16 K and V read plus cache rows written for one new token per sequence."""
    per_row = wl.D * 2 * 2 + KV_BYTES[fmt]
    return wl.B * wl.Hkv * per_row


def make_workload(fmt, seed, T=None, B=None):
    import synth
    if T is None:
        wl = synth.cfg4_nvfp4_70b_32k(seed=seed, B=B or 32)
        if fmt != "nvfp4":
            wl.fmt = fmt
            wl.name = wl.name.replace("nvfp4", fmt)
        return wl
    return synth.cfg5_sweep_cell(fmt, T, B, seed=seed)


# ------------------------------------------------- quantization error (no oracle)
def exact_attention_fp64(wl, ks, vs, seqs, q_bits):
    """fp64 attention of the given sequences over their UNQUANTIZED bf16 K/V
    (plain torch matmul/softmax, q head j reads kv head j // G): the answer an
    unquantized cache would give, against which the quantized formats' outputs
    are compared.  Returns {b: float64 [Hq][D]}."""
    import numpy as np
    import torch
    import synth
    G = wl.Hq // wl.Hkv
    out = {}
    for b in seqs:
        q = torch.from_numpy(synth.bf16_bits_to_float(q_bits[b]).astype(np.float64))  # [Hq][D]
        K = torch.from_numpy(synth.bf16_bits_to_float(ks[b]).astype(np.float64))    # [T][Hkv][D]
        V = torch.from_numpy(synth.bf16_bits_to_float(vs[b]).astype(np.float64))
        o = torch.zeros(wl.Hq, wl.D, dtype=torch.float64)
        if K.shape[0] > 0:
            for h in range(wl.Hkv):
                z = (q[h * G:(h + 1) * G] @ K[:, h].T) * wl.sm_scale
                o[h * G:(h + 1) * G] = torch.softmax(z, dim=-1) @ V[:, h]
        out[b] = o.numpy()
    return out


def quant_error(got_rows, exact):
    """Per (sequence, q head) relative L2 error of an attention output against
    the exact unquantized answer: max and mean over the sampled rows, and the
    largest elementwise error."""
    import numpy as np
    rel, ab = [], 0.0
    for b, ref in exact.items():
        g = got_rows[b]
        den = np.linalg.norm(ref, axis=-1)
        num = np.linalg.norm(g - ref, axis=-1)
        rel.extend(list(np.where(den > 0, num / np.where(den > 0, den, 1), num)))
        ab = max(ab, float(np.abs(g - ref).max()))
    return {"max_rel_l2": float(np.max(rel)), "mean_rel_l2": float(np.mean(rel)), "max_abs": ab,
            "rows": len(rel)}


def out_rows(d_out, seqs):
    import numpy as np
    import synth
    bits = d_out.contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)
    return {b: synth.bf16_bits_to_float(bits[b]).astype(np.float64) for b in seqs}


# --------------------------------------------------------------- oracle timing
def oracle_time(wl, seqs, ks, vs, reps=1):
    """Seconds the CPU oracle takes to run decode attention for `seqs` (after
    storing their tokens, untimed), and the algorithmic bytes it processed."""
    import numpy as np
    import oracle
    c = oracle.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    s = wl.scales(0)
    for b in seqs:
        c.quantize_store(ks[b], vs[b], wl.slots(b), s)
    q = wl.q(0)
    t0 = time.perf_counter()
    for _ in range(reps):
        c.decode_attention(q, wl.page_table, wl.seq_lens, wl.sm_scale, b_list=np.array(seqs))
    dt = (time.perf_counter() - t0) / reps
    nbytes = sum(int(wl.seq_lens[b]) for b in seqs) * wl.Hkv * KV_BYTES[wl.fmt] + \
        len(seqs) * wl.Hq * wl.D * 4
    return dt, nbytes, oracle.num_threads()


def oracle_store_time(n_tokens, seed):
    """Seconds the CPU oracle takes to quantize-and-store an n_tokens prefix of
    one sequence of the FP4 block-16 prefill workload (70B layer, 16K), and the
    algorithmic bytes (bf16 K and V read, cache rows and scales written, slot ids)."""
    import oracle
    import synth
    wl = synth.cfg3_fp4b16_70b(seed=seed)
    k, v = wl.kv(0, 0, 0, n_tokens)
    c = oracle.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    slots = wl.slots(0, 0, n_tokens)
    t0 = time.perf_counter()
    c.quantize_store(k, v, slots, None)
    dt = time.perf_counter() - t0
    nbytes = n_tokens * wl.Hkv * (2 * wl.D * 2 + 2 * (wl.D // 2 + wl.D // 16)) + n_tokens * 8
    return dt, nbytes


def cpu_baseline(wl, ks, vs, seed):
    """The oracle as it stands, on this host's cores: fp64 decode attention of a
    sample of the bench workload (all cores and one thread) and quantize-and-store
    of a sample of the FP4 block-16 prefill (all cores and one thread)."""
    import oracle
    cores = oracle.num_threads()
    seqs = list(range(min(4, wl.B)))
    dt, nb, _ = oracle_time(wl, seqs, ks, vs)
    # one thread: one sequence
    oracle.set_num_threads(1)
    try:
        dt1, nb1, _ = oracle_time(wl, [0], ks, vs)
        st1, sb1 = oracle_store_time(2048, seed)
    finally:
        oracle.set_num_threads(cores)
    st, sb = oracle_store_time(8192, seed)
    ntok = sum(int(wl.seq_lens[b]) for b in seqs)
    return {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle decode attention of sequences {seqs} ({ntok} tokens x "
                      f"{wl.Hkv} kv heads, all {wl.Hq} q heads) of the same workload; {dt:.2f} s",
            "single_thread": {"value": round(nb1 / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"sequence 0 ({int(wl.seq_lens[0])} tokens); {dt1:.2f} s"},
            "store": {"value": round(sb / st / 1e9, 4), "unit": "GB/s", "cores": cores,
                      "single_thread_value": round(sb1 / st1 / 1e9, 4),
                      "sample": f"oracle quantize-and-store (fp4_mx_block16) of the first 8192 "
                                f"(one thread: 2048) tokens of sequence 0 of the 70B-layer 16K x 8 "
                                f"prefill; {st:.2f} s / {st1:.2f} s"}}


# ------------------------------------------------------------------- our arm
PER_FORMAT = ("nvfp4", "fp4_mx_block16", "fp8_e4m3", "fp8_e5m2", "bf16")


def per_format_cells(args, wl, ks, vs, d_q, d_pt, d_sl, exact, dev, peak):
    """Decode attention of the same workload (same K/V draws, every token
    stored) in each cache format: mean CUDA-event time per call issued from
    Python, the device time per call from CUDA-graph replay (the way a serving
    loop replays decode; no host launch gaps), algorithmic GB/s and fraction of
    peak of each, and the quantization error of its output on the sampled
    sequences."""
    import numpy as np
    import torch
    import quantized_paged_kv_store_gb300 as kvq
    kall = synth_to_cuda(np.concatenate(ks))
    vall = synth_to_cuda(np.concatenate(vs))
    slots = torch.from_numpy(np.concatenate([wl.slots(b) for b in range(wl.B)])).to(dev)
    steps = max(20, min(args.steps, 200))
    warm = max(3, min(args.warmup, 10))
    cells = {}
    for f in PER_FORMAT:
        scales = [float(x) for x in wl.scales_for(f, ks, vs)]
        cache = kvq.KVQCache(f, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
        cache.quantize_and_store(0, kall, vall, slots, scales)
        out = torch.empty_like(d_q)
        ws = torch.empty(cache.workspace_size(wl.B, wl.Hq, wl.max_pages), dtype=torch.uint8, device=dev)
        ms = _time_calls(lambda: cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale, out, ws),
                         steps, warm)
        if cache.device_error() != 0:
            raise RuntimeError(f"device error in the {f} per-format decode")
        gus = _graph_us(lambda st: cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale, out, ws,
                                                          stream=st))
        if cache.device_error() != 0:
            raise RuntimeError(f"device error in the {f} per-format decode (graph)")
        nbytes = algorithmic_bytes(wl, f)
        gbs = nbytes / (ms * 1e-3) / 1e9
        ggbs = nbytes / (gus * 1e-6) / 1e9
        cells[f] = {"ms_per_call": round(ms, 5), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
                    "graph_ms_per_call": round(gus * 1e-3, 5), "graph_GBps": round(ggbs, 1),
                    "graph_frac": round(ggbs / peak, 4),
                    "bytes_per_call": nbytes, "calls": steps,
                    "quant_error": {k: (round(v, 6) if isinstance(v, float) else v)
                                    for k, v in quant_error(out_rows(out, exact.keys()), exact).items()}}
        if f in ("fp8_e4m3", "fp8_e5m2"):
            # FP8-domain attention: the query quantized to E4M3 (per-tensor
            # q_scale = amax / 448), QK^T on FP8 tensor cores
            qs = [float(x) for x in wl.q_scales(0)]
            ms = _time_calls(lambda: cache.decode_attention_fp8q(0, d_q, qs, d_pt, d_sl, wl.sm_scale,
                                                                 out, ws), steps, warm)
            gus = _graph_us(lambda st: cache.decode_attention_fp8q(0, d_q, qs, d_pt, d_sl, wl.sm_scale,
                                                                   out, ws, stream=st))
            if cache.device_error() != 0:
                raise RuntimeError(f"device error in the {f} FP8-query decode")
            gbs = nbytes / (ms * 1e-3) / 1e9
            ggbs = nbytes / (gus * 1e-6) / 1e9
            cells[f + "+fp8_query"] = {
                "ms_per_call": round(ms, 5), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
                "graph_ms_per_call": round(gus * 1e-3, 5), "graph_GBps": round(ggbs, 1),
                "graph_frac": round(ggbs / peak, 4),
                "bytes_per_call": nbytes, "calls": steps, "q_scale": qs[0],
                "quant_error": {k: (round(v, 6) if isinstance(v, float) else v)
                                for k, v in quant_error(out_rows(out, exact.keys()), exact).items()}}
        cache.close()
    del kall, vall
    return cells


def run_cell(args, fmt, T=None, B=None, with_cpu=False, with_e2e=True, with_extra=False):
    import numpy as np
    import torch
    import quantized_paged_kv_store_gb300 as kvq
    import synth

    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = make_workload(fmt, args.seed + 7919 * rank, T, B if T is not None else args.batch)
    ks, vs = wl.kv_all(0)
    scales = [float(x) for x in wl.scales(0)]
    cache = kvq.KVQCache(fmt, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
    stream = torch.cuda.current_stream()
    # prefill: every token but the newest of each sequence (untimed)
    for b in range(wl.B):
        T_b = int(wl.seq_lens[b])
        if T_b > 1:
            cache.quantize_and_store(0, synth_to_cuda(ks[b][:T_b - 1]), synth_to_cuda(vs[b][:T_b - 1]),
                                     torch.from_numpy(wl.slots(b, 0, T_b - 1)).to(dev), scales)
    new_k = np.stack([ks[b][int(wl.seq_lens[b]) - 1] for b in range(wl.B)])
    new_v = np.stack([vs[b][int(wl.seq_lens[b]) - 1] for b in range(wl.B)])
    new_slots = np.array([wl.slots(b, int(wl.seq_lens[b]) - 1)[0] for b in range(wl.B)], np.int64)
    q_h = wl.q(0)
    # device-resident step inputs
    d_k, d_v = synth_to_cuda(new_k), synth_to_cuda(new_v)
    d_slots = torch.from_numpy(new_slots).to(dev)
    d_q = synth_to_cuda(q_h)
    d_pt = torch.from_numpy(wl.page_table).to(dev)
    d_sl = torch.from_numpy(wl.seq_lens).to(dev)
    d_out = torch.empty_like(d_q)
    ws = torch.empty(cache.workspace_size(wl.B, wl.Hq, wl.max_pages), dtype=torch.uint8, device=dev)

    def step():
        cache.quantize_and_store(0, d_k, d_v, d_slots, scales)
        cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale, d_out, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if cache.device_error() != 0:
        raise RuntimeError("device error during warm-up: " + kvq.kvq_last_error_string())
    K = args.steps
    # the decode call's own duration: a timing-event pair around it on every
    # DECODE_SAMPLE-th step of the timed region (each pair costs the stream
    # ~3.4 us, which a pair on every step would add to the step time)
    sampled = list(range(0, K, DECODE_SAMPLE))
    d0 = {i: torch.cuda.Event(enable_timing=True) for i in sampled}
    d1 = {i: torch.cuda.Event(enable_timing=True) for i in sampled}
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        e_start.record(stream)
        for i in range(K):
            cache.quantize_and_store(0, d_k, d_v, d_slots, scales)
            if i in d0:
                d0[i].record(stream)
            cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale, d_out, ws)
            if i in d1:
                d1[i].record(stream)
        e_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    local_ms = e_start.elapsed_time(e_end) / K
    decode_ms = statistics.fmean(d0[i].elapsed_time(d1[i]) for i in sampled)
    if cache.device_error() != 0:
        raise RuntimeError("device error during the timed steps: " + kvq.kvq_last_error_string())
    dbytes = algorithmic_bytes(wl, fmt)
    sbytes = store_bytes(wl, fmt)
    ms, gbs = aggregate(local_ms, dbytes + sbytes, dev)
    res = {"wl": wl, "ms": ms, "gbs": gbs, "decode_ms": decode_ms, "decode_bytes": dbytes,
           "clocks": clk.summary(), "launches": 3 * K, "world": world}

    if with_e2e:
        # same step through the public API with pinned host buffers: H2D of the
        # step's inputs, store + decode, D2H of the output, every step.  Steps
        # are pipelined the way a serving loop runs them: two sets of device
        # buffers, uploads and downloads each on their own stream, so that step
        # i + 1's inputs go up and step i - 1's output comes down while step i
        # computes; the clock stops once every step's output is on the host.
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        h_k, h_v = pin(new_k.view(np.int16)), pin(new_v.view(np.int16))
        h_q = pin(q_h.view(np.int16))
        h_slots, h_pt, h_sl = pin(new_slots), pin(wl.page_table), pin(wl.seq_lens)
        NB = 2
        h_out = [torch.empty(d_out.shape, dtype=torch.int16).pin_memory() for _ in range(NB)]
        sets = [dict(k=torch.empty_like(d_k).view(torch.int16), v=torch.empty_like(d_v).view(torch.int16),
                     q=torch.empty_like(d_q).view(torch.int16), slots=torch.empty_like(d_slots),
                     pt=torch.empty_like(d_pt), sl=torch.empty_like(d_sl),
                     out=torch.empty_like(d_out)) for _ in range(NB)]
        h2d = sum(t.numel() * t.element_size() for t in (h_k, h_v, h_q, h_slots, h_pt, h_sl))
        d2h = h_out[0].numel() * h_out[0].element_size()
        xs_in, xs_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_free = [torch.cuda.Event() for _ in range(NB)]   # the set's inputs are no longer read
        ev_in = [torch.cuda.Event() for _ in range(NB)]     # the set's inputs are up
        ev_out = [torch.cuda.Event() for _ in range(NB)]    # the set's output is down
        for e in ev_free + ev_out:
            e.record(stream)

        def e2e_step(i):
            b = i % NB
            d = sets[b]
            xs_in.wait_event(ev_free[b])  # the set's previous step has computed
            with torch.cuda.stream(xs_in):
                d["k"].copy_(h_k, non_blocking=True)
                d["v"].copy_(h_v, non_blocking=True)
                d["q"].copy_(h_q, non_blocking=True)
                d["slots"].copy_(h_slots, non_blocking=True)
                d["pt"].copy_(h_pt, non_blocking=True)
                d["sl"].copy_(h_sl, non_blocking=True)
            ev_in[b].record(xs_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])  # the set's previous output has been read
            cache.quantize_and_store(0, d["k"].view(torch.bfloat16), d["v"].view(torch.bfloat16), d["slots"],
                                     scales, stream=stream)
            cache.decode_attention(0, d["q"].view(torch.bfloat16), d["pt"], d["sl"], wl.sm_scale, d["out"], ws,
                                   stream=stream)
            ev_free[b].record(stream)
            xs_out.wait_event(ev_free[b])
            with torch.cuda.stream(xs_out):
                h_out[b].copy_(d["out"].view(torch.int16), non_blocking=True)
            ev_out[b].record(xs_out)

        for i in range(max(3, args.warmup // 4)):
            e2e_step(i)
        torch.cuda.synchronize()
        Ke = max(10, min(K, 1000))
        barrier()
        t0 = time.perf_counter()
        for i in range(Ke):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_ms_local = (time.perf_counter() - t0) * 1e3 / Ke
        barrier()
        if cache.device_error() != 0:
            raise RuntimeError("device error during the end-to-end steps: " + kvq.kvq_last_error_string())
        if not torch.equal(h_out[(Ke - 1) % NB], d_out.view(torch.int16).cpu()):
            raise RuntimeError("end-to-end output differs from the device-resident step's output")
        e2e_ms, e2e_gbs = aggregate(e2e_ms_local, dbytes + sbytes, dev)
        res["e2e"] = {"value": round(e2e_gbs, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
                      "pipelined": "two buffer sets; uploads and downloads on their own streams overlap compute"}

    if with_extra and rank == 0:
        # quantization error of the timed output against fp64 attention over the
        # unquantized bf16 K/V of two sampled sequences (the longest and one more)
        seqs_q = sorted({int(np.argmax(wl.seq_lens)), 3 % wl.B})
        exact = exact_attention_fp64(wl, ks, vs, seqs_q, q_h)
        qe = quant_error(out_rows(d_out, seqs_q), exact)
        res["quant_error"] = {"format": fmt, "sequences": seqs_q,
                              **{k: (round(v, 6) if isinstance(v, float) else v) for k, v in qe.items()},
                              "reference": "fp64 attention over the unquantized bf16 K/V (plain torch)"}
        if not args.no_per_format:
            cache.close()
            res["per_format"] = per_format_cells(args, wl, ks, vs, d_q, d_pt, d_sl, exact, dev,
                                                 peak_hbm()[0])
    if with_cpu and rank == 0 and world == 1:
        res["cpu_baseline"] = cpu_baseline(wl, ks, vs, args.seed)
    cache.close()
    return res


def synth_to_cuda(bits):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run_ours(args):
    import torch
    rank, world = dist_init("nccl")
    fmt = args.format
    r = run_cell(args, fmt, with_cpu=not args.no_cpu_baseline, with_e2e=not args.no_e2e,
                 with_extra=True)
    wl = r["wl"]
    peak, peak_kind = peak_hbm()
    achieved = r["decode_bytes"] / (r["decode_ms"] * 1e-3) / 1e9
    h = decode_source_hash()
    traffic = NCU_TRAFFIC.get((fmt, h))
    line = {
        "metric": METRIC,
        "value": round(r["gbs"], 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["ms"], 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE[fmt],
        "data": "synthetic",
        "config": {
            "workload": f"{wl.name}: one Llama-3-70B-shaped layer (Hq {wl.Hq}, Hkv {wl.Hkv}, "
                        f"head_dim {wl.D}), {fmt} cache, page_size {wl.P}, batch {wl.B}, ragged "
                        f"context U[24K, 32K] (mean {float(wl.seq_lens.mean()):.0f}), random page "
                        f"tables; step = store newest token + decode attention",
            "format": fmt, "batch": wl.B, "tokens_cached": int(wl.seq_lens.sum()),
            "l2": "no flush: the cache read each step (~%.2f GB) is larger than L2 (129 MB)"
                  % (r["decode_bytes"] / 1e9),
            "parallelism": f"weak: {world} independent rank(s), one batch each",
        },
        "tokens_per_s": round(wl.B * world / (r["ms"] * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "kernel": "decode attention (split-K kernel + LSE merge), one call",
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "bytes_per_launch": r["decode_bytes"],
                     "ms_per_launch": round(r["decode_ms"], 5)},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if "per_format" in r:
        line["per_format"] = r["per_format"]
    if "quant_error" in r:
        line["quant_error"] = r["quant_error"]
    if "e2e" in r:
        line["e2e"] = r["e2e"]
    if "cpu_baseline" in r:
        line["cpu_baseline"] = r["cpu_baseline"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.sweep:
        run_sweep(args)
    if args.store:
        run_store(args)
    barrier()


def run_store(args, steps=None, warmup=None):
    """Quantize-and-store throughput: the 70B-layer prefill of 8 sequences x 16K
    tokens (K and V, 8 kv heads, head_dim 128) stored in one call per step.
    Algorithmic bytes: bf16 K and V read, slot ids read, cache rows and block
    scales written."""
    import numpy as np
    import torch
    import quantized_paged_kv_store_gb300 as kvq
    import synth
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    wl = synth.cfg3_fp4b16_70b(seed=args.seed + 7919 * rank)
    ks, vs = wl.kv_all(0)
    k = synth_to_cuda(np.concatenate(ks))
    v = synth_to_cuda(np.concatenate(vs))
    slots = torch.from_numpy(np.concatenate([wl.slots(b) for b in range(wl.B)])).to(dev)
    n = int(slots.shape[0])
    peak, _ = peak_hbm()
    steps = steps or max(5, min(args.steps, 200))
    warmup = warmup or max(3, min(args.warmup, 10))
    for fmt in (("nvfp4", "fp4_mx_block16", "fp8_e4m3", "fp8_e5m2", "bf16") if args.store_formats is None
                else args.store_formats.split(",")):
        wl.fmt = fmt
        scales = [float(x) for x in wl._scales_from(ks, vs)]
        cache = kvq.KVQCache(fmt, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
        ms = _time_calls(lambda: cache.quantize_and_store(0, k, v, slots, scales), steps, warmup)
        if cache.device_error() != 0:
            raise RuntimeError("device error during the store benchmark")
        row_w = {"bf16": 256, "fp8_e4m3": 128, "fp8_e5m2": 128}.get(fmt, 64 + 8)
        nbytes = n * wl.Hkv * (2 * wl.D * 2 + 2 * row_w) + n * 8
        gbs = nbytes / (ms * 1e-3) / 1e9
        cache.close()
        if rank == 0:
            with open(args.store, "a") as f:
                f.write(json.dumps({"kernel": "quantize-and-store", "format": fmt, "tokens": n,
                                    "kv_heads": wl.Hkv, "head_dim": wl.D, "us_per_call": round(ms * 1e3, 2),
                                    "bytes_per_call": nbytes, "GBps": round(gbs, 1),
                                    "frac": round(gbs / peak, 4)}) + "\n")


def _graph_us(call, reps=20, replays=10):
    """Device time per call: one CUDA graph of `reps` calls, replayed back to back."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                call(s)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * replays)


def run_sweep(args):
    """The format sweep on one 70B layer: contexts 4K / 16K / 32K x batch 1 / 8 /
    32, every format (the K/V draws of a cell are shared by its formats).  Per
    cell: mean CUDA-event time of one decode call issued from Python, and the
    device time per call from CUDA-graph replay (no host launch cost)."""
    import numpy as np
    import torch
    import quantized_paged_kv_store_gb300 as kvq
    import synth
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, _ = peak_hbm()
    want = None
    if args.sweep_cells:
        want = {tuple(c.split(":")) for c in args.sweep_cells.split(",")}
    steps = max(20, min(args.steps, 300))
    for T in (4096, 16384, 32768):
        for B in (1, 8, 32):
            fmts = [f for f in PER_FORMAT if want is None or (f, str(T), str(B)) in want]
            if not fmts:
                continue
            wl = synth.cfg5_sweep_cell("bf16", T, B, seed=args.seed + 7919 * rank)
            ks, vs = wl.kv_all(0)
            kall, vall = synth_to_cuda(np.concatenate(ks)), synth_to_cuda(np.concatenate(vs))
            slots = torch.from_numpy(np.concatenate([wl.slots(b) for b in range(wl.B)])).to(dev)
            d_q = synth_to_cuda(wl.q(0))
            d_pt = torch.from_numpy(wl.page_table).to(dev)
            d_sl = torch.from_numpy(wl.seq_lens).to(dev)
            for fmt in fmts:
                cache = kvq.KVQCache(fmt, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
                cache.quantize_and_store(0, kall, vall, slots, [float(x) for x in wl.scales_for(fmt, ks, vs)])
                out = torch.empty_like(d_q)
                ws = torch.empty(cache.workspace_size(wl.B, wl.Hq, wl.max_pages), dtype=torch.uint8,
                                 device=dev)
                ms = _time_calls(lambda: cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale, out, ws),
                                 steps, 5)
                gus = _graph_us(lambda st: cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale, out,
                                                                  ws, stream=st))
                if cache.device_error() != 0:
                    raise RuntimeError(f"device error in sweep cell {fmt} {T} x {B}")
                nb = algorithmic_bytes(wl, fmt)
                if rank == 0:
                    with open(args.sweep, "a") as f:
                        f.write(json.dumps({
                            "format": fmt, "ctx": T, "batch": B,
                            "decode_us": round(ms * 1e3, 2), "GBps": round(nb / (ms * 1e-3) / 1e9, 1),
                            "frac": round(nb / (ms * 1e-3) / 1e9 / peak, 4),
                            "graph_us": round(gus, 2), "graph_GBps": round(nb / (gus * 1e-6) / 1e9, 1),
                            "graph_frac": round(nb / (gus * 1e-6) / 1e9 / peak, 4),
                            "tokens_per_s": round(B / (gus * 1e-6), 1)}) + "\n")
                cache.close()
            del kall, vall


def _time_calls(fn, steps, warmup):
    """Mean milliseconds per fn() call over `steps` back-to-back calls after
    `warmup`: one CUDA-event pair on the launching stream around all of them
    (a pair around every call would add its own stream cost, ~3.4 us, to each)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_next(args):
    """Per-head scales (calibrated on the device), calibration itself, and extend
    attention, on the benchmark's shapes; one JSON line per measurement."""
    import numpy as np
    import torch
    import quantized_paged_kv_store_gb300 as kvq
    import synth
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, _ = peak_hbm()
    steps = max(20, min(args.steps, 300))
    warm = max(3, min(args.warmup, 10))
    out = []

    def emit(d):
        if rank == 0:
            with open(args.next, "a") as f:
                f.write(json.dumps(d) + "\n")
        out.append(d)

    # 1) decode over a layer whose scales are per kv head (calibrated on the device
    #    from sequence 0's rows) against the same layer with per-tensor scales
    for fmt in ("nvfp4", "fp8_e4m3"):
        wl = make_workload(fmt, args.seed + 7919 * rank, None, args.batch)
        ks, vs = wl.kv_all(0)
        d_q = synth_to_cuda(wl.q(0))
        d_pt = torch.from_numpy(wl.page_table).to(dev)
        d_sl = torch.from_numpy(wl.seq_lens).to(dev)
        d_out = torch.empty_like(d_q)
        dbytes = algorithmic_bytes(wl, fmt)
        for mode in ("per_tensor", "per_head_calibrated"):
            cache = kvq.KVQCache(fmt, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
            if mode == "per_head_calibrated":
                cache.calibrate_scales(0, synth_to_cuda(ks[0]), synth_to_cuda(vs[0]), per_head=True)
                scales = None
            else:
                scales = [float(x) for x in wl.scales(0)]
            for b in range(wl.B):
                cache.quantize_and_store(0, synth_to_cuda(ks[b]), synth_to_cuda(vs[b]),
                                         torch.from_numpy(wl.slots(b)).to(dev), scales)
            ws = torch.empty(cache.workspace_size(wl.B, wl.Hq, wl.max_pages), dtype=torch.uint8,
                             device=dev)
            ms = _time_calls(lambda: cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale, d_out, ws),
                             steps, warm)
            if cache.device_error() != 0:
                raise RuntimeError("device error in the per-head decode measurement")
            gbs = dbytes / (ms * 1e-3) / 1e9
            emit({"path": "decode", "scales": mode, "format": fmt, "workload": wl.name,
                  "batch": wl.B, "tokens_cached": int(wl.seq_lens.sum()), "ms_per_call": round(ms, 5),
                  "GBps": round(gbs, 1), "frac": round(gbs / peak, 4)})
            cache.close()

    # 2) on-device calibration of the 70B-layer 8 x 16K prefill (per kv head):
    #    an amax reduction over K and V; one cache layer per call (a layer's
    #    scales are fixed once)
    wl = synth.cfg3_fp4b16_70b(seed=args.seed + 7919 * rank)
    ks, vs = wl.kv_all(0)
    k = synth_to_cuda(np.concatenate(ks))
    v = synth_to_cuda(np.concatenate(vs))
    n = int(k.shape[0])
    for fmt in ("fp8_e4m3", "nvfp4"):
        cal = kvq.KVQCache(fmt, steps + warm, wl.Hkv, wl.D, 16, 1)
        layer = [0]

        def calibrate():
            cal.calibrate_scales(layer[0], k, v, per_head=True)
            layer[0] += 1

        ms = _time_calls(calibrate, steps, warm)
        if cal.device_error() != 0:
            raise RuntimeError("device error in the calibration measurement")
        nbytes = 2 * n * wl.Hkv * wl.D * 2
        gbs = nbytes / (ms * 1e-3) / 1e9
        emit({"path": "calibrate", "format": fmt, "tokens": n, "kv_heads": wl.Hkv,
              "head_dim": wl.D, "per_head": True, "us_per_call": round(ms * 1e3, 2),
              "bytes_per_call": nbytes, "GBps": round(gbs, 1), "frac": round(gbs / peak, 4)})
        cal.close()

    # 3) extend attention: a 16-token chunk at the end of every sequence of the
    #    32K x 32 NVFP4 workload (512 queries); algorithmic bytes count every
    #    sequence's cached prefix once, so re-reads across a chunk's queries show
    #    as lost efficiency
    fmt, chunk = "nvfp4", 16
    wl = make_workload(fmt, args.seed + 7919 * rank, None, args.batch)
    ks, vs = wl.kv_all(0)
    cache = kvq.KVQCache(fmt, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
    scales = [float(x) for x in wl.scales(0)]
    for b in range(wl.B):
        cache.quantize_and_store(0, synth_to_cuda(ks[b]), synth_to_cuda(vs[b]),
                                 torch.from_numpy(wl.slots(b)).to(dev), scales)
    q_seq = np.repeat(np.arange(wl.B, dtype=np.int32), chunk)
    q_len = np.concatenate([np.arange(int(T) - chunk, int(T)) + 1 for T in wl.seq_lens]).astype(np.int32)
    g = torch.Generator().manual_seed(args.seed)
    d_q = synth_to_cuda(synth.to_bf16_bits(torch.randn(len(q_seq), wl.Hq, wl.D, generator=g)))
    d_qs, d_ql = torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_len).to(dev)
    d_pt = torch.from_numpy(wl.page_table).to(dev)
    d_out = torch.empty_like(d_q)
    wsb = kvq.kvq_extend_workspace_size(cache.handle, len(q_seq), wl.Hq, wl.max_pages)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    ms = _time_calls(lambda: cache.extend_attention(0, d_q, d_qs, d_ql, d_pt, wl.sm_scale, d_out, ws),
                     max(10, steps // 10), warm)
    if cache.device_error() != 0:
        raise RuntimeError("device error in the extend measurement")
    prefix = int(wl.seq_lens.sum()) * wl.Hkv * KV_BYTES[fmt]
    qo = 2 * len(q_seq) * wl.Hq * wl.D * 2
    gbs = (prefix + qo) / (ms * 1e-3) / 1e9
    # QK^T and PV: 2 * 128 multiply-adds per (query row, q head, context token) each
    flops = float(q_len.astype(np.int64).sum()) * wl.Hq * wl.D * 4
    tflops = flops / (ms * 1e-3) / 1e12
    emit({"path": "extend", "format": fmt, "workload": wl.name, "batch": wl.B, "chunk": chunk,
          "queries": len(q_seq), "ms_per_call": round(ms, 4),
          "queries_per_s": round(len(q_seq) / (ms * 1e-3), 1),
          "TFLOPs": round(tflops, 1), "frac_tensor": round(tflops / peak_bf16()[0], 4),
          "GBps_prefix_once": round(gbs, 1), "frac_hbm": round(gbs / peak, 4),
          "workspace_bytes": wsb,
          "note": "tcgen05 kernel: each 64-token K/V chunk dequantized once per 128 (query, q head) "
                  "rows; the contraction is tensor-bound at 16 queries per sequence"})
    cache.close()
    return out


def run_quant_error(args):
    """Quantization error of every format on the specified workloads: for a few
    sampled sequences of each, the GPU decode output of each cache format (all
    q heads) against fp64 attention over the unquantized bf16 K/V.  Scale
    inputs follow each workload's calibration recipe over all its sequences;
    only the sampled sequences are stored and decoded (attention per sequence
    does not depend on the others)."""
    import numpy as np
    import torch
    import quantized_paged_kv_store_gb300 as kvq
    import synth
    rank, world, local = dist_env()
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfgs = [("cfg1 E4M3 1 layer, Hq 32, Hkv 8, 2 x 256", synth.cfg1_e4m3_small(), [0, 1]),
            ("cfg2 Llama-3-8B layer 0, Hq 32, Hkv 8, 8 x U[1K, 4K]",
             synth.cfg2_llama8b_stack(layers=1), [0, 4, 7]),
            ("cfg3 70B layer, 8 x 16K", synth.cfg3_fp4b16_70b(), [1, 6]),
            ("cfg4 70B layer, 32 x U[24K, 32K]", synth.cfg4_nvfp4_70b_32k(), None)]
    for name, wl, seqs in cfgs:
        ks, vs = wl.kv_all(0)
        if seqs is None:
            seqs = sorted({int(np.argmax(wl.seq_lens)), 3})
        q_h = wl.q(0)
        exact = exact_attention_fp64(wl, ks, vs, seqs, q_h)
        sub = np.asarray(seqs)
        d_q = synth_to_cuda(q_h[sub])
        d_pt = torch.from_numpy(np.ascontiguousarray(wl.page_table[sub])).to(dev)
        d_sl = torch.from_numpy(np.ascontiguousarray(wl.seq_lens[sub])).to(dev)
        for f in PER_FORMAT:
            scales = [float(x) for x in wl.scales_for(f, ks, vs)]
            cache = kvq.KVQCache(f, 1, wl.Hkv, wl.D, wl.P, wl.num_pages)
            for b in seqs:
                cache.quantize_and_store(0, synth_to_cuda(ks[b]), synth_to_cuda(vs[b]),
                                         torch.from_numpy(wl.slots(b)).to(dev), scales)
            out = cache.decode_attention(0, d_q, d_pt, d_sl, wl.sm_scale)
            if cache.device_error() != 0:
                raise RuntimeError(f"device error in the quantization-error run ({name}, {f})")
            rows = out_rows(out, range(len(seqs)))
            qe = quant_error({b: rows[i] for i, b in enumerate(seqs)}, exact)
            with open(args.quant_error, "a") as fh:
                fh.write(json.dumps({"workload": name, "format": f, "sequences": seqs,
                                     "tokens": [int(wl.seq_lens[b]) for b in seqs],
                                     "scales": scales, **qe}) + "\n")
            cache.close()


# ------------------------------------------------------------ reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample of the
    same workload (a token prefix of one sequence, all its heads), sized so the
    whole run stays within a few minutes."""
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return
    import numpy as np
    import oracle
    wl = make_workload(args.format, args.seed)
    seqs = [0, 1]
    ks, vs = [], []
    for b in seqs:
        k, v = wl.kv(0, b)
        ks.append(k)
        vs.append(v)
    c = oracle.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    s = wl.scales(0)
    for i, b in enumerate(seqs):
        c.quantize_store(ks[i], vs[i], wl.slots(b), s)
    q = wl.q(0)

    def one(b, T):
        sl = np.zeros_like(wl.seq_lens)
        sl[b] = T
        t0 = time.perf_counter()
        c.decode_attention(q, wl.page_table, sl, wl.sm_scale, b_list=np.array([b]))
        return time.perf_counter() - t0, T * wl.Hkv * KV_BYTES[wl.fmt] + wl.Hq * wl.D * 4

    dt, _ = one(0, 2048)
    budget = max(0.01, min(1.0, 150.0 / max(1, args.steps + args.warmup)))
    T_step = int(max(64, min(int(wl.seq_lens[0]), 2048 * budget / max(dt, 1e-6))))
    for i in range(args.warmup):
        one(seqs[i % 2], T_step)
    tot_t = tot_b = 0.0
    for i in range(args.steps):
        t, nb = one(seqs[i % 2], T_step)
        tot_t += t
        tot_b += nb
    v = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "format": wl.fmt,
                       "sample": f"each step: {T_step}-token prefix of one sequence, all "
                                 f"{wl.Hq} q heads"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"fp64 oracle decode attention, {T_step} tokens x "
                                       f"{wl.Hkv} kv heads per step"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.store_only:
        run_store(args)
        return
    if args.sweep_only and args.sweep:
        run_sweep(args)
        return
    if args.next:
        run_next(args)
        return
    if args.quant_error:
        run_quant_error(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
