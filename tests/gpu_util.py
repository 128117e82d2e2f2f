"""Helpers for the GPU parity tests: run a synthetic workload through the C ABI
(via the Python binding) and through the CPU oracle on the same inputs."""
import numpy as np
import torch

import synth


class DevView:
    """Expose a raw device allocation to torch through __cuda_array_interface__."""

    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3}


def read_device(ptr, nbytes) -> np.ndarray:
    return torch.as_tensor(DevView(ptr, nbytes), device="cuda").cpu().numpy().copy()


def bits_to_cuda(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def cuda_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_cache_for(kvq, wl, layers=None):
    return kvq.KVQCache(wl.fmt, layers or wl.layers, wl.Hkv, wl.D, wl.P, wl.num_pages)


def store_layer(cache, wl, layer=0, seqs=None, chunk=None):
    """Quantize-and-store every token of the given sequences on the GPU (the
    layer's rows are drawn once; the same draws fix its scale inputs)."""
    ks, vs = wl.kv_all(layer)
    s = wl.scales(layer)
    for b in (range(wl.B) if seqs is None else seqs):
        T = int(wl.seq_lens[b])
        step = chunk or max(T, 1)
        for t0 in range(0, T, step):
            t1 = min(T, t0 + step)
            cache.quantize_and_store(layer, bits_to_cuda(ks[b][t0:t1]), bits_to_cuda(vs[b][t0:t1]),
                                     torch.from_numpy(wl.slots(b, t0, t1)).cuda(), list(s))


def oracle_cache_for(orc, wl, layer=0, seqs=None):
    c = orc.OracleCache(wl.fmt, wl.Hkv, wl.D, wl.P, wl.num_pages)
    s = wl.scales(layer)
    for b in (range(wl.B) if seqs is None else seqs):
        k, v = wl.kv(layer, b)
        assert c.quantize_store(k, v, wl.slots(b), s) == 0
    return c


def gpu_pools(cache, layer):
    (kd, vd, ks, vs), st = cache.layout(layer)
    rows = cache.num_pages * cache.kv_heads * cache.page_size
    out = [read_device(kd, rows * st[2]).reshape(rows, st[2]),
           read_device(vd, rows * st[2]).reshape(rows, st[2])]
    if st[3]:
        out += [read_device(ks, rows * st[3]).reshape(rows, st[3]),
                read_device(vs, rows * st[3]).reshape(rows, st[3])]
    return out


def gpu_decode(cache, wl, layer=0, q_bits=None, seq_lens=None, page_table=None):
    q = bits_to_cuda(wl.q(layer) if q_bits is None else q_bits)
    pt = torch.from_numpy(wl.page_table if page_table is None else page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens if seq_lens is None else np.asarray(seq_lens, np.int32)).cuda()
    out = cache.decode_attention(layer, q, pt, sl, wl.sm_scale)
    torch.cuda.synchronize()
    return synth.bf16_bits_to_float(cuda_to_bits(out)).astype(np.float64)


def attention_errors(got: np.ndarray, ref: np.ndarray):
    """Errors of a bf16 attention output against the fp64 reference, in excess
    of the reference's own bf16 rounding (no bf16 output can do better than
    bf16(ref); its rounding alone reaches ~2.3e-3 relative L2 on some vectors):
      rel[b, j] = (||got - ref|| - ||bf16(ref) - ref||) / ||ref||
      absd[...] = |got - ref| - |bf16(ref) - ref|
    Also returns the raw relative L2 error (got vs ref) for reporting."""
    ref_bf16 = synth.bf16_bits_to_float(
        synth.to_bf16_bits(torch.from_numpy(ref.astype(np.float32)))).astype(np.float64)
    floor = np.linalg.norm(ref_bf16 - ref, axis=-1)
    num = np.linalg.norm(got - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    safe = np.where(den > 0, den, 1)
    rel = np.where(den > 0, (num - floor) / safe, num)
    raw = np.where(den > 0, num / safe, num)
    absd = np.abs(got - ref) - np.abs(ref_bf16 - ref)
    return rel, absd, raw


REL_TOL = 2e-3
ABS_TOL = 1e-2


def assert_attention_close(got, ref, where=""):
    rel, absd, raw = attention_errors(got, ref)
    assert np.isfinite(got).all(), where
    assert rel.max() <= REL_TOL, f"{where}: max rel L2 {rel.max():.3e} at {np.unravel_index(rel.argmax(), rel.shape)}"
    assert absd.max() <= ABS_TOL, f"{where}: max abs {absd.max():.3e}"
    return float(rel.max()), float(absd.max()), float(raw.max())
