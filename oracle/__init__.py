"""CPU oracle for the quantized paged KV store -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product (``quantized_paged_kv_store_gb300``)
never imports it, and this package never imports the product.  The arithmetic
lives in ``kvq_oracle.c`` (plain C, fp64 attention, nearest-code encoding);
this module compiles it with gcc and marshals numpy arrays into it.

Cited sources and the readings taken where the pages are silent are listed at
the top of ``kvq_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

FORMATS = {"bf16": 0, "fp8_e4m3": 1, "fp8_e5m2": 2, "fp4_mx_block16": 3, "nvfp4": 4}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into a shared library (gcc, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u32, i32, i64, f64, vp = (ctypes.c_uint32, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_double, ctypes.c_void_p)
            for name in ("orc_dec_e4m3", "orc_dec_e5m2", "orc_dec_e2m1", "orc_dec_e8m0",
                         "orc_dec_bf16"):
                getattr(lib, name).argtypes = [u32]
                getattr(lib, name).restype = f64
            for name in ("orc_enc_e4m3", "orc_enc_e5m2", "orc_enc_e2m1"):
                getattr(lib, name).argtypes = [f64]
                getattr(lib, name).restype = u32
            lib.orc_enc_bf16.argtypes = [ctypes.c_float]
            lib.orc_enc_bf16.restype = u32
            lib.orc_bytes_per_token.argtypes = [i32, i32, i32, i32]
            lib.orc_bytes_per_token.restype = i64
            lib.orc_quantize_store.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, i32, vp,
                                               vp, vp, vp, vp]
            lib.orc_quantize_store.restype = i32
            lib.orc_dequantize.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, vp, vp, vp, i32,
                                           vp, vp]
            lib.orc_dequantize.restype = i32
            lib.orc_decode_attention.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, vp, vp, vp,
                                                 i32, vp, i32, vp, i32, vp, i32, f64, vp]
            lib.orc_decode_attention.restype = i32
            lib.orc_quantize_query.argtypes = [vp, i64, i32, i32, vp, i32, vp]
            lib.orc_quantize_query.restype = i32
            lib.orc_decode_attention_fp8q.argtypes = [i32, i32, i32, i32, i64, vp, vp, vp, vp, vp,
                                                      vp, vp, i32, i32, vp, i32, vp, i32, vp, i32,
                                                      f64, vp]
            lib.orc_decode_attention_fp8q.restype = i32
            lib.orc_calibrate_scales.argtypes = [i32, i32, i32, vp, i32, i32, vp]
            lib.orc_calibrate_scales.restype = i32
            lib.orc_num_threads.argtypes = []
            lib.orc_num_threads.restype = i32
            lib.orc_set_num_threads.argtypes = [i32]
            lib.orc_set_num_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


# --- scalar codecs ---------------------------------------------------------

def dec_e4m3(code: int) -> float:
    return _load().orc_dec_e4m3(code)


def dec_e5m2(code: int) -> float:
    return _load().orc_dec_e5m2(code)


def dec_e2m1(code: int) -> float:
    return _load().orc_dec_e2m1(code)


def dec_e8m0(code: int) -> float:
    return _load().orc_dec_e8m0(code)


def dec_bf16(bits: int) -> float:
    return _load().orc_dec_bf16(bits)


def enc_e4m3(v: float) -> int:
    return _load().orc_enc_e4m3(v)


def enc_e5m2(v: float) -> int:
    return _load().orc_enc_e5m2(v)


def enc_e2m1(v: float) -> int:
    return _load().orc_enc_e2m1(v)


def enc_bf16(v: float) -> int:
    return _load().orc_enc_bf16(v)


def bytes_per_token(fmt, layers: int, kv_heads: int, head_dim: int) -> int:
    return _load().orc_bytes_per_token(_fmt(fmt), layers, kv_heads, head_dim)


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> int:
    """OpenMP threads of later oracle calls; returns the count in effect."""
    return _load().orc_set_num_threads(int(n))


def calibrate_scales(fmt, x_bf16: np.ndarray, per_head: bool) -> np.ndarray:
    """Scale(s) of a format from a batch of bf16 rows x [n][H][D] (reading R16):
    float32 [H] per kv head, or [1] per tensor."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    n, H, D = x.shape
    out = np.zeros(H if per_head else 1, np.float32)
    _load().orc_calibrate_scales(_fmt(fmt), H, D, _ptr(x), n, int(bool(per_head)), _ptr(out))
    return out


def quantize_query(q_bf16: np.ndarray, q_scales) -> np.ndarray:
    """E4M3 codes of a bf16 query [rows][Hq][D] (reading R17): one q_scale per
    tensor ([1]) or per q head ([Hq])."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    rows, Hq, D = q.shape
    s = np.ascontiguousarray(np.asarray(q_scales, np.float32).reshape(-1))
    out = np.zeros((rows, Hq, D), np.uint8)
    rc = _load().orc_quantize_query(_ptr(q), rows, Hq, D, _ptr(s), s.shape[0], _ptr(out))
    assert rc == 0, "q_scales must have 1 or Hq entries"
    return out


# --- cache model ------------------------------------------------------------

def data_row_bytes(fmt, head_dim: int) -> int:
    f = _fmt(fmt)
    return head_dim * 2 if f == 0 else (head_dim if f in (1, 2) else head_dim // 2)


class OracleCache:
    """Host model of one layer of the paged cache (R7 layout)."""

    def __init__(self, fmt, kv_heads: int, head_dim: int, page_size: int, num_pages: int):
        self.fmt = _fmt(fmt)
        self.H, self.D, self.P, self.num_pages = kv_heads, head_dim, page_size, num_pages
        rows = num_pages * kv_heads * page_size
        rb = data_row_bytes(self.fmt, head_dim)
        self.k_data = np.zeros((rows, rb), np.uint8)
        self.v_data = np.zeros((rows, rb), np.uint8)
        self.k_scales = np.zeros((rows, head_dim // 16), np.uint8)
        self.v_scales = np.zeros((rows, head_dim // 16), np.uint8)
        self.scales = np.ones((2, kv_heads), np.float32)   # [K|V][kv head] (reading R15)

    def set_scales(self, scales) -> None:
        """{k, v} per tensor, or a [2][H] array of per-kv-head scales."""
        a = np.asarray(scales, np.float32)
        if a.shape == (2,):   # per tensor: every head takes the tensor's scale
            a = np.repeat(a.reshape(2, 1), self.H, axis=1)
        self.scales = np.ascontiguousarray(a.reshape(2, self.H), dtype=np.float32).copy()

    def quantize_store(self, k_bf16: np.ndarray, v_bf16: np.ndarray, slots: np.ndarray,
                       scales=None) -> int:
        """k, v: uint16 bf16 bits [n][H][D]; slots int64 [n]."""
        k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
        v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
        s = np.ascontiguousarray(slots, dtype=np.int64)
        if scales is not None:
            self.set_scales(scales)
        n = s.shape[0]
        assert k.shape == (n, self.H, self.D) and v.shape == k.shape
        return _load().orc_quantize_store(self.fmt, self.H, self.D, self.P, self.num_pages,
                                          _ptr(k), _ptr(v), _ptr(s), n, _ptr(self.scales),
                                          _ptr(self.k_data), _ptr(self.v_data),
                                          _ptr(self.k_scales), _ptr(self.v_scales))

    def dequantize(self, slots: np.ndarray):
        s = np.ascontiguousarray(slots, dtype=np.int64)
        n = s.shape[0]
        ko = np.zeros((n, self.H, self.D), np.uint16)
        vo = np.zeros((n, self.H, self.D), np.uint16)
        rc = _load().orc_dequantize(self.fmt, self.H, self.D, self.P, self.num_pages,
                                    _ptr(self.k_data), _ptr(self.v_data), _ptr(self.k_scales),
                                    _ptr(self.v_scales), _ptr(self.scales), _ptr(s), n,
                                    _ptr(ko), _ptr(vo))
        return ko, vo, rc

    def decode_attention(self, q_bf16: np.ndarray, page_table: np.ndarray, seq_lens: np.ndarray,
                         sm_scale: float, b_list=None):
        """q: uint16 [B][Hq][D]; returns (out fp64 [B][Hq][D], rc)."""
        q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, D = q.shape
        out = np.zeros((B, Hq, D), np.float64)
        bl = None if b_list is None else np.ascontiguousarray(b_list, dtype=np.int32)
        rc = _load().orc_decode_attention(self.fmt, self.H, self.D, self.P, self.num_pages,
                                          _ptr(self.k_data), _ptr(self.v_data),
                                          _ptr(self.k_scales), _ptr(self.v_scales),
                                          _ptr(self.scales), _ptr(q), Hq, _ptr(pt), pt.shape[1],
                                          _ptr(sl), B, _ptr(bl), 0 if bl is None else bl.shape[0],
                                          float(sm_scale), _ptr(out))
        return out, rc

    def decode_attention_fp8q(self, q_bf16: np.ndarray, q_scales, page_table: np.ndarray,
                              seq_lens: np.ndarray, sm_scale: float, b_list=None):
        """Decode attention in the FP8 domain (reading R17): the query is
        quantized to E4M3 with q_scales ([1] or [Hq]) and attention is exact
        over the dequantized query.  Returns (out fp64 [B][Hq][D], rc)."""
        q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
        s = np.ascontiguousarray(np.asarray(q_scales, np.float32).reshape(-1))
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, D = q.shape
        out = np.zeros((B, Hq, D), np.float64)
        bl = None if b_list is None else np.ascontiguousarray(b_list, dtype=np.int32)
        rc = _load().orc_decode_attention_fp8q(self.fmt, self.H, self.D, self.P, self.num_pages,
                                               _ptr(self.k_data), _ptr(self.v_data),
                                               _ptr(self.k_scales), _ptr(self.v_scales),
                                               _ptr(self.scales), _ptr(q), _ptr(s), s.shape[0], Hq,
                                               _ptr(pt), pt.shape[1], _ptr(sl), B, _ptr(bl),
                                               0 if bl is None else bl.shape[0], float(sm_scale),
                                               _ptr(out))
        return out, rc

    def extend_attention(self, q_bf16: np.ndarray, q_seq: np.ndarray, q_len: np.ndarray,
                         page_table: np.ndarray, sm_scale: float):
        """Extend (chunked-prefill) attention: query token i of sequence q_seq[i]
        attends to that sequence's tokens [0, q_len[i]) (its causal prefix,
        itself included).  This is decode attention with one row per query
        token: page-table row page_table[q_seq[i]] and length q_len[i]."""
        rows = np.asarray(page_table, np.int32)[np.asarray(q_seq, np.int64)]
        return self.decode_attention(q_bf16, rows, np.asarray(q_len, np.int32), sm_scale)

    def row_index(self, slot: int, h: int) -> int:
        return ((slot // self.P) * self.H + h) * self.P + slot % self.P
