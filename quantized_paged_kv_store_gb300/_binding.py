"""ctypes binding of libkvq.so.  Argument marshalling only: torch tensors give
device pointers, torch gives the current stream; the library does the work."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

FORMATS = {"bf16": 0, "fp8_e4m3": 1, "fp8_e5m2": 2, "fp4_mx_block16": 3, "nvfp4": 4}
_STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_OOM",
           4: "KVQ_ERR_CUDA", 5: "KVQ_ERR_SCALE_MISMATCH", 6: "KVQ_ERR_DEVICE_RANGE",
           7: "KVQ_ERR_TIMEOUT"}
_STATUS_CODES = {v: k for k, v in _STATUS.items()}


def library_path() -> str:
    return os.environ.get("KVQ_LIBRARY", _build.LIB)


def _load():
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"libkvq.so not found at {path}; build it with "
            "`python quantized_paged_kv_store_gb300/build.py` (there is no fallback)")
    L = ctypes.CDLL(path)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    sig = {
        "kvq_create_cache": ([i32, i32, i32, i32, i32, i32, ctypes.POINTER(vp)], i32),
        "kvq_destroy_cache": ([vp], i32),
        "kvq_quantize_and_store": ([vp, i32, vp, vp, vp, i32, vp, vp], i32),
        "kvq_quantize_and_store_per_head": ([vp, i32, vp, vp, vp, i32, vp, vp, vp], i32),
        "kvq_calibrate_scales": ([vp, i32, vp, vp, i32, i32, vp], i32),
        "kvq_layer_head_scales": ([vp, i32, ctypes.POINTER(f32), ctypes.POINTER(f32), vp], i32),
        "kvq_decode_attention": ([vp, i32, vp, i32, vp, i32, vp, i32, f32, vp, vp, sz, vp], i32),
        "kvq_decode_workspace_size": ([vp, i32, i32, i32], sz),
        "kvq_extend_workspace_size": ([vp, i32, i32, i32], sz),
        "kvq_decode_attention_fp8q": ([vp, i32, vp, i32, ctypes.POINTER(f32), i32, vp, i32, vp, i32,
                                       f32, vp, vp, sz, vp], i32),
        "kvq_quantize_query": ([vp, i32, i32, i32, ctypes.POINTER(f32), i32, vp, vp], i32),
        "kvq_extend_attention": ([vp, i32, vp, i32, i32, vp, vp, vp, i32, i32, f32, vp, vp, sz, vp],
                                 i32),
        "kvq_decode_attention_noalloc": ([vp, i32, vp, i32, vp, i32, vp, i32, f32, vp, vp], i32),
        "kvq_dequantize": ([vp, i32, vp, i32, vp, vp, vp], i32),
        "kvq_cache_layout": ([vp, i32, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                              ctypes.POINTER(vp), ctypes.POINTER(sz)], i32),
        "kvq_layer_scales": ([vp, i32, ctypes.POINTER(f32)], i32),
        "kvq_bytes_per_token": ([i32, i32, i32, i32], sz),
        "kvq_format_from_name": ([ctypes.c_char_p, ctypes.POINTER(i32)], i32),
        "kvq_format_name": ([i32], ctypes.c_char_p),
        "kvq_get_device_error": ([vp, vp], i32),
        "kvq_last_error_string": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


lib = _load()


class KVQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.code = _STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.code}: {kvq_last_error_string()}")


def _check(st: int, where: str):
    if st != 0:
        raise KVQError(st, where)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def kvq_last_error_string() -> str:
    return lib.kvq_last_error_string().decode()


def kvq_format_name(fmt) -> str | None:
    r = lib.kvq_format_name(_fmt(fmt))
    return None if r is None else r.decode()


def kvq_format_from_name(name: str) -> int:
    out = ctypes.c_int()
    _check(lib.kvq_format_from_name(name.encode(), ctypes.byref(out)), "kvq_format_from_name")
    return out.value


def kvq_bytes_per_token(fmt, layers: int, kv_heads: int, head_dim: int) -> int:
    return lib.kvq_bytes_per_token(_fmt(fmt), layers, kv_heads, head_dim)


def kvq_create_cache(fmt, layers, kv_heads, head_dim, page_size, num_pages) -> int:
    h = ctypes.c_void_p()
    _check(lib.kvq_create_cache(_fmt(fmt), layers, kv_heads, head_dim, page_size, num_pages,
                                ctypes.byref(h)), "kvq_create_cache")
    return h.value


def kvq_destroy_cache(handle: int):
    _check(lib.kvq_destroy_cache(ctypes.c_void_p(handle)), "kvq_destroy_cache")


def kvq_quantize_and_store(handle, layer, k, v, slot_mapping, scales=None, stream=None):
    """k, v: bf16 [n][kv_heads][head_dim] device tensors; slot_mapping int64 [n];
    scales: host sequence of two floats or None."""
    sc = None if scales is None else (ctypes.c_float * 2)(float(scales[0]), float(scales[1]))
    _check(lib.kvq_quantize_and_store(ctypes.c_void_p(handle), layer, _ptr(k), _ptr(v),
                                      _ptr(slot_mapping), int(slot_mapping.shape[0]), sc,
                                      _stream(stream)), "kvq_quantize_and_store")


def kvq_quantize_and_store_per_head(handle, layer, k, v, slot_mapping, k_scales, v_scales,
                                    stream=None):
    """As kvq_quantize_and_store with host sequences of one scale per kv head."""
    def arr(x):
        return None if x is None else (ctypes.c_float * len(x))(*[float(t) for t in x])
    _check(lib.kvq_quantize_and_store_per_head(ctypes.c_void_p(handle), layer, _ptr(k), _ptr(v),
                                               _ptr(slot_mapping), int(slot_mapping.shape[0]),
                                               arr(k_scales), arr(v_scales), _stream(stream)),
           "kvq_quantize_and_store_per_head")


def kvq_calibrate_scales(handle, layer, k, v, per_head: bool, stream=None):
    """Fixes the layer's scales from bf16 K, V device rows [n][kv_heads][head_dim]."""
    _check(lib.kvq_calibrate_scales(ctypes.c_void_p(handle), layer, _ptr(k), _ptr(v),
                                    int(k.shape[0]), int(bool(per_head)), _stream(stream)),
           "kvq_calibrate_scales")


def kvq_layer_head_scales(handle, layer, kv_heads, stream=None):
    ks = (ctypes.c_float * kv_heads)()
    vs = (ctypes.c_float * kv_heads)()
    _check(lib.kvq_layer_head_scales(ctypes.c_void_p(handle), layer, ks, vs, _stream(stream)),
           "kvq_layer_head_scales")
    return [float(x) for x in ks], [float(x) for x in vs]


def kvq_decode_workspace_size(handle, batch, num_q_heads, max_pages_per_seq) -> int:
    n = lib.kvq_decode_workspace_size(ctypes.c_void_p(handle), batch, num_q_heads, max_pages_per_seq)
    if n == 0:
        raise KVQError(2, "kvq_decode_workspace_size")
    return n


def kvq_decode_attention(handle, layer, q, page_table, seq_lens, sm_scale, out, workspace,
                         stream=None):
    """q, out: bf16 [B][Hq][D]; page_table int32 [B][max_pages]; seq_lens int32 [B];
    workspace: uint8 device tensor of kvq_decode_workspace_size bytes."""
    B, Hq, _ = q.shape
    _check(lib.kvq_decode_attention(ctypes.c_void_p(handle), layer, _ptr(q), Hq, _ptr(page_table),
                                    int(page_table.shape[1]), _ptr(seq_lens), B, float(sm_scale),
                                    _ptr(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "kvq_decode_attention")


def _floats(x):
    x = [float(t) for t in x]
    return (ctypes.c_float * len(x))(*x), len(x)


def kvq_decode_attention_fp8q(handle, layer, q, q_scales, page_table, seq_lens, sm_scale, out,
                              workspace, stream=None):
    """FP8-domain decode attention: q bf16 [B][Hq][D] quantized to E4M3 with
    q_scales (host sequence of 1 or Hq floats); otherwise as kvq_decode_attention."""
    B, Hq, _ = q.shape
    qs, nqs = _floats(q_scales)
    _check(lib.kvq_decode_attention_fp8q(ctypes.c_void_p(handle), layer, _ptr(q), Hq, qs, nqs,
                                         _ptr(page_table), int(page_table.shape[1]), _ptr(seq_lens),
                                         B, float(sm_scale), _ptr(out), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream)), "kvq_decode_attention_fp8q")


def kvq_quantize_query(q, q_scales, codes, stream=None):
    """E4M3 codes (uint8 device tensor, q's shape) of a bf16 query [rows][Hq][D]."""
    rows, Hq, D = q.shape
    qs, nqs = _floats(q_scales)
    _check(lib.kvq_quantize_query(_ptr(q), rows, Hq, D, qs, nqs, _ptr(codes), _stream(stream)),
           "kvq_quantize_query")


def kvq_extend_attention(handle, layer, q, q_seq, q_len, page_table, sm_scale, out, workspace,
                         stream=None):
    """q, out: bf16 [n][Hq][D]; q_seq, q_len: int32 [n]; page_table int32 [S][max_pages]."""
    n, Hq, _ = q.shape
    _check(lib.kvq_extend_attention(ctypes.c_void_p(handle), layer, _ptr(q), Hq, n, _ptr(q_seq),
                                    _ptr(q_len), _ptr(page_table), int(page_table.shape[0]),
                                    int(page_table.shape[1]), float(sm_scale), _ptr(out),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "kvq_extend_attention")


def kvq_extend_workspace_size(handle, num_q_tokens, num_q_heads, max_pages_per_seq) -> int:
    """Workspace bytes of the fastest extend plan (0: none needed)."""
    return lib.kvq_extend_workspace_size(ctypes.c_void_p(handle), num_q_tokens, num_q_heads,
                                         max_pages_per_seq)


def kvq_decode_attention_noalloc(handle, layer, q, page_table, seq_lens, sm_scale, out,
                                 stream=None):
    """kvq_decode_attention with the library's static scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    B, Hq, _ = q.shape
    _check(lib.kvq_decode_attention_noalloc(ctypes.c_void_p(handle), layer, _ptr(q), Hq,
                                            _ptr(page_table), int(page_table.shape[1]),
                                            _ptr(seq_lens), B, float(sm_scale), _ptr(out),
                                            _stream(stream)), "kvq_decode_attention_noalloc")


def kvq_dequantize(handle, layer, slot_mapping, k_out, v_out, stream=None):
    _check(lib.kvq_dequantize(ctypes.c_void_p(handle), layer, _ptr(slot_mapping),
                              int(slot_mapping.shape[0]), _ptr(k_out), _ptr(v_out),
                              _stream(stream)), "kvq_dequantize")


def kvq_cache_layout(handle, layer):
    """Returns (k_data, v_data, k_scales, v_scales) device addresses and 4 strides."""
    p = [ctypes.c_void_p() for _ in range(4)]
    st = (ctypes.c_size_t * 4)()
    _check(lib.kvq_cache_layout(ctypes.c_void_p(handle), layer, *[ctypes.byref(x) for x in p], st),
           "kvq_cache_layout")
    return [x.value for x in p], list(st)


def kvq_layer_scales(handle, layer):
    out = (ctypes.c_float * 2)()
    _check(lib.kvq_layer_scales(ctypes.c_void_p(handle), layer, out), "kvq_layer_scales")
    return float(out[0]), float(out[1])


def kvq_get_device_error(handle, stream=None) -> int:
    """Synchronizes the stream; returns the status code (0 = no device error)."""
    return lib.kvq_get_device_error(ctypes.c_void_p(handle), _stream(stream))


class KVQCache:
    """Owning wrapper of a kvq_cache handle (convenience over the functions above)."""

    def __init__(self, fmt, layers, kv_heads, head_dim, page_size, num_pages):
        self.fmt = fmt if isinstance(fmt, str) else kvq_format_name(fmt)
        self.layers, self.kv_heads, self.head_dim = layers, kv_heads, head_dim
        self.page_size, self.num_pages = page_size, num_pages
        self.handle = kvq_create_cache(fmt, layers, kv_heads, head_dim, page_size, num_pages)

    def close(self):
        if self.handle:
            kvq_destroy_cache(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def quantize_and_store(self, layer, k, v, slot_mapping, scales=None, stream=None):
        kvq_quantize_and_store(self.handle, layer, k, v, slot_mapping, scales, stream)

    def quantize_and_store_per_head(self, layer, k, v, slot_mapping, k_scales, v_scales,
                                    stream=None):
        kvq_quantize_and_store_per_head(self.handle, layer, k, v, slot_mapping, k_scales, v_scales,
                                        stream)

    def calibrate_scales(self, layer, k, v, per_head=False, stream=None):
        kvq_calibrate_scales(self.handle, layer, k, v, per_head, stream)

    def layer_head_scales(self, layer, stream=None):
        return kvq_layer_head_scales(self.handle, layer, self.kv_heads, stream)

    def workspace_size(self, batch, num_q_heads, max_pages_per_seq):
        return kvq_decode_workspace_size(self.handle, batch, num_q_heads, max_pages_per_seq)

    def decode_attention(self, layer, q, page_table, seq_lens, sm_scale, out=None, workspace=None,
                         stream=None):
        import torch
        if out is None:
            out = torch.empty_like(q)
        if workspace is None:
            n = self.workspace_size(q.shape[0], q.shape[1], page_table.shape[1])
            workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
        kvq_decode_attention(self.handle, layer, q, page_table, seq_lens, sm_scale, out, workspace,
                             stream)
        return out

    def decode_attention_fp8q(self, layer, q, q_scales, page_table, seq_lens, sm_scale, out=None,
                              workspace=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(q)
        if workspace is None:
            n = self.workspace_size(q.shape[0], q.shape[1], page_table.shape[1])
            workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
        kvq_decode_attention_fp8q(self.handle, layer, q, q_scales, page_table, seq_lens, sm_scale,
                                  out, workspace, stream)
        return out

    def extend_attention(self, layer, q, q_seq, q_len, page_table, sm_scale, out=None,
                         workspace=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(q)
        if workspace is None:
            n = kvq_extend_workspace_size(self.handle, q.shape[0], q.shape[1], page_table.shape[1])
            workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
        kvq_extend_attention(self.handle, layer, q, q_seq, q_len, page_table, sm_scale, out,
                             workspace, stream)
        return out

    def dequantize(self, layer, slot_mapping, stream=None):
        import torch
        n = slot_mapping.shape[0]
        k = torch.empty(n, self.kv_heads, self.head_dim, dtype=torch.bfloat16,
                        device=slot_mapping.device)
        v = torch.empty_like(k)
        kvq_dequantize(self.handle, layer, slot_mapping, k, v, stream)
        return k, v

    def layout(self, layer):
        return kvq_cache_layout(self.handle, layer)

    def layer_scales(self, layer):
        return kvq_layer_scales(self.handle, layer)

    def device_error(self, stream=None) -> int:
        return kvq_get_device_error(self.handle, stream)
