// kvq_api.cu -- host side of the C ABI declared in include/kvq.h.
//
// The cache object follows "SGLang PR #21954 analysis: NVFP4 KV cache", Code
// analysis 1 (create_buffers / quantize_and_store / dequantize_prev_kv): one
// device allocation per cache holds every layer's K and V data pools and block
// scale planes plus a device error word; per-layer scales live on the host and
// reach the kernels as launch arguments.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "kvq_decode_args.cuh"
#include "kvq_internal.h"

struct kvq_cache {
  kvq::Geometry geo;
  int layers;
  int device;
  uint8_t* base;           // single device allocation
  size_t bytes;
  size_t layer_data_bytes; // one K (or V) data pool of one layer
  size_t layer_scale_bytes;
  int* err;                // device error word
  // Scales of each layer ("Quantized KV cache" (vLLM): per-tensor or
  // per-attention-head; fixed by the first store or by calibration).
  std::vector<float> scales;    // [layers][2][kv_heads] host copy (mode kHost)
  std::vector<char> mode;       // [layers] kUnset / kHost / kDevice
  std::vector<char> uniform;    // [layers] every head has the same scales (mode kHost)
  float* dscale;                // [layers][2][kv_heads] device copy
  float* drecip;                // [layers][2][kv_heads] 1 / scale
  unsigned* damax;              // [layers][2][kv_heads] calibration scratch (one slice per layer)
};

namespace {

thread_local char g_msg[512] = "no error";

kvq_status fail(kvq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool valid_format(int f) { return f >= KVQ_BF16 && f <= KVQ_NVFP4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq::LayerView view(const kvq_cache* c, int layer) {
  kvq::LayerView L;
  const size_t per_layer = 2 * c->layer_data_bytes + 2 * c->layer_scale_bytes;
  uint8_t* p = c->base + per_layer * (size_t)layer;
  L.k_data = p;
  L.v_data = p + c->layer_data_bytes;
  if (c->layer_scale_bytes) {
    L.k_scales = p + 2 * c->layer_data_bytes;
    L.v_scales = L.k_scales + c->layer_scale_bytes;
  } else {
    L.k_scales = L.v_scales = nullptr;
  }
  return L;
}

kvq_status check_device(const kvq_cache* c) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != c->device)
    return fail(KVQ_ERR_INVALID_ARG, "cache lives on device %d but device %d is current", c->device, dev);
  return KVQ_OK;
}

kvq_status check_layer(const kvq_cache* c, int layer) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "cache is NULL");
  if (layer < 0 || layer >= c->layers)
    return fail(KVQ_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, c->layers);
  return KVQ_OK;
}

bool uses_scales(kvq_format f) { return f == KVQ_FP8_E4M3 || f == KVQ_FP8_E5M2 || f == KVQ_NVFP4; }

enum : char { kUnset = 0, kHost = 1, kDevice = 2 };

float* host_scales(kvq_cache* c, int layer, int kv) {
  return c->scales.data() + ((size_t)layer * 2 + kv) * c->geo.kv_heads;
}
const float* host_scales(const kvq_cache* c, int layer, int kv) {
  return c->scales.data() + ((size_t)layer * 2 + kv) * c->geo.kv_heads;
}

// Device per-head scales of a layer when its heads differ or were calibrated
// on the device; null pointers (the per-tensor path) otherwise.
kvq::HeadScales head_scales(const kvq_cache* c, int layer) {
  kvq::HeadScales hs;
  const bool ph = uses_scales(c->geo.fmt) &&
                  (c->mode[layer] == kDevice || (c->mode[layer] == kHost && !c->uniform[layer]));
  if (ph) {
    const size_t H = (size_t)c->geo.kv_heads, base = (size_t)layer * 2 * H;
    hs.scale[0] = c->dscale + base;
    hs.scale[1] = c->dscale + base + H;
    hs.recip[0] = c->drecip + base;
    hs.recip[1] = c->drecip + base + H;
  }
  return hs;
}

// Per-tensor scales of a layer for the scalar path (1.0 where none apply).
void tensor_scales(const kvq_cache* c, int layer, float* sk, float* sv) {
  *sk = *sv = 1.0f;
  if (uses_scales(c->geo.fmt) && c->mode[layer] == kHost) {
    *sk = host_scales(c, layer, 0)[0];
    *sv = host_scales(c, layer, 1)[0];
  }
}

kvq_status check_scale_values(const float* s, int n) {
  for (int i = 0; i < n; ++i)
    if (!std::isfinite(s[i]) || !(s[i] > 0.0f))
      return fail(KVQ_ERR_INVALID_ARG, "scales must be finite and > 0 (got %g)", (double)s[i]);
  return KVQ_OK;
}

// FP8-domain attention query scales: host array of 1 (per tensor) or
// num_q_heads (per head) finite positive values, at most kMaxQScales.
kvq_status check_query_scales(const float* q_scales, int n, int num_q_heads) {
  if (!q_scales) return fail(KVQ_ERR_INVALID_ARG, "q_scales is NULL");
  if (n != 1 && n != num_q_heads)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_scales must be 1 or num_q_heads (%d); got %d",
                num_q_heads, n);
  if (n > kvq::kMaxQScales)
    return fail(KVQ_ERR_UNSUPPORTED, "at most %d per-head query scales", kvq::kMaxQScales);
  return check_scale_values(q_scales, n);
}

kvq_status check_rows(const kvq_cache* c, const void* k, const void* v) {
  if (!k || !v) return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
  if (!aligned16(k) || !aligned16(v)) return fail(KVQ_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  return check_device(c);
}

// Fixes a layer's scales from host values (k[H], v[H]) on its first store that
// stores tokens (fix), or checks them against the fixed ones.
kvq_status fix_or_check_scales(kvq_cache* c, int layer, const float* k, const float* v, bool fix,
                               cudaStream_t stream) {
  const int H = c->geo.kv_heads;
  if (c->mode[layer] == kUnset && !fix) return KVQ_OK;
  if (!uses_scales(c->geo.fmt)) {
    if (c->mode[layer] == kUnset) {
      c->mode[layer] = kHost;
      c->uniform[layer] = 1;
    }
    return KVQ_OK;
  }
  if (c->mode[layer] == kDevice)
    return fail(KVQ_ERR_SCALE_MISMATCH,
                "layer %d scales were calibrated on the device; store it with NULL scales", layer);
  if (c->mode[layer] == kHost) {
    for (int h = 0; h < H; ++h)
      if (host_scales(c, layer, 0)[h] != k[h] || host_scales(c, layer, 1)[h] != v[h])
        return fail(KVQ_ERR_SCALE_MISMATCH,
                    "layer %d scales are fixed (kv head %d: {%g, %g}); got {%g, %g}", layer, h,
                    (double)host_scales(c, layer, 0)[h], (double)host_scales(c, layer, 1)[h],
                    (double)k[h], (double)v[h]);
    return KVQ_OK;
  }
  bool uni = true;
  for (int h = 0; h < H; ++h) {
    host_scales(c, layer, 0)[h] = k[h];
    host_scales(c, layer, 1)[h] = v[h];
    uni = uni && k[h] == k[0] && v[h] == v[0];
  }
  const size_t base = (size_t)layer * 2 * H;
  cudaError_t e = kvq::launch_set_head_scales(c->dscale + base, c->drecip + base, k, v, H, stream);
  if (e != cudaSuccess) return cuda_fail(e, "set layer scales");
  c->mode[layer] = kHost;
  c->uniform[layer] = uni;
  return KVQ_OK;
}

kvq_status store_launch(kvq_cache* c, int layer, const void* k_bf16, const void* v_bf16,
                        const int64_t* slot_mapping, int num_tokens, cudaStream_t stream) {
  float sk, sv;
  tensor_scales(c, layer, &sk, &sv);
  cudaError_t e = kvq::launch_store(c->geo, view(c, layer), k_bf16, v_bf16, slot_mapping,
                                    num_tokens, sk, sv, head_scales(c, layer), c->err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "quantize-and-store launch");
  return KVQ_OK;
}

// Reads a layer's per-head scales into k_out / v_out ([kv_heads] each).
kvq_status read_layer_scales(const kvq_cache* c, int layer, float* k_out, float* v_out,
                             cudaStream_t stream, bool sync_device) {
  const int H = c->geo.kv_heads;
  if (c->mode[layer] == kUnset) return fail(KVQ_ERR_INVALID_ARG, "layer %d has no stored data yet", layer);
  if (c->mode[layer] == kHost) {
    std::memcpy(k_out, host_scales(c, layer, 0), sizeof(float) * H);
    std::memcpy(v_out, host_scales(c, layer, 1), sizeof(float) * H);
    return KVQ_OK;
  }
  kvq_status st = check_device(c);
  if (st) return st;
  cudaError_t e = sync_device ? cudaDeviceSynchronize() : cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "synchronize before reading calibrated scales");
  const float* d = c->dscale + (size_t)layer * 2 * H;
  if ((e = cudaMemcpy(k_out, d, sizeof(float) * H, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(v_out, d + H, sizeof(float) * H, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read calibrated scales");
  return KVQ_OK;
}

}  // namespace

namespace kvq {
void set_error_message(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
}
}  // namespace kvq

extern "C" {

const char* kvq_last_error_string(void) { return g_msg; }

const char* kvq_format_name(kvq_format fmt) {
  switch (fmt) {
    case KVQ_BF16: return "bf16";
    case KVQ_FP8_E4M3: return "fp8_e4m3";
    case KVQ_FP8_E5M2: return "fp8_e5m2";
    case KVQ_FP4_BLOCK16: return "fp4_mx_block16";
    case KVQ_NVFP4: return "nvfp4";
  }
  return nullptr;
}

kvq_status kvq_format_from_name(const char* name, kvq_format* out) {
  if (!name || !out) return fail(KVQ_ERR_INVALID_ARG, "NULL argument");
  for (int f = KVQ_BF16; f <= KVQ_NVFP4; ++f) {
    if (std::strcmp(name, kvq_format_name((kvq_format)f)) == 0) {
      *out = (kvq_format)f;
      return KVQ_OK;
    }
  }
  return fail(KVQ_ERR_INVALID_ARG, "unknown format name '%s'", name);
}

size_t kvq_bytes_per_token(kvq_format fmt, int layers, int kv_heads, int head_dim) {
  if (!valid_format(fmt) || layers <= 0 || kv_heads <= 0 || head_dim <= 0 || head_dim % 16) {
    fail(KVQ_ERR_INVALID_ARG, "invalid arguments to kvq_bytes_per_token");
    return 0;
  }
  size_t row = kvq::data_row_bytes(fmt, head_dim) + (kvq::has_block_scales(fmt) ? head_dim / 16 : 0);
  return 2 * (size_t)layers * (size_t)kv_heads * row;
}

kvq_status kvq_create_cache(kvq_format fmt, int layers, int kv_heads, int head_dim, int page_size,
                            int num_pages, kvq_cache** out) {
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "out is NULL");
  if (!valid_format(fmt)) return fail(KVQ_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
  if (layers <= 0 || kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0)
    return fail(KVQ_ERR_INVALID_ARG, "all sizes must be positive");
  if (head_dim % 16) return fail(KVQ_ERR_INVALID_ARG, "head_dim must be a multiple of 16");
  kvq::Geometry g;
  g.fmt = fmt;
  g.kv_heads = kv_heads;
  g.head_dim = head_dim;
  g.page_size = page_size;
  g.num_pages = num_pages;
  g.data_row = kvq::data_row_bytes(fmt, head_dim);
  g.scale_row = kvq::has_block_scales(fmt) ? (size_t)head_dim / 16 : 0;
  const size_t rows = (size_t)num_pages * kv_heads * page_size;
  const size_t ldb = (rows * g.data_row + 255) & ~(size_t)255;
  const size_t lsb = (rows * g.scale_row + 255) & ~(size_t)255;
  const size_t scale_bytes = ((size_t)layers * 2 * kv_heads * sizeof(float) + 255) & ~(size_t)255;
  const size_t amax_bytes = ((size_t)layers * 2 * kv_heads * sizeof(unsigned) + 255) & ~(size_t)255;
  const size_t pools = (2 * ldb + 2 * lsb) * (size_t)layers;
  const size_t total = pools + 2 * scale_bytes + amax_bytes + 256;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const char* fault = std::getenv("KVQ_FAULT");
  uint8_t* base = nullptr;
  if (fault && std::strcmp(fault, "alloc") == 0) {
    return fail(KVQ_ERR_OOM, "device allocation of %zu bytes failed (KVQ_FAULT=alloc)", total);
  }
  e = cudaMalloc(&base, total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(e == cudaErrorMemoryAllocation ? KVQ_ERR_OOM : KVQ_ERR_CUDA,
                "cudaMalloc(%zu): %s", total, cudaGetErrorString(e));
  }
  e = cudaMemset(base, 0, total);
  if (e != cudaSuccess) {
    cudaFree(base);
    return cuda_fail(e, "cudaMemset");
  }
  kvq_cache* c = new (std::nothrow) kvq_cache;
  if (!c) {
    cudaFree(base);
    return fail(KVQ_ERR_OOM, "host allocation failed");
  }
  c->geo = g;
  c->layers = layers;
  c->device = dev;
  c->base = base;
  c->bytes = total;
  c->layer_data_bytes = ldb;
  c->layer_scale_bytes = lsb;
  c->err = reinterpret_cast<int*>(base + total - 256);
  c->dscale = reinterpret_cast<float*>(base + pools);
  c->drecip = reinterpret_cast<float*>(base + pools + scale_bytes);
  c->damax = reinterpret_cast<unsigned*>(base + pools + 2 * scale_bytes);
  c->scales.assign((size_t)layers * 2 * kv_heads, 1.0f);
  c->mode.assign((size_t)layers, kUnset);
  c->uniform.assign((size_t)layers, 1);
  *out = c;
  return KVQ_OK;
}

kvq_status kvq_destroy_cache(kvq_cache* c) {
  if (!c) return KVQ_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(c->device);
  cudaError_t e = cudaDeviceSynchronize();
  cudaError_t e2 = cudaFree(c->base);
  cudaSetDevice(prev);
  delete c;
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFree");
  return KVQ_OK;
}

kvq_status kvq_cache_layout(const kvq_cache* c, int layer, void** k_data, void** v_data,
                            void** k_scales, void** v_scales, size_t strides[4]) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  kvq::LayerView L = view(c, layer);
  if (k_data) *k_data = L.k_data;
  if (v_data) *v_data = L.v_data;
  if (k_scales) *k_scales = L.k_scales;
  if (v_scales) *v_scales = L.v_scales;
  if (strides) {
    const kvq::Geometry& g = c->geo;
    strides[0] = (size_t)g.kv_heads * g.page_size * g.data_row;
    strides[1] = (size_t)g.page_size * g.data_row;
    strides[2] = g.data_row;
    strides[3] = g.scale_row;
  }
  return KVQ_OK;
}

kvq_status kvq_layer_scales(const kvq_cache* c, int layer, float out[2]) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "out is NULL");
  std::vector<float> k(c->geo.kv_heads), v(c->geo.kv_heads);
  if ((st = read_layer_scales(c, layer, k.data(), v.data(), nullptr, true))) return st;
  for (int h = 1; h < c->geo.kv_heads; ++h)
    if (k[h] != k[0] || v[h] != v[0])
      return fail(KVQ_ERR_INVALID_ARG,
                  "layer %d has per-head scales; read them with kvq_layer_head_scales", layer);
  out[0] = k[0];
  out[1] = v[0];
  return KVQ_OK;
}

kvq_status kvq_layer_head_scales(const kvq_cache* c, int layer, float* k_out, float* v_out,
                                 kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (!k_out || !v_out) return fail(KVQ_ERR_INVALID_ARG, "NULL output array");
  return read_layer_scales(c, layer, k_out, v_out, (cudaStream_t)stream, false);
}

kvq_status kvq_quantize_and_store(kvq_cache* c, int layer, const void* k_bf16, const void* v_bf16,
                                  const int64_t* slot_mapping, int num_tokens, const float* scales,
                                  kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  const bool calibrated = c->mode[layer] == kDevice;
  std::vector<float> k(c->geo.kv_heads, 1.0f), v(c->geo.kv_heads, 1.0f);
  if (uses_scales(c->geo.fmt) && scales) {
    if ((st = check_scale_values(scales, 2))) return st;
    if (calibrated)
      return fail(KVQ_ERR_SCALE_MISMATCH,
                  "layer %d scales were calibrated on the device; store it with NULL scales", layer);
    std::fill(k.begin(), k.end(), scales[0]);
    std::fill(v.begin(), v.end(), scales[1]);
  }
  if (num_tokens > 0) {
    if (!slot_mapping) return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
    if ((st = check_rows(c, k_bf16, v_bf16))) return st;
  }
  if (!calibrated && (st = fix_or_check_scales(c, layer, k.data(), v.data(), num_tokens > 0,
                                               (cudaStream_t)stream)))
    return st;
  if (num_tokens == 0) return KVQ_OK;
  return store_launch(c, layer, k_bf16, v_bf16, slot_mapping, num_tokens, (cudaStream_t)stream);
}

kvq_status kvq_quantize_and_store_per_head(kvq_cache* c, int layer, const void* k_bf16,
                                           const void* v_bf16, const int64_t* slot_mapping,
                                           int num_tokens, const float* k_scales,
                                           const float* v_scales, kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  const int H = c->geo.kv_heads;
  std::vector<float> k(H, 1.0f), v(H, 1.0f);
  if (uses_scales(c->geo.fmt)) {
    if (!k_scales || !v_scales) return fail(KVQ_ERR_INVALID_ARG, "per-head scales are NULL");
    if ((st = check_scale_values(k_scales, H)) || (st = check_scale_values(v_scales, H))) return st;
    k.assign(k_scales, k_scales + H);
    v.assign(v_scales, v_scales + H);
  }
  if (num_tokens > 0) {
    if (!slot_mapping) return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
    if ((st = check_rows(c, k_bf16, v_bf16))) return st;
  }
  if ((st = fix_or_check_scales(c, layer, k.data(), v.data(), num_tokens > 0, (cudaStream_t)stream)))
    return st;
  if (num_tokens == 0) return KVQ_OK;
  return store_launch(c, layer, k_bf16, v_bf16, slot_mapping, num_tokens, (cudaStream_t)stream);
}

kvq_status kvq_calibrate_scales(kvq_cache* c, int layer, const void* k_bf16, const void* v_bf16,
                                int num_tokens, int per_head, kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (num_tokens <= 0) return fail(KVQ_ERR_INVALID_ARG, "calibration needs num_tokens > 0");
  if (c->mode[layer] != kUnset)
    return fail(KVQ_ERR_SCALE_MISMATCH, "layer %d scales are already fixed", layer);
  if ((st = check_rows(c, k_bf16, v_bf16))) return st;
  if (!uses_scales(c->geo.fmt)) {  // nothing to calibrate: the layer keeps scale 1.0
    c->mode[layer] = kHost;
    c->uniform[layer] = 1;
    return KVQ_OK;
  }
  const size_t base = (size_t)layer * 2 * c->geo.kv_heads;
  cudaError_t e = kvq::launch_calibrate(c->geo, k_bf16, v_bf16, num_tokens, per_head != 0,
                                        c->damax + base, c->dscale + base, c->drecip + base,
                                        (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "calibration launch");
  c->mode[layer] = kDevice;
  return KVQ_OK;
}

kvq_status kvq_dequantize(kvq_cache* c, int layer, const int64_t* slot_mapping, int num_tokens,
                          void* k_out_bf16, void* v_out_bf16, kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return KVQ_OK;
  if (!slot_mapping || !k_out_bf16 || !v_out_bf16) return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
  if (!aligned16(k_out_bf16) || !aligned16(v_out_bf16))
    return fail(KVQ_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
  if ((st = check_device(c))) return st;
  float sk, sv;
  tensor_scales(c, layer, &sk, &sv);
  cudaError_t e = kvq::launch_dequantize(c->geo, view(c, layer), slot_mapping, num_tokens, sk, sv,
                                         head_scales(c, layer), k_out_bf16, v_out_bf16, c->err,
                                         (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
  return KVQ_OK;
}

size_t kvq_decode_workspace_size(const kvq_cache* c, int batch, int num_q_heads, int max_pages_per_seq) {
  if (!c || batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0) {
    fail(KVQ_ERR_INVALID_ARG, "invalid arguments to kvq_decode_workspace_size");
    return 0;
  }
  kvq::DecodePlan plan;
  const char* why = nullptr;
  if (!kvq::plan_decode(c->geo, batch, num_q_heads, max_pages_per_seq, c->device, &plan, &why)) {
    fail(KVQ_ERR_UNSUPPORTED, "%s", why);
    return 0;
  }
  return plan.ws_bytes;
}

kvq_status kvq_decode_attention(kvq_cache* c, int layer, const void* q_bf16, int num_q_heads,
                                const int32_t* page_table, int max_pages_per_seq,
                                const int32_t* seq_lens, int batch, float sm_scale, void* out_bf16,
                                void* workspace, size_t workspace_bytes, kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0)
    return fail(KVQ_ERR_INVALID_ARG, "invalid batch / num_q_heads / max_pages_per_seq");
  if (!std::isfinite(sm_scale)) return fail(KVQ_ERR_INVALID_ARG, "sm_scale must be finite");
  kvq::DecodePlan plan;
  const char* why = nullptr;
  if (!kvq::plan_decode(c->geo, batch, num_q_heads, max_pages_per_seq, c->device, &plan, &why))
    return fail(KVQ_ERR_UNSUPPORTED, "%s", why);
  if (batch == 0) return KVQ_OK;
  if (!q_bf16 || !page_table || !seq_lens || !out_bf16 || !workspace)
    return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
  if (!aligned16(q_bf16) || !aligned16(out_bf16) || !aligned16(workspace))
    return fail(KVQ_ERR_INVALID_ARG, "q, out and workspace must be 16-byte aligned");
  if (workspace_bytes < plan.ws_bytes)
    return fail(KVQ_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, plan.ws_bytes);
  if ((st = check_device(c))) return st;
  float kf, vf;
  tensor_scales(c, layer, &kf, &vf);
  cudaError_t e = kvq::launch_decode(c->geo, view(c, layer), plan, q_bf16, num_q_heads, page_table,
                                     max_pages_per_seq, seq_lens, batch, sm_scale, kf, vf,
                                     head_scales(c, layer), nullptr, 0, out_bf16, workspace, c->err,
                                     (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  return KVQ_OK;
}

kvq_status kvq_decode_attention_fp8q(kvq_cache* c, int layer, const void* q_bf16, int num_q_heads,
                                     const float* q_scales, int num_q_scales,
                                     const int32_t* page_table, int max_pages_per_seq,
                                     const int32_t* seq_lens, int batch, float sm_scale,
                                     void* out_bf16, void* workspace, size_t workspace_bytes,
                                     kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  if (batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0)
    return fail(KVQ_ERR_INVALID_ARG, "invalid batch / num_q_heads / max_pages_per_seq");
  if (!std::isfinite(sm_scale)) return fail(KVQ_ERR_INVALID_ARG, "sm_scale must be finite");
  if ((st = check_query_scales(q_scales, num_q_scales, num_q_heads))) return st;
  kvq::DecodePlan plan;
  const char* why = nullptr;
  if (!kvq::plan_decode(c->geo, batch, num_q_heads, max_pages_per_seq, c->device, &plan, &why, true))
    return fail(KVQ_ERR_UNSUPPORTED, "%s", why);
  if (batch == 0) return KVQ_OK;
  if (!q_bf16 || !page_table || !seq_lens || !out_bf16 || !workspace)
    return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
  if (!aligned16(q_bf16) || !aligned16(out_bf16) || !aligned16(workspace))
    return fail(KVQ_ERR_INVALID_ARG, "q, out and workspace must be 16-byte aligned");
  if (workspace_bytes < plan.ws_bytes)
    return fail(KVQ_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, plan.ws_bytes);
  if ((st = check_device(c))) return st;
  float kf, vf;
  tensor_scales(c, layer, &kf, &vf);
  cudaError_t e = kvq::launch_decode(c->geo, view(c, layer), plan, q_bf16, num_q_heads, page_table,
                                     max_pages_per_seq, seq_lens, batch, sm_scale, kf, vf,
                                     head_scales(c, layer), nullptr, 0, out_bf16, workspace, c->err,
                                     (cudaStream_t)stream, q_scales, num_q_scales);
  if (e != cudaSuccess) return cuda_fail(e, "FP8-domain decode attention launch");
  return KVQ_OK;
}

kvq_status kvq_quantize_query(const void* q_bf16, int rows, int num_q_heads, int head_dim,
                              const float* q_scales, int num_q_scales, void* q_codes,
                              kvq_stream stream) {
  if (rows < 0 || num_q_heads <= 0 || head_dim <= 0 || head_dim % 16)
    return fail(KVQ_ERR_INVALID_ARG, "invalid rows / num_q_heads / head_dim (a multiple of 16)");
  kvq_status st = check_query_scales(q_scales, num_q_scales, num_q_heads);
  if (st) return st;
  if (rows == 0) return KVQ_OK;
  if (!q_bf16 || !q_codes) return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
  if (!aligned16(q_bf16) || !aligned16(q_codes))
    return fail(KVQ_ERR_INVALID_ARG, "q and q_codes must be 16-byte aligned");
  cudaError_t e = kvq::launch_quantize_query(q_bf16, rows, num_q_heads, head_dim, q_scales,
                                             num_q_scales, q_codes, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "query quantization launch");
  return KVQ_OK;
}

size_t kvq_extend_workspace_size(const kvq_cache* c, int num_q_tokens, int num_q_heads,
                                 int max_pages_per_seq) {
  if (!c || num_q_tokens < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 ||
      num_q_heads % c->geo.kv_heads != 0) {
    fail(KVQ_ERR_INVALID_ARG, "invalid arguments to kvq_extend_workspace_size");
    return 0;
  }
  const int splits = kvq::extend_splits(c->geo, num_q_tokens, num_q_heads, max_pages_per_seq, c->device);
  return kvq::extend_workspace_bytes(splits, num_q_tokens, num_q_heads);
}

kvq_status kvq_extend_attention(kvq_cache* c, int layer, const void* q_bf16, int num_q_heads,
                                int num_q_tokens, const int32_t* q_seq, const int32_t* q_len,
                                const int32_t* page_table, int num_seqs, int max_pages_per_seq,
                                float sm_scale, void* out_bf16, void* workspace,
                                size_t workspace_bytes, kvq_stream stream) {
  kvq_status st = check_layer(c, layer);
  if (st) return st;
  const kvq::Geometry& g = c->geo;
  if (num_q_tokens < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 || num_seqs <= 0)
    return fail(KVQ_ERR_INVALID_ARG, "invalid num_q_tokens / num_q_heads / max_pages / num_seqs");
  if (!std::isfinite(sm_scale)) return fail(KVQ_ERR_INVALID_ARG, "sm_scale must be finite");
  if (g.head_dim != kvq::kHeadDim)
    return fail(KVQ_ERR_UNSUPPORTED, "extend attention supports head_dim == 128 only");
  if (g.page_size % kvq::kTile != 0)
    return fail(KVQ_ERR_UNSUPPORTED, "extend attention needs page_size %% 16 == 0");
  if (num_q_heads % g.kv_heads != 0)
    return fail(KVQ_ERR_UNSUPPORTED, "num_q_heads must be a multiple of kv_heads");
  if (num_q_tokens == 0) return KVQ_OK;
  if (!q_bf16 || !q_seq || !q_len || !page_table || !out_bf16)
    return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer");
  if (!aligned16(q_bf16) || !aligned16(out_bf16) || (workspace && !aligned16(workspace)))
    return fail(KVQ_ERR_INVALID_ARG, "q, out and workspace must be 16-byte aligned");
  if ((st = check_device(c))) return st;
  // context splits: as many as the plan wants and the workspace holds
  int splits = kvq::extend_splits(g, num_q_tokens, num_q_heads, max_pages_per_seq, c->device);
  while (splits > 1 && (!workspace ||
                        kvq::extend_workspace_bytes(splits, num_q_tokens, num_q_heads) > workspace_bytes))
    --splits;
  float kf, vf;
  tensor_scales(c, layer, &kf, &vf);
  cudaError_t e = kvq::launch_extend(g, view(c, layer), q_bf16, num_q_heads, num_q_tokens, q_seq,
                                     q_len, page_table, num_seqs, max_pages_per_seq, sm_scale, kf, vf,
                                     head_scales(c, layer), out_bf16, c->err, splits, workspace,
                                     (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "extend attention launch");
  return KVQ_OK;
}

kvq_status kvq_get_device_error(kvq_cache* c, kvq_stream stream) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "cache is NULL");
  kvq_status st = check_device(c);
  if (st) return st;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, c->err, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (word) {
    const int zero = 0;
    e = cudaMemcpy(c->err, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  }
  if (word & kvq::kErrTimeout) return fail(KVQ_ERR_TIMEOUT, "a kernel's bounded wait ran out");
  if (word & kvq::kErrRange)
    return fail(KVQ_ERR_DEVICE_RANGE, "a kernel saw an out-of-range slot, page id or sequence length");
  return KVQ_OK;
}

}  // extern "C"
