// kvq_store.cu -- quantize-and-store and dequantize-gather kernels.
//
// "SGLang PR #21954 analysis: NVFP4 KV cache", Code analysis 1:
// quantize_and_store quantizes incoming bf16 K/V and writes data plus block
// scales into the cache buffers; dequantize_prev_kv reads them back.
// "Quantized KV Cache" (SGLang documentation), Supported formats and Scaling
// factors: FP8 with a per-tensor scale; FP4 E2M1 with one 8-bit exponent per
// 16-element block computed on the fly; NVFP4 with an fp32 global scale and an
// FP8-E4M3 scale per block.
//
// One thread owns one 16-element block of one (token, kv_head) row: two
// 16-byte loads of bf16, the block amax in registers, encode, and one 16-byte
// (FP8) or 8-byte (FP4) store into the paged row plus one scale byte.  Eight
// consecutive threads cover one 128-element row, so loads and stores of a warp
// are contiguous 1 KB / 512 B / 256 B runs.  The kernel is HBM-bound.
#include "kvq_codecs.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

struct StoreArgs {
  const uint16_t* x[2];  // K, V bf16 [n][H][D]
  uint8_t* data[2];
  uint8_t* scales[2];
  float s[2];            // FP8 scale / NVFP4 global scale per K, V
  const int64_t* slots;
  int64_t items;         // n * H * (D / 16)
  int H, D, P;
  int64_t num_pages;
  int* err;
};

__device__ __forceinline__ void load16(const uint16_t* p, float x[16]) {
  uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_bits_to_float(w[i] & 0xFFFF);
    x[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

template <kvq_format F>
__global__ void __launch_bounds__(256) store_kernel(StoreArgs a) {
  const int kv = blockIdx.y;  // 0: K, 1: V
  const int nb = a.D >> 4;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < a.items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = it / nb;
    const int blk = (int)(it - row * nb);
    const int64_t tok = row / a.H;
    const int h = (int)(row - tok * a.H);
    const int64_t slot = __ldg(a.slots + tok);
    if (slot < 0) continue;
    if (slot >= a.num_pages * a.P) {
      if (blk == 0) atomicOr(a.err, kErrRange);
      continue;
    }
    const int64_t page = slot / a.P, off = slot - page * a.P;
    const int64_t r = (page * a.H + h) * a.P + off;  // destination row
    const uint16_t* src = a.x[kv] + row * a.D + blk * 16;

    if (F == KVQ_BF16) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(a.data[kv] + r * (a.D * 2) + blk * 32);
      d4[0] = __ldg(s4);
      d4[1] = __ldg(s4 + 1);
      continue;
    }

    float x[16];
    load16(src, x);

    if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
      const float s = a.s[kv];
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float x0 = x[4 * i + 2 * j], x1 = x[4 * i + 2 * j + 1];
          const float q0 = x0 / s, q1 = x1 / s;  // IEEE fp32 division
          uint32_t p = (F == KVQ_FP8_E4M3) ? enc2_e4m3(q0, q1) : enc2_e5m2(q0, q1);
          // NaN input: 0x7F with the input's sign
          if (x0 != x0) p = (p & 0xFF00u) | 0x7Fu | ((__float_as_uint(x0) >> 24) & 0x80u);
          if (x1 != x1) p = (p & 0x00FFu) | ((0x7Fu | ((__float_as_uint(x1) >> 24) & 0x80u)) << 8);
          c[2 * j] = p & 0xFF;
          c[2 * j + 1] = p >> 8;
        }
        w[i] = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
      }
      *reinterpret_cast<uint4*>(a.data[kv] + r * a.D + blk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      continue;
    }

    // FP4 formats: block amax, block scale, E2M1 codes.
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    float mul = 1.f, S = 1.f;
    uint32_t scode;
    bool zero = false;
    if (F == KVQ_FP4_BLOCK16) {
      // MX shared exponent: E = clamp(floor(log2 amax) - 2, -127, 127)
      int E = -127;
      if (amax > 0.f) E = max(-127, min(127, floor_log2(amax) - 2));
      scode = (uint32_t)(E + 127);
      mul = exp2i(-E);
    } else {
      // NVFP4: sc = E4M3(amax / (6 g)); S = dec(sc) * g
      const float g = a.s[kv];
      const float ratio = amax / (6.0f * g);
      scode = enc2_e4m3(ratio, 0.f) & 0xFF;
      S = __fmul_rn(dec_e4m3(scode), g);
      zero = (S == 0.f);
    }
    uint32_t w[2] = {0u, 0u};
    if (!zero) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float y0, y1;
        if (F == KVQ_FP4_BLOCK16) {
          y0 = __fmul_rn(x[2 * i], mul);
          y1 = __fmul_rn(x[2 * i + 1], mul);
        } else {
          y0 = x[2 * i] / S;
          y1 = x[2 * i + 1] / S;
        }
        w[i >> 2] |= enc2_e2m1(y0, y1) << (8 * (i & 3));
      }
    }
    *reinterpret_cast<uint2*>(a.data[kv] + r * (a.D / 2) + blk * 8) = make_uint2(w[0], w[1]);
    a.scales[kv][r * nb + blk] = (uint8_t)scode;
  }
}

struct DequantArgs {
  const uint8_t* data[2];
  const uint8_t* scales[2];
  uint16_t* out[2];
  float s[2];
  const int64_t* slots;
  int64_t items;
  int H, D, P;
  int64_t num_pages;
  int* err;
};

template <kvq_format F>
__global__ void __launch_bounds__(256) dequant_kernel(DequantArgs a) {
  const int kv = blockIdx.y;
  const int nb = a.D >> 4;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < a.items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = it / nb;
    const int blk = (int)(it - row * nb);
    const int64_t tok = row / a.H;
    const int h = (int)(row - tok * a.H);
    const int64_t slot = __ldg(a.slots + tok);
    uint4* dst = reinterpret_cast<uint4*>(a.out[kv] + row * a.D + blk * 16);
    const bool in_range = slot >= 0 && slot < a.num_pages * a.P;
    if (!in_range) {
      if (slot >= 0 && blk == 0) atomicOr(a.err, kErrRange);
      dst[0] = make_uint4(0, 0, 0, 0);
      dst[1] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int64_t page = slot / a.P, off = slot - page * a.P;
    const int64_t r = (page * a.H + h) * a.P + off;
    if (F == KVQ_BF16) {
      const uint4* s4 = reinterpret_cast<const uint4*>(a.data[kv] + r * (a.D * 2) + blk * 32);
      dst[0] = __ldg(s4);
      dst[1] = __ldg(s4 + 1);
      continue;
    }
    float v[16];
    if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(a.data[kv] + r * a.D + blk * 16));
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
      const float s = a.s[kv];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2(w[i]) : dec2_e5m2_h2(w[i]);
        const uint32_t hi = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2_hi(w[i]) : dec2_e5m2_h2_hi(w[i]);
        v[4 * i + 0] = __fmul_rn(h2_lo(lo), s);
        v[4 * i + 1] = __fmul_rn(h2_hi(lo), s);
        v[4 * i + 2] = __fmul_rn(h2_lo(hi), s);
        v[4 * i + 3] = __fmul_rn(h2_hi(hi), s);
      }
    } else {
      const uint2 c = __ldg(reinterpret_cast<const uint2*>(a.data[kv] + r * (a.D / 2) + blk * 8));
      const uint32_t sc = a.scales[kv][r * nb + blk];
      const float S = (F == KVQ_FP4_BLOCK16) ? dec_e8m0(sc) : __fmul_rn(dec_e4m3(sc), a.s[kv]);
      const uint32_t w[2] = {c.x, c.y};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t h0 = dec2_e2m1_h2<0>(w[i]), h1 = dec2_e2m1_h2<1>(w[i]);
        const uint32_t h2 = dec2_e2m1_h2<2>(w[i]), h3 = dec2_e2m1_h2<3>(w[i]);
        v[8 * i + 0] = __fmul_rn(h2_lo(h0), S);
        v[8 * i + 1] = __fmul_rn(h2_hi(h0), S);
        v[8 * i + 2] = __fmul_rn(h2_lo(h1), S);
        v[8 * i + 3] = __fmul_rn(h2_hi(h1), S);
        v[8 * i + 4] = __fmul_rn(h2_lo(h2), S);
        v[8 * i + 5] = __fmul_rn(h2_hi(h2), S);
        v[8 * i + 6] = __fmul_rn(h2_lo(h3), S);
        v[8 * i + 7] = __fmul_rn(h2_hi(h3), S);
      }
    }
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = bf16_rne_bits(v[2 * i]) | (bf16_rne_bits(v[2 * i + 1]) << 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

int grid_for(int64_t items) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (items + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;  // grid-stride beyond 8 blocks per SM
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_store(const Geometry& g, const LayerView& L, const void* k, const void* v,
                         const int64_t* slots, int num_tokens, float s_k, float s_v, int* err,
                         cudaStream_t stream) {
  StoreArgs a;
  a.x[0] = static_cast<const uint16_t*>(k);
  a.x[1] = static_cast<const uint16_t*>(v);
  a.data[0] = L.k_data;
  a.data[1] = L.v_data;
  a.scales[0] = L.k_scales;
  a.scales[1] = L.v_scales;
  a.s[0] = s_k;
  a.s[1] = s_v;
  a.slots = slots;
  a.items = (int64_t)num_tokens * g.kv_heads * (g.head_dim / 16);
  a.H = g.kv_heads;
  a.D = g.head_dim;
  a.P = g.page_size;
  a.num_pages = g.num_pages;
  a.err = err;
  if (a.items == 0) return cudaSuccess;
  dim3 grid(grid_for(a.items), 2);
  switch (g.fmt) {
    case KVQ_BF16: store_kernel<KVQ_BF16><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_FP8_E4M3: store_kernel<KVQ_FP8_E4M3><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_FP8_E5M2: store_kernel<KVQ_FP8_E5M2><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_FP4_BLOCK16: store_kernel<KVQ_FP4_BLOCK16><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_NVFP4: store_kernel<KVQ_NVFP4><<<grid, 256, 0, stream>>>(a); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const Geometry& g, const LayerView& L, const int64_t* slots,
                              int num_tokens, float s_k, float s_v, void* k_out, void* v_out,
                              int* err, cudaStream_t stream) {
  DequantArgs a;
  a.data[0] = L.k_data;
  a.data[1] = L.v_data;
  a.scales[0] = L.k_scales;
  a.scales[1] = L.v_scales;
  a.out[0] = static_cast<uint16_t*>(k_out);
  a.out[1] = static_cast<uint16_t*>(v_out);
  a.s[0] = s_k;
  a.s[1] = s_v;
  a.slots = slots;
  a.items = (int64_t)num_tokens * g.kv_heads * (g.head_dim / 16);
  a.H = g.kv_heads;
  a.D = g.head_dim;
  a.P = g.page_size;
  a.num_pages = g.num_pages;
  a.err = err;
  if (a.items == 0) return cudaSuccess;
  dim3 grid(grid_for(a.items), 2);
  switch (g.fmt) {
    case KVQ_BF16: dequant_kernel<KVQ_BF16><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_FP8_E4M3: dequant_kernel<KVQ_FP8_E4M3><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_FP8_E5M2: dequant_kernel<KVQ_FP8_E5M2><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_FP4_BLOCK16: dequant_kernel<KVQ_FP4_BLOCK16><<<grid, 256, 0, stream>>>(a); break;
    case KVQ_NVFP4: dequant_kernel<KVQ_NVFP4><<<grid, 256, 0, stream>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace kvq
