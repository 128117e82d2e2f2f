// kvq_decode.cu -- split-K paged GQA decode attention over the quantized cache.
//
// "Quantized KV Cache" (SGLang documentation), performance warning: an
// attention kernel that does not fuse dequantization is extremely slow, so K
// and V are dequantized in registers inside the attention kernel.
// "SGLang PR #21954 analysis: NVFP4 KV cache", Why is this good? 2: decode is
// bound by KV-cache bandwidth; the kernel reads every cached byte once.
//
// Work decomposition (load balance for ragged lengths):
//   unit u = (sequence b, kv head h, head group hg of <= 8 q heads);
//   a unit has nt_b = ceil(T_b / 16) tiles of 16 tokens;
//   all units' tiles are laid end to end (b-major) into one range of Wtot
//   tiles, and warp worker w takes [w Wtot / NW, (w + 1) Wtot / NW).
//   A worker emits one partial (o normalized, lse in log2 units) per unit it
//   touches into slot u + w (unique, see plan_decode), and the merge kernel
//   combines a unit's partials with the log-sum-exp rule
//     out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s.
#include "kvq_codecs.cuh"
#include "kvq_internal.h"

#include <algorithm>

namespace kvq {
namespace {

constexpr int kWarpsPerCta = 4;
constexpr int kHeadDim = 128;
constexpr int kTile = 16;      // tokens per tile
constexpr int kGroupMax = 8;   // q heads per unit

struct DecodeArgs {
  const uint16_t* q;
  uint16_t* out;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const uint8_t* kd;
  const uint8_t* vd;
  const uint8_t* ks;
  const uint8_t* vs;
  float* part_o;      // [slots][8][128]
  float* part_lse;    // [slots][8]
  long long* meta;    // [0] = Wtot
  int B, H, Hq, G, HG, max_pages, P;
  long long num_pages;
  int num_workers;
  float qscale;       // sm_scale * log2(e) * (k_scale | g_k | 1)
  float v_factor;     // v_scale | g_v | 1
  int* err;
};

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Tiles of sequence b (0 for an empty or invalid length).
__device__ __forceinline__ int tiles_of(const DecodeArgs& a, int b) {
  const int T = __ldg(a.seq_lens + b);
  return (T > 0 && T <= a.max_pages * a.P) ? (T + kTile - 1) / kTile : 0;
}

// First tile of worker w (integer split of [0, total)).
__device__ __forceinline__ long long worker_start(long long total, int w, int nw) {
  return total * w / nw;
}

// Four exact dequantized values of row `row` at head_dim indices 4*lane..+3
// (without the per-tensor factor, which is folded into q or the output).
template <kvq_format F>
__device__ __forceinline__ void load4(const uint8_t* data, const uint8_t* scl, long long row,
                                      int lane, float v[4]) {
  if (F == KVQ_BF16) {
    const uint2 w = *reinterpret_cast<const uint2*>(data + row * (kHeadDim * 2) + lane * 8);
    v[0] = bf16_bits_to_float(w.x & 0xFFFF);
    v[1] = bf16_bits_to_float(w.x >> 16);
    v[2] = bf16_bits_to_float(w.y & 0xFFFF);
    v[3] = bf16_bits_to_float(w.y >> 16);
  } else if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(data + row * kHeadDim + lane * 4);
    const uint32_t lo = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2(w) : dec2_e5m2_h2(w);
    const uint32_t hi = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2_hi(w) : dec2_e5m2_h2_hi(w);
    v[0] = h2_lo(lo);
    v[1] = h2_hi(lo);
    v[2] = h2_lo(hi);
    v[3] = h2_hi(hi);
  } else {
    const uint32_t w = *reinterpret_cast<const uint16_t*>(data + row * (kHeadDim / 2) + lane * 2);
    const uint32_t sc = scl[row * (kHeadDim / 16) + (lane >> 2)];
    const float S = (F == KVQ_FP4_BLOCK16) ? dec_e8m0(sc) : dec_e4m3(sc);
    const uint32_t h0 = dec2_e2m1_h2<0>(w), h1 = dec2_e2m1_h2<1>(w);
    v[0] = h2_lo(h0) * S;
    v[1] = h2_hi(h0) * S;
    v[2] = h2_lo(h1) * S;
    v[3] = h2_hi(h1) * S;
  }
}

// One worker's contribution to unit (b, h, hg) over tiles [t0, t1): simple
// CUDA-core form, lane l owns head_dim indices 4l..4l+3.
template <kvq_format F>
__device__ void segment_simple(const DecodeArgs& a, int w, int b, int h, int hg, int t0, int t1) {
  const int lane = threadIdx.x & 31;
  const int T = __ldg(a.seq_lens + b);
  const int gh = min(kGroupMax, a.G - hg * kGroupMax);
  float q[kGroupMax][4], m[kGroupMax], l[kGroupMax], o[kGroupMax][4];
#pragma unroll
  for (int g = 0; g < kGroupMax; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) { q[g][i] = 0.f; o[g][i] = 0.f; }
    if (g < gh) {
      const uint16_t* qr = a.q + ((long long)b * a.Hq + h * a.G + hg * kGroupMax + g) * kHeadDim;
      const uint2 qw = *reinterpret_cast<const uint2*>(qr + lane * 4);
      q[g][0] = bf16_bits_to_float(qw.x & 0xFFFF) * a.qscale;
      q[g][1] = bf16_bits_to_float(qw.x >> 16) * a.qscale;
      q[g][2] = bf16_bits_to_float(qw.y & 0xFFFF) * a.qscale;
      q[g][3] = bf16_bits_to_float(qw.y >> 16) * a.qscale;
    }
  }
  bool poison = false;
  for (int t = t0; t < t1; ++t) {
    const int tok0 = t * kTile;
    const int page = __ldg(a.page_table + (long long)b * a.max_pages + tok0 / a.P);
    if (page < 0 || page >= a.num_pages) { poison = true; continue; }
    const long long row0 = ((long long)page * a.H + h) * a.P + tok0 % a.P;
    const int ntok = min(kTile, T - tok0);
    for (int j = 0; j < ntok; ++j) {
      float kv[4];
      load4<F>(a.kd, a.ks, row0 + j, lane, kv);
      float z[kGroupMax];
#pragma unroll
      for (int g = 0; g < kGroupMax; ++g)
        z[g] = warp_sum_f(q[g][0] * kv[0] + q[g][1] * kv[1] + q[g][2] * kv[2] + q[g][3] * kv[3]);
      load4<F>(a.vd, a.vs, row0 + j, lane, kv);
#pragma unroll
      for (int g = 0; g < kGroupMax; ++g) {
        const float mn = fmaxf(m[g], z[g]);
        const float al = exp2f(m[g] - mn);
        const float p = exp2f(z[g] - mn);
        l[g] = l[g] * al + p;
#pragma unroll
        for (int i = 0; i < 4; ++i) o[g][i] = o[g][i] * al + p * kv[i];
        m[g] = mn;
      }
    }
  }
  if (poison && lane == 0) atomicOr(a.err, kErrRange);
  const long long u = ((long long)b * a.H + h) * a.HG + hg;
  const long long slot = u + w;
#pragma unroll
  for (int g = 0; g < kGroupMax; ++g) {
    if (g >= gh) break;
    float* po = a.part_o + (slot * kGroupMax + g) * kHeadDim + lane * 4;
    const float inv = poison ? 0.f : a.v_factor / l[g];
    *reinterpret_cast<float4*>(po) = make_float4(o[g][0] * inv, o[g][1] * inv, o[g][2] * inv, o[g][3] * inv);
    if (lane == 0) a.part_lse[slot * kGroupMax + g] = poison ? INFINITY : m[g] + __log2f(l[g]);
  }
}

template <kvq_format F>
__global__ void __launch_bounds__(kWarpsPerCta * 32) decode_kernel(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (w >= a.num_workers) return;
  const long long upb = (long long)a.H * a.HG;  // units per sequence

  // pass 1: total tiles; worker 0 reports invalid lengths and publishes Wtot
  long long total = 0;
  bool bad_len = false;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int b = b0 + lane;
    int nt = 0;
    if (b < a.B) {
      const int T = __ldg(a.seq_lens + b);
      if (T < 0 || T > a.max_pages * a.P) bad_len = true;
      nt = tiles_of(a, b);
    }
    total += warp_sum_i(nt);
  }
  total *= upb;
  if (w == 0) {
    if (__any_sync(0xffffffffu, bad_len) && lane == 0) atomicOr(a.err, kErrRange);
    if (lane == 0) a.meta[0] = total;
  }
  const long long start = worker_start(total, w, a.num_workers);
  const long long end = worker_start(total, w + 1, a.num_workers);
  if (start >= end) return;

  // pass 2: locate the sequence holding `start`
  long long cum = 0;
  int b = 0;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int bb = b0 + lane;
    long long x = (bb < a.B) ? (long long)tiles_of(a, bb) * upb : 0;
    long long incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const long long chunk = __shfl_sync(0xffffffffu, incl, 31);
    if (cum + chunk > start) {
      const unsigned hit = __ballot_sync(0xffffffffu, cum + incl > start);
      const int src = __ffs(hit) - 1;
      const long long excl = __shfl_sync(0xffffffffu, incl - x, src);
      b = b0 + src;
      cum += excl;
      break;
    }
    cum += chunk;
  }
  int nt = tiles_of(a, b);
  long long local = start - cum;
  int ub = (int)(local / nt);
  int tile = (int)(local - (long long)ub * nt);
  long long pos = start;
  while (pos < end) {
    const int n = (int)min((long long)(nt - tile), end - pos);
    segment_simple<F>(a, w, b, ub / a.HG, ub % a.HG, tile, tile + n);
    pos += n;
    tile += n;
    if (tile == nt) {
      tile = 0;
      if (++ub == upb) {
        ub = 0;
        do { ++b; } while (pos < end && (nt = tiles_of(a, b)) == 0);
      }
    }
  }
}

// One CTA per sequence: combine each (unit, head)'s partials.
__global__ void __launch_bounds__(256) merge_kernel(DecodeArgs a) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ long long s_red[8];
  long long part = 0;
  for (int i = threadIdx.x; i < b; i += blockDim.x) part += tiles_of(a, i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) s_red[warp] = part;
  __syncthreads();
  long long cum = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) cum += s_red[i];
  const long long upb = (long long)a.H * a.HG;
  const long long total = a.meta[0];
  const int nt = tiles_of(a, b);
  const int nw = a.num_workers;
  for (int ub = 0; ub < upb; ++ub) {
    const int h = ub / a.HG, hg = ub % a.HG;
    const int g = warp;
    if (g >= min(kGroupMax, a.G - hg * kGroupMax)) continue;
    uint16_t* orow = a.out + ((long long)b * a.Hq + h * a.G + hg * kGroupMax + g) * kHeadDim + lane * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    bool zero = (nt == 0);
    if (!zero) {
      const long long u = (long long)b * upb + ub;
      const long long w0 = cum * upb + (long long)ub * nt;   // first tile of the unit
      const long long w1 = w0 + nt;                          // one past its last tile
      // worker holding tile x: max w with start(w) <= x
      const int wf = (int)(((w0 + 1) * nw - 1) / total);
      const int wl = (int)((w1 * nw - 1) / total);
      float M = -INFINITY;
      for (int w = wf; w <= wl; ++w) {
        if (worker_start(total, w, nw) == worker_start(total, w + 1, nw)) continue;
        const float lse = a.part_lse[(u + w) * kGroupMax + g];
        if (lse == INFINITY) zero = true;
        M = fmaxf(M, lse);
      }
      if (!zero) {
        float den = 0.f;
        for (int w = wf; w <= wl; ++w) {
          if (worker_start(total, w, nw) == worker_start(total, w + 1, nw)) continue;
          const long long s = u + w;
          const float wt = exp2f(a.part_lse[s * kGroupMax + g] - M);
          const float4 po = *reinterpret_cast<const float4*>(a.part_o + (s * kGroupMax + g) * kHeadDim + lane * 4);
          den += wt;
          acc[0] += wt * po.x;
          acc[1] += wt * po.y;
          acc[2] += wt * po.z;
          acc[3] += wt * po.w;
        }
        const float inv = 1.f / den;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] *= inv;
      }
    }
    if (zero) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    uint2 ov;
    ov.x = bf16_rne_bits(acc[0]) | (bf16_rne_bits(acc[1]) << 16);
    ov.y = bf16_rne_bits(acc[2]) | (bf16_rne_bits(acc[3]) << 16);
    *reinterpret_cast<uint2*>(orow) = ov;
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

bool plan_decode(const Geometry& g, int batch, int num_q_heads, int max_pages_per_seq,
                 int device, DecodePlan* plan, const char** why) {
  if (g.head_dim != kHeadDim) { *why = "decode attention supports head_dim == 128 only"; return false; }
  if (g.page_size % kTile != 0) { *why = "decode attention needs page_size % 16 == 0"; return false; }
  if (num_q_heads % g.kv_heads != 0) { *why = "num_q_heads must be a multiple of kv_heads"; return false; }
  const int G = num_q_heads / g.kv_heads;
  if (G > 2 * kGroupMax) { *why = "group size num_q_heads / kv_heads must be <= 16"; return false; }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0) {
    *why = "cannot query the SM count";
    return false;
  }
  plan->group = G;
  plan->head_groups = (G + kGroupMax - 1) / kGroupMax;
  plan->num_units = (int64_t)batch * g.kv_heads * plan->head_groups;
  const int64_t tiles_per_seq = ((int64_t)max_pages_per_seq * g.page_size + kTile - 1) / kTile;
  const int64_t max_tiles = std::max<int64_t>(1, plan->num_units * tiles_per_seq);
  int64_t ctas = (int64_t)sms * 4;
  ctas = std::min<int64_t>(ctas, (max_tiles + kWarpsPerCta - 1) / kWarpsPerCta);
  ctas = std::max<int64_t>(ctas, 1);
  plan->ctas = (int)ctas;
  plan->num_workers = plan->ctas * kWarpsPerCta;
  plan->num_slots = plan->num_units + plan->num_workers;
  plan->ws_bytes = align256((size_t)plan->num_slots * kGroupMax * kHeadDim * sizeof(float)) +
                   align256((size_t)plan->num_slots * kGroupMax * sizeof(float)) + 256;
  return true;
}

cudaError_t launch_decode(const Geometry& g, const LayerView& L, const DecodePlan& plan,
                          const void* q, int num_q_heads, const int32_t* page_table,
                          int max_pages_per_seq, const int32_t* seq_lens, int batch,
                          float sm_scale, float k_factor, float v_factor, void* out,
                          void* workspace, int* err, cudaStream_t stream) {
  DecodeArgs a;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.part_o = reinterpret_cast<float*>(ws);
  ws += align256((size_t)plan.num_slots * kGroupMax * kHeadDim * sizeof(float));
  a.part_lse = reinterpret_cast<float*>(ws);
  ws += align256((size_t)plan.num_slots * kGroupMax * sizeof(float));
  a.meta = reinterpret_cast<long long*>(ws);
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.kd = L.k_data;
  a.vd = L.v_data;
  a.ks = L.k_scales;
  a.vs = L.v_scales;
  a.B = batch;
  a.H = g.kv_heads;
  a.Hq = num_q_heads;
  a.G = plan.group;
  a.HG = plan.head_groups;
  a.max_pages = max_pages_per_seq;
  a.P = g.page_size;
  a.num_pages = g.num_pages;
  a.num_workers = plan.num_workers;
  a.qscale = sm_scale * 1.4426950408889634f * k_factor;
  a.v_factor = v_factor;
  a.err = err;
  if (batch == 0) return cudaSuccess;
  switch (g.fmt) {
    case KVQ_BF16: decode_kernel<KVQ_BF16><<<plan.ctas, kWarpsPerCta * 32, 0, stream>>>(a); break;
    case KVQ_FP8_E4M3: decode_kernel<KVQ_FP8_E4M3><<<plan.ctas, kWarpsPerCta * 32, 0, stream>>>(a); break;
    case KVQ_FP8_E5M2: decode_kernel<KVQ_FP8_E5M2><<<plan.ctas, kWarpsPerCta * 32, 0, stream>>>(a); break;
    case KVQ_FP4_BLOCK16: decode_kernel<KVQ_FP4_BLOCK16><<<plan.ctas, kWarpsPerCta * 32, 0, stream>>>(a); break;
    case KVQ_NVFP4: decode_kernel<KVQ_NVFP4><<<plan.ctas, kWarpsPerCta * 32, 0, stream>>>(a); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  merge_kernel<<<batch, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
