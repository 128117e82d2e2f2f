// kvq_merge.cu -- log-sum-exp merge of the split-K decode partials.
//
// A unit (sequence, kv head, group of <= 8 q heads) is split over the warp
// workers that touched its tiles; each wrote a normalized partial output o_s
// and its log-sum-exp lse_s (log2 units).  The merge combines them:
//   out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s,
// rounded to bf16.  One CTA per unit, one warp per q head, lanes own four
// head_dim elements.  A partial with lse = +inf marks a unit that saw an
// invalid page id: its output is zero.
#include "kvq_codecs.cuh"
#include "kvq_decode_args.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

__global__ void __launch_bounds__(256) merge_kernel(DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long u = blockIdx.x;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long upb = (long long)a.H * a.HG;
  const int b = (int)(u / upb), ub = (int)(u - (long long)b * upb);
  const int h = ub / a.HG, hg = ub - (ub / a.HG) * a.HG;
  if (g >= min(kGroupMax, a.G - hg * kGroupMax)) return;
  uint16_t* orow = a.out + ((long long)b * a.Hq + h * a.G + hg * kGroupMax + g) * kHeadDim + lane * 4;
  const int nt = tiles_of(a, b);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (nt > 0) {
    const long long total = a.meta[0];
    const int nw = a.num_workers;
    const long long w0 = a.prefix[b] * upb + (long long)ub * nt;  // first tile of the unit
    const long long w1 = w0 + nt;                                 // one past its last tile
    // worker holding tile x: max w with start(w) <= x
    const int wf = (int)(((w0 + 1) * nw - 1) / total);
    const int wl = (int)((w1 * nw - 1) / total);
    // with at least one tile per worker no worker in [wf, wl] is empty
    const bool dense = total >= nw;
    auto nonempty = [&](int w) {
      return dense || worker_start(total, w, nw) != worker_start(total, w + 1, nw);
    };
    float M = -INFINITY;
    bool poison = false;
    for (int w = wf + lane; w <= wl; w += 32) {
      if (!nonempty(w)) continue;
      const float lse = a.part_lse[(u + w) * kGroupMax + g];
      poison |= (lse == INFINITY);
      M = fmaxf(M, lse);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    poison = __any_sync(0xffffffffu, poison);
    if (!poison) {
      float den = 0.f;
      const float* base = a.part_o + (u * kGroupMax + g) * kHeadDim + lane * 4;
      for (int c0 = wf; c0 <= wl; c0 += 32) {
        const int w = c0 + lane;
        float wt = 0.f;
        if (w <= wl && nonempty(w)) wt = ex2(a.part_lse[(u + w) * kGroupMax + g] - M);
        den += wt;
        const int cnt = min(32, wl - c0 + 1);
        if (dense) {
          // every slot in range was written: batch the loads
          int j = 0;
          for (; j + 4 <= cnt; j += 4) {
            float4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              v[i] = *reinterpret_cast<const float4*>(base + (long long)(c0 + j + i) * kGroupMax * kHeadDim);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float wj = __shfl_sync(0xffffffffu, wt, j + i);
              acc[0] += wj * v[i].x;
              acc[1] += wj * v[i].y;
              acc[2] += wj * v[i].z;
              acc[3] += wj * v[i].w;
            }
          }
          for (; j < cnt; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wt, j);
            const float4 v = *reinterpret_cast<const float4*>(base + (long long)(c0 + j) * kGroupMax * kHeadDim);
            acc[0] += wj * v.x;
            acc[1] += wj * v.y;
            acc[2] += wj * v.z;
            acc[3] += wj * v.w;
          }
        } else {
          for (int j = 0; j < cnt; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wt, j);
            if (wj != 0.f) {
              const float4 v = *reinterpret_cast<const float4*>(base + (long long)(c0 + j) * kGroupMax * kHeadDim);
              acc[0] += wj * v.x;
              acc[1] += wj * v.y;
              acc[2] += wj * v.z;
              acc[3] += wj * v.w;
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
      const float inv = 1.f / den;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] *= inv;
    }
  }
  uint2 ov;
  ov.x = bf16_rne_bits(acc[0]) | (bf16_rne_bits(acc[1]) << 16);
  ov.y = bf16_rne_bits(acc[2]) | (bf16_rne_bits(acc[3]) << 16);
  *reinterpret_cast<uint2*>(orow) = ov;
}

}  // namespace

cudaError_t launch_merge(const DecodeArgs& a, int64_t num_units, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_units);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, a);
}

}  // namespace kvq
