// kvq_merge.cu -- log-sum-exp merge of the split-K decode partials.
//
// A unit (sequence, kv head, group of <= 8 q heads) is split over the warp
// workers that touched its tiles; each wrote a normalized partial output o_s
// and its log-sum-exp lse_s (log2 units).  The merge combines them:
//   out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s,
// rounded to bf16.  A partial with lse = +inf marks a unit that saw an invalid
// page id (or a wait that ran out): its output is zero.
#include "kvq_codecs.cuh"
#include "kvq_decode_args.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kMergeMaxWarps = 32;

// One CTA per (unit, q head of the unit's group); its warps split the unit's
// partials (warp i takes partials i, i + nwarps, ...), each lane owning four
// head_dim elements, in one pass (every load of a batch in flight together),
// and combine in shared memory.  The warp count is chosen on the host from the
// average number of partials per unit, so a unit split over hundreds of
// workers (small batches) is merged by up to 32 warps.
__global__ void __launch_bounds__(kMergeMaxWarps * 32) merge_kernel(DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // dynamic: nwarps x (32 float4 + den + max), so small CTAs stay small
  extern __shared__ float4 s_dyn[];
  const int nw_cta = blockDim.x >> 5;
  float4(*s_acc)[32] = reinterpret_cast<float4(*)[32]>(s_dyn);
  float* s_den = reinterpret_cast<float*>(s_dyn + 32 * nw_cta);
  float* s_max = s_den + nw_cta;
  const long long u = blockIdx.x / kGroupMax;
  const int g = (int)(blockIdx.x - u * kGroupMax);
  const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5, nwarps = blockDim.x >> 5;
  const long long upb = (long long)a.H * a.HG;
  const int b = (int)(u / upb), ub = (int)(u - (long long)b * upb);
  const int h = ub / a.HG, hg = ub - (ub / a.HG) * a.HG;
  if (g >= min(kGroupMax, a.G - hg * kGroupMax)) return;  // CTA-uniform
  uint16_t* orow = a.out + ((long long)b * a.Hq + h * a.G + hg * kGroupMax + g) * kHeadDim + lane * 4;
  const int nt = tiles_of(a, b);
  if (nt == 0) {
    if (wi == 0) *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
    return;
  }
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

  // ---- one pass: warp wi takes partials wf + wi + k * nwarps, loading each
  // lse with its output slice, and keeps (max, weighted sum, weight) relative
  // to its own running maximum; +inf marks a poisoned partial ----
  const float* base = a.part_o + (u * kGroupMax + g) * kHeadDim + lane * 4;
  const long long pstride = (long long)kGroupMax * kHeadDim;  // floats between slots
  float m = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool poison = false;
  for (int w = wf + wi; w <= wl; w += 4 * nwarps) {
    float l[4];
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int wi2 = w + i * nwarps;
      const bool e = wi2 <= wl && nonempty(wi2);
      l[i] = e ? a.part_lse[(u + wi2) * kGroupMax + g] : -INFINITY;
      v[i] = e ? *reinterpret_cast<const float4*>(base + (long long)wi2 * pstride)
               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mb = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
    poison |= (mb == INFINITY);
    if (mb > m) {  // rescale what this warp has so far
      const float f = (m == -INFINITY) ? 0.f : ex2(m - mb);
      den *= f;
      acc.x *= f;
      acc.y *= f;
      acc.z *= f;
      acc.w *= f;
      m = mb;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float t = (l[i] == -INFINITY || m == INFINITY) ? 0.f : ex2(l[i] - m);
      den += t;
      acc.x += t * v[i].x;
      acc.y += t * v[i].y;
      acc.z += t * v[i].z;
      acc.w += t * v[i].w;
    }
  }
  if (nwarps > 1) {
    s_acc[wi][lane] = acc;
    if (lane == 0) {
      s_den[wi] = den;
      s_max[wi] = poison ? INFINITY : m;
    }
    __syncthreads();
    if (wi != 0) return;
    float M = -INFINITY;
    for (int i = 0; i < nwarps; ++i) M = fmaxf(M, s_max[i]);
    poison = (M == INFINITY);
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    den = 0.f;
    for (int i = 0; i < nwarps; ++i) {
      const float mi = s_max[i];
      const float f = (mi == -INFINITY || poison) ? 0.f : ex2(mi - M);
      const float4 x = s_acc[i][lane];
      den += f * s_den[i];
      acc.x += f * x.x;
      acc.y += f * x.y;
      acc.z += f * x.z;
      acc.w += f * x.w;
    }
  }
  if (poison) {
    *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
    return;
  }
  const float inv = 1.f / den;
  uint2 ov;
  ov.x = bf16_rne_bits(acc.x * inv) | (bf16_rne_bits(acc.y * inv) << 16);
  ov.y = bf16_rne_bits(acc.z * inv) | (bf16_rne_bits(acc.w * inv) << 16);
  *reinterpret_cast<uint2*>(orow) = ov;
}

}  // namespace

cudaError_t launch_merge(const DecodeArgs& a, int64_t num_units, cudaStream_t stream) {
  // about eight partials per warp on average (two batches of loads), 1 to 32
  // warps per CTA; measured at batch 32 x 32K (about 11 partials per unit):
  // two warps per CTA 0.8% faster per decode call than four, eight 1.6% slower
  const int64_t per_unit = (a.num_workers + num_units - 1) / num_units + 1;
  int warps = 1;
  while (warps < kMergeMaxWarps && warps * 8 < per_unit) warps <<= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_units * kGroupMax));
  cfg.blockDim = dim3(32 * warps);
  cfg.dynamicSmemBytes = warps > 1 ? (size_t)warps * (32 * sizeof(float4) + 2 * sizeof(float)) : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, a);
}

}  // namespace kvq
