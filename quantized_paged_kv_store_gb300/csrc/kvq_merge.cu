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
// head_dim elements, and reduce in shared memory.  The warp count is chosen on
// the host from the average number of partials per unit, so a unit split over
// hundreds of workers (small batches) is merged by up to 32 warps.
__global__ void __launch_bounds__(kMergeMaxWarps * 32) merge_kernel(DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float4 s_acc[kMergeMaxWarps][32];
  __shared__ float s_den[kMergeMaxWarps];
  __shared__ float s_max[kMergeMaxWarps];
  __shared__ int s_poison;
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

  // ---- M = max lse over the unit's partials; +inf marks a poisoned partial ----
  float M = -INFINITY;
  bool poison = false;
  for (int w = wf + tid; w <= wl; w += blockDim.x) {
    if (!nonempty(w)) continue;
    const float lse = a.part_lse[(u + w) * kGroupMax + g];
    poison |= (lse == INFINITY);
    M = fmaxf(M, lse);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  poison = __any_sync(0xffffffffu, poison);
  if (tid == 0) s_poison = 0;
  __syncthreads();
  if (lane == 0) {
    s_max[wi] = M;
    if (poison) s_poison = 1;
  }
  __syncthreads();
  for (int i = 0; i < nwarps; ++i) M = fmaxf(M, s_max[i]);
  if (s_poison) {
    if (wi == 0) *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
    return;
  }

  // ---- this warp's share: sum_w 2^(lse_w - M) o_w and the weights ----
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  const float* base = a.part_o + (u * kGroupMax + g) * kHeadDim + lane * 4;
  const long long pstride = (long long)kGroupMax * kHeadDim;  // floats between slots
  int w = wf + wi;
  // two partials per step: both loads in flight together
  for (; w + nwarps <= wl; w += 2 * nwarps) {
    const int w2 = w + nwarps;
    const bool e1 = nonempty(w), e2 = nonempty(w2);
    const float l1 = e1 ? a.part_lse[(u + w) * kGroupMax + g] : -INFINITY;
    const float l2 = e2 ? a.part_lse[(u + w2) * kGroupMax + g] : -INFINITY;
    const float4 v1 = e1 ? *reinterpret_cast<const float4*>(base + (long long)w * pstride)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 v2 = e2 ? *reinterpret_cast<const float4*>(base + (long long)w2 * pstride)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    const float t1 = e1 ? ex2(l1 - M) : 0.f, t2 = e2 ? ex2(l2 - M) : 0.f;
    den += t1 + t2;
    acc.x += t1 * v1.x + t2 * v2.x;
    acc.y += t1 * v1.y + t2 * v2.y;
    acc.z += t1 * v1.z + t2 * v2.z;
    acc.w += t1 * v1.w + t2 * v2.w;
  }
  if (w <= wl && nonempty(w)) {
    const float t1 = ex2(a.part_lse[(u + w) * kGroupMax + g] - M);
    const float4 v1 = *reinterpret_cast<const float4*>(base + (long long)w * pstride);
    den += t1;
    acc.x += t1 * v1.x;
    acc.y += t1 * v1.y;
    acc.z += t1 * v1.z;
    acc.w += t1 * v1.w;
  }
  if (nwarps > 1) {
    s_acc[wi][lane] = acc;
    if (lane == 0) s_den[wi] = den;
    __syncthreads();
    if (wi != 0) return;
    for (int i = 1; i < nwarps; ++i) {
      const float4 v = s_acc[i][lane];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
      den += s_den[i];
    }
  }
  const float inv = 1.f / den;
  uint2 ov;
  ov.x = bf16_rne_bits(acc.x * inv) | (bf16_rne_bits(acc.y * inv) << 16);
  ov.y = bf16_rne_bits(acc.z * inv) | (bf16_rne_bits(acc.w * inv) << 16);
  *reinterpret_cast<uint2*>(orow) = ov;
}

}  // namespace

cudaError_t launch_merge(const DecodeArgs& a, int64_t num_units, cudaStream_t stream) {
  // about four partials per warp on average, 1 to 32 warps per CTA
  const int64_t per_unit = (a.num_workers + num_units - 1) / num_units + 1;
  int warps = 1;
  while (warps < kMergeMaxWarps && warps * 4 < per_unit) warps <<= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_units * kGroupMax));
  cfg.blockDim = dim3(32 * warps);
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
