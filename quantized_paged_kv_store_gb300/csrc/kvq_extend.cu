// kvq_extend.cu -- extend (chunked-prefill) attention over the quantized cache
// on the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// "SGLang PR #21954 analysis: NVFP4 KV cache", Code analysis 1: the prefill /
// extend path reads the previously stored, quantized KV (there through a
// dequantized workspace; here dequantized in shared memory once per K/V chunk
// for all the queries that share it, as "Quantized KV Cache" (SGLang
// documentation), performance warning, asks of an attention kernel).
//
// Query token i of sequence q_seq[i] attends to that sequence's tokens
// [0, q_len[i]).  Rows are (query, q head) pairs laid out query-major; a CTA
// of four warps owns 128 consecutive rows of one kv head (16 queries at 8 q
// heads per kv head) -- one row per thread and per tensor-memory lane -- and
// one split of the context (gridDim.z splits; their partial outputs and
// log-sum-exps are merged by extend_merge_kernel).  Per 64-token chunk:
//   - two copy warps copy the raw K/V rows (and block scales) of the chunk
//     into a ring of raw stages several chunks ahead with cp.async,
//     completing on the stage's mbarrier, and refill a stage once the
//     dequant warps have read it;
//   - every dequant thread dequantizes half a token row of K and of V into f16 (FP8,
//     NVFP4) or bf16 (bf16, FP4 block-16) tiles in the 128-byte-swizzled
//     layout the tensor cores read (exact for every format: the per-tensor /
//     global scale stays out and is applied to the logits and the output);
//   - one elected thread of the MMA warp issues S = Q K^T (M = 128 rows, N = 64 tokens, K = 128 in
//     eight tcgen05.mma kind::f16 steps, fp32 accumulators in tensor memory;
//     A = Q from tensor memory, where each thread stored its row once, so the
//     tensor cores read only K from shared memory; Q in f16 is scaled per row
//     by a power of two that keeps it exact) and commits to an mbarrier;
//   - each thread loads its row of S from tensor memory, runs the online
//     softmax (base 2, lazy rescale when its maximum grows by more than 2^8,
//     causal mask by q_len) and stores P back to tensor memory in f16 (or, for
//     the bf16 operand formats, as a high and a low bf16 part: P = hi + lo to
//     ~2^-16);
//   - one thread issues O += P V (A = P from tensor memory, B = V in the
//     MN-major swizzled layout, two 64-column halves of head_dim).
// Rows of different sequences inside one CTA take one pass per distinct
// sequence (the other rows masked).  Every wait is bounded; a wait that runs
// out records KVQ_ERR_TIMEOUT and the CTA stops issuing work.
#include "kvq_codecs.cuh"
#include "kvq_decode_args.cuh"
#include "kvq_internal.h"

#include <algorithm>
#include <cmath>

namespace kvq {
namespace {

constexpr int kXRows = 128;        // (query, q head) rows per CTA = TMEM lanes
constexpr int kXThreads = 352;     // warps 0-3: rows; 4-7: dequant; 8: MMA issue; 9-10: copies
constexpr int kCopyBase = 288;     // first copy thread
constexpr int kMaxSlots = 4;       // K/V tiles and S slots in flight (per format below)
constexpr int kChunk = 64;         // tokens per chunk (four 16-token tiles)
constexpr int kMaxSplits = 16;
constexpr uint32_t kXWaitLimit = 1u << 22;

// tensor-memory columns: up to four S slots (64 fp32 columns each; P of a
// chunk is written back over its own S slot: f16 in 32 columns, or bf16 high
// and low parts in 64), O (128 fp32 columns, two halves of head_dim) and Q
// (64 columns of f16 / bf16 pairs, the A operand of Q K^T)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 64 * kMaxSlots;
constexpr uint32_t kColQ = kColO + 128;
constexpr uint32_t kTmemCols = 512;
static_assert(kColQ + 64 <= kTmemCols, "tensor-memory columns");

// shared memory (dynamic, 1024-byte aligned offsets)
constexpr int kSKV = 0;                             // slots of [K tile | V tile]
constexpr int kTileKV = 2 * kChunk * 128;           // one K (or V) tile: 2 atoms x 64 tokens x 128 B

template <kvq_format F>
struct XTraits {
  static constexpr int kRow = (F == KVQ_BF16) ? 256 : (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) ? 128 : 64;
  static constexpr bool kScales = (F == KVQ_FP4_BLOCK16 || F == KVQ_NVFP4);
  // f16 operands (FP8 and NVFP4 values are exact in f16; Q prescaled per row
  // by a power of two; P one f16 part); bf16 operands with P split into a
  // high and a low part for the bf16 and FP4 block-16 caches
  static constexpr bool kF16 = (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2 || F == KVQ_NVFP4);
  // raw stage: K rows of 64 tokens, V rows, K scale rows, V scale rows
  static constexpr int kData = kChunk * kRow;
  static constexpr int kScl = kScales ? kChunk * 8 : 0;
  static constexpr int kStage = 2 * kData + 2 * kScl;
  // K/V and S slots in flight: as many as shared memory holds; raw stages:
  // four (more copies in flight per thread made the copy issue slower)
  static constexpr int kSlots = (F == KVQ_BF16) ? 3 : 4;
  static constexpr int kRaw = (F == KVQ_BF16) ? 3 : 4;
  static constexpr int kSRaw = kSKV + kSlots * 2 * kTileKV;  // raw stages
  static constexpr int kSmem = kSRaw + kRaw * kStage + 1024;  // + alignment slack
};

struct ExtendArgs {
  const uint16_t* q;         // [n][Hq][128] bf16
  uint16_t* out;             // [n][Hq][128] bf16
  const int32_t* q_seq;      // [n]
  const int32_t* q_len;      // [n]
  const int32_t* page_table; // [S][max_pages]
  const uint8_t* kd;
  const uint8_t* vd;
  const uint8_t* ks;
  const uint8_t* vs;
  int n, S, max_pages, H, Hq, G, P;
  long long num_pages;
  float qscale;              // |sm_scale| * log2(e) * per-tensor K factor (without it if kfac)
  int neg_q;                 // sm_scale < 0: the query enters negated
  float v_factor;
  const float* kfac;         // per-kv-head K / V scales, or null
  const float* vfac;
  int* err;
  int splits;                // context splits (gridDim.z)
  float* part_o;             // splits > 1: [n * Hq][splits][128]
  float* part_lse;           // splits > 1: [n * Hq][splits] (log2 units)
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  uint32_t polls = 0;
  bool ok = mbar_try_wait(bar, parity);
  while (!ok && ++polls < kXWaitLimit) ok = mbar_try_wait(bar, parity);
  return ok;
}
// Asynchronous global -> shared copy of `bytes` (16 or 4) that reads
// `valid ? bytes : 0` bytes and zero-fills the rest.
__device__ __forceinline__ void cp_async16z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async4z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start
// address, leading byte offset (MN-major operands: the distance between the
// 64-element swizzle atoms along N; unused by K-major ones), stride byte
// offset (the distance between 8-row groups along K), descriptor version 1
// (bits 46-48), layout 2 = 128B swizzle.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t sbo, uint32_t lbo = 16) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16
// (bf = 1) or both f16 (bf = 0), A K-major, B K-major (b_mn = 0) or MN-major
// (1), N and M.
__host__ __device__ constexpr uint32_t idesc_16(uint32_t bf, uint32_t n, uint32_t m, uint32_t b_mn) {
  return (1u << 4) | (bf << 7) | (bf << 10) | (b_mn << 16) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// D (+)= A B with A in tensor memory, issued by one elected lane of a
// converged warp (every lane passes the same, warp-uniform operands: issuing
// from a lane-0 branch instead was 7% slower for the bf16-operand formats).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{ .reg .pred e, p; elect.sync _|e, 0xffffffff; setp.ne.u32 p, %4, 0;\n"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
               :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("{ .reg .pred e; elect.sync _|e, 0xffffffff;\n"
               "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }" ::"r"(bar) : "memory");
}

// 32 consecutive 32-bit tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
               "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                 "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
                 "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
                 "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
                 "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
                 "=r"(v[31])
               : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
               "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                  "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
                  "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
                  "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
                  "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]),
                  "r"(v[31]) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t hmul2x(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float ex2x(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Offset of 16-byte chunk c (0..7) of row `row` in a 128B-swizzled atom.
__device__ __forceinline__ uint32_t sw_off(int row, int c) { return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4)); }

// Raw stage layout of one K (or V) data region: 16-byte piece p of the half
// row (token tt, half hf) sits at natural index n = tt * kRow / 16 + hf * kRow
// / 32 + p, with the low three bits of n XORed by tt & 7 -- a permutation
// inside every 128-byte line, so that eight consecutive tokens (a quarter
// warp of dequant threads) read eight different bank groups.
template <kvq_format F>
__device__ __forceinline__ uint32_t raw_off(int tt, int hf, int p) {
  using Tr = XTraits<F>;
  const uint32_t n = (uint32_t)(tt * (Tr::kRow / 16) + hf * (Tr::kRow / 32) + p);
  return (n ^ (uint32_t)(tt & 7)) << 4;
}

// Dequantizes half a token row (64 head_dim elements, half hf) of K or V from
// the raw stage into 32 packed pairs -- f16x2 for the FP8 and NVFP4 caches,
// bf16x2 for the others -- exactly; the per-tensor / global scale is not
// applied (it multiplies the logits or the output).
template <kvq_format F>
__device__ __forceinline__ void dequant_half(const uint8_t* data, const uint8_t* scl, int tt, int hf,
                                             uint32_t (&o)[32]) {
  using Tr = XTraits<F>;
  auto piece = [&](int p) { return *reinterpret_cast<const uint4*>(data + raw_off<F>(tt, hf, p)); };
  if (F == KVQ_BF16) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = piece(c);
      o[4 * c] = v.x; o[4 * c + 1] = v.y; o[4 * c + 2] = v.z; o[4 * c + 3] = v.w;
    }
  } else if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 v = piece(c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // E4M3 and E5M2 values are exact in f16
        o[8 * c + 2 * i] = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2(w[i]) : dec2_e5m2_h2(w[i]);
        o[8 * c + 2 * i + 1] = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2_hi(w[i]) : dec2_e5m2_h2_hi(w[i]);
      }
    }
  } else {
    const uint4 v0 = piece(0), v1 = piece(1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(scl + tt * 8 + hf * 4);
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      const uint32_t sc = (sc4 >> (8 * blk)) & 0xFF;
      const uint32_t wa = w[2 * blk], wb = w[2 * blk + 1];
      uint32_t h[8] = {dec2_e2m1_h2<0>(wa), dec2_e2m1_h2<1>(wa), dec2_e2m1_h2<2>(wa), dec2_e2m1_h2<3>(wa),
                       dec2_e2m1_h2<0>(wb), dec2_e2m1_h2<1>(wb), dec2_e2m1_h2<2>(wb), dec2_e2m1_h2<3>(wb)};
      if (F == KVQ_NVFP4) {
        // E2M1 x E4M3 block scale: exact in f16 (at most 2688, at least 2^-10)
        const uint32_t s2 = dec2_e4m3_h2(sc | (sc << 8));
#pragma unroll
        for (int i = 0; i < 8; ++i) o[8 * blk + i] = hmul2x(h[i], s2);
      } else {
        // E2M1 x 2^(E - 127): exact in fp32 and in bf16
        const float m = exp2i((int)sc - 127);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[8 * blk + i] = bf2(h2_lo(h[i]) * m, h2_hi(h[i]) * m);
      }
    }
  }
}

// Eleven warps: at most three share one SM sub-partition's register file, so
// the launch bound holds each thread to 168 registers.
template <kvq_format F>
__global__ void __launch_bounds__(kXThreads, 1) extend_kernel(ExtendArgs a) {
  using Tr = XTraits<F>;
  extern __shared__ uint8_t xsm_raw[];
  // mbarriers: per raw stage (landed), per slot (K/V tiles ready, S ready,
  // P ready, PV done)
  constexpr int kMaxRaw = 6;
  constexpr int kSlots = Tr::kSlots;
  constexpr int kSRaw = Tr::kSRaw;
  __shared__ __align__(8) uint64_t bars[kMaxRaw + 4 * kMaxSlots + kMaxRaw];
  __shared__ uint32_t tmem_slot;
  __shared__ int row_seq[kXRows];
  __shared__ int row_len[kXRows];
  __shared__ int pass_seq, pass_max, pass_bad, dead;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool producer = warp >= 4;  // dequant warps 4-7, the MMA warp 8, copy warps 9-10
  const bool mma_warp = warp == 8;
  const bool copy_warp = warp >= 9;
  const int h = blockIdx.y, split = blockIdx.z;
  const long long R0 = (long long)blockIdx.x * kXRows;
  const uint32_t base_u32 = smem_u32(xsm_raw);
  uint8_t* sm = xsm_raw + (((base_u32 + 1023u) & ~1023u) - base_u32);
  const uint32_t sm_u32 = smem_u32(sm);
  static_assert(Tr::kRaw <= kMaxRaw, "raw stages");
  const uint32_t bar_raw = smem_u32(&bars[0]), bar_kv = smem_u32(&bars[kMaxRaw]);
  const uint32_t bar_s = smem_u32(&bars[kMaxRaw + kMaxSlots]), bar_p = smem_u32(&bars[kMaxRaw + 2 * kMaxSlots]);
  const uint32_t bar_o = smem_u32(&bars[kMaxRaw + 3 * kMaxSlots]);
  const uint32_t bar_rfree = smem_u32(&bars[kMaxRaw + 4 * kMaxSlots]);  // raw stage read by the dequant warps

  // ---- rows of this CTA (threads 0..127): (query, q head) = divmod(R0 + tid, G)
  const int rho = tid & (kXRows - 1);
  const long long R = R0 + rho;
  const long long qi = R / a.G;
  const bool qvalid = qi < a.n;
  const int qhead = h * a.G + (int)(R % a.G);
  float qmul = 1.f;
  uint4 qv[16];  // this thread's Q row (row warps), stored to tensor memory below
  if (!producer) {
    int s = -1, T = 0;
    if (qvalid) {
      s = __ldg(a.q_seq + qi);
      T = __ldg(a.q_len + qi);
      if (s < 0 || s >= a.S || T < 0 || T > a.max_pages * a.P) {
        if ((int)(R % a.G) == 0) atomicOr(a.err, kErrRange);
        s = -2;  // invalid: output zeros
      }
    }
    row_seq[rho] = s;
    row_len[rho] = T;
    // Q row as 64 pairs (d, d + 1); for the f16 operand formats the row is
    // scaled by 2^-sq so that its largest magnitude lies in [2^14, 2^15) and
    // every bf16 value of it is exact in f16 (2^sq joins the row's logit scale)
    const uint4* src = reinterpret_cast<const uint4*>(a.q + ((qvalid ? qi : 0) * a.Hq + qhead) * kHeadDim);
#pragma unroll
    for (int c = 0; c < 16; ++c) qv[c] = qvalid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    if (a.neg_q) {  // sm_scale < 0: negate the query (bf16 sign bits), scale by |sm_scale|
      const uint32_t f = 0x80008000u;
#pragma unroll
      for (int c = 0; c < 16; ++c) qv[c] = make_uint4(qv[c].x ^ f, qv[c].y ^ f, qv[c].z ^ f, qv[c].w ^ f);
    }
    if constexpr (Tr::kF16) {
      uint32_t m2 = 0u;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(qv[c].x));
        asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(qv[c].y));
        asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(qv[c].z));
        asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(qv[c].w));
      }
      const float amax = __uint_as_float(max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu) << 16);
      const int sq = (amax > 0.f && amax < INFINITY) ? max(-126, min(126, floor_log2(amax) - 14)) : 0;
      const float mul = exp2i(-sq);
      qmul = exp2i(sq);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
        uint32_t hv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t r;
          asm("cvt.rn.f16x2.f32 %0, %1, %2;"
              : "=r"(r) : "f"(bf16_bits_to_float(w[i] >> 16) * mul), "f"(bf16_bits_to_float(w[i] & 0xFFFF) * mul));
          hv[i] = r;
        }
        qv[c] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      }
    }
  }
  if (tid == 0) {
    // raw stage landed: one release arrival per copy warp (each copy thread
    // adds a pending arrival that its copies complete); K/V and P ready: one
    // per dequant / row warp; raw stage read: one per dequant warp
    for (int i = 0; i < kMaxRaw + 4 * kMaxSlots; ++i) {
      const int grp = i < kMaxRaw ? -1 : (i - kMaxRaw) / kMaxSlots;  // 0 K/V, 1 S, 2 P, 3 O
      mbar_init(smem_u32(&bars[i]), grp < 0 ? 2 : (grp == 0 || grp == 2) ? 4 : 1);
    }
    for (int i = 0; i < kMaxRaw; ++i) mbar_init(smem_u32(&bars[kMaxRaw + 4 * kMaxSlots + i]), 4);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    dead = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lane quarter
  // Q rows into tensor memory: lane = row, column 4c + i = pair i of qv[c]
  if (!producer) {
    uint32_t w0[32], w1[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      w0[4 * c] = qv[c].x; w0[4 * c + 1] = qv[c].y; w0[4 * c + 2] = qv[c].z; w0[4 * c + 3] = qv[c].w;
      w1[4 * c] = qv[8 + c].x; w1[4 * c + 1] = qv[8 + c].y; w1[4 * c + 2] = qv[8 + c].z; w1[4 * c + 3] = qv[8 + c].w;
    }
    tmem_st32(tmem + lane_off + kColQ, w0);
    tmem_st32(tmem + lane_off + kColQ + 32, w1);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const float cs = (a.kfac ? a.qscale * __ldg(a.kfac + h) : a.qscale) * qmul;
  const float vf = a.vfac ? __ldg(a.vfac + h) : a.v_factor;
  constexpr uint32_t kBf = Tr::kF16 ? 0u : 1u;
  constexpr uint32_t kIdQK = idesc_16(kBf, kChunk, kXRows, 0);
  constexpr uint32_t kIdPV = idesc_16(kBf, kHeadDim, kXRows, 1);  // N = all of head_dim

  // chunk counters over the CTA's life: chunk number k uses raw stage
  // k % kRaw and K/V and S slot k % kSlots, with mbarrier phase parity
  // (k / kRaw) & 1 and (k / kSlots) & 1
  uint32_t k_next = 0;  // first chunk number of the current pass
  bool row_done = false;

  // ---- one pass per distinct sequence among the CTA's rows -------------------
  for (;;) {
    if (tid == 0) {
      int s = -1;
      for (int r2 = 0; r2 < kXRows && s < 0; ++r2) s = row_seq[r2] >= 0 ? row_seq[r2] : -1;
      int mx = 0;
      for (int r2 = 0; r2 < kXRows; ++r2)
        if (row_seq[r2] == s && s >= 0) mx = max(mx, row_len[r2]);
      pass_seq = s;
      pass_max = mx;
      pass_bad = 0;
    }
    __syncthreads();
    const int s = pass_seq;
    if (s < 0 || dead) break;
    const int maxT = pass_max;
    const int32_t* prow = a.page_table + (long long)s * a.max_pages;
    const int nc = (maxT + kChunk - 1) / kChunk;
    const int c0 = (int)((long long)nc * split / a.splits), c1 = (int)((long long)nc * (split + 1) / a.splits);
    const uint32_t kbase = k_next;
    const int nch = c1 - c0;
    k_next += (uint32_t)max(nch, 0);

    if (mma_warp) {
      // ================= MMA warp: QK^T and PV issue ==========================
      const uint32_t tmem_u = __shfl_sync(0xffffffffu, tmem, 0);  // warp-uniform operand base
      // O += P V of chunk number kk once its P is ready (acc == 0 starts the pass)
      auto issue_pv = [&](uint32_t kk, bool start) -> bool {
        const uint32_t slot = kk % kSlots;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_p + 8 * slot, (kk / kSlots) & 1u));
        if (!ok) return false;
        tc_fence_after();
        {
          const uint32_t pcol = tmem_u + kColS + 64 * slot;
          const uint32_t vbase = sm_u32 + kSKV + slot * 2 * kTileKV + kTileKV;
          // one MMA per 16 tokens covers both 64-element halves of head_dim
          // (B atoms kChunk * 128 bytes apart along N)
#pragma unroll
          for (int j = 0; j < kChunk / 16; ++j) {
            const uint64_t bd = sw128_desc(vbase + j * 2048, 1024, kChunk * 128);
            mma_ts(tmem_u + kColO, pcol + 8 * j, bd, kIdPV, (start && j == 0) ? 0u : 1u);
            if (!Tr::kF16) mma_ts(tmem_u + kColO, pcol + 32 + 8 * j, bd, kIdPV, 1u);
          }
          mma_commit(bar_o + 8 * slot);
        }
        __syncwarp();
        return true;
      };

      for (int c = c0; c < c1; ++c) {
        const uint32_t kk = kbase + (uint32_t)(c - c0), slot = kk % kSlots;
        // K/V tiles of chunk kk dequantized
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_kv + 8 * slot, (kk / kSlots) & 1u))) {
          if (lane == 0) dead = 1;
          break;
        }
        tc_fence_after();
        {
          // S = Q K^T into S slot `slot`
          const uint32_t kb = sm_u32 + kSKV + slot * 2 * kTileKV;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint64_t bd = sw128_desc(kb + (j >> 2) * (kChunk * 128) + (j & 3) * 32, 1024);
            mma_ts(tmem_u + kColS + 64 * slot, tmem_u + kColQ + 8 * j, bd, kIdQK, j > 0);
          }
          mma_commit(bar_s + 8 * slot);
        }
        __syncwarp();
        // then O += P V of the previous chunk, once its P is ready
        if (c > c0 && !issue_pv(kk - 1, c - 1 == c0)) {
          if (lane == 0) dead = 1;
          break;
        }
      }
      if (nch > 0 && !dead && !issue_pv(kbase + (uint32_t)(nch - 1), nch == 1) && lane == 0) dead = 1;
    } else if (copy_warp) {
      // ======== copy warps: raw K/V rows and block scales of each chunk ========
      // Copy thread ct issues the copies of slices (token tt, half hf) number
      // ct and ct + 64 in the dequant threads' numbering, into the same
      // conflict-free raw layout; a stage is refilled once the four dequant
      // warps have read it.  Absent tokens and bad pages zero-fill.
      const int ct = tid - kCopyBase;
      int ttj[2], hfj[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int p2 = ct + 64 * j;
        ttj[j] = ((p2 >> 5) << 4) | (p2 & 15);
        hfj[j] = (p2 >> 4) & 1;
      }
      auto page_of = [&](int c, int j) -> int {
        const int tok = c * kChunk + ttj[j];
        return (c < c1 && tok < maxT) ? __ldg(prow + tok / a.P) : -1;
      };
      int pg[2] = {page_of(c0, 0), page_of(c0, 1)};
      for (int c = c0; c < c1; ++c) {
        const uint32_t kk = kbase + (uint32_t)(c - c0), st = kk % Tr::kRaw;
        bool ok = true;
        if (kk >= (uint32_t)Tr::kRaw) ok = mbar_wait_bounded(bar_rfree + 8 * st, ((kk - Tr::kRaw) / Tr::kRaw) & 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) dead = 1;
          break;
        }
        const uint32_t stage = sm_u32 + kSRaw + st * Tr::kStage;
        const int npg[2] = {page_of(c + 1, 0), page_of(c + 1, 1)};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tt = ttj[j], hf = hfj[j], page = pg[j];
          const int tok = c * kChunk + tt;
          const bool in_seq = tok < maxT;
          const bool pok = in_seq && page >= 0 && page < a.num_pages;
          if (in_seq && !pok) pass_bad = 1;
          const long long rowi = pok ? ((long long)page * a.H + h) * a.P + tok % a.P : 0;
          constexpr int kHalf = Tr::kRow / 2;
          const uint8_t* sk = a.kd + rowi * Tr::kRow + hf * kHalf;
          const uint8_t* sv = a.vd + rowi * Tr::kRow + hf * kHalf;
#pragma unroll
          for (int i = 0; i < kHalf / 16; ++i) {
            const uint32_t dk = stage + raw_off<F>(tt, hf, i);
            cp_async16z(dk, sk + 16 * i, pok);
            cp_async16z(dk + Tr::kData, sv + 16 * i, pok);
          }
          if constexpr (Tr::kScales) {
            const uint32_t ds = stage + 2 * Tr::kData + tt * 8 + hf * 4;
            cp_async4z(ds, a.ks + rowi * 8 + hf * 4, pok);
            cp_async4z(ds + Tr::kScl, a.vs + rowi * 8 + hf * 4, pok);
          }
        }
        // one pending arrival per thread, completed when its copies land; then
        // one release arrival per copy warp (orders pass_bad before the stage)
        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar_raw + 8 * st) : "memory");
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_raw + 8 * st) : "memory");
        pg[0] = npg[0];
        pg[1] = npg[1];
      }
    } else if (producer) {
      // ======== dequant warps: raw stage -> swizzled K/V tiles ========
      // Thread (token tt of the chunk, head_dim half hf) dequantizes its slice
      // of K and V; a warp holds 16 consecutive tokens x both halves (lanes
      // 0-15 half 0), so a quarter warp writes eight tokens' rows of one
      // swizzled tile: no bank conflicts.
      const int ptid = tid - 128, tt = ((ptid >> 5) << 4) | (ptid & 15), hf = (ptid >> 4) & 1;
      for (int c = c0; c < c1; ++c) {
        const uint32_t kk = kbase + (uint32_t)(c - c0), slot = kk % kSlots;
        const uint32_t rst = kk % Tr::kRaw;
        // raw chunk landed; K/V slot and S slot free (PV of chunk kk - kSlots done)
        bool ok = mbar_wait_bounded(bar_raw + 8 * rst, (kk / Tr::kRaw) & 1u);
        if (ok && c - c0 >= kSlots) ok = mbar_wait_bounded(bar_o + 8 * slot, ((kk - kSlots) / kSlots) & 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) dead = 1;
          break;
        }
        tc_fence_after();
        {
          const uint8_t* stage = sm + kSRaw + rst * Tr::kStage;
          const bool tok_ok = c * kChunk + tt < maxT;
          uint32_t kw[32], vw[32];
          if (tok_ok) {
            dequant_half<F>(stage, stage + 2 * Tr::kData, tt, hf, kw);
            dequant_half<F>(stage + Tr::kData, stage + 2 * Tr::kData + Tr::kScl, tt, hf, vw);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) kw[i] = vw[i] = 0u;
          }
          uint8_t* kv = sm + kSKV + slot * 2 * kTileKV;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const uint32_t off = hf * (kChunk * 128) + sw_off(tt, cc);
            *reinterpret_cast<uint4*>(kv + off) = make_uint4(kw[4 * cc], kw[4 * cc + 1], kw[4 * cc + 2], kw[4 * cc + 3]);
            *reinterpret_cast<uint4*>(kv + kTileKV + off) =
                make_uint4(vw[4 * cc], vw[4 * cc + 1], vw[4 * cc + 2], vw[4 * cc + 3]);
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_kv + 8 * slot) : "memory");
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_rfree + 8 * rst) : "memory");
        }
      }
    } else {
      // ================= rows: online softmax, O rescale, epilogue =============
      const bool act = row_seq[rho] == s;
      const int Tr_ = row_len[rho];
      float m = -INFINITY, l = 0.f;
      for (int c = c0; c < c1; ++c) {
        const uint32_t kk = kbase + (uint32_t)(c - c0), slot = kk % kSlots;
        const bool sok = mbar_wait_bounded(bar_s + 8 * slot, (kk / kSlots) & 1u);
        tc_fence_after();
        if (!__all_sync(0xffffffffu, sok)) {
          if (lane == 0) dead = 1;
          break;
        }
        const uint32_t scol = tmem + lane_off + kColS + 64 * slot;
        uint32_t sv[64];
        {
          uint32_t t0[32], t1[32];
          tmem_ld32(scol, t0);
          tmem_ld32(scol + 32, t1);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            sv[j] = t0[j];
            sv[32 + j] = t1[j];
          }
        }
        float mx = -INFINITY;
        if (act && (c + 1) * kChunk <= Tr_) {  // every token of the chunk is in this row's prefix
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float x = __uint_as_float(sv[j]) * cs;
            sv[j] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int tok = c * kChunk + j;
            const float x = (act && tok < Tr_) ? __uint_as_float(sv[j]) * cs : -INFINITY;
            sv[j] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
        }
        const bool grow = mx > m + 8.f;
        const float m_new = grow ? mx : m;
        if (__any_sync(0xffffffffu, grow && m != -INFINITY && c > c0)) {
          // rescale what O holds: the PV of the previous chunk must be done
          const uint32_t kp = kk - 1;
          const bool pok = mbar_wait_bounded(bar_o + 8 * (kp % kSlots), (kp / kSlots) & 1u);
          tc_fence_after();
          if (!__all_sync(0xffffffffu, pok)) {
            if (lane == 0) dead = 1;
            break;
          }
          const float al = (grow && m != -INFINITY) ? ex2x(m - m_new) : 1.f;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_off + kColO + 32 * q4, ov);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * al);
            tmem_st32(tmem + lane_off + kColO + 32 * q4, ov);
          }
          l *= al;
        } else if (grow && m != -INFINITY) {
          l *= ex2x(m - m_new);
        }
        m = m_new;
        // P over this chunk's S slot
        if constexpr (Tr::kF16) {
          uint32_t ph[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x0 = __uint_as_float(sv[2 * j]), x1 = __uint_as_float(sv[2 * j + 1]);
            const float p0 = (x0 == -INFINITY) ? 0.f : ex2x(x0 - m);
            const float p1 = (x1 == -INFINITY) ? 0.f : ex2x(x1 - m);
            l += p0 + p1;
            uint32_t r;
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(p1), "f"(p0));
            ph[j] = r;
          }
          tmem_st32(scol, ph);
        } else {
          uint32_t ph[32], pl[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x0 = __uint_as_float(sv[2 * j]), x1 = __uint_as_float(sv[2 * j + 1]);
            const float p0 = (x0 == -INFINITY) ? 0.f : ex2x(x0 - m);
            const float p1 = (x1 == -INFINITY) ? 0.f : ex2x(x1 - m);
            l += p0 + p1;
            ph[j] = bf2(p0, p1);
            const float r0 = p0 - bf16_bits_to_float(ph[j] & 0xFFFFu);
            const float r1 = p1 - bf16_bits_to_float(ph[j] >> 16);
            pl[j] = bf2(r0, r1);
          }
          tmem_st32(scol, ph);
          tmem_st32(scol + 32, pl);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_p + 8 * slot) : "memory");
      }
      // ---- O of this pass complete (last PV done); partial or final output ----
      bool has_o = false;
      if (nch > 0 && !dead) {
        const uint32_t kl = kbase + (uint32_t)(nch - 1);
        const bool ook = mbar_wait_bounded(bar_o + 8 * (kl % kSlots), (kl / kSlots) & 1u);
        tc_fence_after();
        if (__all_sync(0xffffffffu, ook)) has_o = true;
        else if (lane == 0) dead = 1;
      }
      has_o = __all_sync(0xffffffffu, has_o);
      const bool poison = pass_bad != 0 || dead != 0;
      const bool has = has_o && l > 0.f;
      const float inv = (has && !poison) ? vf / l : 0.f;
      const long long rowg = qi * a.Hq + qhead;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t ov[32];
        if (has_o) {  // warp-uniform
          tmem_ld32(tmem + lane_off + kColO + 32 * q4, ov);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0u;
        }
        if (act && qvalid) {
          if (a.splits == 1) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + rowg * kHeadDim + 32 * q4);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              dst[j] = bf16_rne_bits(__uint_as_float(ov[2 * j]) * inv) |
                       (bf16_rne_bits(__uint_as_float(ov[2 * j + 1]) * inv) << 16);
          } else {
            float4* dst = reinterpret_cast<float4*>(a.part_o + (rowg * a.splits + split) * kHeadDim + 32 * q4);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(ov[4 * j]) * inv, __uint_as_float(ov[4 * j + 1]) * inv,
                                   __uint_as_float(ov[4 * j + 2]) * inv, __uint_as_float(ov[4 * j + 3]) * inv);
          }
        }
      }
      if (act && qvalid && a.splits > 1)
        a.part_lse[rowg * a.splits + split] = poison ? INFINITY : (has ? m + __log2f(l) : -INFINITY);
      if (act) row_done = true;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      if (pass_bad) atomicOr(a.err, kErrRange);
      for (int r2 = 0; r2 < kXRows; ++r2)
        if (row_seq[r2] == s) row_seq[r2] = -1;
    }
    __syncthreads();
  }
  if (tid == 0 && dead) atomicOr(a.err, kErrTimeout);
  // rows that never ran (invalid, or left after a wait ran out): zero output
  if (!producer && qvalid && !row_done) {
    const long long rowg = qi * a.Hq + qhead;
    if (a.splits == 1) {
      uint4* dst = reinterpret_cast<uint4*>(a.out + rowg * kHeadDim);
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[j] = make_uint4(0u, 0u, 0u, 0u);
    } else {
      a.part_lse[rowg * a.splits + split] = dead ? INFINITY : -INFINITY;
    }
  }
  // after a wait ran out: give MMAs still in flight a bounded chance to
  // complete before the CTA frees its tensor memory and exits; every copy
  // thread waits for its own copies
  if (dead && mma_warp) {
    const uint32_t k0 = k_next > kSlots ? k_next - kSlots : 0;
    for (uint32_t t = k0; t < k_next; ++t) {
      mbar_wait_bounded(bar_s + 8 * (t % kSlots), (t / kSlots) & 1u);
      mbar_wait_bounded(bar_o + 8 * (t % kSlots), (t / kSlots) & 1u);
    }
  }
  if (copy_warp) asm volatile("cp.async.wait_all;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
}

// out[row] = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M) over the splits;
// +inf (poisoned) gives zeros, all -inf (no tokens) gives zeros.  One warp per
// row, lanes own four head_dim elements.
__global__ void __launch_bounds__(256) extend_merge_kernel(ExtendArgs a, long long rows) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float lse = lane < a.splits ? a.part_lse[row * a.splits + lane] : -INFINITY;
  float M = lse;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  uint2 ov = make_uint2(0u, 0u);
  if (M != INFINITY && M != -INFINITY) {
    const float w = (lse == -INFINITY) ? 0.f : ex2x(lse - M);
    float den = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.splits; ++s) {
      const float ws = __shfl_sync(0xffffffffu, w, s);
      if (ws == 0.f) continue;
      const float4 v = *reinterpret_cast<const float4*>(a.part_o + (row * a.splits + s) * kHeadDim + lane * 4);
      acc.x += ws * v.x;
      acc.y += ws * v.y;
      acc.z += ws * v.z;
      acc.w += ws * v.w;
    }
    const float inv = 1.f / den;
    ov.x = bf16_rne_bits(acc.x * inv) | (bf16_rne_bits(acc.y * inv) << 16);
    ov.y = bf16_rne_bits(acc.z * inv) | (bf16_rne_bits(acc.w * inv) << 16);
  }
  *reinterpret_cast<uint2*>(a.out + row * kHeadDim + lane * 4) = ov;
}

template <kvq_format F>
cudaError_t launch_extend_as(const ExtendArgs& a, cudaStream_t stream) {
  static_assert(XTraits<F>::kSmem <= 227 * 1024, "extend tiles exceed shared memory");
  cudaError_t e = cudaFuncSetAttribute(extend_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       XTraits<F>::kSmem);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)a.n * a.G;
  dim3 grid((unsigned)((rows + kXRows - 1) / kXRows), (unsigned)a.H, (unsigned)a.splits);
  extend_kernel<F><<<grid, kXThreads, XTraits<F>::kSmem, stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.splits > 1) {
    const long long orows = (long long)a.n * a.Hq;
    extend_merge_kernel<<<(unsigned)((orows + 7) / 8), 256, 0, stream>>>(a, orows);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

int extend_splits(const Geometry& g, int num_q_tokens, int num_q_heads, int max_pages_per_seq,
                  int device) {
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  const int G = num_q_heads / g.kv_heads;
  const long long ctas = (((long long)num_q_tokens * G + kXRows - 1) / kXRows) * g.kv_heads;
  const long long chunks = ((long long)max_pages_per_seq * g.page_size + kChunk - 1) / kChunk;
  if (ctas <= 0) return 1;
  // one CTA per SM: at least two waves, at least 16 chunks per split, and the
  // split count whose last wave is fullest (waves / ceil(waves) >= 0.9)
  const long long s_max = std::max<long long>(1, std::min<long long>(kMaxSplits, chunks / 16));
  const long long s_min = std::min<long long>(s_max, std::max<long long>(1, (2LL * sms + ctas - 1) / ctas));
  long long best = s_min;
  double best_eff = 0.0;
  for (long long s = s_min; s <= s_max; ++s) {
    const double waves = (double)(ctas * s) / sms;
    const double eff = waves / std::ceil(waves);
    if (eff >= 0.9) return (int)s;
    if (eff > best_eff) { best_eff = eff; best = s; }
  }
  return (int)best;
}

size_t extend_workspace_bytes(int splits, int num_q_tokens, int num_q_heads) {
  if (splits <= 1) return 0;
  const size_t rows = (size_t)num_q_tokens * num_q_heads;
  return ((rows * splits * kHeadDim * sizeof(float) + 255) & ~(size_t)255) +
         ((rows * splits * sizeof(float) + 255) & ~(size_t)255);
}

cudaError_t launch_extend(const Geometry& g, const LayerView& L, const void* q, int num_q_heads,
                          int num_q_tokens, const int32_t* q_seq, const int32_t* q_len,
                          const int32_t* page_table, int num_seqs, int max_pages_per_seq,
                          float sm_scale, float k_factor, float v_factor, const HeadScales& hs,
                          void* out, int* err, int splits, void* workspace, cudaStream_t stream) {
  ExtendArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.q_seq = q_seq;
  a.q_len = q_len;
  a.page_table = page_table;
  a.kd = L.k_data;
  a.vd = L.v_data;
  a.ks = L.k_scales;
  a.vs = L.v_scales;
  a.n = num_q_tokens;
  a.S = num_seqs;
  a.max_pages = max_pages_per_seq;
  a.H = g.kv_heads;
  a.Hq = num_q_heads;
  a.G = num_q_heads / g.kv_heads;
  a.P = g.page_size;
  a.num_pages = g.num_pages;
  a.kfac = hs.scale[0];
  a.vfac = hs.scale[1];
  // the softmax runs on positive logit scales: a negative sm_scale is folded
  // into the query's sign (exact)
  a.neg_q = sm_scale < 0.f;
  a.qscale = std::fabs(sm_scale) * 1.4426950408889634f * (a.kfac ? 1.0f : k_factor);
  a.v_factor = v_factor;
  a.err = err;
  a.splits = std::max(1, splits);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t rows = (size_t)num_q_tokens * num_q_heads;
  a.part_o = reinterpret_cast<float*>(ws);
  a.part_lse = ws ? reinterpret_cast<float*>(ws + ((rows * a.splits * kHeadDim * sizeof(float) + 255) &
                                                   ~(size_t)255))
                  : nullptr;
  if (num_q_tokens == 0) return cudaSuccess;
  switch (g.fmt) {
    case KVQ_BF16: return launch_extend_as<KVQ_BF16>(a, stream);
    case KVQ_FP8_E4M3: return launch_extend_as<KVQ_FP8_E4M3>(a, stream);
    case KVQ_FP8_E5M2: return launch_extend_as<KVQ_FP8_E5M2>(a, stream);
    case KVQ_FP4_BLOCK16: return launch_extend_as<KVQ_FP4_BLOCK16>(a, stream);
    case KVQ_NVFP4: return launch_extend_as<KVQ_NVFP4>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
