// kvq_extend.cu -- extend (chunked-prefill) attention over the quantized cache.
//
// "SGLang PR #21954 analysis: NVFP4 KV cache", Code analysis 1: the prefill /
// extend path reads the previously stored, quantized KV (there through a
// dequantized workspace; here dequantized in place, once per K/V tile for all
// the queries that share it, as "Quantized KV Cache" (SGLang documentation),
// performance warning, asks of an attention kernel).
//
// Query token i of sequence q_seq[i] attends to that sequence's tokens
// [0, q_len[i]).  Rows are (query, q head) pairs laid out query-major; a CTA of
// four warps owns 64 consecutive rows of one kv head (8 queries at G = 8) and
// walks the K/V tiles of their sequence once:
//   - the raw rows of each 16-token tile are copied into shared memory with
//     cp.async, four tiles in flight (absent tokens and bad pages zero-filled);
//   - every thread dequantizes one 16-element block of K and one of V per tile
//     into a shared f16 tile (FP8 / NVFP4, exact) or bf16 tile (bf16 / FP4
//     block-16, exact: E2M1 x 2^(E-127) fits bf16's range);
//   - each warp computes S = Q K^T for its 16 rows with mma.sync.m16n8k16
//     (K fragments by ldmatrix), an online softmax per row (base 2, lazy
//     rescale when a row's maximum grows by more than 2^8), and O += P V
//     (P reused from the S accumulators, V fragments by ldmatrix.trans; for the
//     bf16 instances P is split into high and low bf16 parts).
// Rows of different sequences inside one CTA take one pass per distinct
// sequence (the other rows masked).  No split-K: the output is written once.
#include "kvq_codecs.cuh"
#include "kvq_decode_args.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kXWarps = 4;
constexpr int kXThreads = 32 * kXWarps;
constexpr int kXRows = 16 * kXWarps;           // (query, q head) rows per CTA
constexpr int kXStride = kHeadDim * 2 + 16;    // bytes per shared row (pad: conflict-free ldmatrix)
constexpr int kXTile = kTile * kXStride;       // one dequantized K (or V) tile
static_assert(kXThreads == kTile * (kHeadDim / 16), "one 16-element block per thread per tile");

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
  float qscale;              // sm_scale * log2(e) * per-tensor K factor (without it if kfac)
  float v_factor;
  const float* kfac;         // per-kv-head K / V scales, or null
  const float* vfac;
  int* err;
};

template <kvq_format F>
struct XTraits {
  static constexpr bool kBf16 = (F == KVQ_BF16 || F == KVQ_FP4_BLOCK16);  // bf16 mma
  static constexpr int kRow = (F == KVQ_BF16) ? 256 : (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) ? 128 : 64;
  static constexpr int kBlk = kRow / 8;  // bytes of one 16-element block
  static constexpr bool kScales = (F == KVQ_FP4_BLOCK16 || F == KVQ_NVFP4);
  // raw bytes of one tile as copied: K rows, V rows, K scale rows, V scale rows
  static constexpr int kStageBytes = 2 * kTile * kRow + 2 * kTile * 8;
  static constexpr int kCopies = 2 * kRow + (kScales ? 2 * kTile : 0);  // 16 B data + 8 B scale copies
};
constexpr int kXStages = 4;  // raw tiles in flight per CTA

// Raw bytes of one 16-element block (K or V) held between load and dequant.
struct RawBlock {
  uint4 a, b;   // data (bf16: 32 B; fp8: a = 16 B; fp4: a.x, a.y = 8 B)
  uint32_t sc;  // block scale byte (FP4 formats)
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if (BF16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
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

// Asynchronous global -> shared copies (cp.async); a copy of `valid` false
// reads nothing and fills the destination with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 8 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The raw block (tile token tok, block blk) of K (kv = 0) or V from a raw stage.
template <kvq_format F>
__device__ __forceinline__ RawBlock raw_block(const uint8_t* stage, int kv, int tok, int blk) {
  using Tr = XTraits<F>;
  RawBlock rb;
  const uint8_t* p = stage + kv * kTile * Tr::kRow + tok * Tr::kRow + blk * Tr::kBlk;
  if (F == KVQ_BF16) {
    rb.a = reinterpret_cast<const uint4*>(p)[0];
    rb.b = reinterpret_cast<const uint4*>(p)[1];
  } else if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
    rb.a = reinterpret_cast<const uint4*>(p)[0];
  } else {
    const uint2 v = reinterpret_cast<const uint2*>(p)[0];
    rb.a.x = v.x;
    rb.a.y = v.y;
    rb.sc = stage[2 * kTile * Tr::kRow + kv * kTile * 8 + tok * 8 + blk];
  }
  return rb;
}

// Dequantizes one block into 8 packed pairs (f16x2, or bf16x2 for the bf16
// instances); exact for every format.
template <kvq_format F>
__device__ __forceinline__ void dequant_block(const RawBlock& rb, uint32_t (&o)[8]) {
  if (F == KVQ_BF16) {
    o[0] = rb.a.x; o[1] = rb.a.y; o[2] = rb.a.z; o[3] = rb.a.w;
    o[4] = rb.b.x; o[5] = rb.b.y; o[6] = rb.b.z; o[7] = rb.b.w;
  } else if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
    const uint32_t w[4] = {rb.a.x, rb.a.y, rb.a.z, rb.a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2(w[i]) : dec2_e5m2_h2(w[i]);
      o[2 * i + 1] = (F == KVQ_FP8_E4M3) ? dec2_e4m3_h2_hi(w[i]) : dec2_e5m2_h2_hi(w[i]);
    }
  } else {
    uint32_t h[8];  // E2M1 pairs as f16x2 (even element low)
    h[0] = dec2_e2m1_h2<0>(rb.a.x); h[1] = dec2_e2m1_h2<1>(rb.a.x);
    h[2] = dec2_e2m1_h2<2>(rb.a.x); h[3] = dec2_e2m1_h2<3>(rb.a.x);
    h[4] = dec2_e2m1_h2<0>(rb.a.y); h[5] = dec2_e2m1_h2<1>(rb.a.y);
    h[6] = dec2_e2m1_h2<2>(rb.a.y); h[7] = dec2_e2m1_h2<3>(rb.a.y);
    if (F == KVQ_NVFP4) {  // E2M1 x E4M3 is exact in f16
      const uint32_t s2 = dec2_e4m3_h2(rb.sc | (rb.sc << 8));
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = hmul2x(h[i], s2);
    } else {  // E2M1 x 2^(E - 127), exact in fp32 and in bf16
      const float m = exp2i((int)(rb.sc & 0xFF) - 127);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = pack_bf2(h2_lo(h[i]) * m, h2_hi(h[i]) * m);
    }
  }
}

template <kvq_format F>
__global__ void __launch_bounds__(kXThreads, 4) extend_kernel(ExtendArgs a) {
  using Tr = XTraits<F>;
  constexpr bool BF = Tr::kBf16;
  __shared__ __align__(128) uint8_t sraw[kXStages][Tr::kStageBytes];  // raw tiles in flight
  __shared__ __align__(128) uint8_t sm[2][kXTile];                     // dequantized [K|V] tile
  __shared__ int row_seq[kXRows];                        // sequence of each row, -1: done / none
  __shared__ int row_len[kXRows];
  __shared__ int pass_seq, pass_max, pass_bad;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r4 = lane >> 2, c = lane & 3;
  const int h = blockIdx.y;
  const long long R0 = (long long)blockIdx.x * kXRows;

  // ---- rows of this CTA: (query, head) = divmod(R0 + rho, G) ----------------
  for (int rho = tid; rho < kXRows; rho += kXThreads) {
    const long long R = R0 + rho;
    const long long qi = R / a.G;
    int s = -1, T = 0;
    if (qi < a.n) {
      s = __ldg(a.q_seq + qi);
      T = __ldg(a.q_len + qi);
      if (s < 0 || s >= a.S || T < 0 || T > a.max_pages * a.P) {
        if ((int)(R % a.G) == 0) atomicOr(a.err, kErrRange);
        s = -2;  // invalid: output zeros
      }
    }
    row_seq[rho] = s;
    row_len[rho] = T;
  }

  // ---- this thread's two rows: warp rows r4 and r4 + 8 ----------------------
  long long qrow[2];
  int qhead[2];
  bool qvalid[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const long long R = R0 + warp * 16 + r4 + 8 * i;
    qrow[i] = R / a.G;
    qhead[i] = h * a.G + (int)(R % a.G);
    qvalid[i] = qrow[i] < a.n;
  }
  // Q fragments (A operand): k-step ks covers d = 16 ks .. 16 ks + 15; this
  // thread holds d = 16 ks + 2c, +1 and 16 ks + 2c + 8, +9 of both rows.
  uint32_t qa[8][4];
  float cs[2];
  {
    float qf[2][32];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(
          a.q + ((qvalid[i] ? qrow[i] : 0) * a.Hq + qhead[i]) * kHeadDim);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t w0 = qvalid[i] ? __ldg(src + 8 * ks + c) : 0u;
        const uint32_t w1 = qvalid[i] ? __ldg(src + 8 * ks + 4 + c) : 0u;
        qf[i][4 * ks + 0] = bf16_bits_to_float(w0 & 0xFFFF);
        qf[i][4 * ks + 1] = bf16_bits_to_float(w0 >> 16);
        qf[i][4 * ks + 2] = bf16_bits_to_float(w1 & 0xFFFF);
        qf[i][4 * ks + 3] = bf16_bits_to_float(w1 >> 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float hf = a.kfac ? a.qscale * __ldg(a.kfac + h) : a.qscale;
      if (BF) {
        cs[i] = hf;
      } else {
        // power-of-two prescale: max |q'| in [2^14, 2^15) keeps bf16 values exact in f16
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(qf[i][j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int sq = amax > 0.f ? max(-126, min(126, floor_log2(amax) - 14)) : 0;
        const float mul = exp2i(-sq);
#pragma unroll
        for (int j = 0; j < 32; ++j) qf[i][j] *= mul;
        cs[i] = hf * exp2i(sq);
      }
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      if (BF) {
        qa[ks][0] = pack_bf2(qf[0][4 * ks], qf[0][4 * ks + 1]);
        qa[ks][1] = pack_bf2(qf[1][4 * ks], qf[1][4 * ks + 1]);
        qa[ks][2] = pack_bf2(qf[0][4 * ks + 2], qf[0][4 * ks + 3]);
        qa[ks][3] = pack_bf2(qf[1][4 * ks + 2], qf[1][4 * ks + 3]);
      } else {
        qa[ks][0] = pack_h2(qf[0][4 * ks], qf[0][4 * ks + 1]);
        qa[ks][1] = pack_h2(qf[1][4 * ks], qf[1][4 * ks + 1]);
        qa[ks][2] = pack_h2(qf[0][4 * ks + 2], qf[0][4 * ks + 3]);
        qa[ks][3] = pack_h2(qf[1][4 * ks + 2], qf[1][4 * ks + 3]);
      }
    }
  }

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  bool poison[2] = {false, false};

  const int my_tok = tid >> 3, my_blk = tid & 7;  // the block this thread loads per tile
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(&sm[0][0]);
  const uint32_t sraw_base = (uint32_t)__cvta_generic_to_shared(&sraw[0][0]);
  __syncthreads();

  // ---- one pass per distinct sequence among the CTA's rows ----------------------
  for (;;) {
    if (tid == 0) {
      int s = -1;
      for (int rho = 0; rho < kXRows && s < 0; ++rho) s = row_seq[rho] >= 0 ? row_seq[rho] : -1;
      int mx = 0;
      for (int rho = 0; rho < kXRows; ++rho)
        if (row_seq[rho] == s && s >= 0) mx = max(mx, row_len[rho]);
      pass_seq = s;
      pass_max = mx;
      pass_bad = 0;
    }
    __syncthreads();
    const int s = pass_seq;
    if (s < 0) break;
    const int maxT = pass_max;
    bool act[2];
    int Tr_[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int rho = warp * 16 + r4 + 8 * i;
      act[i] = row_seq[rho] == s;
      Tr_[i] = row_len[rho];
    }
    const int32_t* prow = a.page_table + (long long)s * a.max_pages;
    const int ntiles = (maxT + kTile - 1) / kTile;

    // copy the raw K/V (+ scale) rows of tile t into stage t % kXStages; every
    // thread commits one group per call (empty beyond the last tile)
    auto issue = [&](int t) {
      if (t < ntiles) {
        const uint32_t st = sraw_base + (uint32_t)((t % kXStages) * Tr::kStageBytes);
        const int tt0 = t * kTile;
        const int page = __ldg(prow + tt0 / a.P);  // one page holds the whole tile
        const bool pok = page >= 0 && page < a.num_pages;
        if (!pok) pass_bad = 1;
        const long long row0 = ((long long)(pok ? page : 0) * a.H + h) * a.P + tt0 % a.P;
        constexpr int kChunks = Tr::kRow / 16;  // 16-byte pieces of one row
        for (int i = tid; i < Tr::kCopies; i += kXThreads) {
          if (i < 2 * kTile * kChunks) {
            const int kv = i / (kTile * kChunks), j = i % (kTile * kChunks);
            const int tok = j / kChunks, ch = j % kChunks;
            const bool valid = pok && tt0 + tok < maxT;
            const uint8_t* src = (kv ? a.vd : a.kd) + (row0 + tok) * Tr::kRow + ch * 16;
            cp_async16(st + (uint32_t)(kv * kTile * Tr::kRow + tok * Tr::kRow + ch * 16),
                       valid ? src : a.kd, valid);
          } else {
            const int j = i - 2 * kTile * kChunks, kv = j / kTile, tok = j % kTile;
            const bool valid = pok && tt0 + tok < maxT;
            const uint8_t* src = (kv ? a.vs : a.ks) + (row0 + tok) * 8;
            cp_async8(st + (uint32_t)(2 * kTile * Tr::kRow + kv * kTile * 8 + tok * 8),
                      valid ? src : a.kd, valid);
          }
        }
      }
      cp_async_commit();
    };
#pragma unroll 1
    for (int t = 0; t < kXStages - 1; ++t) issue(t);

    for (int t = 0; t < ntiles; ++t) {
      issue(t + kXStages - 1);
      cp_async_wait<kXStages - 1>();  // this thread's copies of tile t have landed
      __syncthreads();                // ... and every other thread's
      // dequantize tile t (absent tokens and bad pages were zero-filled)
      {
        const uint8_t* stage = &sraw[t % kXStages][0];
        uint32_t ok_[8], ov_[8];
        dequant_block<F>(raw_block<F>(stage, 0, my_tok, my_blk), ok_);
        dequant_block<F>(raw_block<F>(stage, 1, my_tok, my_blk), ov_);
        uint8_t* kdst = &sm[0][my_tok * kXStride + my_blk * 32];
        uint8_t* vdst = &sm[1][my_tok * kXStride + my_blk * 32];
        reinterpret_cast<uint4*>(kdst)[0] = make_uint4(ok_[0], ok_[1], ok_[2], ok_[3]);
        reinterpret_cast<uint4*>(kdst)[1] = make_uint4(ok_[4], ok_[5], ok_[6], ok_[7]);
        reinterpret_cast<uint4*>(vdst)[0] = make_uint4(ov_[0], ov_[1], ov_[2], ov_[3]);
        reinterpret_cast<uint4*>(vdst)[1] = make_uint4(ov_[4], ov_[5], ov_[6], ov_[7]);
      }
      __syncthreads();
      if (!__any_sync(0xffffffffu, act[0] || act[1])) continue;  // no row of this warp in the pass

      const uint32_t kbase = sbase;
      const uint32_t vbase = sbase + (uint32_t)kXTile;
      // ---- S = Q K^T (16 rows x 16 tokens) ----
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mi = lane >> 3, rr = lane & 7;
        const uint32_t lrow = (uint32_t)((rr + 8 * (mi >> 1)) * kXStride + (mi & 1) * 16);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t b00, b01, b10, b11;
          ldsm_x4(kbase + lrow + ks * 32, b00, b01, b10, b11);
          mma16816<BF>(sacc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
          mma16816<BF>(sacc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
        }
      }
      // ---- online softmax (base 2) per row; masked tokens and inactive rows: -inf ----
      float x[2][4];  // [n-tile][c0 c1 (row r4), c2 c3 (row r4 + 8)]
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e >> 1;
          const int tok = t * kTile + nt * 8 + 2 * c + (e & 1);
          x[nt][e] = (act[i] && tok < Tr_[i]) ? sacc[nt][e] * cs[i] : -INFINITY;
        }
      float mx[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mx[i] = fmaxf(fmaxf(x[0][2 * i], x[0][2 * i + 1]), fmaxf(x[1][2 * i], x[1][2 * i + 1]));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      }
      const bool grow0 = mx[0] > m[0] + 8.f, grow1 = mx[1] > m[1] + 8.f;
      if (__any_sync(0xffffffffu, grow0 || grow1)) {
        const float n0 = grow0 ? mx[0] : m[0], n1 = grow1 ? mx[1] : m[1];
        const float al0 = grow0 ? ex2x(m[0] - n0) : 1.f, al1 = grow1 ? ex2x(m[1] - n1) : 1.f;
        l[0] *= al0;
        l[1] *= al1;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          o[j][0] *= al0;
          o[j][1] *= al0;
          o[j][2] *= al1;
          o[j][3] *= al1;
        }
        m[0] = n0;
        m[1] = n1;
      }
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e >> 1;
          p[nt][e] = (x[nt][e] == -INFINITY) ? 0.f : ex2x(x[nt][e] - m[i]);
          l[i] += p[nt][e];
        }
      // ---- O += P V: P from the S accumulators (A operand), V by ldmatrix.trans ----
      uint32_t pa[4], pl[4];
      if (BF) {
        pa[0] = pack_bf2(p[0][0], p[0][1]);
        pa[1] = pack_bf2(p[0][2], p[0][3]);
        pa[2] = pack_bf2(p[1][0], p[1][1]);
        pa[3] = pack_bf2(p[1][2], p[1][3]);
        pl[0] = pack_bf2(p[0][0] - bf16_bits_to_float(pa[0] & 0xFFFF), p[0][1] - bf16_bits_to_float(pa[0] >> 16));
        pl[1] = pack_bf2(p[0][2] - bf16_bits_to_float(pa[1] & 0xFFFF), p[0][3] - bf16_bits_to_float(pa[1] >> 16));
        pl[2] = pack_bf2(p[1][0] - bf16_bits_to_float(pa[2] & 0xFFFF), p[1][1] - bf16_bits_to_float(pa[2] >> 16));
        pl[3] = pack_bf2(p[1][2] - bf16_bits_to_float(pa[3] & 0xFFFF), p[1][3] - bf16_bits_to_float(pa[3] >> 16));
      } else {
        pa[0] = pack_h2(p[0][0], p[0][1]);
        pa[1] = pack_h2(p[0][2], p[0][3]);
        pa[2] = pack_h2(p[1][0], p[1][1]);
        pa[3] = pack_h2(p[1][2], p[1][3]);
        pl[0] = pl[1] = pl[2] = pl[3] = 0u;
      }
      {
        const int mi = lane >> 3, rr = lane & 7;
        const uint32_t lrow = (uint32_t)((rr + 8 * (mi & 1)) * kXStride + (mi >> 1) * 16);
#pragma unroll
        for (int j2 = 0; j2 < 8; ++j2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + lrow + j2 * 32, b0, b1, b2, b3);
          mma16816<BF>(o[2 * j2], pa[0], pa[1], pa[2], pa[3], b0, b1);
          mma16816<BF>(o[2 * j2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
          if (BF) {
            mma16816<BF>(o[2 * j2], pl[0], pl[1], pl[2], pl[3], b0, b1);
            mma16816<BF>(o[2 * j2 + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
          }
        }
      }
    }
    cp_async_wait<0>();  // only empty groups remain; the stages are free
    __syncthreads();     // pass_bad complete; buffers free for the next pass
    if (pass_bad) {
      if (tid == 0) atomicOr(a.err, kErrRange);
      poison[0] = poison[0] || act[0];
      poison[1] = poison[1] || act[1];
    }
    if (tid == 0)
      for (int rho = 0; rho < kXRows; ++rho)
        if (row_seq[rho] == s) row_seq[rho] = -1;
    __syncthreads();
  }

  // ---- normalize and write: row i holds d = 8 j + 2c, +1 -------------------------
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
  }
  const float vf = a.vfac ? __ldg(a.vfac + h) : a.v_factor;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!qvalid[i]) continue;
    const float inv = (poison[i] || !(l[i] > 0.f)) ? 0.f : vf / l[i];
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + (qrow[i] * a.Hq + qhead[i]) * kHeadDim);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      dst[4 * j + c] = bf16_rne_bits(o[j][2 * i] * inv) | (bf16_rne_bits(o[j][2 * i + 1] * inv) << 16);
  }
}

template <kvq_format F>
cudaError_t launch_extend_as(const ExtendArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.n * a.G;
  dim3 grid((unsigned)((rows + kXRows - 1) / kXRows), (unsigned)a.H);
  extend_kernel<F><<<grid, kXThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_extend(const Geometry& g, const LayerView& L, const void* q, int num_q_heads,
                          int num_q_tokens, const int32_t* q_seq, const int32_t* q_len,
                          const int32_t* page_table, int num_seqs, int max_pages_per_seq,
                          float sm_scale, float k_factor, float v_factor, const HeadScales& hs,
                          void* out, int* err, cudaStream_t stream) {
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
  a.qscale = sm_scale * 1.4426950408889634f * (a.kfac ? 1.0f : k_factor);
  a.v_factor = v_factor;
  a.err = err;
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
