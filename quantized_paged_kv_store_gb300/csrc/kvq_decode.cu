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
//   touches into slot u + w (unique), and the merge kernel combines a unit's
//   partials with the log-sum-exp rule
//     out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s.
//
// Per warp worker: a private ring of shared-memory stages; lane 0 stages each
// 16-token (page, kv head) tile of K, V (and their block scales) with 1D bulk
// async copies (TMA engine) completing on an mbarrier, several tiles ahead.
// Each tile then runs, with the lane layout of mma.m16n8k16 (lane = 4 r + q):
//   QK^T on tensor cores: M = 16 tokens, N = 8 q heads of the group, K = d.
//     The contraction index is permuted so that k-step j of thread q reads
//     d = 32 q + 4 j + {0..3}: each thread's K operand is one contiguous
//     byte run of its two token rows; Q is permuted the same way.
//   online softmax per q head (base 2), P to f16, transposed with movmatrix
//     into the B operand of
//   PV on tensor cores: M = 16 head_dim rows (8 tiles), N = 8 q heads,
//     K = 16 tokens.  Thread (r, q) owns head_dim block r (d = 16 r .. +15)
//     of tokens {2q, 2q+1, 2q+8, 2q+9}: code pairs of two tokens are gathered
//     with byte/nibble permutes and converted with cvt.f16x2.{e4m3x2, e5m2x2,
//     e2m1x2}.
// Exactness: E4M3/E5M2 codes and E2M1 x E4M3 products are exact in f16; Q
// (bf16) is scaled by a power of two per head so it is exact in f16; FP4
// block-16 values are held as E2M1 x 2^(E - E_ref) with E_ref the largest
// exponent of the K row / the running largest of the V block, and the 2^E_ref
// factor is applied in fp32.  The bf16 cache uses bf16 MMAs, with P split into
// a high and a low bf16 part.  Per-tensor scales fold into the logit scale
// (K) and the output (V).  Accumulation is fp32.
#include "kvq_codecs.cuh"
#include "kvq_decode_args.cuh"
#include "kvq_internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

namespace kvq {
namespace {

constexpr int kWarpsPerCta = 4;
constexpr int kPidWin = 30;    // page ids prefetched per window (a multiple of every stage size)
constexpr uint32_t kWaitLimit = 1u << 20;  // mbarrier polls before giving up (~1 s)
constexpr uint32_t kFaultWaitLimit = 64;   // polls of the injected never-completing wait

template <kvq_format F>
struct Traits {
  static constexpr int kRow = (F == KVQ_BF16) ? 256 : (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) ? 128 : 64;
  static constexpr bool kScales = (F == KVQ_FP4_BLOCK16 || F == KVQ_NVFP4);
  static constexpr int kData = kTile * kRow;              // one K (or V) tile
  static constexpr int kScale = kScales ? kTile * 8 : 0;  // its block scales
  static constexpr int kTileBytes = 2 * (kData + kScale); // K, V (+ scales) of one tile
  static constexpr int kCopies = kScales ? 4 : 2;         // bulk copies per tile
  static constexpr int kTps = (F == KVQ_BF16) ? 1 : (F == KVQ_NVFP4 || F == KVQ_FP4_BLOCK16) ? 3 : 2;
  static constexpr int kStage = kTps * kTileBytes;
  static constexpr int kStages = (F == KVQ_BF16) ? 3 : 2;
  static constexpr int kWarpSmem = kStages * kStage;
  // per warp: the stage ring, one mbarrier per stage and one that is never
  // armed (the target of the injected wait of the failure-detection test)
  static constexpr int kCtaSmem = kWarpsPerCta * (kWarpSmem + (kStages + 1) * 8);
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }

__device__ __forceinline__ void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// FP8 tensor-core MMA (m16n8k32): A = K codes (E4M3 or E5M2), B = E4M3 query
// codes, fp32 accumulate.
template <kvq_format F>
__device__ __forceinline__ void mma_f8(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1) {
  if (F == KVQ_FP8_E5M2)
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e5m2.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t f32x2_to_h2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t f32x2_to_bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Byte k (compile-time) of x: two E2M1 codes -> half2.
template <int K>
__device__ __forceinline__ uint32_t e2m1_byte_h2(uint32_t x) { return dec2_e2m1_h2<K>(x); }

// half2 of (2^da, 2^db) for da, db <= 15: exact down to 2^-24 (f16 subnormals
// included), 0 below.  Built as fp32 powers of two (exponent field, clamped
// at 2^-126) and rounded to f16 by one convert.
__device__ __forceinline__ uint32_t h2_pow2(int da, int db) {
  const float fa = __uint_as_float((uint32_t)(max(da, -126) + 127) << 23);
  const float fb = __uint_as_float((uint32_t)(max(db, -126) + 127) << 23);
  return f32x2_to_h2(fa, fb);
}

// FP4 block-16 factors without the fp32 route.  Two E8M0 codes b0, b1 held in
// the halves of x (b0 | b1 << 16) and a reference code ref give
//   y = x + (7 - ref) * 0x10001,  halves b - ref + 7
// (one 32-bit add: with every half in [0, 15] no borrow or carry crosses the
// halves).  y is "in window" iff (y & 0xFFF0FFF0) == 0, i.e. both codes lie in
// [ref - 7, ref + 8]; a code outside makes its half >= 16 (an underflow leaves
// 0xFFxx there).  In window, (y << 10) + 0x20002000 is the half2 of
// (2^(b0 - ref), 2^(b1 - ref)): exponent field b - ref + 15, exact.
__device__ __forceinline__ uint32_t e8m0_window(uint32_t x, int ref) {
  return x + (uint32_t)(7 - ref) * 0x10001u;
}
__device__ __forceinline__ uint32_t e8m0_window_h2(uint32_t y) { return (y << 10) + 0x20002000u; }
constexpr uint32_t kWindowMiss = 0xFFF0FFF0u;

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per-warp staging ring.
struct Ring {
  const uint8_t* gsmem;  // generic address of stage 0
  uint32_t smem;         // shared address of stage 0
  uint32_t bar;          // shared address of the first mbarrier (one per stage, then `never`)
  uint32_t pos;          // stages consumed by this warp (monotonic)
  uint32_t issued;       // stages issued by this warp (monotonic)
  uint32_t dead_pos;     // first stage whose wait ran out
  bool dead;             // a wait ran out: issue and wait no more
};

// Logits of one 16-token tile: s = (K^ Q'^T) for rows r, r+8 and heads 2q,
// 2q+1 (before the per-head scale).  FP4 block-16: kf holds the half2 block
// factors 2^(E - kref) of (row r, block 2q), (r, 2q+1), (r+8, 2q), (r+8, 2q+1),
// each broadcast to both halves; 2^kref is applied with the per-head scale.
// QF8 (FP8-domain attention, FP8 caches): qb[j] holds the E4M3 query codes of
// k-step j of m16n8k32 (k = 4q + i <-> d = 32q + 8j + i, k = 16 + 4q + i <->
// d = 32q + 8j + 4 + i), and the K codes enter the MMA unconverted.
template <kvq_format F, bool QF8>
__device__ __forceinline__ void tile_qk(const uint8_t* sK, const uint8_t* sKs, int r, int q,
                                        const uint32_t (&qb)[8][2], float (&s)[4],
                                        const uint32_t (&kf)[4]) {
  s[0] = s[1] = s[2] = s[3] = 0.f;
  if constexpr (QF8) {
    const uint4 x0 = lds128(sK + r * 128 + q * 32), x1 = lds128(sK + r * 128 + q * 32 + 16);
    const uint4 y0 = lds128(sK + (r + 8) * 128 + q * 32), y1 = lds128(sK + (r + 8) * 128 + q * 32 + 16);
    const uint32_t kr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const uint32_t kr8[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      mma_f8<F>(s, kr[2 * j], kr8[2 * j], kr[2 * j + 1], kr8[2 * j + 1], qb[j][0], qb[j][1]);
  } else if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
    const uint4 x0 = lds128(sK + r * 128 + q * 32), x1 = lds128(sK + r * 128 + q * 32 + 16);
    const uint4 y0 = lds128(sK + (r + 8) * 128 + q * 32), y1 = lds128(sK + (r + 8) * 128 + q * 32 + 16);
    const uint32_t kr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const uint32_t kr8[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t a0, a1, a2, a3;
      if (F == KVQ_FP8_E4M3) {
        a0 = dec2_e4m3_h2(kr[j]);
        a2 = dec2_e4m3_h2_hi(kr[j]);
        a1 = dec2_e4m3_h2(kr8[j]);
        a3 = dec2_e4m3_h2_hi(kr8[j]);
      } else {
        a0 = dec2_e5m2_h2(kr[j]);
        a2 = dec2_e5m2_h2_hi(kr[j]);
        a1 = dec2_e5m2_h2(kr8[j]);
        a3 = dec2_e5m2_h2_hi(kr8[j]);
      }
      mma_f16(s, a0, a1, a2, a3, qb[j][0], qb[j][1]);
    }
  } else if (F == KVQ_BF16) {
    uint32_t kr[16], kr8[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 x = lds128(sK + r * 256 + q * 64 + 16 * c);
      const uint4 y = lds128(sK + (r + 8) * 256 + q * 64 + 16 * c);
      kr[4 * c] = x.x; kr[4 * c + 1] = x.y; kr[4 * c + 2] = x.z; kr[4 * c + 3] = x.w;
      kr8[4 * c] = y.x; kr8[4 * c + 1] = y.y; kr8[4 * c + 2] = y.z; kr8[4 * c + 3] = y.w;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) mma_bf16(s, kr[2 * j], kr8[2 * j], kr[2 * j + 1], kr8[2 * j + 1], qb[j][0], qb[j][1]);
  } else {
    const uint4 x = lds128(sK + r * 64 + q * 16);
    const uint4 y = lds128(sK + (r + 8) * 64 + q * 16);
    uint32_t f00, f01, f10, f11;  // f16x2 factors: row r / r+8, block 2q / 2q+1
    if (F == KVQ_NVFP4) {
      const uint32_t sc0 = *reinterpret_cast<const uint16_t*>(sKs + r * 8 + 2 * q);
      const uint32_t sc1 = *reinterpret_cast<const uint16_t*>(sKs + (r + 8) * 8 + 2 * q);
      const uint32_t h0 = dec2_e4m3_h2(sc0), h1 = dec2_e4m3_h2(sc1);
      f00 = __byte_perm(h0, 0, 0x1010);
      f01 = __byte_perm(h0, 0, 0x3232);
      f10 = __byte_perm(h1, 0, 0x1010);
      f11 = __byte_perm(h1, 0, 0x3232);
    } else {
      f00 = kf[0];
      f01 = kf[1];
      f10 = kf[2];
      f11 = kf[3];
    }
    const uint32_t kw[4] = {x.x, x.y, x.z, x.w}, kw8[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t wr = kw[j >> 1], wr8 = kw8[j >> 1];
      uint32_t a0, a1, a2, a3;
      if ((j & 1) == 0) {
        a0 = e2m1_byte_h2<0>(wr);
        a2 = e2m1_byte_h2<1>(wr);
        a1 = e2m1_byte_h2<0>(wr8);
        a3 = e2m1_byte_h2<1>(wr8);
      } else {
        a0 = e2m1_byte_h2<2>(wr);
        a2 = e2m1_byte_h2<3>(wr);
        a1 = e2m1_byte_h2<2>(wr8);
        a3 = e2m1_byte_h2<3>(wr8);
      }
      const uint32_t fr = (j < 4) ? f00 : f01, fr8 = (j < 4) ? f10 : f11;
      a0 = hmul2(a0, fr);
      a2 = hmul2(a2, fr);
      a1 = hmul2(a1, fr8);
      a3 = hmul2(a3, fr8);
      mma_f16(s, a0, a1, a2, a3, qb[j][0], qb[j][1]);
    }
  }

}

// O^T += V^T P^T for one 16-token tile (p* are this thread's P entries:
// rows r, r+8 and heads 2q, 2q+1); nvalid tokens of the tile are real.
template <kvq_format F>
__device__ __forceinline__ void tile_pv(const uint8_t* sV, const uint8_t* sVs, int r, int q, int nvalid,
                                        float p0, float p1, float p2, float p3, float (&o)[8][4],
                                        int& vref) {
  const bool partial = nvalid < kTile;
  const int ta = 2 * q, tb = 2 * q + 1, tc = 2 * q + 8, td = 2 * q + 9;
  if (F == KVQ_BF16) {
    const uint32_t ph0 = f32x2_to_bf2(p0, p1), ph1 = f32x2_to_bf2(p2, p3);
    const float l0a = p0 - bf16_bits_to_float(ph0 & 0xFFFF), l1a = p1 - bf16_bits_to_float(ph0 >> 16);
    const float l2a = p2 - bf16_bits_to_float(ph1 & 0xFFFF), l3a = p3 - bf16_bits_to_float(ph1 >> 16);
    const uint32_t pl0 = f32x2_to_bf2(l0a, l1a), pl1 = f32x2_to_bf2(l2a, l3a);
    const uint32_t bh0 = movm_t(ph0), bh1 = movm_t(ph1), bl0 = movm_t(pl0), bl1 = movm_t(pl1);
    uint32_t va[8], vb[8], vc[8], vd[8];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 A = lds128(sV + ta * 256 + r * 32 + 16 * c), Bv = lds128(sV + tb * 256 + r * 32 + 16 * c);
      const uint4 C = lds128(sV + tc * 256 + r * 32 + 16 * c), D = lds128(sV + td * 256 + r * 32 + 16 * c);
      va[4 * c] = A.x; va[4 * c + 1] = A.y; va[4 * c + 2] = A.z; va[4 * c + 3] = A.w;
      vb[4 * c] = Bv.x; vb[4 * c + 1] = Bv.y; vb[4 * c + 2] = Bv.z; vb[4 * c + 3] = Bv.w;
      vc[4 * c] = C.x; vc[4 * c + 1] = C.y; vc[4 * c + 2] = C.z; vc[4 * c + 3] = C.w;
      vd[4 * c] = D.x; vd[4 * c + 1] = D.y; vd[4 * c + 2] = D.z; vd[4 * c + 3] = D.w;
    }
    if (partial) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (ta >= nvalid) va[k] = 0u;
        if (tb >= nvalid) vb[k] = 0u;
        if (tc >= nvalid) vc[k] = 0u;
        if (td >= nvalid) vd[k] = 0u;
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // rows: d = 16 r + mt (word mt/2 of the block's first half), d = 16 r + 8 + mt
      const uint32_t sel = (mt & 1) ? 0x7632u : 0x5410u;
      const uint32_t a0 = __byte_perm(va[mt >> 1], vb[mt >> 1], sel);
      const uint32_t a1 = __byte_perm(va[4 + (mt >> 1)], vb[4 + (mt >> 1)], sel);
      const uint32_t a2 = __byte_perm(vc[mt >> 1], vd[mt >> 1], sel);
      const uint32_t a3 = __byte_perm(vc[4 + (mt >> 1)], vd[4 + (mt >> 1)], sel);
      mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
      mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
    }
  } else {
    const uint32_t b0 = movm_t(f32x2_to_h2(p0, p1)), b1 = movm_t(f32x2_to_h2(p2, p3));
    if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
      uint4 A = lds128(sV + ta * 128 + r * 16), Bv = lds128(sV + tb * 128 + r * 16);
      uint4 C = lds128(sV + tc * 128 + r * 16), D = lds128(sV + td * 128 + r * 16);
      if (partial) {
        if (ta >= nvalid) A = make_uint4(0, 0, 0, 0);
        if (tb >= nvalid) Bv = make_uint4(0, 0, 0, 0);
        if (tc >= nvalid) C = make_uint4(0, 0, 0, 0);
        if (td >= nvalid) D = make_uint4(0, 0, 0, 0);
      }
      const uint32_t aw[4] = {A.x, A.y, A.z, A.w}, bw[4] = {Bv.x, Bv.y, Bv.z, Bv.w};
      const uint32_t cw[4] = {C.x, C.y, C.z, C.w}, dw[4] = {D.x, D.y, D.z, D.w};
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        // byte mt (row r) and byte 8 + mt (row r + 8) of each token's block
        const uint32_t sel = (mt & 2) ? 0x7362u : 0x5140u;
        const uint32_t pab = __byte_perm(aw[mt >> 2], bw[mt >> 2], sel);
        const uint32_t pab8 = __byte_perm(aw[2 + (mt >> 2)], bw[2 + (mt >> 2)], sel);
        const uint32_t pcd = __byte_perm(cw[mt >> 2], dw[mt >> 2], sel);
        const uint32_t pcd8 = __byte_perm(cw[2 + (mt >> 2)], dw[2 + (mt >> 2)], sel);
        uint32_t a0, a1, a2, a3;
        if (F == KVQ_FP8_E4M3) {
          a0 = (mt & 1) ? dec2_e4m3_h2_hi(pab) : dec2_e4m3_h2(pab);
          a1 = (mt & 1) ? dec2_e4m3_h2_hi(pab8) : dec2_e4m3_h2(pab8);
          a2 = (mt & 1) ? dec2_e4m3_h2_hi(pcd) : dec2_e4m3_h2(pcd);
          a3 = (mt & 1) ? dec2_e4m3_h2_hi(pcd8) : dec2_e4m3_h2(pcd8);
        } else {
          a0 = (mt & 1) ? dec2_e5m2_h2_hi(pab) : dec2_e5m2_h2(pab);
          a1 = (mt & 1) ? dec2_e5m2_h2_hi(pab8) : dec2_e5m2_h2(pab8);
          a2 = (mt & 1) ? dec2_e5m2_h2_hi(pcd) : dec2_e5m2_h2(pcd);
          a3 = (mt & 1) ? dec2_e5m2_h2_hi(pcd8) : dec2_e5m2_h2(pcd8);
        }
        mma_f16(o[mt], a0, a1, a2, a3, b0, b1);
      }
    } else {
      uint2 A = lds64(sV + ta * 64 + r * 8), Bv = lds64(sV + tb * 64 + r * 8);
      uint2 C = lds64(sV + tc * 64 + r * 8), D = lds64(sV + td * 64 + r * 8);
      if (partial) {
        if (ta >= nvalid) A = make_uint2(0, 0);
        if (tb >= nvalid) Bv = make_uint2(0, 0);
        if (tc >= nvalid) C = make_uint2(0, 0);
        if (td >= nvalid) D = make_uint2(0, 0);
      }
      uint32_t sa = sVs[ta * 8 + r], sb = sVs[tb * 8 + r];
      uint32_t sc = sVs[tc * 8 + r], sd = sVs[td * 8 + r];
      if (partial) {  // masked tokens: zero codes, and no say in the reference exponent
        if (ta >= nvalid) sa = 0u;
        if (tb >= nvalid) sb = 0u;
        if (tc >= nvalid) sc = 0u;
        if (td >= nvalid) sd = 0u;
      }
      uint32_t fab, fcd;  // f16x2 block factors (token pair)
      if (F == KVQ_NVFP4) {
        fab = dec2_e4m3_h2(sa | (sb << 8));
        fcd = dec2_e4m3_h2(sc | (sd << 8));
      } else {
        // factors 2^(E - vref) against the running reference exponent of V
        // block r (per lane quad): packed integer path while every code of
        // the warp lies within [vref - 7, vref + 8]; otherwise raise the
        // reference to the quad's maximum (rescaling the accumulator) and
        // build the factors exactly through fp32
        const uint32_t xab = __byte_perm(sa, sb, 0x5410), xcd = __byte_perm(sc, sd, 0x5410);
        const uint32_t yab = e8m0_window(xab, vref), ycd = e8m0_window(xcd, vref);
        if (__any_sync(0xffffffffu, ((yab | ycd) & kWindowMiss) != 0u)) {
          int et = max(max((int)sa, (int)sb), max((int)sc, (int)sd));
          et = max(et, __shfl_xor_sync(0xffffffffu, et, 1));
          et = max(et, __shfl_xor_sync(0xffffffffu, et, 2));
          if (et > vref) {
            const float f = (vref < -127) ? 0.f : exp2i(vref - et);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o[mt][0] *= f;
              o[mt][1] *= f;
              o[mt][2] *= f;
              o[mt][3] *= f;
            }
            vref = et;
          }
          fab = h2_pow2((int)sa - vref, (int)sb - vref);
          fcd = h2_pow2((int)sc - vref, (int)sd - vref);
        } else {
          fab = e8m0_window_h2(yab);
          fcd = e8m0_window_h2(ycd);
        }
      }
      // nibble pairs (token a | token b << 4) for even / odd nibble index
      const uint32_t ev0 = (A.x & 0x0F0F0F0Fu) | ((Bv.x << 4) & 0xF0F0F0F0u);
      const uint32_t od0 = ((A.x >> 4) & 0x0F0F0F0Fu) | (Bv.x & 0xF0F0F0F0u);
      const uint32_t ev1 = (A.y & 0x0F0F0F0Fu) | ((Bv.y << 4) & 0xF0F0F0F0u);
      const uint32_t od1 = ((A.y >> 4) & 0x0F0F0F0Fu) | (Bv.y & 0xF0F0F0F0u);
      const uint32_t ec0 = (C.x & 0x0F0F0F0Fu) | ((D.x << 4) & 0xF0F0F0F0u);
      const uint32_t oc0 = ((C.x >> 4) & 0x0F0F0F0Fu) | (D.x & 0xF0F0F0F0u);
      const uint32_t ec1 = (C.y & 0x0F0F0F0Fu) | ((D.y << 4) & 0xF0F0F0F0u);
      const uint32_t oc1 = ((C.y >> 4) & 0x0F0F0F0Fu) | (D.y & 0xF0F0F0F0u);
#define KVQ_PV_TILE(MT, ODD, BYTE)                                                       \
{                                                                                     \
  const uint32_t a0 = hmul2(e2m1_byte_h2<BYTE>(ODD ? od0 : ev0), fab);                \
  const uint32_t a1 = hmul2(e2m1_byte_h2<BYTE>(ODD ? od1 : ev1), fab);                \
  const uint32_t a2 = hmul2(e2m1_byte_h2<BYTE>(ODD ? oc0 : ec0), fcd);                \
  const uint32_t a3 = hmul2(e2m1_byte_h2<BYTE>(ODD ? oc1 : ec1), fcd);                \
  mma_f16(o[MT], a0, a1, a2, a3, b0, b1);                                             \
}
      KVQ_PV_TILE(0, 0, 0)
      KVQ_PV_TILE(1, 1, 0)
      KVQ_PV_TILE(2, 0, 1)
      KVQ_PV_TILE(3, 1, 1)
      KVQ_PV_TILE(4, 0, 2)
      KVQ_PV_TILE(5, 1, 2)
      KVQ_PV_TILE(6, 0, 3)
      KVQ_PV_TILE(7, 1, 3)
#undef KVQ_PV_TILE
    }
  }

}

// One worker's contribution to unit (b, h, hg) over tiles [t0, t1).
template <kvq_format F, bool QF8>
__device__ void segment(const DecodeArgs& a, Ring& ring, int w, int b, int h, int hg, int t0, int t1) {
  using Tr = Traits<F>;
  constexpr int S = Tr::kStages, TPS = Tr::kTps;
  constexpr float kLazy = 8.f;  // rescale only when a logit beats the max by 2^8
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, q = lane & 3;
  const int T = __ldg(a.seq_lens + b);
  const int gh = min(kGroupMax, a.G - hg * kGroupMax);
  const int n = t1 - t0;
  const int nch = (n + TPS - 1) / TPS;

  // ---- Q fragments (B operand of QK^T) and per-head logit scales ----------
  uint32_t qb[8][2];
  float colscale;  // for head r, then redistributed
  {
    uint32_t w16[16];
    if (r < gh) {
      const uint16_t* qr = a.q + ((long long)b * a.Hq + h * a.G + hg * kGroupMax + r) * kHeadDim + q * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(qr + i * 8);
        w16[4 * i] = v.x;
        w16[4 * i + 1] = v.y;
        w16[4 * i + 2] = v.z;
        w16[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w16[i] = 0u;
    }
    if (a.neg_q) {  // sm_scale < 0: negate the query (bf16 sign bits), scale by |sm_scale|
#pragma unroll
      for (int i = 0; i < 16; ++i) w16[i] ^= 0x80008000u;
    }
    if constexpr (QF8) {
      // FP8-domain attention: E4M3 codes of q / q_scale (the query quantization
      // rule of the store), the B operand of the m16n8k32 FP8 MMAs
      const int head = h * a.G + hg * kGroupMax + r;
      const float qsc = a.qsc[(a.nqs == 1 || r >= gh) ? 0 : head];
      const float rq = 1.0f / qsc;
      uint32_t m2 = 0u;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(w16[i]));
      const float amax = __uint_as_float(max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu) << 16);
      const bool fast = qsc >= 0x1p-80f && qsc <= 0x1p80f && amax * rq < 1e37f;  // NaN: false
      uint32_t c[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        c[i] = quant2_e4m3(bf16_bits_to_float(w16[i] & 0xFFFF), bf16_bits_to_float(w16[i] >> 16),
                           qsc, rq, fast);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        qb[j][0] = c[4 * j] | (c[4 * j + 1] << 16);
        qb[j][1] = c[4 * j + 2] | (c[4 * j + 3] << 16);
      }
#pragma unroll
      for (int j = 4; j < 8; ++j) qb[j][0] = qb[j][1] = 0u;
      const float qs = a.kfac ? a.qscale * __ldg(a.kfac + h) : a.qscale;
      colscale = (r < gh) ? qs * qsc : 1.f;
    } else if (F == KVQ_BF16) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qb[j][0] = w16[2 * j];
        qb[j][1] = w16[2 * j + 1];
      }
      colscale = (r < gh) ? a.qscale : 1.f;  // padded heads: zero q, any positive scale
    } else {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w16[i] & 0xFFFF)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_float(w16[i] >> 16)));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // power-of-two prescale: max |q'| in [2^14, 2^15) keeps bf16 values exact in f16
      const int sq = amax > 0.f ? max(-126, min(126, floor_log2(amax) - 14)) : 0;
      const float mul = exp2i(-sq);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qb[j][0] = f32x2_to_h2(bf16_bits_to_float(w16[2 * j] & 0xFFFF) * mul,
                               bf16_bits_to_float(w16[2 * j] >> 16) * mul);
        qb[j][1] = f32x2_to_h2(bf16_bits_to_float(w16[2 * j + 1] & 0xFFFF) * mul,
                               bf16_bits_to_float(w16[2 * j + 1] >> 16) * mul);
      }
      // per-kv-head K scale (one per unit), else the per-tensor one folded on the host
      const float qs = a.kfac ? a.qscale * __ldg(a.kfac + h) : a.qscale;
      colscale = (r < gh) ? qs * exp2i(sq) : 1.f;
    }
  }
  // D1 columns of this thread are heads 2q, 2q+1 (held by lanes 8q and 8q+4 above)
  const float cs0 = __shfl_sync(0xffffffffu, colscale, 8 * q);
  const float cs1 = __shfl_sync(0xffffffffu, colscale, 8 * q + 4);

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  int vref = -1000;  // FP4 block-16: reference exponent code of V block r
  int kref = -1000;  // FP4 block-16: reference exponent code of the K tiles of a chunk
  float kcs0 = cs0, kcs1 = cs1;  // per-head logit scales, times 2^(kref - 127) for FP4 block-16
  bool poison = false;

  // ---- page ids, prefetched one window (32 tiles) ahead ----------------------
  const int tiles_per_page = a.P / kTile;
  const int32_t* prow = a.page_table + (long long)pt_row_of(a, b) * a.max_pages;
  auto load_pid = [&](int win) -> int {
    const int t = t0 + win * kPidWin + lane;
    return (t < t1) ? __ldg(prow + t / tiles_per_page) : -1;
  };
  int pid_cur = load_pid(0), pid_next = load_pid(1);
  uint32_t bad_mask = 0;  // stages holding an invalid page id (warp-uniform)

  // ---- copy roles: lane = tile * kCopies + kind issues one bulk copy --------
  const int my_tile = lane / Tr::kCopies, my_kind = lane % Tr::kCopies;
  const bool copier = lane < TPS * Tr::kCopies;
  const uint8_t* my_base;
  long long my_page_stride;
  int my_tile_stride;
  uint32_t my_bytes, my_dst;
  {
    const long long page_rows = (long long)a.H * a.P;
    const bool scale_kind = my_kind >= 2;
    const int rowb = scale_kind ? 8 : Tr::kRow;
    const uint8_t* pool = my_kind == 0 ? a.kd : my_kind == 1 ? a.vd : my_kind == 2 ? a.ks : a.vs;
    my_base = pool + (long long)h * a.P * rowb;
    my_page_stride = page_rows * rowb;
    my_tile_stride = kTile * rowb;
    my_bytes = scale_kind ? Tr::kScale : Tr::kData;
    my_dst = (uint32_t)(my_tile * Tr::kTileBytes) +
             (my_kind == 0 ? 0u : my_kind == 1 ? (uint32_t)Tr::kData
                                 : my_kind == 2 ? 2u * Tr::kData : 2u * Tr::kData + Tr::kScale);
  }
  // Per lane: tile (of the sequence) that this lane's copy fetches in the next
  // chunk issued, and the offset of that chunk's first tile in the page-id
  // window; both advance by TPS per chunk (kPidWin is a multiple of TPS).
  int ktile = t0 + my_tile;
  int koff = 0, win = 0;
  const int tpp_mask = (tiles_per_page & (tiles_per_page - 1)) == 0 ? tiles_per_page - 1 : -1;
  const uint32_t npages = (uint32_t)min(a.num_pages, (long long)0x7FFFFFFF);
  const uint32_t page_stride = (uint32_t)my_page_stride;  // < 2^31 (checked at plan time)

  // issue chunk c (tiles c*TPS ..) into stage issued % S; all lanes call
  auto issue = [&](int c) {
    const int ntc = min(TPS, n - c * TPS);
    if (koff == kPidWin) {  // the next window of page ids
      koff = 0;
      ++win;
      pid_cur = pid_next;
      pid_next = load_pid(win + 1);
    }
    const int page = __shfl_sync(0xffffffffu, pid_cur, koff + my_tile);
    const uint32_t st = ring.issued % S;
    const uint32_t bar = ring.bar + 8 * st;
    const bool mine = copier && my_tile < ntc;
    const bool ok = __all_sync(0xffffffffu, !mine || (uint32_t)page < npages);
    bad_mask = ok ? (bad_mask & ~(1u << st)) : (bad_mask | (1u << st));
    if (lane == 0) mbar_arrive_tx(bar, ok ? ntc * Tr::kTileBytes : 0);
    if (ok && mine) {
      const int sb = tpp_mask >= 0 ? (ktile & tpp_mask) : (ktile % tiles_per_page);
      bulk_g2s(ring.smem + st * Tr::kStage + my_dst,
               my_base + (uint64_t)(uint32_t)page * page_stride + (uint32_t)(sb * my_tile_stride), my_bytes,
               bar);
    }
    koff += TPS;
    ktile += TPS;
    ring.issued++;
  };

  if (!ring.dead)
    for (int c = 0; c < min(S, nch); ++c) issue(c);

  // Failure-detection test: the warp's first wait targets the mbarrier that is
  // never armed, with a short limit, so that it runs out while the warp's first
  // copies are in flight (they land in the bounded drain at the kernel's end).
  if (a.fault_wait && ring.pos == 0 && !ring.dead) {
    uint32_t polls = 0;
    bool ok = mbar_try_wait(ring.bar + 8 * S, 0u);
    while (!ok && ++polls < kFaultWaitLimit) ok = mbar_try_wait(ring.bar + 8 * S, 0u);
    if (!__all_sync(0xffffffffu, ok)) {
      ring.dead = true;
      ring.dead_pos = ring.pos;
      if (lane == 0) atomicOr(a.err, kErrTimeout);
    }
  }

  for (int c = 0; c < nch; ++c) {
    const uint32_t st = ring.pos % S;
    const uint32_t parity = (ring.pos / S) & 1u;
    if (!ring.dead) {
      uint32_t polls = 0;
      bool ok = mbar_try_wait(ring.bar + 8 * st, parity);
      while (!ok && ++polls < kWaitLimit) ok = mbar_try_wait(ring.bar + 8 * st, parity);
      if (!__all_sync(0xffffffffu, ok)) {
        ring.dead = true;
        ring.dead_pos = ring.pos;
        if (lane == 0) atomicOr(a.err, kErrTimeout);
      }
    }
    if (ring.dead || (bad_mask >> st) & 1u) {
      poison = true;
      ring.pos++;
      continue;
    }
    const uint8_t* stage = ring.gsmem + st * Tr::kStage;
    const int ntc = min(TPS, n - c * TPS);

    // One chunk of NT tiles; NT is a compile-time constant so the tiles'
    // independent dequant/MMA chains can be interleaved by the compiler.  FULL
    // chunks (every token of every tile valid) carry no masking code at all.
    auto run_chunk = [&](auto nt_const, auto full_const) {
      constexpr int NT = decltype(nt_const)::value;
      constexpr bool FULL = decltype(full_const)::value;
      int nvalid[NT];
#pragma unroll
      for (int tt = 0; tt < NT; ++tt)
        nvalid[tt] = FULL ? kTile : min(kTile, T - (t0 + c * TPS + tt) * kTile);

      // ---- logits of the chunk's tiles ----
      // FP4 block-16: K block factors 2^(E - kref) against one reference code
      // kref; the logits carry 2^(kref - 127) in the per-head scale kcs.  A
      // tile whose codes all lie in kref's window [kref - 7, kref + 8] builds
      // its factors with packed integer ops; otherwise kref is re-anchored at
      // the tile's largest code (earlier tiles of the chunk are rescaled to
      // it) and the tile's factors go through fp32 (exact down to 2^-24).
      float sc[NT][4];
#pragma unroll
      for (int tt = 0; tt < NT; ++tt) {
        const uint8_t* tb = stage + tt * Tr::kTileBytes;
        uint32_t kf[4] = {0u, 0u, 0u, 0u};
        if constexpr (F == KVQ_FP4_BLOCK16) {
          const uint8_t* ks = tb + 2 * Tr::kData;
          uint32_t s0 = *reinterpret_cast<const uint16_t*>(ks + r * 8 + 2 * q);
          uint32_t s1 = *reinterpret_cast<const uint16_t*>(ks + (r + 8) * 8 + 2 * q);
          if (!FULL) {  // rows past the sequence end: no say in the reference
            if (r >= nvalid[tt]) s0 = 0u;
            if (r + 8 >= nvalid[tt]) s1 = 0u;
          }
          const uint32_t x0 = __byte_perm(s0, 0, 0x4140), x1 = __byte_perm(s1, 0, 0x4140);
          uint32_t y0 = e8m0_window(x0, kref), y1 = e8m0_window(x1, kref);
          uint32_t h0, h1;
          if (__any_sync(0xffffffffu, ((y0 | y1) & kWindowMiss) != 0u)) {
            const uint32_t m2 = __vmaxu2(x0, x1);
            uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (kref >= 0) {  // earlier tiles of the chunk: to the new reference
              // 2^(kref - mx) as two factors (the difference spans [-254, 254])
              const int d = kref - (int)mx, d1 = max(-127, min(127, d));
              const float g1 = exp2i(d1), g2 = exp2i(max(-127, min(127, d - d1)));
#pragma unroll
              for (int t2 = 0; t2 < tt; ++t2) {
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[t2][i] = (sc[t2][i] * g1) * g2;
              }
            }
            kref = (int)mx;
            const float f = exp2i(kref - 127);
            kcs0 = cs0 * f;
            kcs1 = cs1 * f;
            h0 = h2_pow2((int)(x0 & 0xFFFFu) - kref, (int)(x0 >> 16) - kref);
            h1 = h2_pow2((int)(x1 & 0xFFFFu) - kref, (int)(x1 >> 16) - kref);
          } else {
            h0 = e8m0_window_h2(y0);
            h1 = e8m0_window_h2(y1);
          }
          kf[0] = __byte_perm(h0, 0, 0x1010);
          kf[1] = __byte_perm(h0, 0, 0x3232);
          kf[2] = __byte_perm(h1, 0, 0x1010);
          kf[3] = __byte_perm(h1, 0, 0x3232);
        }
        tile_qk<F, QF8>(tb, tb + 2 * Tr::kData, r, q, qb, sc[tt], kf);
        if (!FULL && nvalid[tt] < kTile) {
          if (r >= nvalid[tt]) sc[tt][0] = sc[tt][1] = -INFINITY;
          if (r + 8 >= nvalid[tt]) sc[tt][2] = sc[tt][3] = -INFINITY;
        }
      }
      const float c0 = (F == KVQ_FP4_BLOCK16) ? kcs0 : cs0;
      const float c1 = (F == KVQ_FP4_BLOCK16) ? kcs1 : cs1;

      // ---- online softmax on scaled logits cs * s (cs > 0), rescaling lazily ----
      float x0 = fmaxf(sc[0][0], sc[0][2]), x1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
      for (int tt = 1; tt < NT; ++tt) {
        x0 = fmaxf(x0, fmaxf(sc[tt][0], sc[tt][2]));
        x1 = fmaxf(x1, fmaxf(sc[tt][1], sc[tt][3]));
      }
      // scale (c >= 0); an all-masked chunk keeps -inf (its p are set to 0 below)
      x0 = (x0 == -INFINITY) ? x0 : x0 * c0;
      x1 = (x1 == -INFINITY) ? x1 : x1 * c1;
      if (__any_sync(0xffffffffu, x0 > m0 + kLazy || x1 > m1 + kLazy)) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
          x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
        m0 = n0;
        m1 = n1;
      }

      // ---- O^T += V^T P^T ----
#pragma unroll
      for (int tt = 0; tt < NT; ++tt) {
        float p0 = ex2(fmaf(sc[tt][0], c0, -m0)), p1 = ex2(fmaf(sc[tt][1], c1, -m1));
        float p2 = ex2(fmaf(sc[tt][2], c0, -m0)), p3 = ex2(fmaf(sc[tt][3], c1, -m1));
        if (!FULL && nvalid[tt] < kTile) {  // masked tokens: 0 whatever the scale (c = 0 included)
          if (r >= nvalid[tt]) p0 = p1 = 0.f;
          if (r + 8 >= nvalid[tt]) p2 = p3 = 0.f;
        }
        l0 += p0 + p2;
        l1 += p1 + p3;
        const uint8_t* tb = stage + tt * Tr::kTileBytes;
        tile_pv<F>(tb + Tr::kData, tb + 2 * Tr::kData + Tr::kScale, r, q, FULL ? kTile : nvalid[tt], p0,
                   p1, p2, p3, o, vref);
      }
    };
    using False_ = std::false_type;
    if (ntc == TPS && (t0 + c * TPS + TPS) * kTile <= T) {
      run_chunk(std::integral_constant<int, TPS>{}, std::true_type{});
    } else if (ntc == TPS) {
      run_chunk(std::integral_constant<int, TPS>{}, False_{});
    } else if (ntc == 1) {
      run_chunk(std::integral_constant<int, 1>{}, False_{});
    } else {
      if constexpr (TPS >= 3) run_chunk(std::integral_constant<int, 2>{}, False_{});  // 2-tile tail of a 3-tile stage
    }
    static_assert(TPS <= 3, "chunk tails above 2 tiles need their own case");

    // release the stage and refill it with chunk c + S
    __syncwarp();
    ring.pos++;
    if (!ring.dead && c + S < nch) {
      if (lane == 0) fence_proxy_async();
      issue(c + S);
    }
  }

  // ---- partial result of this segment ----------------------------------------
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  poison = __any_sync(0xffffffffu, poison);
  if (poison && lane == 0 && !ring.dead) atomicOr(a.err, kErrRange);
  const long long u = ((long long)b * a.H + h) * a.HG + hg;
  const long long slot = u + w;
  float vscale = a.vfac ? __ldg(a.vfac + h) : a.v_factor;
  if (F == KVQ_FP4_BLOCK16) vscale *= exp2i(max(-127, min(127, vref - 127)));
  const float inv0 = poison ? 0.f : vscale / l0, inv1 = poison ? 0.f : vscale / l1;
  // thread (r, q): heads 2q, 2q+1; d = 16 r + mt (c0, c1) and 16 r + 8 + mt (c2, c3)
  if (2 * q < gh) {
    float* po = a.part_o + (slot * kGroupMax + 2 * q) * kHeadDim + 16 * r;
    reinterpret_cast<float4*>(po)[0] = make_float4(o[0][0] * inv0, o[1][0] * inv0, o[2][0] * inv0, o[3][0] * inv0);
    reinterpret_cast<float4*>(po)[1] = make_float4(o[4][0] * inv0, o[5][0] * inv0, o[6][0] * inv0, o[7][0] * inv0);
    reinterpret_cast<float4*>(po)[2] = make_float4(o[0][2] * inv0, o[1][2] * inv0, o[2][2] * inv0, o[3][2] * inv0);
    reinterpret_cast<float4*>(po)[3] = make_float4(o[4][2] * inv0, o[5][2] * inv0, o[6][2] * inv0, o[7][2] * inv0);
    if (r == 0) a.part_lse[slot * kGroupMax + 2 * q] = poison ? INFINITY : m0 + __log2f(l0);
  }
  if (2 * q + 1 < gh) {
    float* po = a.part_o + (slot * kGroupMax + 2 * q + 1) * kHeadDim + 16 * r;
    reinterpret_cast<float4*>(po)[0] = make_float4(o[0][1] * inv1, o[1][1] * inv1, o[2][1] * inv1, o[3][1] * inv1);
    reinterpret_cast<float4*>(po)[1] = make_float4(o[4][1] * inv1, o[5][1] * inv1, o[6][1] * inv1, o[7][1] * inv1);
    reinterpret_cast<float4*>(po)[2] = make_float4(o[0][3] * inv1, o[1][3] * inv1, o[2][3] * inv1, o[3][3] * inv1);
    reinterpret_cast<float4*>(po)[3] = make_float4(o[4][3] * inv1, o[5][3] * inv1, o[6][3] * inv1, o[7][3] * inv1);
    if (r == 0) a.part_lse[slot * kGroupMax + 2 * q + 1] = poison ? INFINITY : m1 + __log2f(l1);
  }
}

template <kvq_format F, bool QF8>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 4) decode_kernel(DecodeArgs a) {
  using Tr = Traits<F>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int w = blockIdx.x * kWarpsPerCta + warp;
  // let the merge kernel launch early; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;");
  if (w >= a.num_workers) return;
  const long long upb = (long long)a.H * a.HG;  // units per sequence

  Ring ring;
  ring.gsmem = smem_raw + warp * Tr::kWarpSmem;
  ring.smem = smem_addr(smem_raw) + warp * Tr::kWarpSmem;
  ring.dead_pos = 0;
  ring.bar = smem_addr(smem_raw) + kWarpsPerCta * Tr::kWarpSmem + warp * (Tr::kStages + 1) * 8;
  ring.pos = 0;
  ring.issued = 0;
  ring.dead = false;
  if (lane == 0) {
    for (int s = 0; s <= Tr::kStages; ++s) mbar_init(ring.bar + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  __syncwarp();

  // pass 1: total tiles; worker 0 reports invalid lengths and publishes Wtot
  long long total = 0;
  bool bad_len = false;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int b = b0 + lane;
    int nt = 0;
    if (b < a.B) {
      const int T = __ldg(a.seq_lens + b);
      if (T < 0 || T > a.max_pages * a.P || pt_row_of(a, b) < 0) bad_len = true;
      nt = tiles_of(a, b);
    }
    if (w == 0) {  // publish the per-sequence tile prefix for the merge
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b < a.B) a.prefix[b + 1] = total + incl;
    }
    total += warp_sum_i(nt);
  }
  total *= upb;
  if (w == 0) {
    if (__any_sync(0xffffffffu, bad_len) && lane == 0) atomicOr(a.err, kErrRange);
    if (lane == 0) {
      a.meta[0] = total;
      a.prefix[0] = 0;
    }
  }
  const long long start = worker_start(total, w, a.num_workers);
  const long long end = worker_start(total, w + 1, a.num_workers);
  if (start >= end) return;

  // pass 2: locate the sequence holding `start`
  long long cum = 0;
  int b = 0;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int bb = b0 + lane;
    const long long x = (bb < a.B) ? (long long)tiles_of(a, bb) * upb : 0;
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
  const long long local = start - cum;
  int ub = (int)(local / nt);
  int tile = (int)(local - (long long)ub * nt);
  long long pos = start;
  while (pos < end) {
    const int n = (int)min((long long)(nt - tile), end - pos);
    segment<F, QF8>(a, ring, w, b, ub / a.HG, ub % a.HG, tile, tile + n);
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
  // Every issued tile has been consumed, unless a wait ran out: then give the
  // copies still in flight a bounded chance to land before the CTA exits.
  if (ring.dead) {
    for (uint32_t t = ring.dead_pos; t < ring.issued; ++t) {
      const uint32_t bar = ring.bar + 8 * (t % Tr::kStages);
      uint32_t polls = 0;
      while (!mbar_try_wait(bar, (t / Tr::kStages) & 1u) && ++polls < kWaitLimit) {
      }
    }
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

constexpr int kMaxDevices = 64;

// Kernel attributes are per device: the dynamic shared-memory opt-in and the
// occupancy query run once for each (format, device), with that device
// current, under a lock; later calls read the cached CTA count.
template <kvq_format F, bool QF8>
cudaError_t prepare(int device, int* ctas_per_sm) {
  static std::mutex mu;
  static std::atomic<int> cached[kMaxDevices];
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  int n = cached[device].load(std::memory_order_acquire);
  if (n == 0) {
    std::lock_guard<std::mutex> lock(mu);
    n = cached[device].load(std::memory_order_relaxed);
    if (n == 0) {
      int prev = -1;
      cudaError_t e = cudaGetDevice(&prev);
      if (e != cudaSuccess) return e;
      if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
      e = cudaFuncSetAttribute(decode_kernel<F, QF8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Traits<F>::kCtaSmem);
      int occ = 0;
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<F, QF8>, kWarpsPerCta * 32,
                                                          Traits<F>::kCtaSmem);
      if (prev != device) {
        const cudaError_t e2 = cudaSetDevice(prev);
        if (e == cudaSuccess) e = e2;
      }
      if (e != cudaSuccess) return e;
      n = std::max(occ, 1);
      cached[device].store(n, std::memory_order_release);
    }
  }
  *ctas_per_sm = n;
  return cudaSuccess;
}

cudaError_t ctas_per_sm(kvq_format f, bool qf8, int device, int* n) {
  if (qf8) {
    switch (f) {
      case KVQ_FP8_E4M3: return prepare<KVQ_FP8_E4M3, true>(device, n);
      case KVQ_FP8_E5M2: return prepare<KVQ_FP8_E5M2, true>(device, n);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (f) {
    case KVQ_BF16: return prepare<KVQ_BF16, false>(device, n);
    case KVQ_FP8_E4M3: return prepare<KVQ_FP8_E4M3, false>(device, n);
    case KVQ_FP8_E5M2: return prepare<KVQ_FP8_E5M2, false>(device, n);
    case KVQ_FP4_BLOCK16: return prepare<KVQ_FP4_BLOCK16, false>(device, n);
    case KVQ_NVFP4: return prepare<KVQ_NVFP4, false>(device, n);
  }
  return cudaErrorInvalidValue;
}

template <kvq_format F, bool QF8>
cudaError_t launch_f(const DecodeArgs& a, int ctas, cudaStream_t stream) {
  decode_kernel<F, QF8><<<ctas, kWarpsPerCta * 32, Traits<F>::kCtaSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool plan_decode(const Geometry& g, int batch, int num_q_heads, int max_pages_per_seq,
                 int device, DecodePlan* plan, const char** why, bool qf8) {
  if (g.head_dim != kHeadDim) { *why = "decode attention supports head_dim == 128 only"; return false; }
  if (g.page_size % kTile != 0) { *why = "decode attention needs page_size % 16 == 0"; return false; }
  if (num_q_heads % g.kv_heads != 0) { *why = "num_q_heads must be a multiple of kv_heads"; return false; }
  if ((int64_t)g.kv_heads * g.page_size * 2 * g.head_dim >= (int64_t(1) << 31)) {
    *why = "decode attention needs kv_heads * page_size * row bytes < 2^31";
    return false;
  }
  const int G = num_q_heads / g.kv_heads;
  if (G > 2 * kGroupMax) { *why = "group size num_q_heads / kv_heads must be <= 16"; return false; }
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0) {
    *why = "cannot query the SM count";
    return false;
  }
  // the grid (and so the workspace) is sized from the bf16-query kernel of the
  // format; the FP8-query kernel has the same shared memory and register bound
  if (ctas_per_sm(g.fmt, false, device, &per_sm) != cudaSuccess) {
    *why = "cannot configure the decode kernel";
    return false;
  }
  if (qf8) {
    int per_sm_q = 0;
    if (g.fmt != KVQ_FP8_E4M3 && g.fmt != KVQ_FP8_E5M2) {
      *why = "FP8-domain attention needs an fp8_e4m3 or fp8_e5m2 cache";
      return false;
    }
    if (ctas_per_sm(g.fmt, true, device, &per_sm_q) != cudaSuccess) {
      *why = "cannot configure the FP8-domain decode kernel";
      return false;
    }
  }
  plan->group = G;
  plan->head_groups = (G + kGroupMax - 1) / kGroupMax;
  plan->num_units = (int64_t)batch * g.kv_heads * plan->head_groups;
  const int64_t tiles_per_seq = ((int64_t)max_pages_per_seq * g.page_size + kTile - 1) / kTile;
  const int64_t max_tiles = std::max<int64_t>(1, plan->num_units * tiles_per_seq);
  // persistent grid: every resident warp is a worker, each with >= 4 tiles
  int64_t ctas = (int64_t)sms * per_sm;
  ctas = std::min<int64_t>(ctas, (max_tiles + 4 * kWarpsPerCta - 1) / (4 * kWarpsPerCta));
  ctas = std::max<int64_t>(ctas, 1);
  plan->ctas = (int)ctas;
  plan->num_workers = plan->ctas * kWarpsPerCta;
  plan->num_slots = plan->num_units + plan->num_workers;
  plan->ws_bytes = align256((size_t)plan->num_slots * kGroupMax * kHeadDim * sizeof(float)) +
                   align256((size_t)plan->num_slots * kGroupMax * sizeof(float)) + 256 +
                   align256((size_t)(batch + 1) * sizeof(long long));
  return true;
}

cudaError_t launch_decode(const Geometry& g, const LayerView& L, const DecodePlan& plan,
                          const void* q, int num_q_heads, const int32_t* page_table,
                          int max_pages_per_seq, const int32_t* seq_lens, int batch,
                          float sm_scale, float k_factor, float v_factor, const HeadScales& hs,
                          const int32_t* pt_rows, int pt_nrows, void* out, void* workspace,
                          int* err, cudaStream_t stream, const float* q_scales, int num_q_scales) {
  DecodeArgs a;
  const bool qf8 = q_scales != nullptr;
  a.nqs = qf8 ? num_q_scales : 0;
  for (int i = 0; i < kMaxQScales; ++i) a.qsc[i] = (qf8 && i < num_q_scales) ? q_scales[i] : 1.0f;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.part_o = reinterpret_cast<float*>(ws);
  ws += align256((size_t)plan.num_slots * kGroupMax * kHeadDim * sizeof(float));
  a.part_lse = reinterpret_cast<float*>(ws);
  ws += align256((size_t)plan.num_slots * kGroupMax * sizeof(float));
  a.meta = reinterpret_cast<long long*>(ws);
  ws += 256;
  a.prefix = reinterpret_cast<long long*>(ws);
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
  // per-head scales multiply in the kernel, after the same sm_scale * log2(e)
  a.kfac = hs.scale[0];
  a.vfac = hs.scale[1];
  // the softmax runs on positive logit scales: a negative sm_scale is folded
  // into the query's sign (exact)
  a.neg_q = sm_scale < 0.f;
  a.qscale = std::fabs(sm_scale) * 1.4426950408889634f * (a.kfac ? 1.0f : k_factor);
  a.v_factor = v_factor;
  a.pt_rows = pt_rows;
  a.pt_nrows = pt_nrows;
  a.err = err;
  // KVQ_FAULT=wait (failure-detection tests only): every warp's first stage
  // wait gives up, the kernel reports KVQ_ERR_TIMEOUT and zeroes the outputs
  const char* fault = std::getenv("KVQ_FAULT");
  a.fault_wait = fault && std::strcmp(fault, "wait") == 0;
  if (batch == 0) return cudaSuccess;
  cudaError_t e = cudaErrorInvalidValue;
  if (qf8) {
    switch (g.fmt) {
      case KVQ_FP8_E4M3: e = launch_f<KVQ_FP8_E4M3, true>(a, plan.ctas, stream); break;
      case KVQ_FP8_E5M2: e = launch_f<KVQ_FP8_E5M2, true>(a, plan.ctas, stream); break;
      default: break;
    }
  } else {
    switch (g.fmt) {
      case KVQ_BF16: e = launch_f<KVQ_BF16, false>(a, plan.ctas, stream); break;
      case KVQ_FP8_E4M3: e = launch_f<KVQ_FP8_E4M3, false>(a, plan.ctas, stream); break;
      case KVQ_FP8_E5M2: e = launch_f<KVQ_FP8_E5M2, false>(a, plan.ctas, stream); break;
      case KVQ_FP4_BLOCK16: e = launch_f<KVQ_FP4_BLOCK16, false>(a, plan.ctas, stream); break;
      case KVQ_NVFP4: e = launch_f<KVQ_NVFP4, false>(a, plan.ctas, stream); break;
    }
  }
  if (e != cudaSuccess) return e;
  return launch_merge(a, plan.num_units, stream);
}

}  // namespace kvq
