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
// One thread owns an item: one 16-element block of one (token, kv_head) row
// (the bf16 copy) or two, blocks j and j + nb/2 of the row (the quantizing
// formats).  Per block: two 16-byte loads of bf16, the block amax in
// registers, encode, and one 16-byte (FP8) or 8-byte (FP4) store into the
// paged row plus one scale byte.  Consecutive threads take consecutive items,
// so a warp's loads and stores cover contiguous runs of each row half.  The
// kernel is HBM-bound (NVFP4: bound by instruction issue).
#include <algorithm>

#include "kvq_codecs.cuh"
#include "kvq_decode_args.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

struct StoreArgs {
  const uint16_t* x[2];  // K, V bf16 [n][H][D]
  uint8_t* data[2];
  uint8_t* scales[2];
  float s[2];            // FP8 scale / NVFP4 global scale per K, V
  float rs[2];           // FP8: 1 / s (IEEE)
  float s6[2];           // NVFP4: RN(6 g), the block-scale divisor
  float rs6[2];          // NVFP4: RN(1 / RN(6 g))
  const int64_t* slots;
  int64_t n;             // tokens
  int H, D, P;
  int nb;                // blocks per row (D / 16)
  int nb_shift;          // log2(nb) if nb is a power of two, else -1
  int p_shift;           // log2(P) if P is a power of two, else -1
  int hb;                // H * nb: blocks per token
  int ib;                // items per token: hb / blocks per item
  int nbi;               // items per row: nb / blocks per item
  int nbi_shift;         // log2(nbi) if nbi is a power of two, else -1
  bool fast_div;         // scales in [2^-80, 2^80]: reciprocal-based division is exact
  int64_t num_pages;
  int* err;
  const float* hs[2];    // per-kv-head scales of K, V (per-head kernels only)
  const float* hr[2];    // their reciprocals
};

// Largest bf16 magnitude of the 16 values as fp32 bits; NaN propagates, so
// bits >= 0x7F800000 flags a non-finite block.  (max.xorsign.abs takes the
// larger magnitude; the sign it sets is dropped at the end.)
__device__ __forceinline__ uint32_t block_amax_bits(const uint32_t w[8]) {
  uint32_t m = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(w[i]));
  const uint32_t lo = m & 0x7FFFu, hi = (m >> 16) & 0x7FFFu;
  // NaN patterns are larger than every finite magnitude and +inf as integers
  return (lo > hi ? lo : hi) << 16;
}

// Four bytes (the low byte of each word) into one word, c0 lowest.
__device__ __forceinline__ uint32_t pack4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  return __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040), 0x5410);
}

// NVFP4 block-scale table of one tensor: S[c] = RN(dec_E4M3(c) g) for the 128
// non-negative codes, and RN(1 / S[c]) where the corrected quotient is exact
// (S in [2^-80, 2^80]), else 0 (those blocks divide in IEEE arithmetic).
struct NvScaleTable {
  float S[128];
  float rS[128];
};

// Quantizes one 16-element block, already in registers as two 16-byte words of
// bf16, into row r of the cache: data bytes plus (FP4 formats) one scale byte.
template <kvq_format F>
__device__ __forceinline__ void store_block(uint8_t* dat, uint8_t* scl, int64_t r, int blk, int D, int nb,
                                            const uint4 lo, const uint4 hi, float s, float rs,
                                            bool fast_div, const NvScaleTable* tab = nullptr,
                                            float s6 = 0.f, float rs6 = 0.f) {
  if (F == KVQ_BF16) {
    uint4* d4 = reinterpret_cast<uint4*>(dat + r * (D * 2) + blk * 32);
    d4[0] = lo;
    d4[1] = hi;
    return;
  }
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const uint32_t amax_bits = block_amax_bits(w);
  const bool finite = amax_bits < 0x7F800000u;

  if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
    // fast path: every quotient finite, residuals exact near the decisions
    const bool fast = fast_div && finite && __uint_as_float(amax_bits) * rs < 1e37f;
    uint32_t wo[4];
    if (fast) {
      const uint64_t S2 = f2_pack(s, s), R2 = f2_pack(rs, rs), NR2 = f2_pack(-rs, -rs);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t p[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float q0, q1;
          f2_unpack(div2_rn_markstein(bf2_to_f2(w[2 * i + j]), S2, R2, NR2), q0, q1);
          p[j] = ((F == KVQ_FP8_E4M3) ? enc2_e4m3(q0, q1) : enc2_e5m2(q0, q1)) & 0xFFFFu;
        }
        wo[i] = p[0] | (p[1] << 16);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t p[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float x0 = __uint_as_float(w[2 * i + j] << 16);
          const float x1 = __uint_as_float(w[2 * i + j] & 0xFFFF0000u);
          const float q0 = x0 / s, q1 = x1 / s;  // IEEE fp32 division
          uint32_t c = (F == KVQ_FP8_E4M3) ? enc2_e4m3(q0, q1) : enc2_e5m2(q0, q1);
          if (!finite) {  // NaN input: 0x7F with the input's sign
            if (x0 != x0) c = (c & 0xFF00u) | 0x7Fu | ((__float_as_uint(x0) >> 24) & 0x80u);
            if (x1 != x1) c = (c & 0x00FFu) | ((0x7Fu | ((__float_as_uint(x1) >> 24) & 0x80u)) << 8);
          }
          p[j] = c & 0xFFFFu;
        }
        wo[i] = p[0] | (p[1] << 16);
      }
    }
    *reinterpret_cast<uint4*>(dat + r * D + blk * 16) = make_uint4(wo[0], wo[1], wo[2], wo[3]);
    return;
  }

  if constexpr (F == KVQ_FP4_BLOCK16 || F == KVQ_NVFP4) {
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }

  // FP4 formats: block amax, block scale, E2M1 codes.
  const float amax = __uint_as_float(amax_bits);
  float mul = 1.f, S = 1.f, rS = 1.f;
  uint32_t scode;
  bool zero = false, fast = false;
  if (F == KVQ_FP4_BLOCK16) {
    // MX shared exponent: E = clamp(floor(log2 amax) - 2, -127, 127)
    int E = -127;
    if (amax > 0.f) E = max(-127, min(127, floor_log2(amax) - 2));
    scode = (uint32_t)(E + 127);
    mul = exp2i(-E);
  } else if (tab) {
    // NVFP4, per-tensor g: sc = E4M3(amax / RN(6 g)) by the corrected
    // quotient from the precomputed reciprocal; S and 1 / S from the table
    const bool fr = rs6 != 0.f && finite && amax * rs6 < 1e37f;
    const float ratio = fr ? div_rn_markstein(amax, s6, rs6) : amax / s6;
    scode = enc2_e4m3(ratio, 0.f) & 0xFF;
    S = tab->S[scode & 0x7F];
    rS = tab->rS[scode & 0x7F];
    zero = (S == 0.f);
    fast = finite && !zero && rS != 0.f && amax * rS < 1e37f;
    if (fast) {  // packed pairs of corrected quotients
      const uint64_t S2 = f2_pack(S, S), R2 = f2_pack(rS, rS), NR2 = f2_pack(-rS, -rS);
      uint32_t c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float y0, y1;
        f2_unpack(div2_rn_markstein(bf2_to_f2(w[i]), S2, R2, NR2), y0, y1);
        c[i] = enc2_e2m1(y0, y1);
      }
      *reinterpret_cast<uint2*>(dat + r * (D / 2) + blk * 8) =
          make_uint2(pack4(c[0], c[1], c[2], c[3]), pack4(c[4], c[5], c[6], c[7]));
      scl[r * nb + blk] = (uint8_t)scode;
      return;
    }
    if (!zero) rS = 1.f / S;
  } else {
    // NVFP4: sc = E4M3(amax / (6 g)); S = dec(sc) * g
    const float g = s;
    const float ratio = amax / (6.0f * g);
    scode = enc2_e4m3(ratio, 0.f) & 0xFF;
    S = __fmul_rn(dec_e4m3(scode), g);
    zero = (S == 0.f);
    if (!zero) rS = 1.f / S;
    // a saturated block scale can leave x / S beyond the fp32 range: the
    // corrections would turn that inf into NaN, so such blocks divide exactly
    fast = fast_div && finite && !zero && amax * rS < 1e37f;
  }
  uint32_t wo[2] = {0u, 0u};
  if (!zero) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float y0, y1;
      if (F == KVQ_FP4_BLOCK16) {
        y0 = __fmul_rn(x[2 * i], mul);
        y1 = __fmul_rn(x[2 * i + 1], mul);
      } else if (fast) {
        y0 = div_rn_markstein(x[2 * i], S, rS);
        y1 = div_rn_markstein(x[2 * i + 1], S, rS);
      } else {
        y0 = x[2 * i] / S;
        y1 = x[2 * i + 1] / S;
      }
      wo[i >> 2] |= enc2_e2m1(y0, y1) << (8 * (i & 3));
    }
  }
  *reinterpret_cast<uint2*>(dat + r * (D / 2) + blk * 8) = make_uint2(wo[0], wo[1]);
  scl[r * nb + blk] = (uint8_t)scode;
  }
}

// Grid-stride loop over items (token, block-of-16) of one of K / V (blockIdx.y),
// software-pipelined: the next item's 32 input bytes and slot id are loaded
// before the current block is encoded, so every thread keeps a load in flight
// while it computes.  PH: the scale of each item's kv head comes from the
// per-head arrays ("Quantized KV cache" (vLLM), Supported schemes:
// per-attention-head scales) instead of the per-tensor launch argument.
// BPI (blocks per item): the quantizing formats take two blocks of a row per item --
// block j and block j + nb / 2 of one head, so that each of a warp's loads
// and stores covers consecutive blocks -- and share the slot, page and row
// arithmetic and the loop bookkeeping between them.
template <kvq_format F, bool PH, int BPI>
__global__ void __launch_bounds__(256) store_kernel(StoreArgs a) {
  const int kv = blockIdx.y;
  // NVFP4 with a per-tensor global scale: the CTA's block-scale table
  constexpr bool kTable = (F == KVQ_NVFP4) && !PH;
  const NvScaleTable* tab = nullptr;
  if constexpr (kTable) {
    __shared__ NvScaleTable tab_s;
    const float g = kv ? a.s[1] : a.s[0];
    if (threadIdx.x < 128) {
      const float S = __fmul_rn(dec_e4m3(threadIdx.x), g);
      tab_s.S[threadIdx.x] = S;
      tab_s.rS[threadIdx.x] = (S >= 0x1p-80f && S <= 0x1p80f) ? 1.0f / S : 0.f;
    }
    __syncthreads();
    tab = &tab_s;
  }
  // the item index advances by a constant stride, split once into (tokens, blocks)
  const long long S = (long long)gridDim.x * blockDim.x;
  const long long S_tok = S / a.ib;
  const int S_pair = (int)(S - S_tok * a.ib);
  const long long it0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  long long tok = it0 / a.ib;
  int pair = (int)(it0 - tok * a.ib);  // item of the token: blocks BPI pair ..
  if (tok >= a.n) return;
  // select per K/V without indexing the parameter arrays (that would copy them to local memory)
  const float s = kv ? a.s[1] : a.s[0], rs = kv ? a.rs[1] : a.rs[0];
  const uint16_t* const xin = kv ? a.x[1] : a.x[0];
  uint8_t* const dat = kv ? a.data[1] : a.data[0];
  uint8_t* const scl = kv ? a.scales[1] : a.scales[0];
  const float* const hsp = kv ? a.hs[1] : a.hs[0];
  const float* const hrp = kv ? a.hr[1] : a.hr[0];
  const int64_t tok_elems = (int64_t)a.H * a.D;  // input row of one token; item `pair` at pair * 16 BPI
  const int64_t capacity = a.num_pages * a.P;

  // item `pair` = (head h, j): blocks j and j + nbi of the head's row (BPI = 2),
  // so that a warp's first and second loads are each contiguous
  auto item_src = [&](long long t, int it) {
    const int hh = a.nbi_shift >= 0 ? (it >> a.nbi_shift) : it / a.nbi;
    return reinterpret_cast<const uint4*>(xin + t * tok_elems + (int64_t)(it + hh * (a.nb - a.nbi)) * 16);
  };
  const uint4* src = item_src(tok, pair);
  uint4 c[2 * BPI];
#pragma unroll
  for (int i = 0; i < 2 * BPI; ++i) c[i] = __ldg(src + (i >> 1) * (2 * a.nbi) + (i & 1));
  int64_t slot = __ldg(a.slots + tok);
  for (;;) {
    long long ntok = tok + S_tok;
    int npair = pair + S_pair;
    if (npair >= a.ib) {
      npair -= a.ib;
      ++ntok;
    }
    const bool more = ntok < a.n;
    uint4 n[2 * BPI];
#pragma unroll
    for (int i = 0; i < 2 * BPI; ++i) n[i] = make_uint4(0, 0, 0, 0);
    int64_t nslot = -1;
    if (more) {
      const uint4* ns = item_src(ntok, npair);
#pragma unroll
      for (int i = 0; i < 2 * BPI; ++i) n[i] = __ldg(ns + (i >> 1) * (2 * a.nbi) + (i & 1));
      nslot = __ldg(a.slots + ntok);
    }
    const int h = a.nbi_shift >= 0 ? (pair >> a.nbi_shift) : pair / a.nbi;
    const int blk = pair - h * a.nbi;  // blocks blk, blk + nbi
    if (slot >= capacity) {
      if (blk == 0) atomicOr(a.err, kErrRange);
    } else if (slot >= 0) {
      int64_t page, off;
      if (a.p_shift >= 0) {
        page = slot >> a.p_shift;
        off = slot & (a.P - 1);
      } else {
        page = slot / a.P;
        off = slot - page * a.P;
      }
      const int64_t r = (page * a.H + h) * a.P + off;  // destination row
#pragma unroll
      for (int j = 0; j < BPI; ++j) {
        if constexpr (PH) {
          const float sh = __ldg(hsp + h), rh = __ldg(hrp + h);
          store_block<F>(dat, scl, r, blk + j * a.nbi, a.D, a.nb, c[2 * j], c[2 * j + 1], sh, rh,
                         sh >= 0x1p-80f && sh <= 0x1p80f);
        } else if constexpr (kTable) {
          store_block<F>(dat, scl, r, blk + j * a.nbi, a.D, a.nb, c[2 * j], c[2 * j + 1], s, rs, a.fast_div, tab,
                         kv ? a.s6[1] : a.s6[0], kv ? a.rs6[1] : a.rs6[0]);
        } else {
          store_block<F>(dat, scl, r, blk + j * a.nbi, a.D, a.nb, c[2 * j], c[2 * j + 1], s, rs, a.fast_div);
        }
      }
    }
    if (!more) break;
    tok = ntok;
    pair = npair;
#pragma unroll
    for (int i = 0; i < 2 * BPI; ++i) c[i] = n[i];
    slot = nslot;
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
  const float* hs[2];  // per-kv-head scales of K, V, or null (per tensor)
};

template <kvq_format F>
__global__ void __launch_bounds__(256) dequant_kernel(DequantArgs a) {
  const int kv = blockIdx.y;
  const int nb = a.D >> 4;
  const uint8_t* const dat = kv ? a.data[1] : a.data[0];
  const uint8_t* const scl = kv ? a.scales[1] : a.scales[0];
  uint16_t* const outp = kv ? a.out[1] : a.out[0];
  const float s_tensor = kv ? a.s[1] : a.s[0];
  const float* const hsp = kv ? a.hs[1] : a.hs[0];
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < a.items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = it / nb;
    const int blk = (int)(it - row * nb);
    const int64_t tok = row / a.H;
    const int h = (int)(row - tok * a.H);
    const int64_t slot = __ldg(a.slots + tok);
    uint4* dst = reinterpret_cast<uint4*>(outp + row * a.D + blk * 16);
    const bool in_range = slot >= 0 && slot < a.num_pages * a.P;
    if (!in_range) {
      if (slot >= 0 && blk == 0) atomicOr(a.err, kErrRange);
      dst[0] = make_uint4(0, 0, 0, 0);
      dst[1] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int64_t page = slot / a.P, off = slot - page * a.P;
    const int64_t r = (page * a.H + h) * a.P + off;
    const float s_kv = hsp ? __ldg(hsp + h) : s_tensor;
    if (F == KVQ_BF16) {
      const uint4* s4 = reinterpret_cast<const uint4*>(dat + r * (a.D * 2) + blk * 32);
      dst[0] = __ldg(s4);
      dst[1] = __ldg(s4 + 1);
      continue;
    }
    float v[16];
    if (F == KVQ_FP8_E4M3 || F == KVQ_FP8_E5M2) {
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(dat + r * a.D + blk * 16));
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
      const float s = s_kv;
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
      const uint2 c = __ldg(reinterpret_cast<const uint2*>(dat + r * (a.D / 2) + blk * 8));
      const uint32_t sc = scl[r * nb + blk];
      const float S = (F == KVQ_FP4_BLOCK16) ? dec_e8m0(sc) : __fmul_rn(dec_e4m3(sc), s_kv);
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

inline int log2_if_pow2(int v) {
  if (v <= 0 || (v & (v - 1))) return -1;
  int k = 0;
  while ((1 << k) < v) ++k;
  return k;
}

// Resident waves' worth of store CTAs (K and V halves together), never more
// CTAs than there are items: eight for bf16 and FP8 (bf16 at one wave reaches
// 0.72 of the copy bandwidth, at eight 0.97; FP8 at four 0.956, at eight
// 0.998), four for the FP4 formats (NVFP4 at sixteen 0.760, eight 0.798, four
// 0.810, two 0.802).
template <kvq_format F, bool PH, int BPI>
cudaError_t launch_store_bpi(StoreArgs a, int64_t blocks, cudaStream_t stream) {
  a.ib = a.hb / BPI;
  a.nbi = a.nb / BPI;
  a.nbi_shift = log2_if_pow2(a.nbi);
  const int64_t items = blocks / BPI;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, store_kernel<F, PH, BPI>, 256, 0);
  if (e != cudaSuccess) return e;
  constexpr int kWaves = (F == KVQ_FP4_BLOCK16 || F == KVQ_NVFP4) ? 4 : 8;
  const int64_t wave = std::max<int64_t>(1, (int64_t)sms * std::max(per_sm, 1) * kWaves / 2);
  const int64_t need = (items + 255) / 256;
  dim3 grid((unsigned)std::min(wave, need), 2);
  store_kernel<F, PH, BPI><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// The quantizing formats: two blocks per item when the row has an even block
// count (measured on the 131072-token store: NVFP4 0.725 -> 0.811 of the copy
// bandwidth, FP4 block-16 0.867 -> 0.987, FP8 0.950 -> 0.998, with the
// grid sizes above)
template <kvq_format F, bool PH>
cudaError_t launch_store_as(const StoreArgs& a, int64_t blocks, cudaStream_t stream) {
  constexpr bool kPair = (F != KVQ_BF16);
  if (kPair && a.nb % 2 == 0) return launch_store_bpi<F, PH, kPair ? 2 : 1>(a, blocks, stream);
  return launch_store_bpi<F, PH, 1>(a, blocks, stream);
}


cudaError_t launch_store(const Geometry& g, const LayerView& L, const void* k, const void* v,
                         const int64_t* slots, int num_tokens, float s_k, float s_v,
                         const HeadScales& hs, int* err, cudaStream_t stream) {
  StoreArgs a;
  a.x[0] = static_cast<const uint16_t*>(k);
  a.x[1] = static_cast<const uint16_t*>(v);
  a.data[0] = L.k_data;
  a.data[1] = L.v_data;
  a.scales[0] = L.k_scales;
  a.scales[1] = L.v_scales;
  a.s[0] = s_k;
  a.s[1] = s_v;
  a.rs[0] = 1.0f / s_k;
  a.rs[1] = 1.0f / s_v;
  // NVFP4 block-scale divisor 6 g and its reciprocal (0: divide in IEEE
  // arithmetic, outside the range where the corrected quotient is exact)
  const float gs[2] = {s_k, s_v};
  for (int i = 0; i < 2; ++i) {
    a.s6[i] = 6.0f * gs[i];  // one fp32 product, as the quantization rule forms it
    a.rs6[i] = (a.s6[i] >= 0x1p-80f && a.s6[i] <= 0x1p80f) ? 1.0f / a.s6[i] : 0.f;
  }
  a.slots = slots;
  a.n = num_tokens;
  a.H = g.kv_heads;
  a.D = g.head_dim;
  a.P = g.page_size;
  a.nb = g.head_dim / 16;
  a.nb_shift = log2_if_pow2(a.nb);
  a.p_shift = log2_if_pow2(g.page_size);
  a.hb = a.H * a.nb;
  const float lo = 0x1p-80f, hi = 0x1p80f;
  a.fast_div = s_k >= lo && s_k <= hi && s_v >= lo && s_v <= hi;
  a.num_pages = g.num_pages;
  a.err = err;
  const int64_t items = (int64_t)num_tokens * a.hb;
  if (items == 0) return cudaSuccess;
  a.hs[0] = hs.scale[0];
  a.hs[1] = hs.scale[1];
  a.hr[0] = hs.recip[0];
  a.hr[1] = hs.recip[1];
  const bool ph = hs.scale[0] != nullptr;
  switch (g.fmt) {
    case KVQ_BF16: return launch_store_as<KVQ_BF16, false>(a, items, stream);
    case KVQ_FP8_E4M3:
      return ph ? launch_store_as<KVQ_FP8_E4M3, true>(a, items, stream)
                : launch_store_as<KVQ_FP8_E4M3, false>(a, items, stream);
    case KVQ_FP8_E5M2:
      return ph ? launch_store_as<KVQ_FP8_E5M2, true>(a, items, stream)
                : launch_store_as<KVQ_FP8_E5M2, false>(a, items, stream);
    case KVQ_FP4_BLOCK16: return launch_store_as<KVQ_FP4_BLOCK16, false>(a, items, stream);
    case KVQ_NVFP4:
      return ph ? launch_store_as<KVQ_NVFP4, true>(a, items, stream)
                : launch_store_as<KVQ_NVFP4, false>(a, items, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_dequantize(const Geometry& g, const LayerView& L, const int64_t* slots,
                              int num_tokens, float s_k, float s_v, const HeadScales& hs,
                              void* k_out, void* v_out, int* err, cudaStream_t stream) {
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
  a.hs[0] = hs.scale[0];
  a.hs[1] = hs.scale[1];
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


// ---------------------------------------------------------------------------
// Query quantization of FP8-domain attention ("Quantized KV cache" (vLLM),
// FP8 KV cache overview: with an FP8 cache the attention can run in the FP8
// domain, the query quantized to FP8 too; Supported schemes: q_scale per
// tensor or per attention head).  One thread per 16 consecutive elements.
// ---------------------------------------------------------------------------
namespace {

struct QuantQueryArgs {
  const uint16_t* q;  // [rows][Hq][D] bf16
  uint8_t* codes;     // [rows][Hq][D]
  int64_t items;      // rows * Hq * D / 16
  int Hq, nb;         // q heads, 16-element blocks per head row
  int nqs;            // 1 or Hq
  float qs[kMaxQScales];
};

__global__ void __launch_bounds__(256) quantize_query_kernel(QuantQueryArgs a) {
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < a.items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int head = (int)((it / a.nb) % a.Hq);
    const float s = a.qs[a.nqs == 1 ? 0 : head];
    const float rs = 1.0f / s;
    const uint4* src = reinterpret_cast<const uint4*>(a.q + it * 16);
    const uint4 lo = __ldg(src), hi = __ldg(src + 1);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t m2 = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(w[i]));
    const float amax = __uint_as_float(max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu) << 16);
    const bool fast = s >= 0x1p-80f && s <= 0x1p80f && amax * rs < 1e37f;  // NaN: false
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      c[i] = quant2_e4m3(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u), s, rs, fast);
    *reinterpret_cast<uint4*>(a.codes + it * 16) =
        make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16), c[6] | (c[7] << 16));
  }
}

}  // namespace

cudaError_t launch_quantize_query(const void* q, int64_t rows, int num_q_heads, int head_dim,
                                  const float* q_scales, int num_q_scales, void* codes,
                                  cudaStream_t stream) {
  QuantQueryArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.codes = static_cast<uint8_t*>(codes);
  a.nb = head_dim / 16;
  a.Hq = num_q_heads;
  a.items = rows * num_q_heads * a.nb;
  a.nqs = num_q_scales;
  for (int i = 0; i < kMaxQScales; ++i) a.qs[i] = i < num_q_scales ? q_scales[i] : 1.0f;
  if (a.items == 0) return cudaSuccess;
  quantize_query_kernel<<<grid_for(a.items), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-head scales and calibration ("Quantized KV cache" (vLLM features page):
// Supported schemes -- one scale per kv head; Scale calibration approaches --
// scales estimated on the fly from a batch of tokens, then fixed).
// ---------------------------------------------------------------------------
namespace {

constexpr int kSetChunk = 64;  // heads per set-scales launch (values travel as arguments)

struct SetScalesArgs {
  float v[2][kSetChunk];  // K, V scales of heads h0 .. h0 + count - 1
  int H, h0, count;
  float* scale;
  float* recip;
};

__global__ void __launch_bounds__(2 * kSetChunk) set_scales_kernel(SetScalesArgs a) {
  const int kv = threadIdx.x / kSetChunk, j = threadIdx.x % kSetChunk;
  if (j < a.count) {
    const float s = a.v[kv][j];
    a.scale[kv * a.H + a.h0 + j] = s;
    a.recip[kv * a.H + a.h0 + j] = 1.0f / s;  // IEEE division
  }
}

constexpr int kCalSmemHeads = 1024;  // heads reduced in shared memory (more go to global atomics)

struct CalArgs {
  const uint16_t* x[2];  // K, V bf16 [n][H][D]
  int64_t n;
  int H, nb, hb;         // kv heads, 16-element blocks per row, H * nb
  int fixed;             // the grid's thread count is a multiple of hb
  unsigned* amax;        // [2][H] bf16 magnitude bits of the largest finite |x|
};

// Largest finite bf16 magnitude among 16 values, as its 16-bit pattern
// (non-finite values have magnitude patterns >= 0x7F80 and are dropped).
__device__ __forceinline__ uint32_t block_amax_finite(const uint4 lo, const uint4 hi) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t m = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t x = w[i] & 0x7FFF7FFFu;
    x &= ~__vcmpgeu2(x, 0x7F807F80u);
    m = __vmaxu2(m, x);
  }
  return max(m & 0xFFFFu, m >> 16);
}

__global__ void __launch_bounds__(256) calib_amax_kernel(CalArgs a) {
  __shared__ unsigned smax[kCalSmemHeads];
  const int kv = blockIdx.y;
  const int hsm = min(a.H, kCalSmemHeads);
  for (int i = threadIdx.x; i < hsm; i += blockDim.x) smax[i] = 0u;
  __syncthreads();
  const uint16_t* const x = kv ? a.x[1] : a.x[0];
  unsigned* const gmax = a.amax + (size_t)kv * a.H;
  const long long items = a.n * a.hb;
  const long long row = (long long)a.hb * 16;  // elements per token
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (a.fixed) {
    // the thread's block column (head and block) is the same for every token
    // it visits: keep the maximum in a register, one atomic at the end
    const int pair = (int)(g % a.hb);
    const long long tstep = (long long)gridDim.x * blockDim.x / a.hb;
    const uint16_t* src = x + (g / a.hb) * row + (long long)pair * 16;
    const long long sstep = tstep * row;
    uint32_t m = 0u;
#pragma unroll 4
    for (long long tok = g / a.hb; tok < a.n; tok += tstep, src += sstep) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      m = max(m, block_amax_finite(__ldg(s4), __ldg(s4 + 1)));
    }
    const int h = pair / a.nb;
    if (m != 0u) {
      if (h < kCalSmemHeads) atomicMax(&smax[h], m);
      else atomicMax(gmax + h, m);
    }
  }
  for (long long it = a.fixed ? items : g; it < items; it += (long long)gridDim.x * blockDim.x) {
    const long long tok = it / a.hb;
    const int pair = (int)(it - tok * a.hb);
    const int h = pair / a.nb;
    const uint4* src = reinterpret_cast<const uint4*>(x + tok * row + (long long)pair * 16);
    const uint32_t m = block_amax_finite(__ldg(src), __ldg(src + 1));
    if (m != 0u) {
      if (h < kCalSmemHeads) atomicMax(&smax[h], m);
      else atomicMax(gmax + h, m);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < hsm; i += blockDim.x)
    if (smax[i] != 0u) atomicMax(gmax + i, smax[i]);
}

// scale = amax / fmt_max (IEEE fp32 division), 1 when amax is 0; per tensor:
// the largest amax over the heads serves every head.  The amax words are left
// zero for the layer's next calibration (they start zero with the cache).
__global__ void __launch_bounds__(256) calib_finalize_kernel(unsigned* amax, int H,
                                                             bool per_head, float fmt_max,
                                                             float* scale, float* recip) {
  __shared__ unsigned tmax[2];
  if (threadIdx.x < 2) tmax[threadIdx.x] = 0u;
  __syncthreads();
  if (!per_head)
    for (int i = threadIdx.x; i < 2 * H; i += blockDim.x) atomicMax(&tmax[i / H], amax[i]);
  __syncthreads();
  for (int i = threadIdx.x; i < 2 * H; i += blockDim.x) {
    const unsigned bits = per_head ? amax[i] : tmax[i / H];
    const float am = __uint_as_float(bits << 16);
    const float sc = am > 0.f ? am / fmt_max : 1.0f;
    scale[i] = sc;
    recip[i] = 1.0f / sc;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2 * H; i += blockDim.x) amax[i] = 0u;
}

}  // namespace

cudaError_t launch_set_head_scales(float* scale, float* recip, const float* k, const float* v,
                                   int H, cudaStream_t stream) {
  for (int h0 = 0; h0 < H; h0 += kSetChunk) {
    SetScalesArgs a;
    a.H = H;
    a.h0 = h0;
    a.count = std::min(kSetChunk, H - h0);
    for (int j = 0; j < kSetChunk; ++j) {
      a.v[0][j] = j < a.count ? k[h0 + j] : 1.0f;
      a.v[1][j] = j < a.count ? v[h0 + j] : 1.0f;
    }
    a.scale = scale;
    a.recip = recip;
    set_scales_kernel<<<1, 2 * kSetChunk, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_calibrate(const Geometry& g, const void* k, const void* v, int n, bool per_head,
                             unsigned* amax_scratch, float* scale, float* recip,
                             cudaStream_t stream) {
  const float fmt_max = g.fmt == KVQ_FP8_E4M3 ? 448.0f
                        : g.fmt == KVQ_FP8_E5M2 ? 57344.0f
                                                : 6.0f * 448.0f;  // NVFP4: E2M1 max x E4M3 max
  // amax_scratch is zero here: zeroed with the cache, and again by every
  // finalize after it has read it
  cudaError_t e = cudaSuccess;
  CalArgs a;
  a.x[0] = static_cast<const uint16_t*>(k);
  a.x[1] = static_cast<const uint16_t*>(v);
  a.n = n;
  a.H = g.kv_heads;
  a.nb = g.head_dim / 16;
  a.hb = a.H * a.nb;
  a.amax = amax_scratch;
  const int64_t items = (int64_t)n * a.hb;
  if (items > 0) {
    // one resident wave of CTAs (K and V halves together), rounded down to a
    // multiple of the CTA count whose threads span whole token rows (hb
    // blocks each)
    int dev = 0, sms = 148, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, calib_amax_kernel, 256, 0)) != cudaSuccess)
      return e;
    int64_t unit = a.hb;
    for (int t = 0; t < 8 && unit % 2 == 0; ++t) unit /= 2;  // hb / gcd(hb, 256)
    const int64_t ctas = std::max<int64_t>(1, (int64_t)sms * std::max(per_sm, 1) / 2 / unit) * unit;
    a.fixed = ctas <= 65535;
    dim3 grid(a.fixed ? (unsigned)ctas : (unsigned)grid_for(items), 2);
    calib_amax_kernel<<<grid, 256, 0, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  calib_finalize_kernel<<<1, 256, 0, stream>>>(amax_scratch, g.kv_heads, per_head, fmt_max, scale,
                                               recip);
  return cudaGetLastError();
}

}  // namespace kvq
