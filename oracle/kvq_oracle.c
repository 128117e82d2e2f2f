/*
 * kvq_oracle.c -- plain, slow CPU oracle for the quantized paged KV store.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * path: every format is decoded here from its bit definition and encoded by
 * an exhaustive nearest-value search, and attention is evaluated in fp64.
 *
 * Sources (web pages, cited by title and section):
 *   [QKV]   "Quantized KV Cache" (SGLang documentation, mirrored on the
 *           data-sketchers wiki): Supported formats / FP8 formats, FP4 formats;
 *           Scaling factors; Performance considerations / Memory savings.
 *   [TRAPS] "KV cache quantization: mechanism and traps" (hrletsgo.me):
 *           INT8, FP8, INT4: measured numbers; When to enable.
 *   [NVFP4] "SGLang PR #21954 analysis: NVFP4 KV cache" (secrett2633 blog):
 *           Code analysis 1 (fp4_kv_cache_quant_method.py), Review feedback.
 *   [VLLM]  "Quantized KV cache" (vLLM features page on the data-sketchers
 *           wiki): Supported schemes; Scale calibration approaches.
 *   The formats themselves are the OCP 8-bit floating point (OFP8) and OCP
 *   Microscaling (MX) v1.0 definitions that [QKV] names.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   R1  E4M3 is the "fn" variant (bias 7, no infinities, S.1111.111 = NaN,
 *       max 448).  [QKV] prints +-240 for E4M3, the maximum of the IEEE-style
 *       variant; the target format of this library is E4M3fn.
 *   R2  Encoding is round-to-nearest, ties to the even code, with saturation
 *       to the largest finite magnitude (values at or beyond it, including
 *       +-Inf, give +-max).  The sign bit is copied from the input, so -0 and
 *       negatives that round to zero give the sign-set zero code.  NaN gives
 *       0x7F with the input's sign for both FP8 formats.
 *   R3  FP8 quantization divides in IEEE fp32: code = enc(x / s).
 *   R4  FP4 block-16 (E2M1 + E8M0): E = clamp(floor(log2(amax)) - 2, -127, 127),
 *       the MX v1.0 shared-exponent rule with emax(E2M1) = 2 applied to a
 *       16-element block; amax == 0 gives E = -127.  Codes: enc(x * 2^-E).
 *   R5  NVFP4: g is the per-tensor fp32 global scale.  Block scale code
 *       sc = enc_E4M3(amax / (6 * g)) (fp32 ops, RNE); S = dec(sc) * g (fp32);
 *       S == 0 gives all-zero codes (0x0); otherwise codes = enc_E2M1(x / S).
 *   R6  FP4 packing: even head_dim index in the low nibble, odd in the high.
 *   R7  Layout: data rows at [page][kv_head][token_in_page][head_dim] and a
 *       separate scale plane [page][kv_head][token_in_page][head_dim / 16].
 *   R8  Dequantize: out = bf16_RNE(fp32(dec(code) * S)).
 *   R9  Attention: q head j reads kv head floor(j / G), G = Hq / Hkv; a
 *       sequence of length 0 gives an all-zero output.
 *   R15 Per-attention-head scales ([VLLM] Supported schemes): the FP8
 *       scale (and the NVFP4 global scale) of kv head h is scales[h] of K or
 *       V; per-tensor scales are the case where every head has the same one.
 *   R16 Calibration from a batch of K or V rows ([VLLM] Scale calibration
 *       approaches, random-token mode; [QKV] Scaling factors): amax over the
 *       finite values (per tensor, or per kv head); scale = amax / M in fp32
 *       with M = 448 (E4M3), 57344 (E5M2), 6 * 448 = 2688 (NVFP4 global scale,
 *       so the largest block scale lands on the E4M3 maximum); amax == 0
 *       gives 1.0, the pages' default scale.
 *   R17 FP8-domain attention ([VLLM] FP8 KV cache overview; Supported
 *       schemes): the query is quantized to E4M3 with q_scale (per tensor or
 *       per q head) by the R2/R3 rule; attention is then exact over the
 *       dequantized query (the softmax weights are not quantized).
 *   Non-finite K/V values are outside the contract for the FP4 formats.
 *
 * Parity pins: R4 and R5 are this library's own definitions; the pages give
 * no worked example of either, so their parity against the pages is
 * "parity unpinned" beyond the invariants the tests check.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -ffp-contract=off (no fused
 * multiply-add may change an fp32 rounding that decides a code).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Format numbering used by this oracle's entry points (same meaning as the
 * names "bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4" from
 * [QKV] Usage). */
enum { ORC_BF16 = 0, ORC_E4M3 = 1, ORC_E5M2 = 2, ORC_FP4B16 = 3, ORC_NVFP4 = 4 };

/* ------------------------------------------------------------------------ */
/* Decoding from the bit definitions                                         */
/* ------------------------------------------------------------------------ */

/* E4M3fn: s eeee mmm, bias 7.  e == 0: subnormal m/8 * 2^-6.
 * S.1111.111 is NaN; there is no infinity.  Max finite 0x7E = 448. */
double orc_dec_e4m3(uint32_t code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 0xF, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = (m / 8.0) * ldexp(1.0, -6);
  else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
  return s ? -v : v;
}

/* E5M2: s eeeee mm, bias 15 (IEEE-like).  e == 0: m/4 * 2^-14.
 * e == 31: m == 0 is +-Inf, otherwise NaN.  Max finite 0x7B = 57344. */
double orc_dec_e5m2(uint32_t code) {
  int s = (code >> 7) & 1, e = (code >> 2) & 0x1F, m = code & 3;
  double v;
  if (e == 31) v = (m == 0) ? INFINITY : NAN;
  else if (e == 0) v = (m / 4.0) * ldexp(1.0, -14);
  else v = (1.0 + m / 4.0) * ldexp(1.0, e - 15);
  return s ? -v : v;
}

/* E2M1 (4 bits): s ee m, bias 1.  e == 0: m * 0.5.  Max 0x7 = 6. */
double orc_dec_e2m1(uint32_t code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double v;
  if (e == 0) v = m * 0.5;
  else v = (1.0 + m / 2.0) * ldexp(1.0, e - 1);
  return s ? -v : v;
}

/* E8M0 (unsigned power of two): 2^(c - 127); 0xFF is NaN. */
double orc_dec_e8m0(uint32_t code) {
  if ((code & 0xFF) == 0xFF) return NAN;
  return ldexp(1.0, (int)(code & 0xFF) - 127);
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double orc_dec_bf16(uint32_t bits) {
  uint32_t u = (bits & 0xFFFFu) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------------------------ */
/* Encoding: exhaustive nearest search, ties to the even code (R2)           */
/* ------------------------------------------------------------------------ */


/* Decode tables of the non-negative codes, filled once from the bit-level
 * decoders above; the encoders search them exhaustively. */
static double tab_e4m3[0x7F], tab_e5m2[0x7C], tab_e2m1[0x8];

__attribute__((constructor)) static void build_tables(void) {
  for (uint32_t c = 0; c <= 0x7E; ++c) tab_e4m3[c] = orc_dec_e4m3(c);
  for (uint32_t c = 0; c <= 0x7B; ++c) tab_e5m2[c] = orc_dec_e5m2(c);
  for (uint32_t c = 0; c <= 0x7; ++c) tab_e2m1[c] = orc_dec_e2m1(c);
}

/* Nearest non-negative code to magnitude a among codes [0, max_code]
 * (all finite, increasing with the code), ties to the even code. */
static uint32_t nearest_code(double a, const double* tab, uint32_t max_code) {
  uint32_t lo = 0, hi = max_code, c;
  if (a >= tab[max_code]) return max_code;   /* saturate (satfinite) */
  /* lo = largest code with value <= a, hi = smallest code with value >= a */
  for (c = 0; c <= max_code; ++c)
    if (tab[c] <= a && tab[c] >= tab[lo]) lo = c;
  for (c = max_code + 1; c-- > 0;)
    if (tab[c] >= a && tab[c] <= tab[hi]) hi = c;
  if (tab[lo] == a) return lo;
  {
    double mid = 0.5 * (tab[lo] + tab[hi]);  /* exact: both have few bits */
    if (a < mid) return lo;
    if (a > mid) return hi;
    return (lo & 1u) ? hi : lo;              /* tie: even mantissa */
  }
}

static uint32_t enc_fp8(double v, const double* tab, uint32_t max_code) {
  uint32_t sign = signbit(v) ? 0x80u : 0u;
  if (isnan(v)) return 0x7Fu | sign;
  return nearest_code(fabs(v), tab, max_code) | sign;
}

uint32_t orc_enc_e4m3(double v) { return enc_fp8(v, tab_e4m3, 0x7E); }
uint32_t orc_enc_e5m2(double v) { return enc_fp8(v, tab_e5m2, 0x7B); }

/* E2M1 has no NaN; NaN inputs are outside the contract (mapped to +-6). */
uint32_t orc_enc_e2m1(double v) {
  uint32_t sign = signbit(v) ? 0x8u : 0u;
  if (isnan(v)) return 0x7u | sign;
  return nearest_code(fabs(v), tab_e2m1, 0x7) | sign;
}

/* bfloat16 round-to-nearest-even of a binary32 value.  The two candidates are
 * the truncation of the value and the next bfloat16 away from zero; an
 * overflow past the largest finite value rounds to infinity as in IEEE.
 * Any NaN gives the canonical quiet NaN 0x7FC0 (the sign of a NaN produced by
 * arithmetic is not portable, so it is not part of the contract). */
uint32_t orc_enc_bf16(float v) {
  uint32_t u, lo, hi;
  double a, alo, ahi, mid;
  memcpy(&u, &v, sizeof u);
  if (isnan(v)) return 0x7FC0u;
  lo = u >> 16;
  if ((u & 0xFFFFu) == 0) return lo;
  hi = lo + 1;
  a = fabs((double)v);
  alo = fabs(orc_dec_bf16(lo));
  ahi = ((hi & 0x7FFFu) == 0x7F80u) ? ldexp(1.0, 128) : fabs(orc_dec_bf16(hi));
  mid = 0.5 * (alo + ahi);
  if (a < mid) return lo;
  if (a > mid) return hi;
  return (lo & 1u) ? hi : lo;
}

/* ------------------------------------------------------------------------ */
/* Cache geometry (R7)                                                       */
/* ------------------------------------------------------------------------ */

/* Bytes of one (page, kv_head, token) data row. */
static size_t data_row_bytes(int fmt, int D) {
  switch (fmt) {
    case ORC_BF16: return (size_t)D * 2;
    case ORC_E4M3:
    case ORC_E5M2: return (size_t)D;
    default: return (size_t)D / 2;
  }
}

static int has_block_scales(int fmt) { return fmt == ORC_FP4B16 || fmt == ORC_NVFP4; }

/* KV bytes per token for a model ([TRAPS] "When to enable": 2 (K and V) x
 * layers x kv_heads x head_dim x element bytes); the block formats add one
 * scale byte per 16 elements ([QKV] Memory savings: FP4 block 16 with an
 * 8-bit scale is 4.5 bits per element). */
int64_t orc_bytes_per_token(int fmt, int layers, int kv_heads, int head_dim) {
  int64_t per_head = (int64_t)data_row_bytes(fmt, head_dim);
  if (has_block_scales(fmt)) per_head += head_dim / 16;
  return 2LL * layers * kv_heads * per_head;
}

/* ------------------------------------------------------------------------ */
/* Quantize-and-store (R3-R7)                                                */
/* ------------------------------------------------------------------------ */

/*
 * k, v: bf16 bits [num_tokens][H][D].  slots[i] = page * P + offset, or -1
 * to skip token i.  scales: [2][H] (K heads, then V heads): FP8 scales or
 * NVFP4 global scales per kv head (R15), NULL for 1.0; ignored by bf16 and
 * FP4 block-16.  Writes the data rows and (block formats) scale rows.
 * Returns 0, or -1 if a slot is out of range (that token is skipped).
 */
static int store_one(int fmt, int H, int D, int P, int64_t num_pages, const uint16_t* x,
                     const int64_t* slots, int num_tokens, const float* sh, uint8_t* data,
                     uint8_t* scl) {
  int bad = 0;
  size_t drow = data_row_bytes(fmt, D), srow = (size_t)D / 16;
  /* tokens are independent when their slots are distinct (duplicate slots in
   * one call leave unspecified which token's row is stored) */
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int i = 0; i < num_tokens; ++i) {
    int64_t slot = slots[i];
    if (slot < 0) continue;
    if (slot >= num_pages * P) { bad = 1; continue; }
    int64_t page = slot / P, off = slot % P;
    for (int h = 0; h < H; ++h) {
      const float s = sh[h];                             /* R15: scale of kv head h */
      const uint16_t* row = x + ((size_t)i * H + h) * D;
      size_t r = ((size_t)page * H + h) * P + (size_t)off;
      uint8_t* out = data + r * drow;
      uint8_t* so = scl ? scl + r * srow : NULL;
      if (fmt == ORC_BF16) {
        memcpy(out, row, (size_t)D * 2);
      } else if (fmt == ORC_E4M3 || fmt == ORC_E5M2) {
        for (int d = 0; d < D; ++d) {
          float xv = bf16_to_float(row[d]);
          float q = xv / s;                              /* R3: fp32 division */
          if (isnan(xv))                                 /* R2: sign taken from x */
            out[d] = (uint8_t)(0x7Fu | (signbit(xv) ? 0x80u : 0u));
          else
            out[d] = (uint8_t)(fmt == ORC_E4M3 ? orc_enc_e4m3(q) : orc_enc_e5m2(q));
        }
      } else {
        for (int b = 0; b < D / 16; ++b) {
          float amax = 0.0f;
          uint32_t codes[16];
          for (int e = 0; e < 16; ++e) {
            float a = fabsf(bf16_to_float(row[b * 16 + e]));
            if (a > amax) amax = a;
          }
          if (fmt == ORC_FP4B16) {
            int E;                                         /* R4 */
            if (amax == 0.0f) {
              E = -127;
            } else {
              int ex;
              (void)frexpf(amax, &ex);                      /* amax = m 2^ex, m in [0.5,1) */
              E = (ex - 1) - 2;                             /* floor(log2 amax) - emax(E2M1) */
              if (E < -127) E = -127;
              if (E > 127) E = 127;
            }
            so[b] = (uint8_t)(E + 127);
            float p2 = ldexpf(1.0f, -E);
            for (int e = 0; e < 16; ++e)
              codes[e] = orc_enc_e2m1(bf16_to_float(row[b * 16 + e]) * p2);
          } else {                                         /* NVFP4, R5 */
            float denom = 6.0f * s;
            float ratio = amax / denom;
            uint32_t sc = orc_enc_e4m3(ratio);
            float S = (float)orc_dec_e4m3(sc) * s;
            so[b] = (uint8_t)sc;
            for (int e = 0; e < 16; ++e)
              codes[e] = (S == 0.0f) ? 0u : orc_enc_e2m1(bf16_to_float(row[b * 16 + e]) / S);
          }
          for (int e = 0; e < 16; e += 2)                  /* R6: even d low nibble */
            out[b * 8 + e / 2] = (uint8_t)((codes[e] & 0xF) | ((codes[e + 1] & 0xF) << 4));
        }
      }
    }
  }
  return bad ? -1 : 0;
}

/* H ones (the scales when none are given); caller frees */
static float* ones_for(int H) {
  float* o = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
  for (int h = 0; h < H; ++h) o[h] = 1.0f;
  return o;
}

int orc_quantize_store(int fmt, int H, int D, int P, int64_t num_pages, const uint16_t* k,
                       const uint16_t* v, const int64_t* slots, int num_tokens,
                       const float* scales, uint8_t* k_data, uint8_t* v_data, uint8_t* k_scl,
                       uint8_t* v_scl) {
  float* ones;
  int rk, rv;
  if (D % 16 != 0 || fmt < 0 || fmt > 4) return -2;
  ones = scales ? NULL : ones_for(H);
  rk = store_one(fmt, H, D, P, num_pages, k, slots, num_tokens, scales ? scales : ones,
                 k_data, has_block_scales(fmt) ? k_scl : NULL);
  rv = store_one(fmt, H, D, P, num_pages, v, slots, num_tokens, scales ? scales + H : ones,
                 v_data, has_block_scales(fmt) ? v_scl : NULL);
  free(ones);
  return (rk || rv) ? -1 : 0;
}

/* Calibration (R16): scale(s) from the amax of x [n][H][D] (bf16 bits) over
 * the finite values, per kv head (out[0..H-1]) or per tensor (out[0]). */
int orc_calibrate_scales(int fmt, int H, int D, const uint16_t* x, int n, int per_head,
                         float* out) {
  float M;
  if (fmt == ORC_E4M3) M = 448.0f;
  else if (fmt == ORC_E5M2) M = 57344.0f;
  else if (fmt == ORC_NVFP4) M = 6.0f * 448.0f;
  else M = 0.0f;                                     /* no per-tensor scale: 1.0 */
  for (int h = 0; h < (per_head ? H : 1); ++h) out[h] = 0.0f;
  for (int i = 0; i < n; ++i)
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d) {
        float a = fabsf(bf16_to_float(x[((size_t)i * H + h) * D + d]));
        float* o = &out[per_head ? h : 0];
        if (isfinite(a) && a > *o) *o = a;
      }
  for (int h = 0; h < (per_head ? H : 1); ++h)
    out[h] = (M > 0.0f && out[h] > 0.0f) ? out[h] / M : 1.0f;   /* fp32 division */
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization                                                            */
/* ------------------------------------------------------------------------ */

/* Exact real value of element d of a stored row (fp64; every product here is
 * exact in binary64).  Used by attention (fp64 path). */
static double element_value(int fmt, const uint8_t* drow, const uint8_t* srow, int d, float s) {
  switch (fmt) {
    case ORC_BF16: return orc_dec_bf16((uint32_t)drow[2 * d] | ((uint32_t)drow[2 * d + 1] << 8));
    case ORC_E4M3: return orc_dec_e4m3(drow[d]) * (double)s;
    case ORC_E5M2: return orc_dec_e5m2(drow[d]) * (double)s;
    default: {
      uint32_t nib = (d & 1) ? (drow[d / 2] >> 4) : (drow[d / 2] & 0xF);
      double e = orc_dec_e2m1(nib);
      if (fmt == ORC_FP4B16) return e * orc_dec_e8m0(srow[d / 16]);
      return e * orc_dec_e4m3(srow[d / 16]) * (double)s;
    }
  }
}

/* fp32 scale S of element d (R8). */
static float element_scale_f32(int fmt, const uint8_t* srow, int d, float s) {
  if (fmt == ORC_E4M3 || fmt == ORC_E5M2) return s;
  if (fmt == ORC_FP4B16) return (float)orc_dec_e8m0(srow[d / 16]);
  return (float)orc_dec_e4m3(srow[d / 16]) * s;
}

/* out = bf16_RNE(fp32(dec(code) * S)); slots < 0 give a zero row. */
static int dequant_one(int fmt, int H, int D, int P, int64_t num_pages, const uint8_t* data,
                       const uint8_t* scl, const int64_t* slots, int n, const float* sh,
                       uint16_t* out) {
  int bad = 0;
  size_t drow = data_row_bytes(fmt, D), srow = (size_t)D / 16;
  for (int i = 0; i < n; ++i) {
    int64_t slot = slots[i];
    int valid = slot >= 0 && slot < num_pages * P;
    if (slot >= 0 && !valid) bad = 1;
    for (int h = 0; h < H; ++h) {
      const float s = sh[h];
      uint16_t* o = out + ((size_t)i * H + h) * D;
      if (!valid) { memset(o, 0, (size_t)D * 2); continue; }
      size_t r = ((size_t)(slot / P) * H + h) * P + (size_t)(slot % P);
      const uint8_t* dr = data + r * drow;
      const uint8_t* sr = scl ? scl + r * srow : NULL;
      for (int d = 0; d < D; ++d) {
        if (fmt == ORC_BF16) {
          o[d] = (uint16_t)(dr[2 * d] | (dr[2 * d + 1] << 8));
        } else {
          double code_val;
          if (fmt == ORC_E4M3) code_val = orc_dec_e4m3(dr[d]);
          else if (fmt == ORC_E5M2) code_val = orc_dec_e5m2(dr[d]);
          else code_val = orc_dec_e2m1((d & 1) ? (dr[d / 2] >> 4) : (dr[d / 2] & 0xF));
          float prod = (float)code_val * element_scale_f32(fmt, sr, d, s);  /* fp32 product */
          o[d] = (uint16_t)orc_enc_bf16(prod);
        }
      }
    }
  }
  return bad ? -1 : 0;
}

int orc_dequantize(int fmt, int H, int D, int P, int64_t num_pages, const uint8_t* k_data,
                   const uint8_t* v_data, const uint8_t* k_scl, const uint8_t* v_scl,
                   const float* scales, const int64_t* slots, int n, uint16_t* k_out,
                   uint16_t* v_out) {
  float* ones = scales ? NULL : ones_for(H);
  int bs = has_block_scales(fmt);
  int rk = dequant_one(fmt, H, D, P, num_pages, k_data, bs ? k_scl : NULL, slots, n,
                       scales ? scales : ones, k_out);
  int rv = dequant_one(fmt, H, D, P, num_pages, v_data, bs ? v_scl : NULL, slots, n,
                       scales ? scales + H : ones, v_out);
  free(ones);
  return (rk || rv) ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention in fp64 (R9)                                             */
/* ------------------------------------------------------------------------ */

/*
 * Attention core over exact query values qv: fp64 [B][Hq][D].
 * page_table: int32 [B][max_pages]; token t of sequence b lives in page
 * page_table[b][t / P] at offset t % P.  For every b in b_list (or every b
 * when b_list is NULL) and every q head j:
 *   z_t = sm_scale * sum_d qv[b][j][d] * K^[t][d],  t < seq_lens[b]
 *   out[b][j][:] = sum_t softmax(z)_t * V^[t][:]
 * with K^, V^ the exact dequantized values (scales [2][H] as for the store).
 * Output rows of sequences not in b_list are left untouched.  Returns 0, or
 * -1 if a page id or length is out of range (the affected rows are set to
 * zero).
 */
static int attention_core(int fmt, int H, int D, int P, int64_t num_pages, const uint8_t* k_data,
                          const uint8_t* v_data, const uint8_t* k_scl, const uint8_t* v_scl,
                          const float* scales, const double* qv, int Hq,
                          const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                          int B, const int32_t* b_list, int nb, double sm_scale, double* out) {
  int G, bad = 0;
  int nsel = b_list ? nb : B;
  size_t drow = data_row_bytes(fmt, D), srow = (size_t)D / 16;
  int bs = has_block_scales(fmt);
  if (H <= 0 || Hq % H != 0) return -2;
  G = Hq / H;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t w = 0; w < (int64_t)nsel * H; ++w) {
    int b = b_list ? b_list[w / H] : (int)(w / H);
    int h = (int)(w % H);
    const float sk = scales ? scales[h] : 1.0f, sv = scales ? scales[H + h] : 1.0f;  /* R15 */
    int T = seq_lens[b];
    double* z = NULL;
    double* kv = (double*)malloc(sizeof(double) * (size_t)D);
    double* acc = (double*)calloc((size_t)G * D, sizeof(double));
    double* m = (double*)malloc(sizeof(double) * (size_t)G);
    double* l = (double*)calloc((size_t)G, sizeof(double));
    const double* qd = qv + ((size_t)b * Hq + (size_t)h * G) * D;   /* the group's G heads */
    int ok = 1;
    if (T < 0 || T > max_pages * P) ok = 0;
    if (ok && T > 0) z = (double*)malloc(sizeof(double) * (size_t)G * T);
    /* pass 1: logits */
    for (int t = 0; ok && t < T; ++t) {
      int32_t page = page_table[(size_t)b * max_pages + t / P];
      if (page < 0 || page >= num_pages) { ok = 0; break; }
      size_t r = ((size_t)page * H + h) * P + (size_t)(t % P);
      for (int d = 0; d < D; ++d)
        kv[d] = element_value(fmt, k_data + r * drow, bs ? k_scl + r * srow : NULL, d, sk);
      for (int g = 0; g < G; ++g) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[g * D + d] * kv[d];
        z[(size_t)g * T + t] = sm_scale * dot;
      }
    }
    /* softmax weights */
    for (int g = 0; ok && g < G; ++g) {
      m[g] = -INFINITY;
      for (int t = 0; t < T; ++t)
        if (z[(size_t)g * T + t] > m[g]) m[g] = z[(size_t)g * T + t];
      for (int t = 0; t < T; ++t) {
        double e = exp(z[(size_t)g * T + t] - m[g]);
        z[(size_t)g * T + t] = e;
        l[g] += e;
      }
    }
    /* pass 2: weighted sum of values */
    for (int t = 0; ok && t < T; ++t) {
      int32_t page = page_table[(size_t)b * max_pages + t / P];
      size_t r = ((size_t)page * H + h) * P + (size_t)(t % P);
      for (int d = 0; d < D; ++d)
        kv[d] = element_value(fmt, v_data + r * drow, bs ? v_scl + r * srow : NULL, d, sv);
      for (int g = 0; g < G; ++g) {
        double wgt = z[(size_t)g * T + t];
        for (int d = 0; d < D; ++d) acc[g * D + d] += wgt * kv[d];
      }
    }
    for (int g = 0; g < G; ++g) {
      double* o = out + ((size_t)b * Hq + (size_t)h * G + g) * D;
      for (int d = 0; d < D; ++d) o[d] = (ok && T > 0) ? acc[g * D + d] / l[g] : 0.0;
    }
    if (!ok) bad = 1;
    free(z); free(kv); free(acc); free(m); free(l);
  }
  return bad ? -1 : 0;
}

/* Decode attention of a bf16 query q: bits [B][Hq][D] (R9); see attention_core. */
int orc_decode_attention(int fmt, int H, int D, int P, int64_t num_pages, const uint8_t* k_data,
                         const uint8_t* v_data, const uint8_t* k_scl, const uint8_t* v_scl,
                         const float* scales, const uint16_t* q, int Hq,
                         const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                         int B, const int32_t* b_list, int nb, double sm_scale, double* out) {
  size_t n = (size_t)B * Hq * D;
  double* qv = (double*)malloc(sizeof(double) * (n ? n : 1));
  int rc;
  for (size_t i = 0; i < n; ++i) qv[i] = orc_dec_bf16(q[i]);
  rc = attention_core(fmt, H, D, P, num_pages, k_data, v_data, k_scl, v_scl, scales, qv, Hq,
                      page_table, max_pages, seq_lens, B, b_list, nb, sm_scale, out);
  free(qv);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Attention in the FP8 domain with a quantized query (R17)                  */
/* ------------------------------------------------------------------------ */

/*
 * [VLLM] FP8 KV cache overview: with an FP8 cache on the Flash Attention 3
 * backend the attention itself runs in the quantized (FP8) domain and the
 * query is quantized to FP8 as well; Supported schemes: q_scale is one value
 * per tensor ([1]) or one per attention head ([num_heads]).
 * R17: the query is quantized like the cache's FP8 E4M3 store (R2, R3):
 *   code = enc_E4M3(q / q_scale) (fp32 division, nearest, ties to even,
 *   saturating; NaN gives 0x7F with its sign), q_scale = q_scales[0] for
 *   nq == 1, else q_scales[j] for q head j.
 * q: bf16 bits [rows][Hq][D]; codes: [rows][Hq][D] bytes.
 */
int orc_quantize_query(const uint16_t* q, int64_t rows, int Hq, int D, const float* q_scales,
                       int nq, uint8_t* codes) {
  if (nq != 1 && nq != Hq) return -2;
  for (int64_t i = 0; i < rows * Hq; ++i) {
    const float s = q_scales[nq == 1 ? 0 : (int)(i % Hq)];
    for (int d = 0; d < D; ++d) {
      float x = bf16_to_float(q[i * D + d]);
      float y = x / s;                                         /* R3: fp32 division */
      codes[i * D + d] = isnan(x) ? (uint8_t)(0x7Fu | (signbit(x) ? 0x80u : 0u))
                                  : (uint8_t)orc_enc_e4m3(y);
    }
  }
  return 0;
}

/* Decode attention with the query quantized by orc_quantize_query: the same
 * attention over the exact query values dec_E4M3(code) * q_scale (fp64). */
int orc_decode_attention_fp8q(int fmt, int H, int D, int P, int64_t num_pages,
                              const uint8_t* k_data, const uint8_t* v_data, const uint8_t* k_scl,
                              const uint8_t* v_scl, const float* scales, const uint16_t* q,
                              const float* q_scales, int nq, int Hq, const int32_t* page_table,
                              int max_pages, const int32_t* seq_lens, int B, const int32_t* b_list,
                              int nb, double sm_scale, double* out) {
  size_t n = (size_t)B * Hq * D;
  uint8_t* codes = (uint8_t*)malloc(n ? n : 1);
  double* qv = (double*)malloc(sizeof(double) * (n ? n : 1));
  int rc = orc_quantize_query(q, B, Hq, D, q_scales, nq, codes);
  if (rc == 0) {
    for (size_t i = 0; i < n; ++i) {
      const size_t j = (i / (size_t)D) % (size_t)Hq;
      qv[i] = orc_dec_e4m3(codes[i]) * (double)q_scales[nq == 1 ? 0 : j];
    }
    rc = attention_core(fmt, H, D, P, num_pages, k_data, v_data, k_scl, v_scl, scales, qv, Hq,
                        page_table, max_pages, seq_lens, B, b_list, nb, sm_scale, out);
  }
  free(codes);
  free(qv);
  return rc;
}

/* Threads the OpenMP runtime will use (reported beside timings). */
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Sets the OpenMP thread count of later calls (n >= 1), for single-thread
 * timings of the baseline; returns the count now in effect. */
int orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
  return orc_num_threads();
}
