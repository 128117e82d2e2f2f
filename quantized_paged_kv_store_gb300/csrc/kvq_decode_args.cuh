// kvq_decode_args.cuh -- launch arguments and helpers shared by the split-K
// decode kernel (kvq_decode.cu) and the merge kernel (kvq_merge.cu).
#pragma once

#include <cstdint>

namespace kvq {

constexpr int kHeadDim = 128;
constexpr int kTile = 16;     // tokens per tile
constexpr int kGroupMax = 8;  // q heads per unit
constexpr int kMaxQScales = 256;  // FP8-domain attention: q scales carried in the launch

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
  long long* prefix;  // [B + 1]: tiles of sequences before b (written by worker 0)
  int B, H, Hq, G, HG, max_pages, P;
  long long num_pages;
  int num_workers;
  float qscale;       // sm_scale * log2(e) * (k_scale | g_k | 1); without the factor if kfac
  float v_factor;     // v_scale | g_v | 1 (per tensor)
  int* err;
  const float* kfac;  // per-kv-head K scales (or null: per tensor)
  const float* vfac;  // per-kv-head V scales (or null)
  const int32_t* pt_rows;  // extend: page-table row of each query token b (or null: row b)
  int pt_nrows;            // rows of the page table when pt_rows is set
  int fault_wait;          // failure-detection test: each warp's first stage wait runs out
  int neg_q;               // sm_scale < 0: the query enters negated and qscale holds |sm_scale|
  int nqs;                 // FP8-domain attention: 1 (per tensor) or Hq q scales in qsc
  float qsc[kMaxQScales];  // FP8-domain attention: q_scale per tensor / per q head
};


// 2^x by the hardware approximation; results below 2^-126 flush to zero,
// which is harmless for softmax weights that small.
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Page-table row of query b: b itself for decode; for extend attention the
// row its q_seq entry names, or -1 if that is out of range.
__device__ __forceinline__ int pt_row_of(const DecodeArgs& a, int b) {
  if (!a.pt_rows) return b;
  const int r = __ldg(a.pt_rows + b);
  return (r >= 0 && r < a.pt_nrows) ? r : -1;
}

// Tiles of sequence (query) b (0 for an empty or invalid length or row).
__device__ __forceinline__ int tiles_of(const DecodeArgs& a, int b) {
  const int T = __ldg(a.seq_lens + b);
  if (pt_row_of(a, b) < 0) return 0;
  return (T > 0 && T <= a.max_pages * a.P) ? (T + kTile - 1) / kTile : 0;
}

// First tile of worker w (integer split of [0, total)).
__device__ __forceinline__ long long worker_start(long long total, int w, int nw) {
  return total * w / nw;
}


// Launches the merge kernel after the split kernel on `stream` (programmatic
// dependent launch: it starts while the split kernel drains).
cudaError_t launch_merge(const DecodeArgs& a, int64_t num_units, cudaStream_t stream);

}  // namespace kvq
