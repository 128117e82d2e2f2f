// kvq_internal.h -- definitions shared by the host C-ABI and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "kvq.h"

namespace kvq {

// Bits of the device error word.
constexpr int kErrRange = 1;    // out-of-range slot, page id or sequence length
constexpr int kErrTimeout = 2;  // a bounded wait ran out

// Rows of one layer's pool: [num_pages][kv_heads][page_size][row bytes].
struct LayerView {
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_scales;  // nullptr unless the format has block scales
  uint8_t* v_scales;
};

struct Geometry {
  kvq_format fmt;
  int kv_heads;
  int head_dim;
  int page_size;
  int64_t num_pages;
  size_t data_row;   // bytes per token row of a data pool
  size_t scale_row;  // bytes per token row of a scale plane (0: none)
};

inline size_t data_row_bytes(kvq_format f, int head_dim) {
  switch (f) {
    case KVQ_BF16: return (size_t)head_dim * 2;
    case KVQ_FP8_E4M3:
    case KVQ_FP8_E5M2: return (size_t)head_dim;
    default: return (size_t)head_dim / 2;
  }
}
inline bool has_block_scales(kvq_format f) { return f == KVQ_FP4_BLOCK16 || f == KVQ_NVFP4; }

// Sets the thread-local message returned by kvq_last_error_string().
void set_error_message(const char* fmt, ...);

// Per-kv-head scales of one layer in device memory: scale[0] / scale[1] are
// the K / V scales ([kv_heads] floats each), recip the IEEE reciprocals.
// Null pointers select the per-tensor path (scalar scales in the launch).
struct HeadScales {
  const float* scale[2] = {nullptr, nullptr};
  const float* recip[2] = {nullptr, nullptr};
};

// ---- launchers (defined in the .cu files; return a CUDA error code) -------

cudaError_t launch_store(const Geometry& g, const LayerView& L, const void* k, const void* v,
                         const int64_t* slots, int num_tokens, float s_k, float s_v,
                         const HeadScales& hs, int* err, cudaStream_t stream);

cudaError_t launch_dequantize(const Geometry& g, const LayerView& L, const int64_t* slots,
                              int num_tokens, float s_k, float s_v, const HeadScales& hs,
                              void* k_out, void* v_out, int* err, cudaStream_t stream);

// Writes host-given per-head scales (k[H], v[H]) and their reciprocals into
// scale / recip ([2][H] each) with kernel launches on `stream` (the values
// travel as launch arguments, so the call is capturable in a CUDA graph).
cudaError_t launch_set_head_scales(float* scale, float* recip, const float* k, const float* v,
                                   int H, cudaStream_t stream);

// Calibration: amax over the finite values of bf16 K and V rows [n][H][D],
// per kv head or per tensor, turned into scale = amax / fmt_max (1 if amax is
// 0) and its reciprocal in scale / recip ([2][H]).  amax_scratch: 2 * H words,
// zero on entry and left zero (the calibration clears what it read).
cudaError_t launch_calibrate(const Geometry& g, const void* k, const void* v, int n, bool per_head,
                             unsigned* amax_scratch, float* scale, float* recip,
                             cudaStream_t stream);

// Extend attention (kvq_extend.cu): per 128 (query, q head) rows of a kv head
// and per split of each sequence's context, one pass over its K/V chunks on
// the tcgen05 tensor cores; with splits > 1 the workspace holds the partial
// outputs (extend_workspace_bytes) and a merge kernel combines them.
int extend_splits(const Geometry& g, int num_q_tokens, int num_q_heads, int max_pages_per_seq,
                  int device);
size_t extend_workspace_bytes(int splits, int num_q_tokens, int num_q_heads);
cudaError_t launch_extend(const Geometry& g, const LayerView& L, const void* q, int num_q_heads,
                          int num_q_tokens, const int32_t* q_seq, const int32_t* q_len,
                          const int32_t* page_table, int num_seqs, int max_pages_per_seq,
                          float sm_scale, float k_factor, float v_factor, const HeadScales& hs,
                          void* out, int* err, int splits, void* workspace, cudaStream_t stream);

// Decode attention plan: how many warp workers and how much workspace.
struct DecodePlan {
  int group;          // q heads per kv head (G)
  int head_groups;    // ceil(G / 8): units per (sequence, kv head)
  int num_workers;    // warps that share the page-tile range
  int ctas;           // thread blocks launched
  int64_t num_units;  // batch * kv_heads * head_groups
  int64_t num_slots;  // num_units + num_workers partial slots
  size_t ws_bytes;    // total workspace bytes
};

// Fills `plan` for a call; returns false (with a message) if unsupported.
// qf8: the FP8-domain attention kernel (FP8 caches only) will be launched.
bool plan_decode(const Geometry& g, int batch, int num_q_heads, int max_pages_per_seq,
                 int device, DecodePlan* plan, const char** why, bool qf8 = false);

// q_scales (host, num_q_scales = 1 or num_q_heads, <= 256) selects FP8-domain
// attention with the query quantized to E4M3; nullptr: the bf16 query path.
cudaError_t launch_decode(const Geometry& g, const LayerView& L, const DecodePlan& plan,
                          const void* q, int num_q_heads, const int32_t* page_table,
                          int max_pages_per_seq, const int32_t* seq_lens, int batch,
                          float sm_scale, float k_factor, float v_factor, const HeadScales& hs,
                          const int32_t* pt_rows, int pt_nrows, void* out, void* workspace,
                          int* err, cudaStream_t stream, const float* q_scales = nullptr,
                          int num_q_scales = 0);

// E4M3 codes of a bf16 query [rows][num_q_heads][head_dim] quantized with
// q_scales (host, 1 or num_q_heads, <= 256): the FP8-domain attention's rule.
cudaError_t launch_quantize_query(const void* q, int64_t rows, int num_q_heads, int head_dim,
                                  const float* q_scales, int num_q_scales, void* codes,
                                  cudaStream_t stream);

}  // namespace kvq
