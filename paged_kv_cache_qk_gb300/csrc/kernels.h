// Internal launch interface between the C-ABI host layer (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkvqk {

struct NormRopeAppendArgs {
  __nv_bfloat16* q;
  int64_t q_stride_t, q_stride_h;
  const __nv_bfloat16* k;
  int64_t k_stride_t, k_stride_h;
  const __nv_bfloat16* v;
  int64_t v_stride_t, v_stride_h;
  const int64_t* positions;
  const int64_t* slot_mapping;
  const __nv_bfloat16* gamma_q;
  const __nv_bfloat16* gamma_k;
  float eps;
  double inv_freq[64];             // theta^(-2i/D), i < D/2, computed on the host in float64
  float sincos_tab[51][4];         // sin/cos(k/64) as float-float pairs (rope_math.cuh)
  int32_t num_tokens, num_q_heads, num_kv_heads;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  int64_t num_blocks;
  int32_t block_size;
  int64_t block_stride, slot_stride, head_stride;
  int32_t* status_flags;
  // optional: sin/cos of positions 0 .. table_positions-1 from
  // launch_rope_table_build (nullptr / 0: every token computes its own)
  const float4* rope_table;
  int32_t table_positions;
};

cudaError_t launch_norm_rope_append(const NormRopeAppendArgs& a, cudaStream_t stream);

// Fills table[pos][l][4] (l < 16: float4s cos_hi, cos_lo, sin_hi, sin_lo of
// frequencies 4l .. 4l+3) for pos < positions with the values the append
// kernel computes for a token at pos.
cudaError_t launch_rope_table_build(float4* table, int32_t positions, const double (&inv_freq)[64],
                                    const float (&sincos_tab)[51][4], cudaStream_t stream);

struct DecodeArgs {
  const __nv_bfloat16* q;
  int64_t q_stride_t, q_stride_h;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* seq_lens;
  int32_t batch, q_len, num_q_heads, num_kv_heads, group;
  int32_t block_size;
  int64_t num_blocks;
  int32_t num_splits;            // 0: balanced persistent schedule; >= 1: split schedule
  int32_t chunk_pages;           // split schedule: pages per split
  int32_t groups;                // kv-head groups (num_kv_heads / heads per CTA)
  int32_t rows_per_unit;         // q_len * heads per CTA * group: rows of one (seq, group)
  float scale_log2;              // softmax scale * log2(e)
  __nv_bfloat16* out;            // final bf16 output
  float* lse_out;                // optional final lse
  float* ws_o;                   // partial outputs (split / balanced schedules)
  float* ws_lse;                 // partial lse
  int2* unit_info;               // balanced: first and last CTA of every (seq, group) unit
  int32_t* status_flags;
};

// Kernel family chosen by the host for a decode call.
struct DecodePlan {
  int heads_per_cta;   // kv heads handled by one CTA (divides num_kv_heads)
  bool tensor_core;    // mma tiles (rows per kv head > 2) vs CUDA-core dots
  int rows;            // q_len * group
  int tile_keys;       // keys per TMA tile (8 or 16)
  int ctas_per_sm;     // resident CTAs per SM the shared-memory ring allows
};

DecodePlan plan_decode(int num_kv_heads, int rows);

// grid_ctas: CTAs of the balanced schedule (one per SM); unused otherwise.
cudaError_t launch_paged_decode(const DecodePlan& plan, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const DecodeArgs& a, int grid_ctas,
                                cudaStream_t stream);

cudaError_t launch_lse_combine(const float* ws_o, const float* ws_lse, int rows, int num_splits,
                               __nv_bfloat16* out, float* lse_out, cudaStream_t stream);

// Merge of the balanced schedule's partials (units cut across CTAs only).
cudaError_t launch_balanced_combine(const DecodeArgs& a, int heads_per_cta, cudaStream_t stream);

}  // namespace pkvqk
