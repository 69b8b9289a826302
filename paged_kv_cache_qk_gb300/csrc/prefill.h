// Internal launch interface of the multi-query (chunked-prefill) attention
// kernel.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkvqk {

// Packed (token, q head) rows of one kv head that one CTA covers.
constexpr int kPrefillRowsPerCta = 256;

struct PrefillArgs {
  const __nv_bfloat16* q;          // [tokens, Hq, 128] (strided tokens / heads)
  int64_t q_stride_t, q_stride_h;
  const int32_t* block_tables;     // [B, max_blocks_per_seq]
  int32_t max_blocks_per_seq;
  const int32_t* seq_lens;         // [B], counting the q_len new tokens
  int32_t batch, q_len, num_q_heads, num_kv_heads, group;
  // varlen: sequence b's new tokens are rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
  // of q/out (q_len is then their maximum); NULL: every sequence has q_len, at
  // rows b * q_len ..
  const int32_t* cu_seqlens_q;
  int64_t total_q;                 // rows of q/out (rows past it are never written)
  int32_t block_size;
  int64_t num_blocks;
  int32_t num_splits;              // >= 1
  int32_t chunk_pages;             // pages per split
  int32_t m_tiles;                 // ceil(q_len * group / kPrefillRowsPerCta)
  float scale_log2;                // softmax scale * log2(e)
  __nv_bfloat16* out;              // num_splits == 1: [tokens, Hq, 128]
  float* lse_out;                  // num_splits == 1: optional [tokens, Hq]
  float* ws_o;                     // num_splits > 1: [rows, S, 128] normalised partials
  float* ws_lse;                   // num_splits > 1: [rows, S]
  int32_t* status_flags;
  // set by launch_paged_prefill: q rows arrive by TMA through qmap, and whole
  // row tiles of out (num_splits == 1) leave by TMA through omap
  int32_t q_tma, o_tma;
  // set by launch_paged_prefill: the grid runs over (row tile descending,
  // sequence, kv head, split) instead of (sequence, split, kv head, row tile
  // descending)
  int32_t mt_major;
  int32_t group_shift;             // set by launch_paged_prefill: log2(group), or -1
};

// Shared-memory bytes one CTA of the kernel takes (one CTA per SM).
int prefill_smem_bytes();

// Tensor maps: 5-D cache views with a box of (64 dims, b slots, 1 half, 1 head,
// 1 block), b = the largest power of two dividing block_size, at most 128.
// The q and out row-tile maps are built here (where the layouts allow them).
cudaError_t launch_paged_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const PrefillArgs& a, cudaStream_t stream);

}  // namespace pkvqk
