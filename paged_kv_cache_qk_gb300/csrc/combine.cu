// Log-sum-exp merge of split-KV partials.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, ...", section "概述 / Summary", item 1 ("splitkv"): the
// splits of a sequence each produce a normalised partial output o_j and its
// log-sum-exp lse_j; the merged row is sum_j w_j o_j / sum_j w_j with
// w_j = exp(lse_j - max_k lse_k).
//
// One warp per output row; lane l owns dims [4l, 4l+4) and reads each split's
// partial as one float4 (a warp reads a 512-byte partial row per split, eight
// splits in flight).  Lane j computes split j's weight once; the others get it
// by shuffle.  Launched as a programmatic dependent of the decode kernel, so
// its launch overlaps the decode tail; it waits for the partials before
// reading them.
#include "combine_row.cuh"
#include "device_common.cuh"
#include "kernels.h"

namespace pkvqk {

namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
lse_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, int rows,
                   int S, __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  pdl_launch_dependents();
  pdl_wait();                                   // the partials come from the decode kernel
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  combine_row(ws_o, ws_lse, row * S, 1, S, out + row * kHeadDim,
              lse_out != nullptr ? lse_out + row : nullptr, lane);
}

// Balanced schedule: output row -> its (sequence, head group) unit; units cut
// across CTAs c_first..c_last left partials in slots c + unit, at row
// (t * HPC + hh) * group + gi of the slot.
__global__ void __launch_bounds__(kWarps * 32)
balanced_combine_kernel(const DecodeArgs a, int hpc) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(a.batch) * a.q_len * a.num_q_heads;
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int per_seq = a.q_len * a.num_q_heads;
  const int b = static_cast<int>(row / per_seq), rem = static_cast<int>(row % per_seq);
  const int t = rem / a.num_q_heads, h = rem % a.num_q_heads;
  const int kvh = h / a.group, gi = h % a.group;
  const int hg = kvh / hpc, hh = kvh % hpc;
  const int u = hg * a.batch + b;
  const int2 info = a.unit_info[u];
  if (info.x == info.y) return;                 // written whole by one CTA
  const long long srow = (t * hpc + hh) * a.group + gi;
  const long long base = (static_cast<long long>(info.x) + u) * a.rows_per_unit + srow;
  combine_row(a.ws_o, a.ws_lse, base, a.rows_per_unit, info.y - info.x + 1,
              a.out + row * kHeadDim, a.lse_out != nullptr ? a.lse_out + row : nullptr, lane);
}

}  // namespace

cudaError_t launch_lse_combine(const float* ws_o, const float* ws_lse, int rows, int num_splits,
                               __nv_bfloat16* out, float* lse_out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int blocks = (rows + kWarps - 1) / kWarps;
  return launch_pdl(lse_combine_kernel, dim3(blocks), dim3(kWarps * 32), 0, stream, ws_o, ws_lse,
                    rows, num_splits, out, lse_out);
}

cudaError_t launch_balanced_combine(const DecodeArgs& a, int heads_per_cta, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.batch) * a.q_len * a.num_q_heads;
  if (rows == 0) return cudaSuccess;
  const int blocks = static_cast<int>((rows + kWarps - 1) / kWarps);
  return launch_pdl(balanced_combine_kernel, dim3(blocks), dim3(kWarps * 32), 0, stream, a,
                    heads_per_cta);
}

}  // namespace pkvqk
