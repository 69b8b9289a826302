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
#include "device_common.cuh"
#include "kernels.h"

namespace pkvqk {

namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

// Merge of n partial rows at ws index base + j * stride (j < n) into one
// bf16 output row (+ lse); one warp.
__device__ __forceinline__ void combine_row(const float* __restrict__ ws_o,
                                            const float* __restrict__ ws_lse, long long base,
                                            long long stride, int n, __nv_bfloat16* out_row,
                                            float* lse_dst, int lane) {
  // pass 1: the row's max lse (lane j holds split j, j + 32, ...)
  float M = -INFINITY;
  for (int j = lane; j < n; j += 32) M = fmaxf(M, __ldg(ws_lse + base + j * stride));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  // pass 2: weights in the lanes that own the splits, partial rows summed
  // with 8 independent float4 loads in flight per lane
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int jl = j0 + lane;
      const float lj = jl < n ? __ldg(ws_lse + base + jl * stride) : -INFINITY;
      const float wl = (lj == -INFINITY) ? 0.f : exp2f((lj - M) * kLog2e);
      wsum += wl;
      const int cnt = min(32, n - j0);
      for (int jj = 0; jj < cnt; jj += 8) {
        float4 v[8];
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wl, (jj + u) & 31);
          const long long idx = base + static_cast<long long>(j0 + jj + u) * stride;
          v[u] = (jj + u < cnt)
                     ? __ldg(reinterpret_cast<const float4*>(ws_o + idx * kHeadDim + 4 * lane))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float ww = (jj + u < cnt) ? w[u] : 0.f;
          acc.x = fmaf(ww, v[u].x, acc.x);
          acc.y = fmaf(ww, v[u].y, acc.y);
          acc.z = fmaf(ww, v[u].z, acc.z);
          acc.w = fmaf(ww, v[u].w, acc.w);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(out_row + 4 * lane) = packed;
  if (lane == 0 && lse_dst != nullptr) *lse_dst = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

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
