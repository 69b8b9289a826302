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

__global__ void __launch_bounds__(kWarps * 32)
lse_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, int rows,
                   int S, __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  pdl_launch_dependents();
  pdl_wait();                                   // the partials come from the decode kernel
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* lse = ws_lse + row * S;
  const float* o = ws_o + row * S * static_cast<int64_t>(kHeadDim) + 4 * lane;

  // pass 1: the row's max lse (lane j holds split j, j + 32, ...)
  float M = -INFINITY;
  for (int j = lane; j < S; j += 32) M = fmaxf(M, __ldg(lse + j));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  // pass 2: weights in the lanes that own the splits, partial rows summed
  // with 8 independent float4 loads in flight per lane
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int j0 = 0; j0 < S; j0 += 32) {
      const int jl = j0 + lane;
      const float lj = jl < S ? __ldg(lse + jl) : -INFINITY;
      const float wl = (lj == -INFINITY) ? 0.f : exp2f((lj - M) * kLog2e);
      wsum += wl;
      const int n = min(32, S - j0);
      for (int jj = 0; jj < n; jj += 8) {
        float4 v[8];
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wl, (jj + u) & 31);
          v[u] = (jj + u < n) ? __ldg(reinterpret_cast<const float4*>(o + (j0 + jj + u) *
                                                                             kHeadDim))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float ww = (jj + u < n) ? w[u] : 0.f;
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
  *reinterpret_cast<uint2*>(out + row * kHeadDim + 4 * lane) = packed;
  if (lane == 0 && lse_out != nullptr) lse_out[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_lse_combine(const float* ws_o, const float* ws_lse, int rows, int num_splits,
                               __nv_bfloat16* out, float* lse_out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int blocks = (rows + kWarps - 1) / kWarps;
  return launch_pdl(lse_combine_kernel, dim3(blocks), dim3(kWarps * 32), 0, stream, ws_o, ws_lse,
                    rows, num_splits, out, lse_out);
}

}  // namespace pkvqk
