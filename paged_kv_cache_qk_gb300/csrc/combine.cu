// Log-sum-exp merge of split-KV partials.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, ...", section "概述 / Summary", item 1 ("splitkv"): the
// splits of a sequence each produce a normalised partial output o_j and its
// log-sum-exp lse_j; the merged row is sum_j w_j o_j / sum_j w_j with
// w_j = exp(lse_j - max_k lse_k).
//
// One warp per output row; lane l owns dims [4l, 4l+4) and reads each split's
// partial as one float4 (a warp reads a 512-byte partial row per split).
#include "device_common.cuh"
#include "kernels.h"

namespace pkvqk {

namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(kWarps * 32)
lse_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, int rows,
                   int S, __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* lse = ws_lse + row * S;

  float M = -INFINITY;
  for (int j = lane; j < S; j += 32) M = fmaxf(M, __ldg(lse + j));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    const float* o = ws_o + row * S * static_cast<int64_t>(kHeadDim) + 4 * lane;
    for (int j = 0; j < S; ++j) {
      const float lj = __ldg(lse + j);
      const float w = (lj == -INFINITY) ? 0.f : exp2f((lj - M) * kLog2e);
      wsum += w;
      if (w != 0.f) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(o + j * kHeadDim));
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
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
  lse_combine_kernel<<<blocks, kWarps * 32, 0, stream>>>(ws_o, ws_lse, rows, num_splits, out,
                                                          lse_out);
  return cudaGetLastError();
}

}  // namespace pkvqk
