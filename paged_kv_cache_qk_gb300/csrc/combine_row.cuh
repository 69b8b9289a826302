// Log-sum-exp merge of split-KV partials for one output row (one warp),
// shared by the split and the balanced combine kernels.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, ...", section "概述 / Summary", item 1 ("splitkv"): the
// splits of a sequence each produce a normalised partial output o_j and its
// log-sum-exp lse_j; the merged row is sum_j w_j o_j / sum_j w_j with
// w_j = exp(lse_j - max_k lse_k).  Lane l owns dims [4l, 4l+4); lane j
// computes split j's weight once and the others get it by shuffle; eight
// float4 partial loads are kept in flight per lane.
#pragma once

#include "device_common.cuh"

namespace pkvqk {

constexpr float kLog2e = 1.4426950408889634f;

// Merge of n partial rows at ws index base + j * stride (j < n) into one
// bf16 output row (+ lse); one warp.  The partials come from the previous
// kernel in the stream, so the read-only path may cache them.
__device__ __forceinline__ void combine_row(const float* __restrict__ ws_o,
                                            const float* __restrict__ ws_lse, long long base,
                                            long long stride, int n, __nv_bfloat16* out_row,
                                            float* lse_dst, int lane) {
  auto ld_part = [](const float* ptr) { return __ldg(ptr); };
  auto ld_part4 = [](const float4* ptr) { return __ldg(ptr); };
  // pass 1: the row's max lse (lane j holds split j, j + 32, ...)
  float M = -INFINITY;
  for (int j = lane; j < n; j += 32) M = fmaxf(M, ld_part(ws_lse + base + j * stride));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  // pass 2: weights in the lanes that own the splits, partial rows summed
  // with 8 independent float4 loads in flight per lane
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int jl = j0 + lane;
      const float lj = jl < n ? ld_part(ws_lse + base + jl * stride) : -INFINITY;
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
                     ? ld_part4(reinterpret_cast<const float4*>(ws_o + idx * kHeadDim + 4 * lane))
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


}  // namespace pkvqk
