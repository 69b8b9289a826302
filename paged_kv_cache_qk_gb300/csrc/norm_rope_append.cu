// Fused per-head RMSNorm + neox RoPE on q and k, with the k/v cache append.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, fused rms_norm_rope, ...", section "概述 / Summary",
// item 2 (per-head RMSNorm + full-rotary RoPE in one op) and item 1 (the
// BSHD paged cache the decode kernel reads).
//
// One CTA per token.  The token's 64 rotation angles are computed once, in
// float64 with an explicit 2*pi reduction (positions reach 3e4 rad, where a
// float32 angle would be off by ~2e-3 rad), then sin/cos of the reduced
// float32 angle go to shared memory for every head of the token.  Each head
// vector (D = 128 bf16 = 256 B) is handled by a half-warp: lane l holds
// elements [8l, 8l+8) as one 16-byte load; the sum of squares is a 4-step
// xor-shuffle reduction inside the half-warp, and the rotate-half partner of
// lane l is lane l ^ 8.
#include "device_common.cuh"
#include "kernels.h"

namespace pkvqk {

namespace {

constexpr int kThreads = 256;
constexpr double kTwoPi = 6.283185307179586476925286766559;

__global__ void __launch_bounds__(kThreads)
norm_rope_append_kernel(NormRopeAppendArgs a) {
  __shared__ float s_cos[kHeadDim / 2];
  __shared__ float s_sin[kHeadDim / 2];

  const int t = blockIdx.x;
  const int64_t pos = a.positions[t];
  const int64_t slot = a.slot_mapping[t];
  const int64_t nslots = a.num_blocks * static_cast<int64_t>(a.block_size);

  if (threadIdx.x < kHeadDim / 2) {
    const int i = threadIdx.x;
    const double inv_freq = pow(static_cast<double>(a.theta), -2.0 * i / kHeadDim);
    const double ang = static_cast<double>(pos) * inv_freq;
    const double turns = rint(ang * (1.0 / kTwoPi));
    const double red = fma(-turns, kTwoPi, ang);        // in [-pi, pi]
    float sn, cs;
    sincosf(static_cast<float>(red), &sn, &cs);
    s_cos[i] = cs;
    s_sin[i] = sn;
  }
  if (threadIdx.x == 0 && slot >= nslots) report(a.status_flags, kFlagBadSlot);
  __syncthreads();

  const bool write_cache = slot >= 0 && slot < nslots;
  const int64_t blk = write_cache ? slot / a.block_size : 0;
  const int64_t off = write_cache ? slot % a.block_size : 0;
  const int64_t cache_row = blk * a.block_stride + off * a.slot_stride;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;          // which vector of the warp's pair
  const int l = lane & 15;             // lane within the half-warp
  const int num_vec = a.num_q_heads + a.num_kv_heads;
  const float inv_d = 1.0f / kHeadDim;

  // warp-uniform trip count: both halves run every shuffle
  for (int base = warp * 2; base < num_vec; base += (kThreads / 32) * 2) {
    const int h = base + half;
    const bool active = h < num_vec;
    const bool is_q = h < a.num_q_heads;
    const int hk = h - a.num_q_heads;

    __nv_bfloat16* xrow;
    const __nv_bfloat16* gamma;
    if (is_q) {
      xrow = a.q + t * a.q_stride_t + static_cast<int64_t>(h) * a.q_stride_h;
      gamma = a.gamma_q;
    } else {
      xrow = const_cast<__nv_bfloat16*>(a.k) + t * a.k_stride_t +
             static_cast<int64_t>(hk) * a.k_stride_h;
      gamma = a.gamma_k;
    }

    uint4 xv = make_uint4(0, 0, 0, 0), gv = make_uint4(0, 0, 0, 0);
    if (active) {
      xv = *reinterpret_cast<const uint4*>(xrow + l * 8);
      gv = __ldg(reinterpret_cast<const uint4*>(gamma + l * 8));
    }
    float x[8], g[8];
    unpack8(xv, x);
    unpack8(gv, g);

    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(fmaf(ss, inv_d, a.eps));

    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = x[j] * r * g[j];

    // rotate-half: lanes 0..7 hold y[i], lanes 8..15 hold y[i + D/2]
    const int fbase = (l & 7) * 8;
    float out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float partner = __shfl_xor_sync(0xffffffffu, y[j], 8);
      const float c = s_cos[fbase + j], s = s_sin[fbase + j];
      out[j] = (l < 8) ? fmaf(y[j], c, -partner * s) : fmaf(y[j], c, partner * s);
    }
    uint4 ov;
    ov.x = pack_bf16x2(out[0], out[1]);
    ov.y = pack_bf16x2(out[2], out[3]);
    ov.z = pack_bf16x2(out[4], out[5]);
    ov.w = pack_bf16x2(out[6], out[7]);

    if (!active) continue;
    if (is_q) {
      *reinterpret_cast<uint4*>(xrow + l * 8) = ov;
    } else if (write_cache) {
      const int64_t dst = cache_row + static_cast<int64_t>(hk) * a.head_stride + l * 8;
      *reinterpret_cast<uint4*>(a.k_cache + dst) = ov;
      const uint4 vv = *reinterpret_cast<const uint4*>(
          a.v + t * a.v_stride_t + static_cast<int64_t>(hk) * a.v_stride_h + l * 8);
      *reinterpret_cast<uint4*>(a.v_cache + dst) = vv;
    }
  }
}

}  // namespace

cudaError_t launch_norm_rope_append(const NormRopeAppendArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  norm_rope_append_kernel<<<a.num_tokens, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkvqk
