// Fused per-head RMSNorm + neox RoPE on q and k, with the k/v cache append.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, fused rms_norm_rope, ...", section "概述 / Summary",
// item 2 (per-head RMSNorm + full-rotary RoPE in one op) and item 1 (the
// BSHD paged cache the decode kernel reads).
//
// One CTA per token.  Numerics, chosen so the rounded bf16 result is within
// one ulp of the correctly rounded exact value even where the rotation
// cancels (y_i cos - y_{i+D/2} sin close to 0):
//  * the token's 64 angles pos * inv_freq_i (inv_freq from the host, float64)
//    are reduced by 2*pi and their sin/cos evaluated in float64 once per
//    token, then kept in shared memory as float-float pairs (hi + lo);
//  * per element a = x * gamma is exact in fp32 (two 8-bit significands);
//    the rotation a_i c - a_j s is formed with error-free products
//    (p = a*c_hi, e = fma(a, c_hi, -p)) so cancellation loses nothing;
//  * the RMS scale r = rsqrt(mean(x^2) + eps) multiplies the rotated value
//    last (a common factor, it contributes only relative error).
// Each head vector (D = 128 bf16 = 256 B) is handled by a half-warp: lane l
// holds elements [8l, 8l+8) as one 16-byte load; the sum of squares is a
// 4-step xor-shuffle reduction inside the half-warp, and the rotate-half
// partner of lane l is lane l ^ 8.
#include "device_common.cuh"
#include "kernels.h"

namespace pkvqk {

namespace {

constexpr int kThreads = 256;
constexpr double kTwoPiHi = 6.283185307179586232;          // 2*pi rounded to double
constexpr double kTwoPiLo = 2.4492935982947064e-16;          // 2*pi - kTwoPiHi
constexpr double kInvTwoPi = 0.15915494309189535;

__global__ void __launch_bounds__(kThreads)
norm_rope_append_kernel(NormRopeAppendArgs a) {
  __shared__ float s_cos_hi[kHeadDim / 2], s_cos_lo[kHeadDim / 2];
  __shared__ float s_sin_hi[kHeadDim / 2], s_sin_lo[kHeadDim / 2];

  const int t = blockIdx.x;
  const int64_t pos = a.positions[t];
  const int64_t slot = a.slot_mapping[t];
  const int64_t nslots = a.num_blocks * static_cast<int64_t>(a.block_size);

  if (threadIdx.x < kHeadDim / 2) {
    const int i = threadIdx.x;
    const double ang = static_cast<double>(pos) * a.inv_freq[i];
    const double turns = rint(ang * kInvTwoPi);
    double red = fma(-turns, kTwoPiHi, ang);             // Cody-Waite: 2*pi = hi + lo
    red = fma(-turns, kTwoPiLo, red);                     // |red| <= pi (+ rounding)
    double sn, cs;
    sincos(red, &sn, &cs);
    const float ch = static_cast<float>(cs), sh = static_cast<float>(sn);
    s_cos_hi[i] = ch;
    s_cos_lo[i] = static_cast<float>(cs - static_cast<double>(ch));
    s_sin_hi[i] = sh;
    s_sin_lo[i] = static_cast<float>(sn - static_cast<double>(sh));
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

    // x*gamma is exact in fp32; x^2 is exact, the sum rounds
    float ss = 0.f, ag[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ss = fmaf(x[j], x[j], ss);
      ag[j] = x[j] * g[j];
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(fmaf(ss, inv_d, a.eps));

    // rotate-half: lanes 0..7 hold a[i], lanes 8..15 hold a[i + D/2];
    // out_i = a_i c - a_{i+D/2} s,  out_{i+D/2} = a_{i+D/2} c + a_i s
    const int fbase = (l & 7) * 8;
    const float sgn = (l < 8) ? -1.f : 1.f;
    float out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float b = sgn * __shfl_xor_sync(0xffffffffu, ag[j], 8);
      const float ch = s_cos_hi[fbase + j], cl = s_cos_lo[fbase + j];
      const float sh = s_sin_hi[fbase + j], sl = s_sin_lo[fbase + j];
      const float p1 = ag[j] * ch, e1 = fmaf(ag[j], ch, -p1);   // a*c_hi = p1 + e1 exactly
      const float p2 = b * sh, e2 = fmaf(b, sh, -p2);           // b*s_hi = p2 + e2 exactly
      const float tail = fmaf(ag[j], cl, b * sl) + (e1 + e2);
      out[j] = r * ((p1 + p2) + tail);
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
