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
//    are formed and reduced by quarter turns in float64, and their sin/cos
//    evaluated once per token in float-float arithmetic on the float32 pipe
//    to ~2e-14 (rope_math.cuh: a 51-knot table, copied to shared memory
//    first, and the addition theorems), one angle per lane of warps 0 and 1,
//    then kept in shared memory as float-float pairs (hi + lo);
//  * per element a = x * gamma is exact in fp32 (two 8-bit significands);
//    the rotation a_i c - a_j s is formed with error-free products
//    (p = a*c_hi, e = fma(a, c_hi, -p)) so cancellation loses nothing;
//  * the RMS scale r = rsqrt(mean(x^2) + eps) multiplies the rotated value
//    last (a common factor, it contributes only relative error).
// Each head vector (D = 128 bf16 = 256 B) is handled by a half-warp: lane l
// holds elements [8l, 8l+8) as one 16-byte load; the sum of squares is a
// 4-step xor-shuffle reduction inside the half-warp, and the rotate-half
// partner of lane l is lane l ^ 8.  A half-warp takes up to kHoist vectors of
// its token, and issues all their loads before the angle work.  Few tokens
// (decode): one half-warp per vector, the shortest path per token.  Many
// tokens (prefill chunks): three or more warps per token and up to four
// vectors per half-warp, so several tokens per SM overlap their latencies.
#include "device_common.cuh"
#include "kernels.h"
#include "rope_math.cuh"

namespace pkvqk {

namespace {

constexpr int kMaxThreads = 512;
constexpr int kHoist = 4;            // vectors per half-warp whose loads go first
constexpr int kManyTokens = 1024;    // from here on, narrow CTAs
// Narrow CTAs of at most kManyThreads threads, kManyMinBlocks of them per SM:
// the compiler then keeps a thread at 80 registers, 8 tokens per SM (measured
// on GB300, 8192 tokens: 6 per SM at 96 registers 55.4 us, 8 at 80 49.6 us,
// 10 at 64 registers with spills 53.4 us).
constexpr int kManyThreads = 96;
constexpr int kManyMinBlocks = 8;

struct Loaded {
  uint4 x, v;
};

// Loads x (and for k heads the v row) of head vector h of token t.
__device__ __forceinline__ Loaded load_vector(const NormRopeAppendArgs& a, int t, int h, int l) {
  Loaded r;
  r.x = r.v = make_uint4(0, 0, 0, 0);
  if (h < a.num_q_heads) {
    r.x = *reinterpret_cast<const uint4*>(a.q + t * a.q_stride_t +
                                          static_cast<int64_t>(h) * a.q_stride_h + l * 8);
  } else if (h < a.num_q_heads + a.num_kv_heads) {
    const int hk = h - a.num_q_heads;
    r.x = __ldg(reinterpret_cast<const uint4*>(a.k + t * a.k_stride_t +
                                               static_cast<int64_t>(hk) * a.k_stride_h + l * 8));
    r.v = __ldg(reinterpret_cast<const uint4*>(a.v + t * a.v_stride_t +
                                               static_cast<int64_t>(hk) * a.v_stride_h + l * 8));
  }
  return r;
}

// Norm + rotation + stores of one head vector; both half-warps of the warp
// call it together (every shuffle is warp-wide).
__device__ __forceinline__ void finish_vector(const NormRopeAppendArgs& a, int t, int h, int l,
                                              const Loaded& in, const uint4& gq, const uint4& gk,
                                              int64_t cache_row,
                                              bool write_cache, const float* s_cos_hi,
                                              const float* s_cos_lo, const float* s_sin_hi,
                                              const float* s_sin_lo) {
  const int num_vec = a.num_q_heads + a.num_kv_heads;
  float x[8], g[8];
  unpack8(in.x, x);
  unpack8(h < a.num_q_heads ? gq : gk, g);
  // x*gamma is exact in fp32; x^2 is exact, the sum rounds
  float ss = 0.f, ag[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ss = fmaf(x[j], x[j], ss);
    ag[j] = x[j] * g[j];
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(fmaf(ss, 1.0f / kHeadDim, a.eps));

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

  if (h >= num_vec) return;
  if (h < a.num_q_heads) {
    *reinterpret_cast<uint4*>(a.q + t * a.q_stride_t + static_cast<int64_t>(h) * a.q_stride_h +
                              l * 8) = ov;
  } else if (write_cache) {
    const int hk = h - a.num_q_heads;
    const int64_t dst = cache_row + static_cast<int64_t>(hk) * a.head_stride + l * 8;
    *reinterpret_cast<uint4*>(a.k_cache + dst) = ov;
    *reinterpret_cast<uint4*>(a.v_cache + dst) = in.v;
  }
}

template <int kThreadsBound, int kMinBlocks>
__global__ void __launch_bounds__(kThreadsBound, kMinBlocks)
norm_rope_append_kernel(const __grid_constant__ NormRopeAppendArgs a) {
  __shared__ float s_cos_hi[kHeadDim / 2], s_cos_lo[kHeadDim / 2];
  __shared__ float s_sin_hi[kHeadDim / 2], s_sin_lo[kHeadDim / 2];
  __shared__ float s_tab[kSinCosKnots][4];

  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int l = lane & 15;                       // lane within the half-warp
  const int vec_per_pass = (blockDim.x >> 5) * 2;
  const int h0 = warp * 2 + (lane >> 4);         // this half-warp's first head vector

  // launched as a programmatic dependent: wait for the kernel that produced
  // q/k/v before reading them, but let the next kernel begin its launch now
  pdl_launch_dependents();
  pdl_wait();

  // every independent global load first
  const int64_t pos = a.positions[t];
  const int64_t slot = a.slot_mapping[t];
  Loaded in[kHoist];
#pragma unroll
  for (int p = 0; p < kHoist; ++p) in[p] = load_vector(a, t, h0 + p * vec_per_pass, l);
  // the gains are the same for every token and head: one load per lane
  const uint4 gq = __ldg(reinterpret_cast<const uint4*>(a.gamma_q + l * 8));
  const uint4 gk = __ldg(reinterpret_cast<const uint4*>(a.gamma_k + l * 8));
  // the sin/cos knots to shared memory while those loads are in flight: the
  // lookups below take a different knot in every lane, and indexing the
  // parameter copy that way costs one constant-cache access per distinct
  // address (cold misses included) on the angle's critical path
  for (int e = threadIdx.x; e < kSinCosKnots * 4; e += blockDim.x)
    (&s_tab[0][0])[e] = (&a.sincos_tab[0][0])[e];
  __syncthreads();

  // the token's 64 angles, one per lane of warps 0 and 1 (every lane of a
  // float64 instruction busy): float64 angle and quarter-turn reduction,
  // float-float sin/cos
  if (warp < 2) {
    const int i = threadIdx.x;
    FF x, sn, cs;
    const int quadrant = reduce_angle(static_cast<double>(pos), a.inv_freq[i], &x);
    sincos_ff(x, quadrant, s_tab, &sn, &cs);
    s_cos_hi[i] = cs.hi;
    s_cos_lo[i] = cs.lo;
    s_sin_hi[i] = sn.hi;
    s_sin_lo[i] = sn.lo;
  }
  const int64_t nslots = a.num_blocks * static_cast<int64_t>(a.block_size);
  if (threadIdx.x == 0 && slot >= nslots) report(a.status_flags, kFlagBadSlot);
  const bool write_cache = slot >= 0 && slot < nslots;
  const int64_t blk = write_cache ? slot / a.block_size : 0;
  const int64_t off = write_cache ? slot % a.block_size : 0;
  const int64_t cache_row = blk * a.block_stride + off * a.slot_stride;
  __syncthreads();

  // warp-uniform: both half-warps of a warp share `base`
  const int num_vec = a.num_q_heads + a.num_kv_heads;
#pragma unroll
  for (int p = 0; p < kHoist; ++p) {
    const int base = warp * 2 + p * vec_per_pass;
    if (base < num_vec)
      finish_vector(a, t, base + (lane >> 4), l, in[p], gq, gk, cache_row, write_cache, s_cos_hi,
                    s_cos_lo, s_sin_hi, s_sin_lo);
  }
  // more head vectors than kHoist passes cover (Hq + Hkv > 2 * kHoist * warps)
  for (int base = warp * 2 + kHoist * vec_per_pass; base < num_vec; base += vec_per_pass) {
    const int h = base + (lane >> 4);
    const Loaded in = load_vector(a, t, h, l);
    finish_vector(a, t, h, l, in, gq, gk, cache_row, write_cache, s_cos_hi, s_cos_lo, s_sin_hi,
                  s_sin_lo);
  }
}

}  // namespace

cudaError_t launch_norm_rope_append(const NormRopeAppendArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  // few tokens: one half-warp per head vector; many: up to kHoist vectors per
  // half-warp; at least 2 warps (one angle per lane of warps 0 and 1)
  const int num_vec = a.num_q_heads + a.num_kv_heads;
  const bool many = a.num_tokens >= kManyTokens;
  const int per_half_warp = many ? kHoist : 1;
  int warps = (num_vec + 2 * per_half_warp - 1) / (2 * per_half_warp);
  warps = warps < 2 ? 2 : (warps > kMaxThreads / 32 ? kMaxThreads / 32 : warps);
  if (many && warps * 32 <= kManyThreads)
    return launch_pdl(norm_rope_append_kernel<kManyThreads, kManyMinBlocks>, dim3(a.num_tokens),
                      dim3(warps * 32), 0, stream, a);
  return launch_pdl(norm_rope_append_kernel<kMaxThreads, 1>, dim3(a.num_tokens), dim3(warps * 32),
                    0, stream, a);
}

}  // namespace pkvqk
