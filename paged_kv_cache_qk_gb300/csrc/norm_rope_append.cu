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
// holds elements [4l, 4l+4) and their rotate-half partners [64+4l, 64+4l+4)
// (two 8-byte loads), so a rotation needs no shuffle, and keeps the sin/cos
// of its four frequencies in registers for every vector of the token; the
// sum of squares is a 4-step xor-shuffle reduction inside the half-warp.  A
// half-warp takes up to kHoist vectors of its token, and issues all their
// loads before the angle work.  Few tokens
// (decode): one half-warp per vector, the shortest path per token.  Many
// tokens (prefill chunks): three or more warps per token and up to four
// vectors per half-warp, so several tokens per SM overlap their latencies.
//
// The angles depend on the position alone, so a caller may build them once
// (launch_rope_table_build: the same float64 reduction and float-float sin/cos,
// kept per position as the float4s a lane reads) and pass the table: a token
// whose position is in it loads its lane's 64 bytes with the q/k/v loads and
// skips the angle phase; any other token computes its angles as above.  Both
// ways give the same bits.
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
// With the angles from a table, 10 CTAs per SM at 64 registers (a few bytes
// of spill, in the per-token angle fallback): 8192 tokens with the scalar
// rotation 34.0 us at 8 per SM, 32.2 at 9, 31.0 at 10, 33.8 at 11; with the
// packed rotation 31.6 at 8, 31.1 at 9, 29.0 at 10 (measured on GB300).
constexpr int kTableMinBlocks = 10;

// A lane's part of one head vector: elements [4l, 4l + 4) and their
// rotate-half partners [64 + 4l, 64 + 4l + 4), as raw bf16 (x, and v for kv
// heads).
struct Loaded {
  uint2 x0, x1, v0, v1;
};

// sin/cos of this lane's four frequencies 4l .. 4l+3, float-float pairs.
struct Trig {
  float4 ch, cl, sh, sl;
};

__device__ __forceinline__ void unpack4(const uint2& u, float* f) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x);
  f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
}

// Loads x (and for k heads the v row) of head vector h of token t.
__device__ __forceinline__ Loaded load_vector(const NormRopeAppendArgs& a, int t, int h, int l) {
  Loaded r;
  r.x0 = r.x1 = r.v0 = r.v1 = make_uint2(0, 0);
  if (h < a.num_q_heads) {
    const __nv_bfloat16* src = a.q + t * a.q_stride_t + static_cast<int64_t>(h) * a.q_stride_h;
    r.x0 = *reinterpret_cast<const uint2*>(src + 4 * l);
    r.x1 = *reinterpret_cast<const uint2*>(src + 64 + 4 * l);
  } else if (h < a.num_q_heads + a.num_kv_heads) {
    const int hk = h - a.num_q_heads;
    const __nv_bfloat16* ks = a.k + t * a.k_stride_t + static_cast<int64_t>(hk) * a.k_stride_h;
    const __nv_bfloat16* vs = a.v + t * a.v_stride_t + static_cast<int64_t>(hk) * a.v_stride_h;
    r.x0 = __ldg(reinterpret_cast<const uint2*>(ks + 4 * l));
    r.x1 = __ldg(reinterpret_cast<const uint2*>(ks + 64 + 4 * l));
    r.v0 = __ldg(reinterpret_cast<const uint2*>(vs + 4 * l));
    r.v1 = __ldg(reinterpret_cast<const uint2*>(vs + 64 + 4 * l));
  }
  return r;
}

__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// r * (a c - b s) for c = ch + cl, s = sh + sl, two elements at once (packed
// f32x2, each lane rounded as the scalar instruction rounds it): the products
// a*ch and b*sh error-free (p1 = a ch rounded, its error -(p1 - a ch) from
// one fma against -ch; q2 = b sh rounded, the error of -b sh as q2 - b sh),
// the low parts and the error terms added last.  nch, nsh, nsl are -ch, -sh,
// -sl (exact), so no negation is spent per element.
__device__ __forceinline__ uint64_t rotate2(uint64_t a, uint64_t b, uint64_t ch, uint64_t nch,
                                            uint64_t cl, uint64_t sh, uint64_t nsh, uint64_t nsl,
                                            uint64_t r) {
  const uint64_t p1 = mul2(a, ch);
  const uint64_t m1 = fma2(a, nch, p1);
  const uint64_t q2 = mul2(b, sh);
  const uint64_t e2 = fma2(b, nsh, q2);
  const uint64_t tail = add2(fma2(a, cl, mul2(b, nsl)), sub2(e2, m1));
  return mul2(r, add2(sub2(p1, q2), tail));
}

// Norm + rotation + stores of one head vector; both half-warps of the warp
// call it together (the sum-of-squares shuffles are warp-wide).
__device__ __forceinline__ void finish_vector(const NormRopeAppendArgs& a, int t, int h, int l,
                                              const Loaded& in, const uint2 (&gq)[2],
                                              const uint2 (&gk)[2], int64_t cache_row,
                                              bool write_cache, const Trig& tr) {
  const int num_vec = a.num_q_heads + a.num_kv_heads;
  float x0[4], x1[4], g0[4], g1[4];
  unpack4(in.x0, x0);
  unpack4(in.x1, x1);
  const bool is_q = h < a.num_q_heads;
  unpack4(is_q ? gq[0] : gk[0], g0);
  unpack4(is_q ? gq[1] : gk[1], g1);
  // x*gamma is exact in fp32; x^2 is exact, the sum rounds
  float ss = 0.f, a0[4], a1[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    ss = fmaf(x0[j], x0[j], ss);
    ss = fmaf(x1[j], x1[j], ss);
    a0[j] = x0[j] * g0[j];
    a1[j] = x1[j] * g1[j];
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(fmaf(ss, 1.0f / kHeadDim, a.eps));

  // rotate-half, pair (i, i + D/2) in this lane:
  //   out_i = a_i c - a_{i+D/2} s,   out_{i+D/2} = a_{i+D/2} c + a_i s
  const float ch[4] = {tr.ch.x, tr.ch.y, tr.ch.z, tr.ch.w};
  const float cl[4] = {tr.cl.x, tr.cl.y, tr.cl.z, tr.cl.w};
  const float sh[4] = {tr.sh.x, tr.sh.y, tr.sh.z, tr.sh.w};
  const float sl[4] = {tr.sl.x, tr.sl.y, tr.sl.z, tr.sl.w};
  const uint64_t r2 = pack2(r, r);
  float o0[4], o1[4];
#pragma unroll
  for (int j = 0; j < 4; j += 2) {
    const uint64_t x0 = pack2(a0[j], a0[j + 1]), x1 = pack2(a1[j], a1[j + 1]);
    const uint64_t c = pack2(ch[j], ch[j + 1]), nc = pack2(-ch[j], -ch[j + 1]);
    const uint64_t c_lo = pack2(cl[j], cl[j + 1]);
    const uint64_t s = pack2(sh[j], sh[j + 1]), ns = pack2(-sh[j], -sh[j + 1]);
    const uint64_t s_lo = pack2(sl[j], sl[j + 1]), ns_lo = pack2(-sl[j], -sl[j + 1]);
    // out_i = r (a_i c - a_{i+64} s);  out_{i+64} = r (a_{i+64} c - (-a_i) s)
    unpack2(rotate2(x0, x1, c, nc, c_lo, s, ns, ns_lo, r2), o0[j], o0[j + 1]);
    unpack2(rotate2(x1, x0, c, nc, c_lo, ns, s, s_lo, r2), o1[j], o1[j + 1]);
  }
  const uint2 w0 = make_uint2(pack_bf16x2(o0[0], o0[1]), pack_bf16x2(o0[2], o0[3]));
  const uint2 w1 = make_uint2(pack_bf16x2(o1[0], o1[1]), pack_bf16x2(o1[2], o1[3]));

  if (h >= num_vec) return;
  if (is_q) {
    __nv_bfloat16* dst = a.q + t * a.q_stride_t + static_cast<int64_t>(h) * a.q_stride_h;
    *reinterpret_cast<uint2*>(dst + 4 * l) = w0;
    *reinterpret_cast<uint2*>(dst + 64 + 4 * l) = w1;
  } else if (write_cache) {
    const int hk = h - a.num_q_heads;
    const int64_t row = cache_row + static_cast<int64_t>(hk) * a.head_stride;
    *reinterpret_cast<uint2*>(a.k_cache + row + 4 * l) = w0;
    *reinterpret_cast<uint2*>(a.k_cache + row + 64 + 4 * l) = w1;
    *reinterpret_cast<uint2*>(a.v_cache + row + 4 * l) = in.v0;
    *reinterpret_cast<uint2*>(a.v_cache + row + 64 + 4 * l) = in.v1;
  }
}

// The token's sin/cos through shared memory: the knots copied in, 64 angles
// (one per lane of warps 0 and 1: every lane of a float64 instruction busy),
// float64 angle and quarter-turn reduction, float-float sin/cos.  CTA-wide.
__device__ __forceinline__ Trig angles_in_cta(const NormRopeAppendArgs& a, int64_t pos, int l,
                                              float (*s_tab)[4], float* s_cos_hi,
                                              float* s_cos_lo, float* s_sin_hi,
                                              float* s_sin_lo) {
  // the sin/cos knots to shared memory: the lookups below take a different
  // knot in every lane, and indexing the parameter copy that way costs one
  // constant-cache access per distinct address (cold misses included) on the
  // angle's critical path
  for (int e = threadIdx.x; e < kSinCosKnots * 4; e += blockDim.x)
    (&s_tab[0][0])[e] = (&a.sincos_tab[0][0])[e];
  __syncthreads();
  if (threadIdx.x < kHeadDim / 2) {
    const int i = threadIdx.x;
    FF x, sn, cs;
    const int quadrant = reduce_angle(static_cast<double>(pos), a.inv_freq[i], &x);
    sincos_ff(x, quadrant, s_tab, &sn, &cs);
    s_cos_hi[i] = cs.hi;
    s_cos_lo[i] = cs.lo;
    s_sin_hi[i] = sn.hi;
    s_sin_lo[i] = sn.lo;
  }
  __syncthreads();
  // this lane's four frequencies, for every head vector it finishes
  Trig tr;
  tr.ch = *reinterpret_cast<const float4*>(s_cos_hi + 4 * l);
  tr.cl = *reinterpret_cast<const float4*>(s_cos_lo + 4 * l);
  tr.sh = *reinterpret_cast<const float4*>(s_sin_hi + 4 * l);
  tr.sl = *reinterpret_cast<const float4*>(s_sin_lo + 4 * l);
  return tr;
}

template <int kThreadsBound, int kMinBlocks, bool kTable>
__global__ void __launch_bounds__(kThreadsBound, kMinBlocks)
norm_rope_append_kernel(const __grid_constant__ NormRopeAppendArgs a) {
  __shared__ __align__(16) float s_cos_hi[kHeadDim / 2], s_cos_lo[kHeadDim / 2];
  __shared__ __align__(16) float s_sin_hi[kHeadDim / 2], s_sin_lo[kHeadDim / 2];
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
  // the gains are the same for every token and head: loaded once per lane
  const uint2 gq[2] = {__ldg(reinterpret_cast<const uint2*>(a.gamma_q + 4 * l)),
                       __ldg(reinterpret_cast<const uint2*>(a.gamma_q + 64 + 4 * l))};
  const uint2 gk[2] = {__ldg(reinterpret_cast<const uint2*>(a.gamma_k + 4 * l)),
                       __ldg(reinterpret_cast<const uint2*>(a.gamma_k + 64 + 4 * l))};
  // uniform over the CTA (one token)
  const bool from_table = kTable && pos >= 0 && pos < a.table_positions;
  Trig tr;
  if (from_table) {
    const float4* row = a.rope_table + (pos * (kHeadDim / 8) + l) * 4;
    tr.ch = __ldg(row);
    tr.cl = __ldg(row + 1);
    tr.sh = __ldg(row + 2);
    tr.sl = __ldg(row + 3);
  } else {
    tr = angles_in_cta(a, pos, l, s_tab, s_cos_hi, s_cos_lo, s_sin_hi, s_sin_lo);
  }
  const int64_t nslots = a.num_blocks * static_cast<int64_t>(a.block_size);
  if (threadIdx.x == 0 && slot >= nslots) report(a.status_flags, kFlagBadSlot);
  const bool write_cache = slot >= 0 && slot < nslots;
  const int64_t blk = write_cache ? slot / a.block_size : 0;
  const int64_t off = write_cache ? slot % a.block_size : 0;
  const int64_t cache_row = blk * a.block_stride + off * a.slot_stride;

  // warp-uniform: both half-warps of a warp share `base`
  const int num_vec = a.num_q_heads + a.num_kv_heads;
#pragma unroll
  for (int p = 0; p < kHoist; ++p) {
    const int base = warp * 2 + p * vec_per_pass;
    if (base < num_vec)
      finish_vector(a, t, base + (lane >> 4), l, in[p], gq, gk, cache_row, write_cache, tr);
  }
  // more head vectors than kHoist passes cover (Hq + Hkv > 2 * kHoist * warps)
  for (int base = warp * 2 + kHoist * vec_per_pass; base < num_vec; base += vec_per_pass) {
    const int h = base + (lane >> 4);
    const Loaded in = load_vector(a, t, h, l);
    finish_vector(a, t, h, l, in, gq, gk, cache_row, write_cache, tr);
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
  const bool table = a.rope_table != nullptr && a.table_positions > 0;
  if (many && warps * 32 <= kManyThreads)
    return launch_pdl(table ? norm_rope_append_kernel<kManyThreads, kTableMinBlocks, true>
                            : norm_rope_append_kernel<kManyThreads, kManyMinBlocks, false>,
                      dim3(a.num_tokens), dim3(warps * 32), 0, stream, a);
  return launch_pdl(table ? norm_rope_append_kernel<kMaxThreads, 1, true>
                          : norm_rope_append_kernel<kMaxThreads, 1, false>,
                    dim3(a.num_tokens), dim3(warps * 32), 0, stream, a);
}

namespace {

struct RopeTableArgs {
  float4* table;
  int32_t positions;
  double inv_freq[64];
  float sincos_tab[kSinCosKnots][4];
};

// One CTA per position, thread i = frequency i: the same steps as the append
// kernel's angle phase, stored where lane i/4 of a half-warp reads them.
__global__ void __launch_bounds__(64) rope_table_kernel(const __grid_constant__ RopeTableArgs a) {
  __shared__ float s_tab[kSinCosKnots][4];
  for (int e = threadIdx.x; e < kSinCosKnots * 4; e += blockDim.x)
    (&s_tab[0][0])[e] = (&a.sincos_tab[0][0])[e];
  __syncthreads();
  const int64_t pos = blockIdx.x;
  const int i = threadIdx.x;
  FF x, sn, cs;
  const int quadrant = reduce_angle(static_cast<double>(pos), a.inv_freq[i], &x);
  sincos_ff(x, quadrant, s_tab, &sn, &cs);
  float* row = reinterpret_cast<float*>(a.table + (pos * (kHeadDim / 8) + i / 4) * 4);
  row[0 * 4 + (i & 3)] = cs.hi;
  row[1 * 4 + (i & 3)] = cs.lo;
  row[2 * 4 + (i & 3)] = sn.hi;
  row[3 * 4 + (i & 3)] = sn.lo;
}

}  // namespace

cudaError_t launch_rope_table_build(float4* table, int32_t positions, const double (&inv_freq)[64],
                                    const float (&sincos_tab)[51][4], cudaStream_t stream) {
  if (positions <= 0) return cudaSuccess;
  RopeTableArgs a;
  a.table = table;
  a.positions = positions;
  for (int i = 0; i < 64; ++i) a.inv_freq[i] = inv_freq[i];
  for (int k = 0; k < kSinCosKnots; ++k)
    for (int c = 0; c < 4; ++c) a.sincos_tab[k][c] = sincos_tab[k][c];
  rope_table_kernel<<<positions, 64, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkvqk
