// Split-KV paged decode attention with 3..16 query rows per kv head (GQA-4,
// GQA-8 decode, speculative verify) on the 5th-generation tensor cores, in
// the swapped-operand form: the keys, not the few query rows, fill the MMA's
// 128-row M dimension.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, fused rms_norm_rope, ...", section "概述 / Summary",
// items 1 (paged split-KV decode with GQA) and 4 (verify of k+1 tokens, causal
// among them) — the same attention as the mma.sync kernel in decode.cu, on
// the same segment schedules (decode_schedule.cuh).
//
// A tile is 128 rows (page p, kv head h, slot s) of the CTA's HPC kv heads:
// 8 / HPC consecutive 16-key pages.  The cache is read through a tensor map
// whose dimensions are (64 dims, slot, head, dim half, block), so one box per
// (page, half) lands as [HPC heads][16 slots][128 B] and a tile's K (and V)
// is [2 dim halves][128 rows][64 bf16], 128-byte swizzled.  With the
// segment's q rows n = h * R8 + j (j = t * group + gi < q_len * group, R8 the
// row count padded to 8) in Q^T [2 halves][128][64]:
//   S^T = K Q^T        M 128 rows, N = HPC * R8, K 128 dims (tensor memory)
//   O^T += V^T P^T     M 128 dims, N = HPC * R8, K 128 rows (tensor memory)
// Row (p, h, s) of S^T holds the scores of head h's key against every q row;
// only the columns of head h's rows are used.  P^T is block-diagonal: the
// softmax thread of row (p, h, s) writes its key's probabilities into head
// h's columns, every other column of P^T stays zero, so one K = 128 MMA chain
// computes every head's output at once.  The tensor core does HPC times the
// useful work, which costs nothing here: decode moves 2-10 flop per K/V byte.
//
// Warps: 0-3 softmax (thread r owns tensor-memory lane r: key row r of S^T,
// and dim r of O^T in the epilogue), 4 the TMA producer, 5 allocates the
// tensor memory and one lane issues the MMAs.  Per tile: MMA1 -> softmax
// (row max over the head's keys, lazy reference max that moves only when the
// tile max exceeds it by 2^8, O^T rescaled in tensor memory then, P^T into
// shared memory) -> MMA2.  Each tile carries 64 KB of K and V, ~1.4 us of HBM
// time per SM, far longer than this chain.  Every wait is bounded; on a
// timeout the CTA reports PKVQK_FLAG_WAIT_TIMEOUT, lets its copies and MMAs in
// flight finish (bounded), frees its tensor memory and exits.
#include "decode_schedule.cuh"
#include "device_common.cuh"
#include "kernels.h"
#include "tc5.cuh"

#include <cmath>

namespace pkvqk {

namespace {

using namespace sched;

constexpr int kRows = 128;                     // tile rows = tensor-memory lanes
constexpr int kHalf = kRows * 128;             // [128 rows][64 bf16], bytes
constexpr int kTile = 2 * kHalf;               // K, V, P^T or Q^T tile, bytes
constexpr int kStages = 2;
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kOffP = kOffV + kStages * kTile;
constexpr int kOffQ = kOffP + kTile;
constexpr int kDataBytes = kOffQ + kTile;      // 192 KiB
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;                  // S^T: N <= 128 columns
constexpr uint32_t kColO = 128;                // O^T: N <= 128 columns
constexpr float kRescaleLog2 = 8.f;
constexpr float kLn2 = 0.6931471805599453f;

struct Bars {
  uint64_t full_k[kStages], full_v[kStages];   // TMA landed
  uint64_t empty[kStages];                     // MMA2 of the stage's tile finished
  uint64_t s_full;                             // S^T of the tile written
  uint64_t p_full;                             // P^T written (and O^T rescaled)
  uint64_t pv_full;                            // O^T += V^T P^T finished
  uint64_t q_full;                             // Q^T of the segment loaded (O^T read out)
  uint64_t drain;                              // MMA thread's own completion (timeout path)
  uint32_t tmem_base;
  int32_t abort;
  int32_t issued;
  // cross-warp exchange of per-(page, head, row) tile maxima and sums
  float xmax[8][16];
  float xsum[8][16];
  // per segment column n: reference max, row sum, rescale factor
  float m_ref[kRows];
  float l_sum[kRows];
  float alpha[kRows];
};
constexpr int kSmemBytes = kDataBytes + static_cast<int>(sizeof(Bars)) + 1024;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t s = smem_addr(p);
  return p + (((s + 1023u) & ~1023u) - s);
}

// [128 rows][128 bf16] K-major operand in two 64-wide swizzled halves: step kk
// (16 elements) is 32 bytes into the rows of half kk/4; 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_k_major(uint32_t tile, int kk) {
  return tc5::smem_desc_sw128(tile + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
}

// [128 rows][128 bf16] MN-major operand (the 128 elements of a row are the M or
// N index, the rows are K): the two 64-wide halves kHalf apart, 8-row groups
// 1024 B apart; step ks (16 rows) starts 2048 bytes on.
__device__ __forceinline__ uint64_t desc_mn_major(uint32_t tile, int ks) {
  return tc5::smem_desc_sw128(tile + ks * 2048, kHalf, 1024);
}

// kind::f16 instruction descriptor with both operands' majorness.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
  return tc5::idesc_bf16_f32(M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Named barrier of the 128 softmax threads.
__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// The same barrier, returning whether any of the 128 threads passed true.
__device__ __forceinline__ bool softmax_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

// A wait of the four softmax warps whose outcome they agree on: if any warp
// timed out, all of them see the failure (and leave together, so that none
// is left at a named barrier).
__device__ __forceinline__ bool softmax_wait(uint64_t* bar, uint32_t parity) {
  return !softmax_sync_or(!warp_wait(bar, parity));
}

__device__ __forceinline__ int tiles_of(const Segment& seg, int tk) {
  return seg.k1 > seg.k0 ? (seg.k1 - seg.k0 + tk - 1) / tk : 0;
}

// ------------------------------------------------------------- producer

template <int HPC>
__device__ void produce(const DecodeArgs& a, const Plan* plan, const CUtensorMap* kmap,
                        const CUtensorMap* vmap, uint8_t* smem, Bars* bars, int* issued_out) {
  constexpr int PPT = 8 / HPC;                 // pages per tile
  constexpr int TK = 16 * PPT;
  constexpr int kBox = HPC * 16 * 128;         // one (page, half) box, bytes
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first_policy();
  if (lane == 0) {
    prefetch_tensormap(kmap);
    prefetch_tensormap(vmap);
  }
  SegmentSource src;
  src.init(a, plan, TK);
  Segment seg;
  int it = 0;
  bool ok = true;
  while (ok && src.next(seg)) {
    const int32_t* bt = a.block_tables + static_cast<int64_t>(seg.b) * a.max_blocks_per_seq;
    const int n = tiles_of(seg, TK);
    for (int i = 0; i < n && ok; ++i) {
      const int s = it % kStages;
      // lane q < boxes: the 16-key page box q of the tile (an out-of-range
      // block id reads zeros and is reported)
      const int key0 = seg.k0 + i * TK;
      const int boxes = min(PPT, (seg.k1 - key0 + 15) / 16);
      int blk = 0, slot0 = 0;
      const int key = key0 + lane * 16;
      if (lane < boxes) {
        const int page = key / a.block_size;
        slot0 = key - page * a.block_size;
        blk = __ldg(bt + page);
        if (blk < 0 || blk >= a.num_blocks) report(a.status_flags, kFlagBadBlock);
      }
      int good = 1;
      if (lane == 0 && it >= kStages) good = mbar_wait(&bars->empty[s], ((it / kStages) - 1) & 1);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->full_k[s], boxes * 2 * kBox);
        mbar_arrive_expect_tx(&bars->full_v[s], boxes * 2 * kBox);
      }
      __syncwarp();
      if (lane < boxes) {
        uint8_t* kt = smem + kOffK + s * kTile + lane * kBox;
        uint8_t* vt = smem + kOffV + s * kTile + lane * kBox;
        // coordinates: (dim lo, slot, kv head, dim half, block)
        tma_load_5d(kt, kmap, &bars->full_k[s], 0, slot0, seg.hg * HPC, 0, blk, pol);
        tma_load_5d(kt + kHalf, kmap, &bars->full_k[s], 0, slot0, seg.hg * HPC, 1, blk, pol);
        tma_load_5d(vt, vmap, &bars->full_v[s], 0, slot0, seg.hg * HPC, 0, blk, pol);
        tma_load_5d(vt + kHalf, vmap, &bars->full_v[s], 0, slot0, seg.hg * HPC, 1, blk, pol);
      }
      ++it;
    }
  }
  if (!ok && lane == 0) {
    bars->abort = 1;
    report(a.status_flags, kFlagTimeout);
  }
  if (lane == 0) *issued_out = it;
}

// ------------------------------------------------------------ MMA issue

template <int HPC, int R8>
__device__ void issue_mmas(const DecodeArgs& a, const Plan* plan, uint8_t* smem, Bars* bars,
                           uint32_t tmem) {
  constexpr int N = HPC * R8;
  constexpr int TK = 16 * (8 / HPC);
  const uint32_t id_s = idesc(kRows, N, false, false);
  const uint32_t id_o = idesc(kRows, N, true, true);
  const uint32_t qt = smem_addr(smem + kOffQ);
  const uint32_t pt = smem_addr(smem + kOffP);
  SegmentSource src;
  src.init(a, plan, TK);
  Segment seg;
  int it = 0, sg = 0;
  bool ok = true;
  while (ok && src.next(seg)) {
    const int n = tiles_of(seg, TK);
    if (n == 0) continue;                      // nothing to multiply; no Q^T is loaded
    // Q^T of this segment loaded (and O^T of the previous one read out)
    if (!mbar_wait(&bars->q_full, sg & 1)) {
      ok = false;
      break;
    }
    ++sg;
    for (int i = 0; i < n; ++i, ++it) {
      const int s = it % kStages;
      const uint32_t par = (it / kStages) & 1;
      if (!mbar_wait(&bars->full_k[s], par)) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      const uint32_t kt = smem_addr(smem + kOffK + s * kTile);
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        tc5::mma_f16(tmem + kColS, desc_k_major(kt, kk), desc_k_major(qt, kk), id_s,
                     kk > 0 ? 1u : 0u);
      tc5::commit(&bars->s_full);
      // P^T of this tile written (the softmax also waited for V and zeroed
      // the rows no query sees)
      if (!mbar_wait(&bars->p_full, it & 1) || !mbar_wait(&bars->full_v[s], par)) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      const uint32_t vt = smem_addr(smem + kOffV + s * kTile);
#pragma unroll
      for (int ks = 0; ks < kRows / 16; ++ks)
        tc5::mma_f16(tmem + kColO, desc_mn_major(vt, ks), desc_mn_major(pt, ks), id_o,
                     (i > 0 || ks > 0) ? 1u : 0u);
      tc5::commit(&bars->pv_full);
      tc5::commit(&bars->empty[s]);
    }
  }
  if (!ok) {
    bars->abort = 1;
    report(a.status_flags, kFlagTimeout);
    tc5::commit(&bars->drain);                 // everything issued so far ...
    mbar_wait(&bars->drain, 0);                // ... has finished
  }
}

// --------------------------------------------------------------- softmax

// Q^T of a segment: row n = h * R8 + j holds q row j (token t = j / group,
// head gi = j % group) of kv head h of the segment's group; rows past the
// segment's rows are zero.
template <int HPC, int R8>
__device__ void load_q(const DecodeArgs& a, const Segment& seg, uint8_t* smem, int R) {
  const int n = threadIdx.x;                   // 0..127
  const int h = n / R8, j = n - h * R8;
  const bool valid = h < HPC && j < R;
  const int t = valid ? j / a.group : 0, gi = valid ? j - t * a.group : 0;
  const uint4* src = reinterpret_cast<const uint4*>(
      a.q + (static_cast<int64_t>(seg.b) * a.q_len + t) * a.q_stride_t +
      static_cast<int64_t>((seg.hg * HPC + (valid ? h : 0)) * a.group + gi) * a.q_stride_h);
  uint8_t* qt = smem + kOffQ;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(qt + (c >> 3) * kHalf + swz128(n, c & 7)) = v;
  }
}

// The segment's outputs from O^T: thread d writes dim d of every row.
template <int HPC, int R8>
__device__ void write_out(const DecodeArgs& a, const Segment& seg, Bars* bars, uint32_t tmem,
                          int R, bool have_o) {
  constexpr int N = HPC * R8;
  const int d = threadIdx.x;
  const uint32_t lanes = tmem + (static_cast<uint32_t>((d >> 5) * 32) << 16) + kColO;
  for (int c0 = 0; c0 < N; c0 += 32) {
    float o[32];
    if (have_o) {
      tc5::tmem_ld32(lanes + c0, o);
      tc5::wait_ld();
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int n = c0 + e;
      const int h = n / R8, j = n - h * R8;
      if (n >= N || j >= R) continue;
      const int t = j / a.group, gi = j - t * a.group;
      const float l = bars->l_sum[n];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float v = have_o ? o[e] * inv : 0.f;
      const float lse = l > 0.f ? (bars->m_ref[n] + log2f(l)) * kLn2 : -INFINITY;
      const int hq = (seg.hg * HPC + h) * a.group + gi;
      const long long row = (static_cast<long long>(seg.b) * a.q_len + t) * a.num_q_heads + hq;
      if (seg.dest == kDestFinal) {
        a.out[row * kHeadDim + d] = __float2bfloat16_rn(v);
        if (d == 0 && a.lse_out != nullptr) a.lse_out[row] = lse;
      } else {
        const long long idx = seg.dest == kDestSplit
                                  ? row * a.num_splits + seg.split
                                  : seg.slot * a.rows_per_unit + (t * HPC + h) * a.group + gi;
        a.ws_o[idx * kHeadDim + d] = v;
        if (d == 0) a.ws_lse[idx] = lse;
      }
    }
  }
}

template <int HPC, int R8>
__device__ void softmax(const DecodeArgs& a, const Plan* plan, uint8_t* smem, Bars* bars,
                        uint32_t tmem, int R) {
  constexpr int N = HPC * R8;
  constexpr int PPT = 8 / HPC;
  constexpr int TK = 16 * PPT;
  const int r = threadIdx.x;                   // tensor-memory lane: tile row
  const int warp = r >> 5, lane = r & 31;
  const int p = r / (HPC * 16), h = (r / 16) % HPC, slot = r % 16;
  // the warp's two heads' columns, and this thread's offset among them
  const int h_lo = h & ~1;
  const uint32_t s_cols = tmem + (static_cast<uint32_t>(warp * 32) << 16) + kColS + h_lo * R8;
  const bool odd = h != h_lo;                  // this head's columns follow the other head's
  const float sl2 = a.scale_log2;

  SegmentSource src;
  src.init(a, plan, TK);
  Segment seg;
  int it = 0;
  bool ok = true;
  while (ok && src.next(seg)) {
    const int n_tiles = tiles_of(seg, TK);
    if (n_tiles > 0) {
      load_q<HPC, R8>(a, seg, smem, R);
      tc5::fence_smem_for_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_full);
    }
    float m_ref[16], l[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      m_ref[j] = -INFINITY;
      l[j] = 0.f;
    }
    for (int i = 0; i < n_tiles; ++i, ++it) {
      const int s = it % kStages;
      if (!softmax_wait(&bars->s_full, it & 1)) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      float sv[32];
      tc5::tmem_ld32(s_cols, sv);
      tc5::wait_ld();
      const int key = seg.k0 + i * TK + p * 16 + slot;
      float x[16];
      float tmax[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = j / a.group;
        const bool vis = j < R && key < seg.k1 && key < seg.seq_len - a.q_len + t + 1;
        const float sj = (odd && j + R8 < 32) ? sv[(j + R8) & 31] : sv[j];
        x[j] = vis ? sj * sl2 : -INFINITY;
        // max over the head's 16 keys of this page (a half-warp)
        float mx = x[j];
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        tmax[j] = mx;
      }
      if constexpr (PPT > 1) {
        // the head's keys of the other pages of the tile sit in other warps
        if (slot == 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) bars->xmax[p * HPC + h][j] = tmax[j];
        }
        softmax_sync();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float mx = -INFINITY;
#pragma unroll
          for (int q = 0; q < PPT; ++q) mx = fmaxf(mx, bars->xmax[q * HPC + h][j]);
          tmax[j] = mx;
        }
      }
      // lazy reference: moves only when the tile max exceeds it by 2^8
      bool grow_any = false;
      float alpha[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const bool grow = tmax[j] > m_ref[j] + kRescaleLog2;
        alpha[j] = grow ? ex2_approx(m_ref[j] - tmax[j]) : 1.f;
        if (grow) m_ref[j] = tmax[j];
        grow_any |= grow && i > 0;
      }
      // MMA2 of the previous tile finished: O^T is stable and P^T is free
      if (i > 0 && !softmax_wait(&bars->pv_full, (it - 1) & 1)) {
        ok = false;
        break;
      }
      if (softmax_sync_or(grow_any)) {
        // rescale O^T: columns of (h, j) by alpha; thread r is dim r here
        if (slot == 0 && p == 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (h * R8 + j < N && j < R8) bars->alpha[h * R8 + j] = alpha[j];
        }
        softmax_sync();
        const uint32_t o_cols = tmem + (static_cast<uint32_t>(warp * 32) << 16) + kColO;
        for (int c0 = 0; c0 < N; c0 += 32) {
          float o[32];
          tc5::tmem_ld32(o_cols + c0, o);
          tc5::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + e < N) o[e] *= bars->alpha[c0 + e];
          tc5::tmem_st32(o_cols + c0, o);
        }
        tc5::wait_st();
        softmax_sync();
      }
      // P = 2^(x - m_ref) in this head's columns of row r of P^T
      float ps[16];
      uint32_t pk[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const float u0 = m_ref[j] == -INFINITY ? 0.f : m_ref[j];
        const float u1 = m_ref[j + 1] == -INFINITY ? 0.f : m_ref[j + 1];
        const float p0 = ex2_approx(x[j] - u0), p1 = ex2_approx(x[j + 1] - u1);
        ps[j] = p0;
        ps[j + 1] = p1;
        pk[j / 2] = pack_bf16x2(p0, p1);
      }
      uint8_t* prow = smem + kOffP;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c * 8 >= R8) break;
        const int col = h * R8 + c * 8;        // first of 8 columns (16 bytes)
        *reinterpret_cast<uint4*>(prow + (col >> 6) * kHalf + swz128(r, (col & 63) >> 3)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      // row sums over the head's keys of the tile
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float sm = ps[j];
        sm += __shfl_xor_sync(0xffffffffu, sm, 8);
        sm += __shfl_xor_sync(0xffffffffu, sm, 4);
        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
        ps[j] = sm;
      }
      if constexpr (PPT > 1) {
        if (slot == 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) bars->xsum[p * HPC + h][j] = ps[j];
        }
        softmax_sync();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float sm = 0.f;
#pragma unroll
          for (int q = 0; q < PPT; ++q) sm += bars->xsum[q * HPC + h][j];
          ps[j] = sm;
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) l[j] = l[j] * alpha[j] + ps[j];
      // keys no query of the segment sees (past its end): their K and V rows
      // may hold anything (a partial tile keeps an earlier tile's rows, an
      // unwritten cache slot any bits); P is 0 there, but 0 x NaN is NaN, so
      // their V rows are zeroed before MMA2 reads them
      if (!softmax_wait(&bars->full_v[s], (it / kStages) & 1)) {
        ok = false;
        break;
      }
      if (key >= seg.k1) {
        uint8_t* vrow = smem + kOffV + s * kTile;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + swz128(r, c)) = z;
          *reinterpret_cast<uint4*>(vrow + kHalf + swz128(r, c)) = z;
        }
      }
      tc5::fence_smem_for_async();
      tc5::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
      if constexpr (PPT > 1) softmax_sync();   // the exchange buffers are reused next tile
    }
    if (!ok) break;
    // the segment's last MMA2, then its outputs
    if (n_tiles > 0 && !softmax_wait(&bars->pv_full, (it - 1) & 1)) {
      ok = false;
      break;
    }
    tc5::fence_after_sync();
    if (slot == 0 && p == 0) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j < R8 && h * R8 + j < N) {
          bars->m_ref[h * R8 + j] = m_ref[j];
          bars->l_sum[h * R8 + j] = l[j];
        }
      }
    }
    softmax_sync();
    write_out<HPC, R8>(a, seg, bars, tmem, R, n_tiles > 0);
    tc5::fence_before_sync();
    softmax_sync();                            // O^T read out before the next segment's MMA2
  }
  if (!ok) {
    bars->abort = 1;
    report(a.status_flags, kFlagTimeout);
  }
}

// ------------------------------------------------------------------ kernel

template <int HPC, int R8>
__global__ void __launch_bounds__(kThreads, 1)
paged_decode_tc5_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = reinterpret_cast<Bars*>(smem + kDataBytes);
  __shared__ Plan plan;
  __shared__ long long wsum[32];
  const int warp = threadIdx.x >> 5;
  const int R = a.q_len * a.group;

  if (threadIdx.x == kProducerWarp * 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full_k[s], 1);
      mbar_init(&bars->full_v[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, kSoftmaxWarps);
    mbar_init(&bars->pv_full, 1);
    mbar_init(&bars->q_full, kSoftmaxWarps);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->issued = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tc5::tmem_alloc(&bars->tmem_base, kTmemCols);
  if (warp < kSoftmaxWarps) {
    // P^T starts at zero: the softmax only ever writes a head's own columns
    uint4* pz = reinterpret_cast<uint4*>(smem + kOffP);
    for (int i = threadIdx.x; i < kTile / 16; i += kSoftmaxWarps * 32)
      pz[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  // launched as a programmatic dependent: everything below may read what the
  // previous kernel in the stream wrote (q, appended K/V, tables, lengths)
  pdl_launch_dependents();
  pdl_wait();
  if (a.num_splits == 0) {
    make_plan(a, &plan, wsum);
    write_empty_units(a, HPC);
  }
  const uint32_t tmem = bars->tmem_base;

  if (warp < kSoftmaxWarps) {
    softmax<HPC, R8>(a, &plan, smem, bars, tmem, R);
  } else if (warp == kProducerWarp) {
    int n = 0;
    produce<HPC>(a, &plan, &kmap, &vmap, smem, bars, &n);
    if ((threadIdx.x & 31) == 0) bars->issued = n;
  } else {
    if ((threadIdx.x & 31) == 0) issue_mmas<HPC, R8>(a, &plan, smem, bars, tmem);
    __syncwarp();
  }
  tc5::fence_before_sync();
  __syncthreads();
  if (bars->abort && threadIdx.x == kProducerWarp * 32) {
    // wait (bounded) for the copies last issued into each stage
    const int n = bars->issued;
    for (int i = n - kStages < 0 ? 0 : n - kStages; i < n; ++i) {
      mbar_wait(&bars->full_k[i % kStages], (i / kStages) & 1);
      mbar_wait(&bars->full_v[i % kStages], (i / kStages) & 1);
    }
  }
  if (warp == kMmaWarp) {
    tc5::fence_after_sync();
    tc5::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int HPC, int R8>
cudaError_t launch_hpc(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeArgs& a,
                       int grid_ctas, cudaStream_t stream) {
  auto kern = paged_decode_tc5_kernel<HPC, R8>;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = set_smem_limit_once(kern, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid = a.num_splits == 0 ? dim3(grid_ctas, 1, 1)
                                      : dim3(a.num_splits, a.num_kv_heads / HPC, a.batch);
  return launch_pdl(kern, grid, dim3(kThreads), kSmemBytes, stream, kmap, vmap, a);
}

}  // namespace

cudaError_t launch_paged_decode_tc5(int heads_per_cta, const CUtensorMap& kmap,
                                    const CUtensorMap& vmap, const DecodeArgs& a, int grid_ctas,
                                    cudaStream_t stream) {
  const int R = a.q_len * a.group;               // 3..16 query rows per kv head
  if (R < 1 || R > 16) return cudaErrorInvalidValue;
  const bool wide = R > 8;                        // rows padded to 16, else to 8
  switch (heads_per_cta) {
    case 8:
      return wide ? launch_hpc<8, 16>(kmap, vmap, a, grid_ctas, stream)
                  : launch_hpc<8, 8>(kmap, vmap, a, grid_ctas, stream);
    case 4:
      return wide ? launch_hpc<4, 16>(kmap, vmap, a, grid_ctas, stream)
                  : launch_hpc<4, 8>(kmap, vmap, a, grid_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkvqk
