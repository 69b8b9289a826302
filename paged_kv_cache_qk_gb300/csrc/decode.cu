// Split-KV paged decode attention with GQA (and the causal multi-query
// verify variant), sm_103a.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, fused rms_norm_rope, ...", section "概述 / Summary":
// item 1 (pure decode through a paged split-KV kernel that reads the
// FlashAttention BSHD cache through strided views) and item 4 (one verify
// forward over k+1 tokens per sequence, causal among the draft tokens).
//
// A CTA owns HPC kv heads ("head group") of some sequences and walks a list
// of segments — runs of 16-key tiles of one (sequence, head group).  Two
// schedules produce the segment list:
//   * split   (num_splits >= 1): grid (S, head groups, batch), one segment
//     per CTA: split j of the sequence (chunk_pages pages per split, the last
//     split takes the rest);
//   * balanced (num_splits == 0): a persistent grid (0.84 CTAs per SM); the
//     pages of all (head group, sequence) units are laid end to end and CTA c
//     takes pages [c*TP/G, (c+1)*TP/G) of that list (G = min(grid, TP)), crossing sequence
//     boundaries without refilling its pipeline.  A unit that one CTA covers
//     whole is written straight to the output; a unit cut across CTAs leaves
//     one partial per CTA in slot (cta + unit), merged by the combine kernel.
// Warp HPC is the producer: it walks the same segment list, its lanes fetch
// 32 block-table entries at a time and lane 0 issues, per 16-key tile, one
// 5-D TMA box for K and one for V (HPC heads x 16 slots x 128 dims each,
// 128-byte swizzled) into a ring of STAGES shared-memory stages guarded by
// full/empty mbarriers; the ring runs on across segments.  Warps 0..HPC-1
// consume, one per kv head, every q row that reads their kv head
// (rows = q_len * group):
//   * rows <= 2 ("simt", GQA-2 and multi-head decode): 8 lanes per key, 4
//     keys per warp instruction; each lane holds 16 of the 128 dims, its
//     part of q.k and of the P V update in packed fp32x2 FMAs (two dims per
//     instruction), the q.k dot finished by a 3-step xor-shuffle reduction;
//     every 8-lane key group keeps its own online softmax and the four groups
//     are merged by shuffles at the end of a segment.
//   * rows 3..16 ("tc", GQA-4 and GQA-8 decode, verify): the 16 padded rows
//     x 16 keys score tile and the 16 rows x 128 dims output tile are
//     mma.sync m16n8k16 bf16 contractions fed by ldmatrix from the swizzled
//     stages (conflict-free).  From 3 rows on the per-row dot products make
//     the CUDA-core form issue-bound below the HBM rate (measured on GB300,
//     32 x 8192 at 4 rows: 255 us with one warp per kv head, 225 us with
//     two; mma tiles 166 us, the HBM bound).
// Every wait on an mbarrier is bounded; on a timeout the CTA reports
// PKVQK_FLAG_WAIT_TIMEOUT, drains its own copies in flight and exits.
#include "combine_row.cuh"
#include "device_common.cuh"
#include "kernels.h"

#include <cmath>

namespace pkvqk {

namespace {

constexpr float kLn2 = 0.693147180559945309f;

// HPC kv heads per CTA, TK keys per tile (one TMA box covers TK consecutive
// slots of a page), stage ring of at most BUDGET_KB kilobytes.
template <int HPC, int TK, int BUDGET_KB>
struct Geometry {
  static constexpr int kHalfTileBytes = TK * 128;       // (kv head, 64-dim half): TK rows x 128 B
  static constexpr int kHeadTileBytes = 2 * kHalfTileBytes;
  static constexpr int kStageBytes = 2 * HPC * kHeadTileBytes;        // K + V tiles
  static constexpr int kStagesRaw = (BUDGET_KB * 1024) / kStageBytes;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;      // + alignment slack
  static constexpr int kConsumers = HPC;
  static constexpr int kThreads = (kConsumers + 1) * 32;
};

constexpr int kDestFinal = 0;   // bf16 output + lse
constexpr int kDestSplit = 1;   // partial at [row][split] (split schedule)
constexpr int kDestSlot = 2;    // partial at [slot][row in unit] (balanced schedule)

// A run of 16-key tiles of one (sequence, head group): keys [k0, k1).
struct Segment {
  int b, hg, seq_len, k0, k1, ntiles, dest, split;
  long long slot;
};

__device__ __forceinline__ int clamped_len(const DecodeArgs& a, int b) {
  int L = a.seq_lens[b];
  if (L < 0) L = 0;
  const long long cap = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
  if (L > cap) {
    report(a.status_flags, kFlagBadBlock);
    L = static_cast<int>(cap);
  }
  return L;
}

__device__ __forceinline__ long long unit_pages(const DecodeArgs& a, int u) {
  const int L = clamped_len(a, u % a.batch);
  return (L + a.block_size - 1) / a.block_size;
}

__device__ __forceinline__ void set_range(Segment& s, int k0, int k1, int tk) {
  s.k0 = k0;
  s.k1 = k1;
  s.ntiles = k1 > k0 ? (k1 - k0 + tk - 1) / tk : 0;
}

// Balanced schedule of this CTA: its page range and where its walk starts.
struct Plan {
  long long tp, lo, hi;     // total pages; this CTA's pages [lo, hi)
  long long g_eff;          // CTAs that get pages: min(grid, total pages)
  int u_start;              // first unit with pages at or after lo
  long long s_start;        // pages before unit u_start
};

// Produces the CTA's segments in order; producer and consumers each run
// their own copy and see the same sequence.
struct SegmentSource {
  const DecodeArgs* a;
  const Plan* plan;
  int tk;                   // keys per tile
  int balanced;
  int done;
  int u;
  long long s;              // pages before unit u

  __device__ void init(const DecodeArgs& args, const Plan* p, int tile_keys) {
    a = &args;
    plan = p;
    tk = tile_keys;
    balanced = args.num_splits == 0;
    done = 0;
    u = 0;
    s = 0;
    if (balanced) {
      u = p->u_start;
      s = p->s_start;
    }
  }

  __device__ bool next(Segment& seg) {
    if (!balanced) {
      if (done) return false;
      done = 1;
      seg.b = blockIdx.z;
      seg.hg = blockIdx.y;
      seg.split = blockIdx.x;
      seg.slot = 0;
      seg.seq_len = clamped_len(*a, seg.b);
      const int P = (seg.seq_len + a->block_size - 1) / a->block_size;
      int p0 = seg.split * a->chunk_pages;
      int p1 = (seg.split == a->num_splits - 1) ? P : p0 + a->chunk_pages;
      p0 = min(p0, P);
      p1 = min(p1, P);
      set_range(seg, p0 * a->block_size, min(p1 * a->block_size, seg.seq_len), tk);
      seg.dest = a->num_splits == 1 ? kDestFinal : kDestSplit;
      return true;
    }
    const int U = a->batch * a->groups;
    while (u < U && s < plan->hi) {
      const int cur = u;
      const long long start = s;
      const long long P = unit_pages(*a, cur);
      u += 1;
      s += P;
      const long long plo = max(start, plan->lo) - start;
      const long long phi = min(s, plan->hi) - start;
      if (phi <= plo) continue;                            // empty unit or no overlap
      seg.b = cur % a->batch;
      seg.hg = cur / a->batch;
      seg.split = 0;
      seg.seq_len = clamped_len(*a, seg.b);
      set_range(seg, static_cast<int>(plo) * a->block_size,
                min(static_cast<int>(phi) * a->block_size, seg.seq_len), tk);
      const bool whole = plo == 0 && phi == P;
      seg.dest = whole ? kDestFinal : kDestSlot;
      seg.slot = static_cast<long long>(blockIdx.x) + cur;
      // the CTA holding the unit's first page records which CTAs cut it:
      // page x belongs to CTA floor(((x + 1) * G' - 1) / TP), G' = g_eff
      if (start >= plan->lo && threadIdx.x == 0) {
        const int c_last = static_cast<int>((s * plan->g_eff - 1) / plan->tp);
        a->unit_info[cur] = make_int2(blockIdx.x, c_last);
      }
      return true;
    }
    return false;
  }
};

// Block-wide plan of the balanced schedule (every thread takes part).
__device__ void make_plan(const DecodeArgs& a, Plan* plan, long long* wsum) {
  const int U = a.batch * a.groups;
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = nt >> 5;
  const int chunk = (U + nt - 1) / nt;
  const int u_lo = min(U, tid * chunk), u_hi = min(U, u_lo + chunk);
  long long mine = 0;
  for (int u = u_lo; u < u_hi; ++u) mine += unit_pages(a, u);
  long long v = mine;                                       // inclusive warp scan
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) wsum[warp] = v;
  if (tid == 0) plan->u_start = U;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < nwarps) wsum[lane] = w;
  }
  __syncthreads();
  const long long tp = wsum[nwarps - 1];
  const long long before = (warp ? wsum[warp - 1] : 0) + v - mine;   // pages before u_lo
  // with fewer pages than CTAs only the first tp CTAs get pages, so that
  // every CTA between a unit's first and last owner holds some of it
  const long long G = min(static_cast<long long>(gridDim.x), tp > 0 ? tp : 1);
  const long long c = blockIdx.x;
  const long long lo = c < G ? c * tp / G : tp, hi = c < G ? (c + 1) * tp / G : tp;
  long long run = before;
  for (int u = u_lo; u < u_hi; ++u) {
    const long long P = unit_pages(a, u);
    if (run + P > lo) {
      atomicMin(&plan->u_start, u);
      break;
    }
    run += P;
  }
  __syncthreads();
  run = before;
  for (int u = u_lo; u < u_hi; ++u) {
    if (u == plan->u_start) plan->s_start = run;
    run += unit_pages(a, u);
  }
  if (tid == 0) {
    plan->tp = tp;
    plan->lo = lo;
    plan->hi = hi;
    plan->g_eff = G;
    if (plan->u_start == U) plan->s_start = tp;
  }
  __syncthreads();
}

// Units without any key: zero output, lse -inf, nothing to combine.  Unit u
// is handled by CTA u mod G (all threads of the CTA).
__device__ void write_empty_units(const DecodeArgs& a, int hpc) {
  const int U = a.batch * a.groups;
  for (int u = blockIdx.x; u < U; u += gridDim.x) {
    if (unit_pages(a, u) != 0) continue;
    const int b = u % a.batch, hg = u / a.batch;
    const int rows = a.rows_per_unit;
    for (int idx = threadIdx.x; idx < rows * (kHeadDim / 8); idx += blockDim.x) {
      const int r = idx / (kHeadDim / 8), c8 = idx % (kHeadDim / 8);
      // unit row r = (t * HPC + hh) * group + gi
      const int gi = r % a.group, th = r / a.group, hh = th % hpc, t = th / hpc;
      const int h = (hg * hpc + hh) * a.group + gi;
      const long long row = (static_cast<long long>(b) * a.q_len + t) * a.num_q_heads + h;
      *reinterpret_cast<uint4*>(a.out + row * kHeadDim + c8 * 8) = make_uint4(0, 0, 0, 0);
      if (c8 == 0 && a.lse_out != nullptr) a.lse_out[row] = -INFINITY;
    }
    if (threadIdx.x == 0) a.unit_info[u] = make_int2(blockIdx.x, blockIdx.x);
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t off = (1024u - (smem_addr(p) & 1023u)) & 1023u;
  return p + off;
}

// ----------------------------------------------------------------- producer

template <int HPC, int TK, int BUDGET, int STAGES>
__device__ void produce(const CUtensorMap* kmap, const CUtensorMap* vmap, const DecodeArgs& a,
                        const Plan* plan, uint8_t* stages, uint64_t* full, uint64_t* empty,
                        volatile int* abort_flag, int* issued_out) {
  using Geo = Geometry<HPC, TK, BUDGET>;
  constexpr int kStageBytes = Geo::kStageBytes;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    prefetch_tensormap(kmap);
    prefetch_tensormap(vmap);
  }
  const uint64_t pol = l2_evict_first_policy();
  SegmentSource src;
  src.init(a, plan, TK);
  Segment seg;
  int it = 0;                      // tiles issued so far (ring position)
  bool ok = true;
  while (ok && src.next(seg)) {
    const int32_t* bt = a.block_tables + static_cast<int64_t>(seg.b) * a.max_blocks_per_seq;
    for (int i0 = 0; i0 < seg.ntiles && ok; i0 += 32) {
      int blk = 0, slot0 = 0;
      const int i = i0 + lane;
      if (i < seg.ntiles) {
        const int key = seg.k0 + i * TK;
        const int page = key / a.block_size;
        slot0 = key - page * a.block_size;
        blk = __ldg(bt + page);
        if (blk < 0 || blk >= a.num_blocks) report(a.status_flags, kFlagBadBlock);
      }
      const int n = min(32, seg.ntiles - i0);
      for (int j = 0; j < n; ++j) {
        const int bj = __shfl_sync(0xffffffffu, blk, j);
        const int sj = __shfl_sync(0xffffffffu, slot0, j);
        int good = 1;
        if (lane == 0) {
          const int s = it % STAGES;
          if (it >= STAGES) good = mbar_wait(&empty[s], ((it / STAGES) - 1) & 1) ? 1 : 0;
          if (good) {
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            uint8_t* dst = stages + s * kStageBytes;
            // coordinates: (dim lo, slot, dim half, kv head, block)
            tma_load_5d(dst, kmap, &full[s], 0, sj, 0, seg.hg * HPC, bj, pol);
            tma_load_5d(dst + HPC * Geo::kHeadTileBytes, vmap, &full[s], 0, sj, 0, seg.hg * HPC,
                        bj, pol);
          } else {
            *abort_flag = 1;
            report(a.status_flags, kFlagTimeout);
          }
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        ++it;
      }
    }
  }
  if (lane == 0) *issued_out = it;
}

// After a timeout: wait (bounded) for the last copy issued into every stage
// so that no TMA write lands in shared memory after the CTA exits.
template <int STAGES>
__device__ void drain(uint64_t* full, int issued) {
  for (int s = 0; s < STAGES; ++s) {
    if (issued <= s) continue;
    const int last = s + ((issued - 1 - s) / STAGES) * STAGES;
    mbar_wait(&full[s], (last / STAGES) & 1);
  }
}

// -------------------------------------------------------- row destinations

struct RowDest {
  __nv_bfloat16* out;   // final bf16 row (or null)
  float* lse;           // final lse (or null)
  float* po;            // partial fp32 row (or null)
  float* plse;          // partial lse (or null)
};

template <int HPC>
__device__ __forceinline__ RowDest row_dest(const DecodeArgs& a, const Segment& seg, int t,
                                            int hh, int gi) {
  RowDest d{nullptr, nullptr, nullptr, nullptr};
  const int h = (seg.hg * HPC + hh) * a.group + gi;
  const long long row = (static_cast<long long>(seg.b) * a.q_len + t) * a.num_q_heads + h;
  if (seg.dest == kDestFinal) {
    d.out = a.out + row * kHeadDim;
    d.lse = a.lse_out != nullptr ? a.lse_out + row : nullptr;
  } else {
    const long long idx = seg.dest == kDestSplit
                              ? row * a.num_splits + seg.split
                              : seg.slot * a.rows_per_unit + (t * HPC + hh) * a.group + gi;
    d.po = a.ws_o + idx * kHeadDim;
    d.plse = a.ws_lse + idx;
  }
  return d;
}

__device__ __forceinline__ float final_lse(float m, float l) {
  return l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------ CUDA-core consumer

template <int HPC, int TK, int BUDGET, int STAGES, int R>
__device__ void consume_simt(const DecodeArgs& a, const Plan* plan, const uint8_t* stages,
                             uint64_t* full, uint64_t* empty, volatile int* abort_flag) {
  using Geo = Geometry<HPC, TK, BUDGET>;
  constexpr int kStageBytes = Geo::kStageBytes;
  constexpr int kHalfTileBytes = Geo::kHalfTileBytes;
  constexpr int kHeadTileBytes = Geo::kHeadTileBytes;
  constexpr int kQuads = TK / 4;   // 4 keys per warp step
  const int lane = threadIdx.x & 31;
  const int hh = threadIdx.x >> 5;
  const int kg = lane >> 3;        // key group: key 4*q4 + kg of the tile
  const int p = lane & 7;          // 16-byte chunk p of each 64-dim half

  SegmentSource src;
  src.init(a, plan, TK);
  Segment seg;
  int it = 0;                      // tiles consumed so far (ring position)
  bool aborted = false;
  while (!aborted && src.next(seg)) {
    const int kvh = seg.hg * HPC + hh;
    float qf[R][16], acc[R][16], m[R], l[R];
    int limit[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const int t = rr / a.group, gi = rr - t * a.group;
      const __nv_bfloat16* qrow = a.q +
                                  (static_cast<int64_t>(seg.b) * a.q_len + t) * a.q_stride_t +
                                  static_cast<int64_t>(kvh * a.group + gi) * a.q_stride_h;
      const uint4 u0 = __ldg(reinterpret_cast<const uint4*>(qrow + 8 * p));
      const uint4 u1 = __ldg(reinterpret_cast<const uint4*>(qrow + 64 + 8 * p));
      unpack8(u0, qf[rr]);
      unpack8(u1, qf[rr] + 8);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        qf[rr][j] *= a.scale_log2;
        acc[rr][j] = 0.f;
      }
      m[rr] = -INFINITY;
      l[rr] = 0.f;
      limit[rr] = seg.seq_len - a.q_len + t + 1;
    }

    for (int i = 0; i < seg.ntiles; ++i, ++it) {
      const int s = it % STAGES;
      if (!mbar_wait(&full[s], (it / STAGES) & 1)) {
        *abort_flag = 1;
        report(a.status_flags, kFlagTimeout);
        aborted = true;
        break;
      }
      const uint8_t* kt = stages + s * kStageBytes + hh * kHeadTileBytes;
      const uint8_t* vt = kt + HPC * kHeadTileBytes;
      const int key0 = seg.k0 + i * TK;

      float sc[R][kQuads];
#pragma unroll
      for (int q4 = 0; q4 < kQuads; ++q4) {
        const int row = q4 * 4 + kg;
        const uint4 k0 = *reinterpret_cast<const uint4*>(kt + swz128(row, p));
        const uint4 k1 = *reinterpret_cast<const uint4*>(kt + kHalfTileBytes + swz128(row, p));
        float kf[16];
        unpack8(k0, kf);
        unpack8(k1, kf + 8);
        const int n = key0 + row;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
          // 16 products in 8 packed fp32x2 FMAs (even and odd dims), then one add
          uint64_t d2 = pack2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            d2 = fma2(pack2(qf[rr][2 * j], qf[rr][2 * j + 1]), pack2(kf[2 * j], kf[2 * j + 1]), d2);
          float d0, d1;
          unpack2(d2, d0, d1);
          float d = d0 + d1;
          d += __shfl_xor_sync(0xffffffffu, d, 4);
          d += __shfl_xor_sync(0xffffffffu, d, 2);
          d += __shfl_xor_sync(0xffffffffu, d, 1);
          sc[rr][q4] = (n < limit[rr]) ? d : -INFINITY;
        }
      }

      float pr[R][kQuads];
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        float mt = sc[rr][0];
#pragma unroll
        for (int q4 = 1; q4 < kQuads; ++q4) mt = fmaxf(mt, sc[rr][q4]);
        const float mn = fmaxf(m[rr], mt);
        const float mu = (mn == -INFINITY) ? 0.f : mn;
        const float alpha = exp2f(m[rr] - mu);
        m[rr] = mn;
        float ls = l[rr] * alpha;
#pragma unroll
        for (int q4 = 0; q4 < kQuads; ++q4) {
          pr[rr][q4] = exp2f(sc[rr][q4] - mu);
          ls += pr[rr][q4];
        }
        l[rr] = ls;
        const uint64_t alpha2 = pack2(alpha, alpha);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint64_t a2 = mul2(pack2(acc[rr][2 * j], acc[rr][2 * j + 1]), alpha2);
          unpack2(a2, acc[rr][2 * j], acc[rr][2 * j + 1]);
        }
      }

#pragma unroll
      for (int q4 = 0; q4 < kQuads; ++q4) {
        const int row = q4 * 4 + kg;
        const uint4 v0 = *reinterpret_cast<const uint4*>(vt + swz128(row, p));
        const uint4 v1 = *reinterpret_cast<const uint4*>(vt + kHalfTileBytes + swz128(row, p));
        float vf[16];
        unpack8(v0, vf);
        unpack8(v1, vf + 8);
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
          const uint64_t p2 = pack2(pr[rr][q4], pr[rr][q4]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint64_t a2 = fma2(p2, pack2(vf[2 * j], vf[2 * j + 1]),
                                     pack2(acc[rr][2 * j], acc[rr][2 * j + 1]));
            unpack2(a2, acc[rr][2 * j], acc[rr][2 * j + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // merge the four key groups (lanes 8 and 16 apart)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[rr], off);
        const float lo = __shfl_xor_sync(0xffffffffu, l[rr], off);
        const float mn = fmaxf(m[rr], mo);
        const float mu = (mn == -INFINITY) ? 0.f : mn;
        const float ea = exp2f(m[rr] - mu), eb = exp2f(mo - mu);
        l[rr] = l[rr] * ea + lo * eb;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          acc[rr][j] = acc[rr][j] * ea + __shfl_xor_sync(0xffffffffu, acc[rr][j], off) * eb;
        m[rr] = mn;
      }
    }

    if (kg == 0) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const int t = rr / a.group, gi = rr - t * a.group;
        const RowDest d = row_dest<HPC>(a, seg, t, hh, gi);
        const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
        const float lse = final_lse(m[rr], l[rr]);
        if (d.out != nullptr) {
          uint4 w0, w1;
          w0.x = pack_bf16x2(acc[rr][0] * inv, acc[rr][1] * inv);
          w0.y = pack_bf16x2(acc[rr][2] * inv, acc[rr][3] * inv);
          w0.z = pack_bf16x2(acc[rr][4] * inv, acc[rr][5] * inv);
          w0.w = pack_bf16x2(acc[rr][6] * inv, acc[rr][7] * inv);
          w1.x = pack_bf16x2(acc[rr][8] * inv, acc[rr][9] * inv);
          w1.y = pack_bf16x2(acc[rr][10] * inv, acc[rr][11] * inv);
          w1.z = pack_bf16x2(acc[rr][12] * inv, acc[rr][13] * inv);
          w1.w = pack_bf16x2(acc[rr][14] * inv, acc[rr][15] * inv);
          *reinterpret_cast<uint4*>(d.out + 8 * p) = w0;
          *reinterpret_cast<uint4*>(d.out + 64 + 8 * p) = w1;
          if (p == 0 && d.lse != nullptr) *d.lse = lse;
        } else {
          float4* o0 = reinterpret_cast<float4*>(d.po + 8 * p);
          float4* o1 = reinterpret_cast<float4*>(d.po + 64 + 8 * p);
          o0[0] = make_float4(acc[rr][0] * inv, acc[rr][1] * inv, acc[rr][2] * inv,
                              acc[rr][3] * inv);
          o0[1] = make_float4(acc[rr][4] * inv, acc[rr][5] * inv, acc[rr][6] * inv,
                              acc[rr][7] * inv);
          o1[0] = make_float4(acc[rr][8] * inv, acc[rr][9] * inv, acc[rr][10] * inv,
                              acc[rr][11] * inv);
          o1[1] = make_float4(acc[rr][12] * inv, acc[rr][13] * inv, acc[rr][14] * inv,
                              acc[rr][15] * inv);
          if (p == 0) *d.plse = lse;
        }
      }
    }
  }
}

// ---------------------------------------------------- tensor-core consumer

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A (16x16, row) * B (16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int HPC, int TK, int BUDGET, int STAGES>
__device__ void consume_tc(const DecodeArgs& a, const Plan* plan, const uint8_t* stages,
                           uint64_t* full, uint64_t* empty, volatile int* abort_flag) {
  static_assert(TK == 16, "the mma tiles take 16 keys per tile");
  using Geo = Geometry<HPC, TK, BUDGET>;
  constexpr int kStageBytes = Geo::kStageBytes;
  constexpr int kHalfTileBytes = Geo::kHalfTileBytes;
  constexpr int kHeadTileBytes = Geo::kHeadTileBytes;
  const int lane = threadIdx.x & 31;
  const int hh = threadIdx.x >> 5;           // kv head within the CTA
  const int g = lane >> 2;         // fragment row group
  const int c = lane & 3;          // thread in group
  const int R = a.q_len * a.group;
  const int rA = g, rB = g + 8;    // the two q rows this thread's fragments touch
  const bool vA = rA < R, vB = rB < R;
  const int mat = lane >> 3;       // which 8x8 matrix this lane addresses in ldmatrix.x4
  const int mrow = lane & 7;

  SegmentSource src;
  src.init(a, plan, TK);
  Segment seg;
  int it = 0;                      // tiles consumed so far (ring position)
  bool aborted = false;
  while (!aborted && src.next(seg)) {
    const int kvh = seg.hg * HPC + hh;
    auto qrow_ptr = [&](int rr) {
      const int t = rr / a.group, gi = rr - t * a.group;
      return a.q + (static_cast<int64_t>(seg.b) * a.q_len + t) * a.q_stride_t +
             static_cast<int64_t>(kvh * a.group + gi) * a.q_stride_h;
    };
    const __nv_bfloat16* qA = vA ? qrow_ptr(rA) : a.q;
    const __nv_bfloat16* qB = vB ? qrow_ptr(rB) : a.q;
    const int limA = vA ? seg.seq_len - a.q_len + rA / a.group + 1 : 0;
    const int limB = vB ? seg.seq_len - a.q_len + rB / a.group + 1 : 0;

    uint32_t qa[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d0 = 16 * kk + 2 * c;
      qa[kk][0] = vA ? __ldg(reinterpret_cast<const uint32_t*>(qA + d0)) : 0u;
      qa[kk][1] = vB ? __ldg(reinterpret_cast<const uint32_t*>(qB + d0)) : 0u;
      qa[kk][2] = vA ? __ldg(reinterpret_cast<const uint32_t*>(qA + d0 + 8)) : 0u;
      qa[kk][3] = vB ? __ldg(reinterpret_cast<const uint32_t*>(qB + d0 + 8)) : 0u;
    }

    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    for (int i = 0; i < seg.ntiles; ++i, ++it) {
      const int s = it % STAGES;
      if (!mbar_wait(&full[s], (it / STAGES) & 1)) {
        *abort_flag = 1;
        report(a.status_flags, kFlagTimeout);
        aborted = true;
        break;
      }
      const uint32_t kt = smem_addr(stages + s * kStageBytes + hh * kHeadTileBytes);
      const uint32_t vt = kt + HPC * kHeadTileBytes;
      const int key0 = seg.k0 + i * TK;

      // S (16 rows x 16 keys) = Q K^T over 8 k-steps of 16 dims
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int key = ((mat >> 1) << 3) + mrow;
        const int ch = 2 * kk + (mat & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt + (ch >> 3) * kHalfTileBytes + swz128(key, ch & 7), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[kk], b0, b1);
        mma_bf16(sc[1], qa[kk], b2, b3);
      }

#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = key0 + 8 * nt + 2 * c + (e & 1);
          const int lim = (e < 2) ? limA : limB;
          sc[nt][e] = (key < lim) ? sc[nt][e] * a.scale_log2 : -INFINITY;
        }

      float tA = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float tB = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 1));
      tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 2));
      tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 1));
      tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 2));
      const float nA = fmaxf(mA, tA), nB = fmaxf(mB, tB);
      const float uA = (nA == -INFINITY) ? 0.f : nA;
      const float uB = (nB == -INFINITY) ? 0.f : nB;
      const float alA = exp2f(mA - uA), alB = exp2f(mB - uB);
      mA = nA;
      mB = nB;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - uA);
        sc[nt][1] = exp2f(sc[nt][1] - uA);
        sc[nt][2] = exp2f(sc[nt][2] - uB);
        sc[nt][3] = exp2f(sc[nt][3] - uB);
      }
      lA = lA * alA + (sc[0][0] + sc[0][1]) + (sc[1][0] + sc[1][1]);
      lB = lB * alB + (sc[0][2] + sc[0][3]) + (sc[1][2] + sc[1][3]);
      // rescale O in packed fp32 pairs (elements 0, 1: row A; 2, 3: row B)
      const uint64_t alA2 = pack2(alA, alA), alB2 = pack2(alB, alB);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const uint64_t ta = mul2(pack2(o[nt][0], o[nt][1]), alA2);
        const uint64_t tb = mul2(pack2(o[nt][2], o[nt][3]), alB2);
        unpack2(ta, o[nt][0], o[nt][1]);
        unpack2(tb, o[nt][2], o[nt][3]);
      }
      uint32_t pa[4];
      pa[0] = pack_bf16x2(sc[0][0], sc[0][1]);
      pa[1] = pack_bf16x2(sc[0][2], sc[0][3]);
      pa[2] = pack_bf16x2(sc[1][0], sc[1][1]);
      pa[3] = pack_bf16x2(sc[1][2], sc[1][3]);

      // O (16 rows x 128 dims) += P V
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int key = ((mat & 1) << 3) + mrow;
        const int ch = 2 * dp + (mat >> 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(vt + (ch >> 3) * kHalfTileBytes + swz128(key, ch & 7), v0, v1, v2, v3);
        mma_bf16(o[2 * dp], pa, v0, v1);
        mma_bf16(o[2 * dp + 1], pa, v2, v3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);

#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int rr = half ? rB : rA;
      if (rr >= R) continue;
      const float l = half ? lB : lA;
      const float m = half ? mB : mA;
      const int t = rr / a.group, gi = rr - t * a.group;
      const RowDest d = row_dest<HPC>(a, seg, t, hh, gi);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (d.out != nullptr) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          *reinterpret_cast<uint32_t*>(d.out + 8 * nt + 2 * c) =
              pack_bf16x2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (c == 0 && d.lse != nullptr) *d.lse = final_lse(m, l);
      } else {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          *reinterpret_cast<float2*>(d.po + 8 * nt + 2 * c) =
              make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (c == 0) *d.plse = final_lse(m, l);
      }
    }
  }
}

// Before the dependency wait the previous kernel (the append) is still
// running and HBM is mostly idle: start this CTA's first ring of K/V tiles
// (split schedule), or the line(s) of sequence lengths the plan reads
// (balanced schedule), towards L2.  A prefetch binds no value -- the loads
// after the wait read L2, which the previous kernel's writes update -- so a
// block table or length that the previous kernel rewrites costs only a wasted
// prefetch.  The two values read here go through L2 only (ld.global.cg), so
// no L1 copy of them outlives the wait.
template <int HPC, int TK, int NT>
__device__ void prefetch_before_wait(const CUtensorMap* kmap, const CUtensorMap* vmap,
                                     const DecodeArgs& a) {
  const int lane = threadIdx.x & 31;
  if (a.num_splits == 0) {
    for (int i = lane * 32; i < a.batch; i += 32 * 32) prefetch_l2(a.seq_lens + i);
    return;
  }
  if (lane >= NT) return;
  const int b = blockIdx.z, hg = blockIdx.y, j = blockIdx.x;
  const long long cap = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
  long long L = __ldcg(a.seq_lens + b);
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const long long chunk = static_cast<long long>(a.chunk_pages) * a.block_size;
  const long long k0 = static_cast<long long>(j) * chunk;
  const long long k1 = (j == a.num_splits - 1) ? L : min(L, k0 + chunk);
  const long long key = k0 + static_cast<long long>(lane) * TK;
  if (key >= k1) return;
  const long long page = key / a.block_size;
  const int blk = __ldcg(a.block_tables + static_cast<long long>(b) * a.max_blocks_per_seq + page);
  if (blk < 0 || blk >= a.num_blocks) return;
  const int slot = static_cast<int>(key - page * a.block_size);
  tma_prefetch_5d(kmap, 0, slot, 0, hg * HPC, blk);
  tma_prefetch_5d(vmap, 0, slot, 0, hg * HPC, blk);
}

// ------------------------------------------------------------------ kernel

template <int HPC, int TK, int BUDGET, int R, bool TC>
__global__ void __launch_bounds__(Geometry<HPC, TK, BUDGET>::kThreads, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using Geo = Geometry<HPC, TK, BUDGET>;
  constexpr int STAGES = Geo::kStages;
  constexpr int kProducer = Geo::kConsumers;    // warp index of the producer
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES];
  __shared__ uint64_t empty[STAGES];
  __shared__ int abort_flag;
  __shared__ int issued;
  __shared__ Plan plan;
  __shared__ long long wsum[32];
  uint8_t* stages = align1024(smem_raw);

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], Geo::kConsumers);
    }
    abort_flag = 0;
    issued = 0;
    fence_barrier_init();
  }
  if (warp == kProducer) prefetch_before_wait<HPC, TK, STAGES>(&kmap, &vmap, a);
  __syncthreads();
  // launched as a programmatic dependent: everything below may read what the
  // previous kernel in the stream wrote (q, appended K/V, tables, lengths)
  pdl_launch_dependents();
  pdl_wait();

  if (a.num_splits == 0) {
    make_plan(a, &plan, wsum);
    write_empty_units(a, HPC);
  }
  if (warp == kProducer) {
    produce<HPC, TK, BUDGET, STAGES>(&kmap, &vmap, a, &plan, stages, full, empty, &abort_flag,
                                     &issued);
  } else {
    if constexpr (TC) {
      consume_tc<HPC, TK, BUDGET, STAGES>(a, &plan, stages, full, empty, &abort_flag);
    } else {
      consume_simt<HPC, TK, BUDGET, STAGES, R>(a, &plan, stages, full, empty, &abort_flag);
    }
  }
  __syncthreads();
  if (abort_flag && threadIdx.x == kProducer * 32) drain<STAGES>(full, issued);
}

template <int HPC, int TK, int BUDGET, int R, bool TC>
cudaError_t launch_one(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeArgs& a,
                       int grid_ctas, cudaStream_t stream) {
  using Geo = Geometry<HPC, TK, BUDGET>;
  auto kern = paged_decode_kernel<HPC, TK, BUDGET, R, TC>;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = set_smem_limit_once(kern, Geo::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid = a.num_splits == 0 ? dim3(grid_ctas, 1, 1)
                                      : dim3(a.num_splits, a.num_kv_heads / HPC, a.batch);
  return launch_pdl(kern, grid, dim3(Geo::kThreads), Geo::kSmemBytes, stream, kmap, vmap, a);
}

// Per head count: the CUDA-core path's tile and ring, and the mma path's.
template <int HPC>
struct Config;
template <>
struct Config<8> {
  static constexpr int kSimtTK = 16, kSimtBudget = 192;
  static constexpr int kTcBudget = 192;
};
template <>
struct Config<4> {
  static constexpr int kSimtTK = 16, kSimtBudget = 192;
  static constexpr int kTcBudget = 192;
};
template <>
struct Config<2> {
  static constexpr int kSimtTK = 16, kSimtBudget = 96;
  static constexpr int kTcBudget = 96;
};
template <>
struct Config<1> {
  static constexpr int kSimtTK = 16, kSimtBudget = 64;
  static constexpr int kTcBudget = 64;
};

template <int HPC>
cudaError_t launch_hpc(const DecodePlan& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const DecodeArgs& a, int grid_ctas, cudaStream_t stream) {
  using C = Config<HPC>;
  if (p.tensor_core)
    return launch_one<HPC, 16, C::kTcBudget, 16, true>(kmap, vmap, a, grid_ctas, stream);
  constexpr int TK = C::kSimtTK, B = C::kSimtBudget;
  switch (p.rows) {
    case 1: return launch_one<HPC, TK, B, 1, false>(kmap, vmap, a, grid_ctas, stream);
    case 2: return launch_one<HPC, TK, B, 2, false>(kmap, vmap, a, grid_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int HPC>
void fill_plan(DecodePlan& p) {
  using C = Config<HPC>;
  const int tk = p.tensor_core ? 16 : C::kSimtTK;
  const int budget = p.tensor_core ? C::kTcBudget : C::kSimtBudget;
  p.tile_keys = tk;
  const int stage = 2 * HPC * 2 * tk * 128;
  int stages = budget * 1024 / stage;
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  const int smem = stages * stage + 1024 + 512;       // + static shared memory
  p.ctas_per_sm = smem > 0 ? (228 * 1024) / smem : 1;
  if (p.ctas_per_sm < 1) p.ctas_per_sm = 1;
}

}  // namespace

DecodePlan plan_decode(int num_kv_heads, int rows) {
  DecodePlan p;
  int hpc = 8;
  while (hpc > 1 && (num_kv_heads % hpc) != 0) hpc >>= 1;
  p.heads_per_cta = hpc;
  p.tensor_core = rows > 2;
  p.rows = rows;
  switch (hpc) {
    case 8: fill_plan<8>(p); break;
    case 4: fill_plan<4>(p); break;
    case 2: fill_plan<2>(p); break;
    default: fill_plan<1>(p); break;
  }
  return p;
}

cudaError_t launch_paged_decode(const DecodePlan& p, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const DecodeArgs& a, int grid_ctas,
                                cudaStream_t stream) {
  switch (p.heads_per_cta) {
    case 8: return launch_hpc<8>(p, kmap, vmap, a, grid_ctas, stream);
    case 4: return launch_hpc<4>(p, kmap, vmap, a, grid_ctas, stream);
    case 2: return launch_hpc<2>(p, kmap, vmap, a, grid_ctas, stream);
    case 1: return launch_hpc<1>(p, kmap, vmap, a, grid_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkvqk
