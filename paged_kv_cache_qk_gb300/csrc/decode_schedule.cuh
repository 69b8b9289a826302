// Segment schedules of the split-KV decode kernels (shared by the CUDA-core /
// mma.sync kernel and the tcgen05 kernel): which runs of keys of which
// (sequence, kv-head group) a CTA works through, and where each run's result
// goes.
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, ...", section "概述 / Summary", item 1 (split-KV decode
// over the paged cache).
//   * split schedule (num_splits >= 1): CTA (split, head group, sequence)
//     takes split `split` of the sequence: chunk_pages pages per split, the
//     last split takes the rest;
//   * balanced schedule (num_splits == 0): the pages of all units laid end to
//     end; CTA c takes pages [c*TP/G, (c+1)*TP/G) (G = min(grid, TP)),
//     crossing sequence boundaries; a unit covered whole by one CTA is written
//     to the output, a unit cut across CTAs leaves one partial per CTA in slot
//     (cta + unit), merged by the balanced combine kernel.
#pragma once

#include "device_common.cuh"
#include "kernels.h"

namespace pkvqk {
namespace sched {

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
__device__ inline void make_plan(const DecodeArgs& a, Plan* plan, long long* wsum) {
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
__device__ inline void write_empty_units(const DecodeArgs& a, int hpc) {
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


}  // namespace sched
}  // namespace pkvqk
