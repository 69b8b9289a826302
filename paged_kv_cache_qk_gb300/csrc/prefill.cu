// Causal multi-query attention over the paged K/V cache -- the chunked-prefill
// step (many new tokens of one sequence at once) and, as its small case, the
// speculative-verify step -- on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory, operands staged by TMA).
//
// Operation: InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid
// attention backend, fused rms_norm_rope, chunked prefill + prompt-lookup spec
// decoding", section "概述 / Summary", items 1 and 4: new token t of sequence
// b (t < q_len) sits at position seq_len - q_len + t and attends to the keys
// n <= seq_len - q_len + t of its own sequence, gathered page by page through
// the block table; q head h reads kv head h / group; softmax scale D^-1/2
// unless the caller gives one.  q_len is either one value for the batch or,
// varlen (the FlashAttention-2 varlen role of Summary item 1), per sequence
// from cumulative row offsets; the grid covers the longest, and row tiles past
// a shorter sequence's rows do nothing.  Launch order: a (sequence, kv head)'s
// row tiles last-first (the most keys first); varlen grids run every
// sequence's last row tiles first.
//
// One CTA = two tiles A and B of 128 packed rows r = t * group + (h % group)
// of one (sequence, kv head) -- 256 consecutive rows -- restricted to one
// split of the key range.  Keys stream in tiles of 128 through two-stage TMA
// rings (K and V separately); both row tiles use every key tile, and the
// tensor core alternates between them so that one tile's softmax runs while
// the other tile's MMAs do (ping-pong).  Warp roles:
//   warps 0-7 / 8-15  softmax of tile A / B, two threads per row: warp
//              8x + 4h + q owns lanes 32q..32q+31 (rows) and keys 64h..64h+63
//              of every key tile.  Reads its half of the score row S = Q K^T
//              from tensor memory, keeps the running max and sum, writes P
//              (bf16 pairs) back over the S columns it has read, swaps its
//              reference max with the other half once per tile, rescales its
//              half of O in tensor memory only when the max grew by more than
//              2^8 (P <= 2^8 otherwise), and writes its 64 output dims;
//   warp 16    TMA producer: Q tile A at set-up (one box per 64-dim half,
//              where q's layout allows), then one box per (page, 64-dim half)
//              of K and one per page of V, Q tile B right after K(0) (the SM's
//              TMA unit takes the boxes one after another, so S_A(0) waits for
//              two boxes less);
//   warp 17    allocates the tensor memory; lane 0 issues the MMAs in the
//              order  S_A(0) S_B(0) | PV_A(i) S_A(i+1) PV_B(i) S_B(i+1) | ...
//              S_x = Q_x K_i^T  (M 128 rows, N 128 keys, K 128 dims; both
//                               operands in shared memory),
//              O_x += P_x V_i   (M 128 rows, N 128 dims, K 128 keys; P from
//                               tensor memory, V from shared memory).
// Output: a whole row tile (inside its sequence, single split) is staged as
// bf16 in its Q tile's shared memory and leaves as two TMA boxes; partial
// tiles and split partials are stored by the softmax threads.
// S_x(i+1) overwrites the columns that held P_x(i): the MMAs of one thread
// run in issue order, and PV_x(i) is issued first.  The commit that signals
// S_x(i+1) also covers PV_x(i), so softmax x may rescale O_x as soon as it
// sees S_x(i+1).
//
// Shared memory (1024-byte aligned, 128-byte swizzle everywhere, the layout
// the MMA descriptors describe):
//   Q_A, Q_B  [2 dim halves][128 rows][64 bf16]      2 x 32 KiB
//   K stage s [2 dim halves][128 keys][64 bf16]      2 x 32 KiB
//   V stage s [128 / tb boxes][2 dim halves][tb keys][64 bf16], tb the
//             slots per box (16 at 16-key pages)     2 x 32 KiB
//   pair-swap slots [tile][parity][half][128 rows] fp32  4 KiB
// Tensor memory: S_A at columns 0-127 (P_A over columns 0-31 and 64-95), S_B
// 128-255 (P_B likewise), O_A 256-383, O_B 384-511.
//
// Every wait is bounded: on a timeout the CTA reports PKVQK_FLAG_WAIT_TIMEOUT,
// lets its own copies and MMAs in flight finish (bounded), frees its tensor
// memory and exits.
#include "device_common.cuh"
#include "prefill.h"
#include "tc5.cuh"

#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

namespace pkvqk {

namespace {

constexpr int kM = 128;                        // rows per row tile
constexpr int kN = 128;                        // keys per key tile
static_assert(2 * kM == kPrefillRowsPerCta, "two row tiles per CTA");
constexpr int kHalf = 128 * 128;               // [128 rows][64 bf16] sub-tile, bytes
constexpr int kTile = 2 * kHalf;               // [128 rows][128 bf16], bytes
constexpr int kStages = 2;
constexpr int kOffQ = 0;                       // Q_A, Q_B
constexpr int kOffK = 2 * kTile;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kDataBytes = kOffV + kStages * kTile;
constexpr int kSoftmaxWarps = 16;             // 8 per row tile, two per lane quadrant
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                  // + x * kN
constexpr uint32_t kColO = 256;                // + x * kN
constexpr float kRescaleLog2 = 8.f;
constexpr float kLn2 = 0.6931471805599453f;

struct Bars {
  uint64_t full_k[kStages], full_v[kStages];     // TMA landed
  uint64_t empty_k[kStages], empty_v[kStages];   // the MMAs reading a stage finished
  uint64_t s_full[2];                            // S_x written (and the PV before it done)
  uint64_t p_full[2];                            // P_x written (and O_x rescaled)
  uint64_t pv_done[2];                           // the last O_x += P_x V finished
  uint64_t drain;                                // MMA thread's own completion (timeout path)
  uint64_t xch[2][4];                            // warp pair (tile, lane quadrant) swaps
  uint64_t q_full[2];                            // Q tile x landed (TMA)
  uint64_t o_staged[2];                          // tile x's output rows staged for TMA
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");
constexpr int kOffSlots = kDataBytes + 256;   // pair-swap slots [tile][parity][half][row]
constexpr int kSlotBytes = 2 * 2 * 2 * kM * 4;
constexpr int kSmemBytes = kOffSlots + kSlotBytes + 1024;   // + alignment slack

// x / group for x >= 0: a shift where the group is a power of two (the
// usual case), else the division.
__device__ __forceinline__ int div_group(const PrefillArgs& a, int x) {
  return a.group_shift >= 0 ? (x >> a.group_shift) : x / a.group;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t s = smem_addr(p);
  return p + (((s + 1023u) & ~1023u) - s);
}

// A [128 rows][128 bf16] operand stored as two 64-wide swizzled halves, read
// K-major in 16-element steps: step kk is 32 bytes into the rows of half kk/4;
// 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_k_major(uint32_t tile, int kk) {
  return tc5::smem_desc_sw128(tile + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
}

// Slots per cache box: the largest power of two dividing the page size, at
// most a key tile; a tile's boxes start at multiples of it, so none crosses a
// page.  Returns log2.
__device__ __forceinline__ int box_shift(int block_size) {
  return __ffs(min(block_size & -block_size, kN)) - 1;
}

// V stage as the MN-major B operand of O += P V (N = dims, K = keys), one
// TMA box per tb = 2^tbs keys holding both dim halves: box j at 256 tb j,
// [2 dim halves][tb keys][64 bf16 swizzled], so the halves are 128 tb bytes
// apart (leading offset) and 8-key groups 1024 apart (stride offset); the
// 16-key step ks starts in box 16 ks / tb, 16 ks % tb rows in.  One box per
// page instead of one per (page, half): at 16-key pages the SM's TMA unit
// costs ~50 cycles a box on top of ~2.2 a 128-byte row, and V's boxes were
// half of what held up K.
__device__ __forceinline__ uint32_t v_step_offset(int ks, int tbs) {
  const int k = ks * 16;
  return static_cast<uint32_t>(((k >> tbs) << (tbs + 8)) + ((k & ((1 << tbs) - 1)) << 7));
}
__device__ __forceinline__ uint32_t v_row_offset(int key, int half, int tbs) {
  return static_cast<uint32_t>(((key >> tbs) << (tbs + 8)) + (half << (tbs + 7)) +
                               ((key & ((1 << tbs) - 1)) << 7));
}

// 5-D tiled TMA load without an L2 hint: K/V tiles are read by every row tile
// of their (sequence, kv head), so they should stay in L2 meanwhile.
__device__ __forceinline__ void tma_load_5d_keep(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                 int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_addr(bar))
      : "memory");
}

// One box of a row-tile map (q): 64 dims x group heads x 128 / group tokens.
__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* map, uint64_t* bar,
                                              int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// The same box from shared memory to out, then wait until shared memory has
// been read (the CTA may leave after that).
__device__ __forceinline__ void tma_store_rows(const void* src, const CUtensorMap* map, int c0,
                                               int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
      : "memory");
}
__device__ __forceinline__ void tma_store_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

struct Work {
  int b, g, j, mt;
  int L;         // keys of the sequence (clamped to the table)
  int k0, k1;    // the split's key range
  int key_end;   // keys at or past key_end are visible to no row of the CTA
  int ntiles;
  int q_len;     // this sequence's new tokens
  long long q0;  // row of q/out holding its token 0
  int rows;      // q_len * group
  bool has_b;    // row tile B holds rows
};

__device__ Work decode_work(const PrefillArgs& a) {
  Work w;
  if (a.mt_major) {
    // the launch order runs over all sequences' last row tiles first: for
    // fresh prompts a row tile's keys grow with its index, so this hands the
    // longest work out first
    const int per_mt = gridDim.y * a.num_kv_heads * a.num_splits;
    int x = blockIdx.y * gridDim.x + blockIdx.x;
    w.mt = a.m_tiles - 1 - x / per_mt;
    x %= per_mt;
    w.b = x / (a.num_kv_heads * a.num_splits);
    x %= a.num_kv_heads * a.num_splits;
    w.g = x / a.num_splits;
    w.j = x % a.num_splits;
  } else {
    // within a (sequence, kv head) the last row tile (the most keys) first
    int x = blockIdx.x;
    w.mt = a.m_tiles - 1 - x % a.m_tiles;
    x /= a.m_tiles;
    w.g = x % a.num_kv_heads;
    w.j = x / a.num_kv_heads;
    w.b = blockIdx.y;
  }
  const long long cap = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
  const long long L = min(static_cast<long long>(max(a.seq_lens[w.b], 0)), cap);
  w.L = static_cast<int>(L);
  const long long chunk_keys = static_cast<long long>(a.chunk_pages) * a.block_size;
  w.k0 = static_cast<int>(min(L, w.j * chunk_keys));
  w.k1 = (w.j == a.num_splits - 1) ? w.L : static_cast<int>(min(L, (w.j + 1) * chunk_keys));
  if (a.cu_seqlens_q != nullptr) {
    const long long c0 = a.cu_seqlens_q[w.b], c1 = a.cu_seqlens_q[w.b + 1];
    w.q0 = c0;
    w.q_len = static_cast<int>(max(0ll, min(c1 - c0, static_cast<long long>(a.q_len))));
  } else {
    w.q0 = static_cast<long long>(w.b) * a.q_len;
    w.q_len = a.q_len;
  }
  w.rows = w.q_len * a.group;
  const int row0 = w.mt * 2 * kM;
  w.has_b = row0 + kM < w.rows;
  const int last_row = min(row0 + 2 * kM - 1, w.rows - 1);
  const int t_last = div_group(a, max(last_row, 0));   // rows == 0: no tiles either way
  w.key_end = max(w.k0, min(w.k1, w.L - w.q_len + t_last + 1));
  w.ntiles = row0 < w.rows ? (w.key_end - w.k0 + kN - 1) / kN : 0;
  return w;
}

// ------------------------------------------------------------- producer

__device__ void produce(const PrefillArgs& a, const Work& w, const CUtensorMap* kmap,
                        const CUtensorMap* vmap, const CUtensorMap* qmap, uint8_t* smem,
                        Bars* bars, int* issued_out) {
  const int lane = threadIdx.x & 31;
  const int bs = a.block_size;
  const int tbs = box_shift(bs);
  const int tb = 1 << tbs;
  const int ppt = kN >> tbs;                    // boxes per key tile
  const int32_t* bt = a.block_tables + static_cast<long long>(w.b) * a.max_blocks_per_seq;
  const int oob = static_cast<int>(a.num_blocks);   // past the extent: TMA fills zeros
  // page id of box `lane` of tile i, when the box holds a visible key; loaded
  // one tile ahead, so that its latency is not in the chain V(i) -> K(i+1)
  auto box_visible = [&](int i) { return lane < ppt && w.k0 + i * kN + lane * tb < w.key_end; };
  auto page_id = [&](int i) {
    return box_visible(i) ? __ldg(bt + (w.k0 + i * kN + lane * tb) / bs) : oob;
  };
  int id_next = w.ntiles > 0 ? page_id(0) : oob;
  int issued = 0;
  for (int i = 0; i < w.ntiles; ++i) {
    const int s = i & 1;
    const uint32_t rel = ((i >> 1) - 1) & 1;         // release of tile i - 2
    uint8_t* kt = smem + kOffK + s * kTile;
    uint8_t* vt = smem + kOffV + s * kTile;
    int blk = id_next;
    if (box_visible(i) && (blk < 0 || static_cast<long long>(blk) >= a.num_blocks)) {
      report(a.status_flags, kFlagBadBlock);
      blk = oob;
    }
    if (i + 1 < w.ntiles) id_next = page_id(i + 1);
    int slot0 = 0;
    if (lane < ppt) {
      const int key = w.k0 + i * kN + lane * tb;   // first key of box `lane`
      slot0 = key - (key / bs) * bs;
    }
    bool ok = true;
    if (lane == 0 && i >= 2) ok = mbar_wait(&bars->empty_k[s], rel);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        bars->abort = 1;
        report(a.status_flags, kFlagTimeout);
      }
      break;
    }
    if (lane == 0) mbar_arrive_expect_tx(&bars->full_k[s], kTile);
    __syncwarp();
    if (lane < ppt) {
      tma_load_5d_keep(kt + lane * tb * 128, kmap, &bars->full_k[s], 0, slot0, 0, w.g, blk);
      tma_load_5d_keep(kt + kHalf + lane * tb * 128, kmap, &bars->full_k[s], 0, slot0, 1, w.g,
                       blk);
    }
    if (i == 0 && a.q_tma && w.has_b && lane == 0) {
      mbar_arrive_expect_tx(&bars->q_full[1], kTile);
      const int tok = static_cast<int>(w.q0 + div_group(a, w.mt * 2 * kM + kM));
      for (int dh = 0; dh < 2; ++dh)
        tma_load_rows(smem + kOffQ + kTile + dh * kHalf, qmap, &bars->q_full[1], dh * 64,
                      w.g * a.group, tok);
    }
    if (lane == 0 && i >= 2) ok = mbar_wait(&bars->empty_v[s], rel);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        bars->abort = 1;
        report(a.status_flags, kFlagTimeout);
      }
      issued = -(i + 1);                            // K of tile i is in flight, V is not
      break;
    }
    if (lane == 0) mbar_arrive_expect_tx(&bars->full_v[s], kTile);
    __syncwarp();
    if (lane < ppt)
      tma_load_5d_keep(vt + lane * tb * 256, vmap, &bars->full_v[s], 0, slot0, 0, w.g, blk);
    issued = i + 1;
  }
  *issued_out = issued;
}

// After a timeout: wait (bounded) for the last copies issued into each stage.
__device__ void drain_copies(Bars* bars, int issued) {
  const bool v_missing = issued < 0;
  const int n = v_missing ? -issued : issued;
  for (int i = n - 2 < 0 ? 0 : n - 2; i < n; ++i) {
    const int s = i & 1;
    mbar_wait(&bars->full_k[s], (i >> 1) & 1);
    if (!(v_missing && i == n - 1)) mbar_wait(&bars->full_v[s], (i >> 1) & 1);
  }
}

// ------------------------------------------------------------ MMA issue

__device__ void issue_mmas(const PrefillArgs& a, const Work& w, uint8_t* smem, Bars* bars,
                           uint32_t tmem) {
  const int last = w.has_b ? 1 : 0;            // the row tile that reads a stage last
  const int n = w.ntiles;
  constexpr uint32_t idesc_s = tc5::idesc_bf16_f32(kM, kN, false);
  constexpr uint32_t idesc_pv = tc5::idesc_bf16_f32(kM, kHeadDim, true);
  // Descriptors as 32-bit halves; every operand of this kernel shares the high
  // half (stride offset 1024, version, 128-byte swizzle), and a 16-element
  // step moves only the low half's start address.
  const uint64_t d0 = desc_k_major(smem_addr(smem + kOffQ), 0);
  const uint32_t hi = static_cast<uint32_t>(d0 >> 32);
  const uint32_t q_lo = static_cast<uint32_t>(d0);
  const uint32_t k_lo = static_cast<uint32_t>(desc_k_major(smem_addr(smem + kOffK), 0));
  const int tbs = box_shift(a.block_size);
  const uint32_t v_lo = static_cast<uint32_t>(
      tc5::smem_desc_sw128(smem_addr(smem + kOffV), 128u << tbs, 1024));
  uint32_t v_step[kN / 16];
#pragma unroll
  for (int ks = 0; ks < kN / 16; ++ks) v_step[ks] = v_step_offset(ks, tbs) >> 4;
  // S_x(i) = Q_x K_i^T  (the caller has waited for K_i)
  auto mma_s = [&](int x, int i) {
    const int s = i & 1;
    const uint32_t qa = q_lo + (x * kTile >> 4), kb = k_lo + (s * kTile >> 4);
    const uint32_t dst = tmem + kColS + x * kN;
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      const uint32_t step = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
      tc5::mma_f16_lh(dst, qa + step, hi, kb + step, hi, idesc_s, kk > 0 ? 1u : 0u);
    }
    tc5::commit(&bars->s_full[x]);
    if (x == last) tc5::commit(&bars->empty_k[s]);
  };
  // O_x += P_x V_i  (the caller has waited for P_x and V_i)
  auto mma_pv = [&](int x, int i) {
    const int s = i & 1;
    const uint32_t vb = v_lo + (s * kTile >> 4);
    const uint32_t dst = tmem + kColO + x * kN, p0 = tmem + kColS + x * kN;
    // P_x: 16 keys per step = 8 columns of bf16 pairs; keys 64h.. at column 64h
#pragma unroll
    for (int ks = 0; ks < kN / 16; ++ks)
      tc5::mma_f16_ts_lh(dst, p0 + (ks >> 2) * (kN / 2) + (ks & 3) * 8, vb + v_step[ks], hi,
                         idesc_pv, (i > 0 || ks > 0) ? 1u : 0u);
    if (i == n - 1) tc5::commit(&bars->pv_done[x]);
    if (x == last) tc5::commit(&bars->empty_v[s]);
  };
  bool ok = true;
  // Q tile A by TMA (issued at set-up), tile B after K(0)
  if (a.q_tma && n > 0) ok = mbar_wait(&bars->q_full[0], 0);
  if (ok && n > 0) ok = mbar_wait(&bars->full_k[0], 0);
  if (ok && n > 0) {
    tc5::fence_after_sync();
    mma_s(0, 0);
    if (w.has_b) {
      if (a.q_tma) ok = mbar_wait(&bars->q_full[1], 0);
      if (ok) {
        tc5::fence_after_sync();
        mma_s(1, 0);
      }
    }
  }
  for (int i = 0; i < n && ok; ++i) {
    // V_i and K_(i+1) first, while the softmax still works on P_A(i): they
    // have almost always landed, and a wait between PV_A(i) and S_A(i+1)
    // left the tensor pipe idle (~330 cycles a tile, even on a completed
    // barrier)
    ok = mbar_wait(&bars->full_v[i & 1], (i >> 1) & 1);
    if (ok && i + 1 < n) ok = mbar_wait(&bars->full_k[(i + 1) & 1], ((i + 1) >> 1) & 1);
    if (ok) ok = mbar_wait(&bars->p_full[0], i & 1);
    if (!ok) break;
    tc5::fence_after_sync();
    mma_pv(0, i);
    if (i + 1 < n) mma_s(0, i + 1);
    if (w.has_b) {
      ok = mbar_wait(&bars->p_full[1], i & 1);
      if (!ok) break;
      tc5::fence_after_sync();
      mma_pv(1, i);
      if (i + 1 < n) mma_s(1, i + 1);
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
//
// Two threads per row: the warp pair (tile x, lane quadrant q, half 0/1)
// shares tensor-memory lanes 32q..32q+31, and half h owns keys 64h..64h+63 of
// every key tile and dims 64h..64h+63 of O.  Each thread keeps a reference
// max m_ref (log2 units, an integer once set) and writes P = 2^(s sl2 - m_ref)
// as bf16 pairs over the S columns it has already read: half h's keys
// 64h + 2j, +1 land in column 64h + j, which is where the PV MMA reads them.
// A 32-key chunk's max is taken from registers before its exponentials; if
// it exceeds m_ref by more than 2^8 the reference is raised to the ceiling of
// that max first, so P <= 2^8 always, and P already written for the tile is
// scaled by the (exact, power-of-two) ratio.  After the tile the two halves
// swap their references and the lower one scales its P the same way, so both
// use one reference for the row; O is rescaled only when that reference rose.

// 2^x on the SFU (relative error ~2^-22; -inf -> +0).  P is rounded to bf16
// right after, so the approximate unit is accurate enough.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^d for an integer-valued d <= 0: exact, 0 below the normal range (and for
// d = -inf).
__device__ __forceinline__ float pow2_int(float d) {
  return d < -126.f ? 0.f : __int_as_float((127 + static_cast<int>(d)) << 23);
}

// Multiply the bf16 pairs in kWords columns at taddr by the power of two f
// (exact unless a value drops below the normal range).
template <int kWords>
__device__ __forceinline__ void scale_p(uint32_t taddr, float f) {
  tc5::wait_st();                              // this thread's P stores to these columns
  float w[32];
  if (kWords == 16) tc5::tmem_ld16(taddr, w);
  else tc5::tmem_ld32(taddr, w);
  tc5::wait_ld();
  uint32_t p[kWords];
#pragma unroll
  for (int j = 0; j < kWords; ++j) {
    const uint32_t u = __float_as_uint(w[j]);
    p[j] = pack_bf16x2(bf16lo(u) * f, bf16hi(u) * f);
  }
  if (kWords == 16) tc5::tmem_st16(taddr, p);
  else tc5::tmem_st32u(taddr, p);
}

// This thread's 64 keys of one key tile: S from scol (two 32-column chunks),
// P pairs to pcol (16 columns per chunk).  kbase = the first key's index in the
// tile; keys kbase + e >= nvis are masked.  Returns the sum of P (before
// rounding) against the m_ref in force at the end.
// One pass over this thread's 64 keys of key tile i: two 32-column chunks,
// each with its max, a rise of the reference when the chunk's max passes it
// by more than 2^8, the exponentials and the P stores.  The reference is
// final once the second chunk's max is in: `publish` hands it to the other
// half of the row there, so that the exchange overlaps that chunk's
// exponentials instead of following them.
template <bool kMasked, typename Publish>
__device__ __forceinline__ float half_tile(uint32_t scol, uint32_t pcol, int kbase, int nvis,
                                           float sl2, float& m_ref, Publish&& publish) {
  float psum = 0.f;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float v[32];
    tc5::tmem_ld32(scol + c * 32, v);
    tc5::wait_ld();
    if (kMasked) {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = (kbase + c * 32 + e < nvis) ? v[e] : -INFINITY;
    }
    float m4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) m4[j] = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; e += 2) m4[(e >> 1) & 3] = max3(m4[(e >> 1) & 3], v[e], v[e + 1]);
    const float mt = max3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;
    const bool grow = mt > m_ref + kRescaleLog2;
    if (__any_sync(0xffffffffu, grow)) {
      const float m_new = grow ? ceilf(mt) : m_ref;
      const float f = grow ? pow2_int(m_ref - m_new) : 1.f;
      if (c == 1) scale_p<16>(pcol, f);
      psum *= f;
      m_ref = m_new;
    }
    if (c == 1) publish(m_ref);
    const float u = (m_ref == -INFINITY) ? 0.f : m_ref;
    const uint64_t scale2 = pack2(sl2, sl2), shift2 = pack2(-u, -u);
    uint64_t acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = pack2(0.f, 0.f);
    uint32_t pk[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      float x0, x1;
      unpack2(fma2(pack2(v[2 * q], v[2 * q + 1]), scale2, shift2), x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);   // masked: 2^-inf = 0
      acc[q & 3] = add2(acc[q & 3], pack2(p0, p1));
      pk[q] = pack_bf16x2(p0, p1);
    }
    tc5::tmem_st16(pcol + c * 16, pk);
    const uint64_t t = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
    float t0, t1;
    unpack2(t, t0, t1);
    psum += t0 + t1;
  }
  return psum;
}

// Swap one value per row with the other half of the warp pair, in two parts
// so that work can run in between: publish v in this half's slot of the
// current parity and arrive on the pair's barrier; then wait (bounded) for
// the partner's arrival and read its slot.  Slots alternate by parity, so a
// slot is rewritten only after the partner's next arrival, which follows its
// read.
__device__ __forceinline__ void swap_publish(float v, float* slots, uint64_t* bar,
                                             uint32_t uses, int half, int r) {
  const int p = uses & 1;
  slots[(p * 2 + half) * kM + r] = v;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ float swap_read(float* slots, uint64_t* bar, uint32_t& uses, int half,
                                           int r, bool& ok) {
  const int p = uses & 1;
  ok = warp_wait(bar, p) && ok;
  ++uses;
  return slots[(p * 2 + (half ^ 1)) * kM + r];
}

__device__ __forceinline__ float pair_swap(float v, float* slots, uint64_t* bar, uint32_t& uses,
                                           int half, int r, bool& ok) {
  swap_publish(v, slots, bar, uses, half, r);
  return swap_read(slots, bar, uses, half, r, ok);
}

// This thread's half of an output row of tile x: O / l for dims 64h..64h+63
// (bf16, or the fp32 partial of the split), and the log-sum-exp (half 0).
// Inline: out of line, its code was cold in the SM's instruction cache at
// every CTA's end (1.2 us from the last swap to the first output load,
// against 0.5 inline), which cost more than the few spills inlining brings
// at 96 registers.
__device__ __forceinline__ void write_rows(const PrefillArgs& a, const Work& w, uint32_t tmem,
                                        uint8_t* smem, Bars* bars, const CUtensorMap* omap,
                                        int x, int half, float m_ref, float l) {
  const int r = ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31);
  const int rg = w.mt * 2 * kM + x * kM + r;
  const int t0 = div_group(a, rg);
  // rows outside the sequence, or (inconsistent offsets) outside q/out: no write;
  // every lane still takes part in the warp-wide tensor-memory loads below
  const bool valid = rg < w.rows && w.q0 + t0 >= 0 && w.q0 + t0 < a.total_q;
  const int t = valid ? t0 : 0;
  const int hh = valid ? rg - t * a.group : 0;
  const uint32_t o_cols = tmem + (static_cast<uint32_t>((r >> 5) * 32) << 16) + kColO +
                          x * kN + half * (kHeadDim / 2);
  const int h = w.g * a.group + hh;
  const long long row = (w.q0 + t) * a.num_q_heads + h;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
  const bool have_o = w.ntiles > 0;            // uniform over the CTA
  const int d0 = half * (kHeadDim / 2);
  // a whole row tile inside the sequence and inside out (uniform over the
  // tile): staged in Q_x's shared memory (no MMA reads it any more), then one
  // TMA store per 64-dim half
  const int row0 = w.mt * 2 * kM + x * kM;
  const long long tok0 = w.q0 + div_group(a, row0);
  const bool whole_tile = a.o_tma && a.num_splits == 1 && row0 + kM <= w.rows && tok0 >= 0 &&
                          w.q0 + div_group(a, row0 + kM - 1) < a.total_q;
  if (whole_tile) {
    uint8_t* stage = smem + kOffQ + x * kTile + half * kHalf;
#pragma unroll 1
    for (int c = 0; c < kHeadDim / 64; ++c) {
      float o[32];
      if (have_o) {
        tc5::tmem_ld32(o_cols + c * 32, o);
        tc5::wait_ld();
      }
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint4 pk;
        const float* y = o + q8 * 8;
        pk.x = have_o ? pack_bf16x2(y[0] * inv, y[1] * inv) : 0u;
        pk.y = have_o ? pack_bf16x2(y[2] * inv, y[3] * inv) : 0u;
        pk.z = have_o ? pack_bf16x2(y[4] * inv, y[5] * inv) : 0u;
        pk.w = have_o ? pack_bf16x2(y[6] * inv, y[7] * inv) : 0u;
        *reinterpret_cast<uint4*>(stage + swz128(r, c * 4 + q8)) = pk;
      }
    }
    tc5::fence_smem_for_async();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&bars->o_staged[x]);
    if (half == 0 && a.lse_out != nullptr) a.lse_out[row] = lse;
    if (threadIdx.x == x * 2 * kM) {           // warp 8x, lane 0
      if (mbar_wait(&bars->o_staged[x], 0)) {
        const uint8_t* src = smem + kOffQ + x * kTile;
        const int hc = w.g * a.group, tc = static_cast<int>(tok0);
        tma_store_rows(src, omap, 0, hc, tc);
        tma_store_rows(src + kHalf, omap, 64, hc, tc);
        tma_store_commit_and_wait_read();
      } else {
        bars->abort = 1;
        report(a.status_flags, kFlagTimeout);
      }
    }
    return;
  }
  if (a.num_splits == 1) {
    __nv_bfloat16* orow = a.out + row * kHeadDim + d0;
#pragma unroll 1
    for (int c = 0; c < kHeadDim / 64; ++c) {
      float o[32];
      if (have_o) {
        tc5::tmem_ld32(o_cols + c * 32, o);
        tc5::wait_ld();
      }
      if (valid) {
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          uint4 pk;
          const float* y = o + q8 * 8;
          pk.x = have_o ? pack_bf16x2(y[0] * inv, y[1] * inv) : 0u;
          pk.y = have_o ? pack_bf16x2(y[2] * inv, y[3] * inv) : 0u;
          pk.z = have_o ? pack_bf16x2(y[4] * inv, y[5] * inv) : 0u;
          pk.w = have_o ? pack_bf16x2(y[6] * inv, y[7] * inv) : 0u;
          *reinterpret_cast<uint4*>(orow + c * 32 + q8 * 8) = pk;
        }
      }
    }
    if (valid && half == 0 && a.lse_out != nullptr) a.lse_out[row] = lse;
  } else {
    const long long prow = row * a.num_splits + w.j;
    float* po = a.ws_o + prow * kHeadDim + d0;
#pragma unroll 1
    for (int c = 0; c < kHeadDim / 64; ++c) {
      float o[32];
      if (have_o) {
        tc5::tmem_ld32(o_cols + c * 32, o);
        tc5::wait_ld();
      }
      if (valid) {
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float* y = o + q4 * 4;
          *reinterpret_cast<float4*>(po + c * 32 + q4 * 4) =
              have_o ? make_float4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    if (valid && half == 0) a.ws_lse[prow] = lse;
  }
}

__device__ void softmax_rows(const PrefillArgs& a, const Work& w, uint8_t* smem, Bars* bars,
                             const CUtensorMap* omap, float* xslots, uint32_t tmem, int x,
                             int half) {
  const int wq = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int r = wq * 32 + lane;                // row of tile x = tensor-memory lane
  const int rg = w.mt * 2 * kM + x * kM + r;
  const bool valid = rg < w.rows;
  const int t = valid ? div_group(a, rg) : 0;
  // keys [k0, lim) are visible to this row
  const int lim = valid ? max(w.k0, min(w.k1, w.L - w.q_len + t + 1)) : w.k0;
  const uint32_t lanes = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t s_cols = lanes + kColS + x * kN + half * (kN / 2);
  const uint32_t o_cols = lanes + kColO + x * kN + half * (kHeadDim / 2);
  const float sl2 = a.scale_log2;
  float* slots = xslots + x * 4 * kM;          // [parity][half][row] of tile x
  uint64_t* xbar = &bars->xch[x][wq];
  uint32_t uses = 0;

  // decided once: interior tiles end at or before every row's limit (the
  // warp's smallest), and only the last tile can reach past key_end (tile A
  // zeroes the V rows there)
  int lim_min = lim;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lim_min = min(lim_min, __shfl_xor_sync(0xffffffffu, lim_min, o));
  const int n = w.ntiles;
  const int k0 = w.k0;
  const int tail_tile = (x == 0 && k0 + n * kN > w.key_end) ? n - 1 : -1;

  float m_ref = -INFINITY;                     // reference max (log2 units), integer once set
  float l = 0.f;                               // this half's sum of P
  bool ok = true;
  for (int i = 0; i < n; ++i) {
    // S_x(i) landed, and with it PV_x(i - 1): O_x is complete up to tile i - 1
    if (!warp_wait(&bars->s_full[x], i & 1)) {
      ok = false;
      break;
    }
    tc5::fence_after_sync();
    const int kb = k0 + i * kN;
    const int nvis = min(kN, max(0, lim - kb));   // keys kb .. kb + nvis - 1 visible
    // interior tiles (every row of the warp sees all 128 keys) skip the masks
    const bool whole = lim_min >= kb + kN;
    const float m_start = m_ref;
    auto publish = [&](float m) { swap_publish(m, slots, xbar, uses, half, r); };
    float psum = whole ? half_tile<false>(s_cols, s_cols, half * (kN / 2), nvis, sl2, m_ref, publish)
                       : half_tile<true>(s_cols, s_cols, half * (kN / 2), nvis, sl2, m_ref, publish);
    // one reference per row: the higher of the two halves'
    const float m_other = swap_read(slots, xbar, uses, half, r, ok);
    if (!ok) break;
    if (__all_sync(0xffffffffu, m_ref == m_start && m_other == m_start)) {
      l += psum;                               // neither half moved (the usual tile)
    } else {
      const float m_row = fmaxf(m_ref, m_other);
      if (__any_sync(0xffffffffu, m_ref < m_row)) {
        const float f = m_ref < m_row ? pow2_int(m_ref - m_row) : 1.f;
        scale_p<32>(s_cols, f);
        psum *= f;
      }
      m_ref = m_row;
      const bool rose = m_row > m_start;       // -inf -> finite counts
      const float alpha = rose ? pow2_int(m_start - m_row) : 1.f;
      if (i > 0 && __any_sync(0xffffffffu, rose)) {
#pragma unroll 1
        for (int c = 0; c < kHeadDim / 64; ++c) {
          float o[32];
          tc5::tmem_ld32(o_cols + c * 32, o);
          tc5::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tc5::tmem_st32(o_cols + c * 32, o);
        }
      }
      l = l * alpha + psum;
    }
    // Tail tile: cache slots past the last visible key may hold anything
    // (stale or never-written rows); P is 0 there, but 0 x NaN is NaN, so
    // their V rows are zeroed (by tile A, each half its dims, before either
    // PV reads them).
    if (i == tail_tile) {
      const int s = i & 1;
      if (!warp_wait(&bars->full_v[s], (i >> 1) & 1)) {
        ok = false;
        break;
      }
      if (kb + r >= w.key_end) {
        uint8_t* vrow = smem + kOffV + s * kTile + v_row_offset(r, half, box_shift(a.block_size));
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + c * 16) = z;
      }
      tc5::fence_smem_for_async();
    }
    tc5::wait_st();
    tc5::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->p_full[x]);
  }
  // O_x is complete once the last PV has finished
  if (ok && w.ntiles > 0) {
    ok = warp_wait(&bars->pv_done[x], 0);
    tc5::fence_after_sync();
  }
  // the row's sum of P: both halves'
  if (ok) l += pair_swap(l, slots, xbar, uses, half, r, ok);
  if (!ok) {
    bars->abort = 1;
    report(a.status_flags, kFlagTimeout);
    return;
  }
  write_rows(a, w, tmem, smem, bars, omap, x, half, m_ref, l);
}

// ------------------------------------------------------------------ kernel

// 18 warps: two of the SM's four sub-partitions hold five of them, so a
// thread gets at most 96 registers (16,384 per sub-partition).
__global__ void __maxnreg__(96)
paged_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap omap,
                     const __grid_constant__ PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = reinterpret_cast<Bars*>(smem + kDataBytes);
  __shared__ int issued;
  const int warp = threadIdx.x >> 5;

  // launched as a programmatic dependent: q, the appended K/V, the tables and
  // the lengths may come from the previous kernel in the stream
  pdl_wait();
  const Work w = decode_work(a);
  // row tiles past this sequence's rows (varlen grids cover the longest
  // sequence): nothing to compute or write; leave before any set-up
  if (w.mt * 2 * kM >= w.rows) return;

  if (threadIdx.x == kProducerWarp * 32) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full_k[s], 1);
      mbar_init(&bars->full_v[s], 1);
      mbar_init(&bars->empty_k[s], 1);
      mbar_init(&bars->empty_v[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->p_full[x], kSoftmaxWarps / 2);
      for (int q = 0; q < 4; ++q) mbar_init(&bars->xch[x][q], 2);
      mbar_init(&bars->pv_done[x], 1);
      mbar_init(&bars->o_staged[x], kSoftmaxWarps / 2);
    }
    mbar_init(&bars->q_full[0], 1);
    mbar_init(&bars->q_full[1], 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    issued = 0;
    fence_barrier_init();
    // Q by TMA: one box per (row tile, 64-dim half), rows past q or
    // before it read as zeros, rows of a following sequence are masked
    if (a.q_tma && w.ntiles > 0) {
      prefetch_tensormap(&qmap);
      // tile A now; tile B after K(0), so that S_A(0) waits for two boxes less
      mbar_arrive_expect_tx(&bars->q_full[0], kTile);
      const int tok = static_cast<int>(w.q0 + div_group(a, w.mt * 2 * kM));
      for (int dh = 0; dh < 2; ++dh)
        tma_load_rows(smem + kOffQ + dh * kHalf, &qmap, &bars->q_full[0], dh * 64,
                      w.g * a.group, tok);
    }
  }
  if (warp == kMmaWarp) tc5::tmem_alloc(&bars->tmem_base, kTmemCols);

  if (warp < kSoftmaxWarps && !a.q_tma) {
    // Q tiles: thread i loads 64 dims (half i / 256) of row i % 128 of tile
    // (i / 128) % 2 (row = (token, q head of the group)), one swizzled half
    const int row = threadIdx.x % (2 * kM), dh = threadIdx.x / (2 * kM);
    const int x = row / kM, r = row % kM;
    const int rg = w.mt * 2 * kM + row;
    const int t0 = div_group(a, rg);
    const bool valid = rg < w.rows && w.q0 + t0 >= 0 && w.q0 + t0 < a.total_q;
    const int t = valid ? t0 : 0;
    const int hh = valid ? rg - t * a.group : 0;
    const uint4* src = reinterpret_cast<const uint4*>(
        a.q + (valid ? w.q0 + t : 0) * a.q_stride_t +
        static_cast<long long>(w.g * a.group + hh) * a.q_stride_h);
    uint8_t* qt = smem + kOffQ + x * kTile;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = valid ? __ldg(src + dh * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(qt + dh * kHalf + swz128(r, c)) = v;
    }
    tc5::fence_smem_for_async();
  }
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  pdl_launch_dependents();
  const uint32_t tmem = bars->tmem_base;

  if (warp < kSoftmaxWarps) {
    // warp = 8 x + 4 half + lane quadrant
    const int x = warp >> 3, half = (warp >> 2) & 1;
    if (x == 0 || w.has_b)
      softmax_rows(a, w, smem, bars, &omap, reinterpret_cast<float*>(smem + kOffSlots), tmem, x,
                   half);
  } else if (warp == kProducerWarp) {
    int n = 0;
    produce(a, w, &kmap, &vmap, &qmap, smem, bars, &n);
    if (threadIdx.x == kProducerWarp * 32) {
      issued = n;
      // the Q copies have landed before the CTA can leave (done long ago
      // unless the MMA thread gave up)
      if (a.q_tma && w.ntiles > 0) {
        mbar_wait(&bars->q_full[0], 0);
        if (w.has_b) mbar_wait(&bars->q_full[1], 0);
      }
    }
  } else {
    if ((threadIdx.x & 31) == 0) issue_mmas(a, w, smem, bars, tmem);
    __syncwarp();
  }
  tc5::fence_before_sync();
  __syncthreads();
  if (bars->abort && threadIdx.x == kProducerWarp * 32) drain_copies(bars, issued);
  if (warp == kMmaWarp) {
    tc5::fence_after_sync();
    tc5::tmem_dealloc(tmem, kTmemCols);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, looked up
// once; nullptr if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 row_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D view (128 dims, heads, tokens) of q or out, strides in bytes, with a box
// of (64 dims, group heads, 128 / group tokens) and 128-byte swizzle: one box
// is one 64-dim half of a 128-row tile in the packed row order
// r = t * group + h % group, laid out as the MMA operand (and the output
// staging) expects.  False where the layout does not allow such a box (group
// not a power of two up to 128, base or strides not multiples of 16 bytes).
bool encode_rows_map(CUtensorMap* map, const void* base, long long tokens, int heads,
                     long long stride_h, long long stride_t, int group) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = row_map_encoder();
  if (encode == nullptr || base == nullptr || tokens < 1 || group < 1 || group > 128 ||
      (group & (group - 1)) != 0 || heads < group)
    return false;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || stride_h % 16 != 0 || stride_t % 16 != 0 ||
      stride_h <= 0 || stride_t <= 0)
    return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride_h), static_cast<cuuint64_t>(stride_t)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(kM / group)};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int prefill_smem_bytes() { return kSmemBytes; }

cudaError_t launch_paged_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const PrefillArgs& args, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = set_smem_limit_once(paged_prefill_kernel, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  PrefillArgs a = args;
  CUtensorMap qmap, omap;
  std::memset(&qmap, 0, sizeof(qmap));
  std::memset(&omap, 0, sizeof(omap));
  a.mt_major = a.cu_seqlens_q != nullptr ? 1 : 0;
  a.group_shift = -1;
  if (a.group > 0 && (a.group & (a.group - 1)) == 0)
    for (int s = 0; s < 31; ++s)
      if ((1 << s) == a.group) a.group_shift = s;
  a.q_tma = encode_rows_map(&qmap, a.q, a.total_q, a.num_q_heads, a.q_stride_h * 2,
                            a.q_stride_t * 2, a.group) ? 1 : 0;
  a.o_tma = (a.num_splits == 1 &&
             encode_rows_map(&omap, a.out, a.total_q, a.num_q_heads, kHeadDim * 2,
                             static_cast<long long>(a.num_q_heads) * kHeadDim * 2, a.group))
                ? 1 : 0;
  const long long gx = static_cast<long long>(a.m_tiles) * a.num_kv_heads * a.num_splits;
  return launch_pdl(paged_prefill_kernel, dim3(static_cast<unsigned>(gx), a.batch),
                    dim3(kThreads), kSmemBytes, stream, kmap, vmap, qmap, omap, a);
}

}  // namespace pkvqk
