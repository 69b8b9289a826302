// C-ABI host layer of pkvqk: argument validation, TMA descriptor encoding,
// the split-count heuristic and kernel launches on the caller's stream.
//
// Nothing here allocates device memory, synchronises or reads device memory;
// every decision comes from host arguments (InfiniLM PR #585, "概述 /
// Summary" item 3: decode routing decided on the host with zero device sync),
// so every entry point can be recorded into a CUDA graph.
#include "pkvqk.h"
#include "kernels.h"
#include "prefill.h"
#include "rope_math.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace {

thread_local std::string g_last_error;

pkvqk_status fail(pkvqk_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

pkvqk_status ok() {
  g_last_error.clear();
  return PKVQK_OK;
}

pkvqk_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKVQK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device pointer check (InfiniLM issue #498 review notes: host-resident vs
// device-resident arguments are checked before use).
pkvqk_status check_device_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(PKVQK_ERR_INVALID_ARG, "%s is NULL", name);
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) cur = -1;
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(PKVQK_ERR_POINTER_RESIDENCY, "%s: cudaPointerGetAttributes failed (%s)", name,
                cudaGetErrorName(e));
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(PKVQK_ERR_POINTER_RESIDENCY, "%s is not device memory", name);
  if (cur >= 0 && attr.type == cudaMemoryTypeDevice && attr.device != cur)
    return fail(PKVQK_ERR_POINTER_RESIDENCY, "%s lives on device %d, current device is %d", name,
                attr.device, cur);
  return PKVQK_OK;
}

#define PKVQK_TRY(expr)                      \
  do {                                       \
    pkvqk_status _s = (expr);                \
    if (_s != PKVQK_OK) return _s;           \
  } while (0)

pkvqk_status check_layout(const pkvqk_cache_layout* L) {
  if (L == nullptr) return fail(PKVQK_ERR_INVALID_ARG, "layout is NULL");
  if (L->head_dim != 128) return fail(PKVQK_ERR_UNSUPPORTED, "head_dim %d (only 128)", L->head_dim);
  if (L->num_blocks < 1 || L->num_blocks > (int64_t(1) << 31) - 1)
    return fail(PKVQK_ERR_INVALID_ARG, "num_blocks %lld out of range",
                static_cast<long long>(L->num_blocks));
  if (L->block_size < 16 || L->block_size > 256 || (L->block_size % 16) != 0)
    return fail(PKVQK_ERR_UNSUPPORTED, "block_size %d (multiple of 16 in [16, 256])",
                L->block_size);
  if (L->num_kv_heads < 1 || L->num_kv_heads > 256)
    return fail(PKVQK_ERR_INVALID_ARG, "num_kv_heads %d", L->num_kv_heads);
  const int64_t st[3] = {L->block_stride, L->slot_stride, L->head_stride};
  const char* nm[3] = {"block_stride", "slot_stride", "head_stride"};
  for (int i = 0; i < 3; ++i) {
    if (st[i] <= 0 || (st[i] % 8) != 0 || st[i] * 2 >= (int64_t(1) << 40))
      return fail(PKVQK_ERR_INVALID_ARG, "%s %lld must be a positive multiple of 8 elements", nm[i],
                  static_cast<long long>(st[i]));
  }
  return PKVQK_OK;
}

// ------------------------------------------------------- TMA descriptors

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

pkvqk_status get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr)
    return fail(PKVQK_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                cudaGetErrorName(g_encode_err));
  return PKVQK_OK;
}

// 5-D view of a paged cache for the kernels' TMA boxes:
//   dims (inner first) = (64 dims, slot, dim half, kv head, block),
// box = (64, tile_keys slots, halves, heads_per_cta, 1 block), 128-byte
// swizzle, so the shared-memory tile of one (kv head, half) is tile_keys rows
// of 128 B.  The decode kernel and the prefill kernel's V take both halves
// per box; the prefill kernel's K takes one (it places the halves of all
// pages of a key tile in two blocks, as its K-major operand needs).
pkvqk_status encode_cache_map(CUtensorMap* map, const void* base, const pkvqk_cache_layout& L,
                              int heads_per_cta, int tile_keys, int halves = 2) {
  PKVQK_TRY(get_encoder());
  cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(L.block_size), 2,
                        static_cast<cuuint64_t>(L.num_kv_heads),
                        static_cast<cuuint64_t>(L.num_blocks)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(L.slot_stride) * 2, 128,
                           static_cast<cuuint64_t>(L.head_stride) * 2,
                           static_cast<cuuint64_t>(L.block_stride) * 2};
  cuuint32_t box[5] = {64, static_cast<cuuint32_t>(tile_keys), static_cast<cuuint32_t>(halves),
                       static_cast<cuuint32_t>(heads_per_cta), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PKVQK_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  return PKVQK_OK;
}

// ---------------------------------------------------------------- SM count

int sm_count_current() {
  static std::atomic<int> cache[64] = {};      // 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Rotary table: per position, 16 lanes x 4 float4s (cos hi, cos lo, sin hi,
// sin lo of four frequencies) = 1 KiB; up to 2^21 positions (2 GiB).
constexpr size_t kRopeTableRowBytes = 16 * 4 * 16;
constexpr int32_t kRopeTableMaxPositions = 1 << 21;

// Split schedule: fp32 partials [rows][S][128], then partial lse [rows][S].
size_t partial_bytes(int64_t rows, int S) {
  const size_t raw = static_cast<size_t>(rows) * S * (128 + 1) * sizeof(float);
  return (raw + 255) & ~size_t(255);
}

// Balanced schedule: fp32 partials [slot rows][128] and lse [slot rows]
// (slot = CTA + unit), then the int2 table [units] of the first and last CTA
// of every unit.
size_t balanced_bytes(int64_t slot_rows, int64_t units) {
  const size_t raw = align16(static_cast<size_t>(slot_rows) * 129 * 4) +
                     static_cast<size_t>(units) * 8;
  return (raw + 255) & ~size_t(255);
}

struct DecodeCall {
  const void* q;
  int64_t q_stride_t, q_stride_h;
  const void* k_cache;
  const void* v_cache;
  const pkvqk_cache_layout* layout;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* seq_lens;
  int32_t batch, q_len, num_q_heads, num_splits, max_seq_len_hint;
  float scale;
  void* out;
  float* lse_out;
  void* workspace;
  size_t workspace_bytes;
  int32_t* status_flags;
  cudaStream_t stream;
  bool partials_only;
};

pkvqk_status run_prefill(const DecodeCall& c, const int32_t* cu_seqlens_q, int64_t total_q);

pkvqk_status run_decode(const DecodeCall& c) {
  PKVQK_TRY(check_layout(c.layout));
  const pkvqk_cache_layout& L = *c.layout;
  if (c.batch < 0 || c.batch > 65535) return fail(PKVQK_ERR_INVALID_ARG, "batch %d", c.batch);
  if (c.q_len < 1 || c.q_len > 16) return fail(PKVQK_ERR_INVALID_ARG, "q_len %d (1..16)", c.q_len);
  if (c.num_q_heads < 1 || (c.num_q_heads % L.num_kv_heads) != 0)
    return fail(PKVQK_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                c.num_q_heads, L.num_kv_heads);
  const int group = c.num_q_heads / L.num_kv_heads;
  const int rows = c.q_len * group;
  if (c.max_blocks_per_seq < 1) return fail(PKVQK_ERR_INVALID_ARG, "max_blocks_per_seq < 1");
  if (c.max_seq_len_hint < 0) return fail(PKVQK_ERR_INVALID_ARG, "max_seq_len_hint < 0");
  if (c.num_splits < 0 || c.num_splits > 256)
    return fail(PKVQK_ERR_INVALID_ARG, "num_splits %d (0..256)", c.num_splits);
  if (c.partials_only && c.num_splits < 2)
    return fail(PKVQK_ERR_INVALID_ARG, "partials need an explicit num_splits >= 2");
  if (c.q_stride_t % 8 || c.q_stride_h % 8 || c.q_stride_h < 1 || c.q_stride_t < 0)
    return fail(PKVQK_ERR_INVALID_ARG, "q strides must be multiples of 8 elements");
  if (!std::isfinite(c.scale)) return fail(PKVQK_ERR_INVALID_ARG, "scale is not finite");
  if (rows > 16) {
    // More query rows per kv head than the decode kernel's register tiles
    // hold: the tensor-core multi-query kernel computes the same rows, with
    // the same split boundaries and partial layout.  The balanced schedule
    // has no counterpart there; it becomes a split count whose partials fit
    // the balanced workspace bound ((SMs + batch) x q_len x Hq rows).
    DecodeCall p = c;
    if (p.num_splits == 0) {
      const int64_t cap = static_cast<int64_t>(c.max_blocks_per_seq) * L.block_size;
      const int hint = c.max_seq_len_hint > 0
                           ? c.max_seq_len_hint
                           : static_cast<int>(std::min<int64_t>(cap, INT32_MAX));
      const int S = pkvqk_choose_prefill_splits(c.batch, L.num_kv_heads, c.q_len, group, hint, 0);
      p.num_splits = std::max(1, std::min(S, 1 + sm_count_current() / std::max(1, c.batch)));
    }
    return run_prefill(p, nullptr, static_cast<int64_t>(c.batch) * c.q_len);
  }

  const int64_t cap_tokens = static_cast<int64_t>(c.max_blocks_per_seq) * L.block_size;
  const int hint = c.max_seq_len_hint > 0
                       ? c.max_seq_len_hint
                       : static_cast<int>(std::min<int64_t>(cap_tokens, INT32_MAX));
  const int S = c.num_splits;                   // 0: balanced schedule
  const pkvqk::DecodePlan plan = pkvqk::plan_decode(L.num_kv_heads, rows);
  const int64_t nrows = static_cast<int64_t>(c.batch) * c.q_len * c.num_q_heads;
  // balanced schedule: 0.84 CTAs per SM, the share the split heuristic also
  // keeps in flight (measured on GB300 against one CTA per SM: decode call
  // GQA-8 mixed batch 86.7 -> 83.9 us, verify 32 x 5 116.2 -> 113.7 us,
  // 64 x 8192 315.7 -> 311.9 us; 112-144 CTAs within 1 %)
  const int grid_ctas = std::max(1, static_cast<int>(std::lround(0.84 * sm_count_current())));
  const int groups = L.num_kv_heads / plan.heads_per_cta;
  const int64_t units = static_cast<int64_t>(c.batch) * groups;
  const int64_t rows_per_unit = static_cast<int64_t>(c.q_len) * plan.heads_per_cta * group;
  const int64_t slot_rows = (grid_ctas + units) * rows_per_unit;
  size_t need = 0;
  if (S == 0) need = balanced_bytes(slot_rows, units);
  else if (c.partials_only || S > 1) need = partial_bytes(nrows, S);
  if (need > 0 && c.workspace_bytes < need)
    return fail(PKVQK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed",
                c.workspace_bytes, need);
  if (c.batch == 0) return ok();

  PKVQK_TRY(check_device_ptr(c.q, "q"));
  PKVQK_TRY(check_device_ptr(c.k_cache, "k_cache"));
  PKVQK_TRY(check_device_ptr(c.v_cache, "v_cache"));
  PKVQK_TRY(check_device_ptr(c.block_tables, "block_tables"));
  PKVQK_TRY(check_device_ptr(c.seq_lens, "seq_lens"));
  if (!aligned16(c.q)) return fail(PKVQK_ERR_INVALID_ARG, "q not 16-byte aligned");
  if (!aligned16(c.k_cache) || !aligned16(c.v_cache))
    return fail(PKVQK_ERR_INVALID_ARG, "cache base not 16-byte aligned");
  if (!c.partials_only) {
    PKVQK_TRY(check_device_ptr(c.out, "out"));
    if (!aligned16(c.out)) return fail(PKVQK_ERR_INVALID_ARG, "out not 16-byte aligned");
    if (c.lse_out != nullptr) PKVQK_TRY(check_device_ptr(c.lse_out, "lse_out"));
  }
  if (need > 0) {
    PKVQK_TRY(check_device_ptr(c.workspace, "workspace"));
    if (!aligned16(c.workspace)) return fail(PKVQK_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  }
  if (c.status_flags != nullptr) PKVQK_TRY(check_device_ptr(c.status_flags, "status_flags"));

  CUtensorMap kmap, vmap;
  PKVQK_TRY(encode_cache_map(&kmap, c.k_cache, L, plan.heads_per_cta, plan.tile_keys));
  PKVQK_TRY(encode_cache_map(&vmap, c.v_cache, L, plan.heads_per_cta, plan.tile_keys));

  const int hint_pages = (hint + L.block_size - 1) / L.block_size;
  pkvqk::DecodeArgs a;
  a.q = static_cast<const __nv_bfloat16*>(c.q);
  a.q_stride_t = c.q_stride_t;
  a.q_stride_h = c.q_stride_h;
  a.block_tables = c.block_tables;
  a.max_blocks_per_seq = c.max_blocks_per_seq;
  a.seq_lens = c.seq_lens;
  a.batch = c.batch;
  a.q_len = c.q_len;
  a.num_q_heads = c.num_q_heads;
  a.num_kv_heads = L.num_kv_heads;
  a.group = group;
  a.block_size = L.block_size;
  a.num_blocks = L.num_blocks;
  a.num_splits = S;
  a.chunk_pages = S > 0 ? std::max(1, (hint_pages + S - 1) / S) : 0;
  a.groups = groups;
  a.rows_per_unit = static_cast<int32_t>(rows_per_unit);
  const float scale = c.scale > 0.f ? c.scale : 1.0f / std::sqrt(128.0f);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<__nv_bfloat16*>(c.out);
  a.lse_out = c.lse_out;
  a.ws_o = nullptr;
  a.ws_lse = nullptr;
  a.unit_info = nullptr;
  if (S == 0) {
    char* base = static_cast<char*>(c.workspace);
    a.ws_o = reinterpret_cast<float*>(base);
    a.ws_lse = a.ws_o + slot_rows * 128;
    a.unit_info = reinterpret_cast<int2*>(base + align16(static_cast<size_t>(slot_rows) * 129 * 4));
  } else if (need > 0) {
    a.ws_o = static_cast<float*>(c.workspace);
    a.ws_lse = a.ws_o + nrows * S * 128;
  }
  a.status_flags = c.status_flags;

  cudaError_t e = pkvqk::launch_paged_decode(plan, kmap, vmap, a, grid_ctas, c.stream);
  if (e != cudaSuccess) return cuda_fail(e, "paged decode launch");
  if (S == 0) {
    e = pkvqk::launch_balanced_combine(a, plan.heads_per_cta, c.stream);
    if (e != cudaSuccess) return cuda_fail(e, "balanced combine launch");
  } else if (S > 1 && !c.partials_only) {
    e = pkvqk::launch_lse_combine(a.ws_o, a.ws_lse, static_cast<int>(nrows), S, a.out, c.lse_out,
                                  c.stream);
    if (e != cudaSuccess) return cuda_fail(e, "lse combine launch");
  }
  return ok();
}

// --------------------------------------------------------------- prefill

size_t prefill_bytes(int64_t rows, int S) {
  if (S <= 1) return 0;
  const size_t raw = static_cast<size_t>(rows) * S * (128 + 1) * sizeof(float);
  return (raw + 255) & ~size_t(255);
}

// cu_seqlens_q == nullptr: every sequence has c.q_len new tokens (total_q is
// then batch * q_len); else varlen with c.q_len the longest.
pkvqk_status run_prefill(const DecodeCall& c, const int32_t* cu_seqlens_q, int64_t total_q) {
  PKVQK_TRY(check_layout(c.layout));
  const pkvqk_cache_layout& L = *c.layout;
  if (c.batch < 0 || c.batch > 65535) return fail(PKVQK_ERR_INVALID_ARG, "batch %d", c.batch);
  if (c.q_len < 1 || c.q_len > 16384)
    return fail(PKVQK_ERR_INVALID_ARG, "%s %d (1..16384)",
                cu_seqlens_q != nullptr ? "max_q_len" : "q_len", c.q_len);
  if (total_q < 0 || total_q > INT32_MAX)
    return fail(PKVQK_ERR_INVALID_ARG, "total_q %lld (0..2^31-1)", static_cast<long long>(total_q));
  if (c.num_q_heads < 1 || (c.num_q_heads % L.num_kv_heads) != 0)
    return fail(PKVQK_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                c.num_q_heads, L.num_kv_heads);
  const int group = c.num_q_heads / L.num_kv_heads;
  const int64_t rows = static_cast<int64_t>(c.q_len) * group;
  if (rows > 65536)
    return fail(PKVQK_ERR_UNSUPPORTED, "q_len * group = %lld rows per kv head (max 65536)",
                static_cast<long long>(rows));
  if (c.max_blocks_per_seq < 1) return fail(PKVQK_ERR_INVALID_ARG, "max_blocks_per_seq < 1");
  const int64_t cap_tokens = static_cast<int64_t>(c.max_blocks_per_seq) * L.block_size;
  if (cap_tokens > INT32_MAX)
    return fail(PKVQK_ERR_INVALID_ARG, "max_blocks_per_seq * block_size exceeds 2^31 - 1");
  if (c.max_seq_len_hint < 0) return fail(PKVQK_ERR_INVALID_ARG, "max_seq_len_hint < 0");
  if (c.num_splits < 1 || c.num_splits > 256)
    return fail(PKVQK_ERR_INVALID_ARG, "num_splits %d (1..256)", c.num_splits);
  if (c.q_stride_t % 8 || c.q_stride_h % 8 || c.q_stride_h < 1 || c.q_stride_t < 0)
    return fail(PKVQK_ERR_INVALID_ARG, "q strides must be multiples of 8 elements");
  if (!std::isfinite(c.scale)) return fail(PKVQK_ERR_INVALID_ARG, "scale is not finite");
  const int S = c.num_splits;
  const int m_tiles = static_cast<int>((rows + pkvqk::kPrefillRowsPerCta - 1) /
                                       pkvqk::kPrefillRowsPerCta);
  const int64_t grid_x = static_cast<int64_t>(m_tiles) * L.num_kv_heads * S;
  if (grid_x > INT32_MAX) return fail(PKVQK_ERR_UNSUPPORTED, "too many CTAs (%lld)",
                                      static_cast<long long>(grid_x));
  const int64_t nrows = total_q * c.num_q_heads;
  if (nrows > INT32_MAX)
    return fail(PKVQK_ERR_UNSUPPORTED, "total_q * num_q_heads exceeds 2^31 - 1");
  const size_t need = prefill_bytes(nrows, S);
  if (need > 0 && c.workspace_bytes < need)
    return fail(PKVQK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed",
                c.workspace_bytes, need);
  if (c.batch == 0 || total_q == 0) return ok();

  PKVQK_TRY(check_device_ptr(c.q, "q"));
  PKVQK_TRY(check_device_ptr(c.k_cache, "k_cache"));
  PKVQK_TRY(check_device_ptr(c.v_cache, "v_cache"));
  PKVQK_TRY(check_device_ptr(c.block_tables, "block_tables"));
  PKVQK_TRY(check_device_ptr(c.seq_lens, "seq_lens"));
  if (cu_seqlens_q != nullptr) PKVQK_TRY(check_device_ptr(cu_seqlens_q, "cu_seqlens_q"));
  if (!c.partials_only) {
    PKVQK_TRY(check_device_ptr(c.out, "out"));
    if (c.lse_out != nullptr) PKVQK_TRY(check_device_ptr(c.lse_out, "lse_out"));
    if (!aligned16(c.out)) return fail(PKVQK_ERR_INVALID_ARG, "out not 16-byte aligned");
  }
  if (!aligned16(c.q)) return fail(PKVQK_ERR_INVALID_ARG, "q not 16-byte aligned");
  if (!aligned16(c.k_cache) || !aligned16(c.v_cache))
    return fail(PKVQK_ERR_INVALID_ARG, "cache base not 16-byte aligned");
  if (need > 0) {
    PKVQK_TRY(check_device_ptr(c.workspace, "workspace"));
    if (!aligned16(c.workspace)) return fail(PKVQK_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  }
  if (c.status_flags != nullptr) PKVQK_TRY(check_device_ptr(c.status_flags, "status_flags"));

  // largest power of two dividing the page size, at most 128 (the kernel's
  // key tile): no box crosses a page
  const int box_slots = std::min(L.block_size & -L.block_size, 128);
  CUtensorMap kmap, vmap;
  PKVQK_TRY(encode_cache_map(&kmap, c.k_cache, L, 1, box_slots, 1));
  PKVQK_TRY(encode_cache_map(&vmap, c.v_cache, L, 1, box_slots, 2));

  const int hint = c.max_seq_len_hint > 0 ? c.max_seq_len_hint : static_cast<int>(cap_tokens);
  const int hint_pages = (hint + L.block_size - 1) / L.block_size;
  pkvqk::PrefillArgs a;
  a.q = static_cast<const __nv_bfloat16*>(c.q);
  a.q_stride_t = c.q_stride_t;
  a.q_stride_h = c.q_stride_h;
  a.block_tables = c.block_tables;
  a.max_blocks_per_seq = c.max_blocks_per_seq;
  a.seq_lens = c.seq_lens;
  a.batch = c.batch;
  a.q_len = c.q_len;
  a.num_q_heads = c.num_q_heads;
  a.num_kv_heads = L.num_kv_heads;
  a.group = group;
  a.cu_seqlens_q = cu_seqlens_q;
  a.total_q = total_q;
  a.block_size = L.block_size;
  a.num_blocks = L.num_blocks;
  a.num_splits = S;
  a.chunk_pages = std::max(1, (hint_pages + S - 1) / S);
  a.m_tiles = m_tiles;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / std::sqrt(128.0f);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<__nv_bfloat16*>(c.out);
  a.lse_out = c.lse_out;
  a.ws_o = S > 1 ? static_cast<float*>(c.workspace) : nullptr;
  a.ws_lse = S > 1 ? a.ws_o + nrows * S * 128 : nullptr;
  a.status_flags = c.status_flags;

  cudaError_t e = pkvqk::launch_paged_prefill(kmap, vmap, a, c.stream);
  if (e != cudaSuccess) return cuda_fail(e, "paged prefill launch");
  if (S > 1 && !c.partials_only) {
    e = pkvqk::launch_lse_combine(a.ws_o, a.ws_lse, static_cast<int>(nrows), S, a.out, c.lse_out,
                                  c.stream);
    if (e != cudaSuccess) return cuda_fail(e, "lse combine launch");
  }
  return ok();
}

}  // namespace

namespace pkvqk {
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace pkvqk

extern "C" {

const char* pkvqk_last_error(void) { return g_last_error.c_str(); }

int32_t pkvqk_abi_version(void) { return 1; }

namespace {

// theta^(-2i/D) in float64 and the float-float sin/cos knots: the inputs of
// both the append kernel's angle phase and the table build.
void rope_constants(float theta, double (&inv_freq)[64], float (&tab)[pkvqk::kSinCosKnots][4]) {
  for (int i = 0; i < 64; ++i) inv_freq[i] = std::pow(static_cast<double>(theta), -2.0 * i / 128.0);
  static float s_tab[pkvqk::kSinCosKnots][4];
  static std::once_flag s_tab_once;
  std::call_once(s_tab_once, [] { pkvqk::build_sincos_table(s_tab); });
  std::memcpy(tab, s_tab, sizeof(s_tab));
}

pkvqk_status run_append(void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                        int64_t k_stride_t, int64_t k_stride_h, const void* v, int64_t v_stride_t,
                        int64_t v_stride_h, const int64_t* positions, const int64_t* slot_mapping,
                        const void* gamma_q, const void* gamma_k, float theta, float eps,
                        int32_t num_tokens, int32_t num_q_heads, void* k_cache, void* v_cache,
                        const pkvqk_cache_layout* layout, const void* rope_table,
                        int32_t table_positions, int32_t* status_flags, pkvqk_stream_t stream) {
  PKVQK_TRY(check_layout(layout));
  const pkvqk_cache_layout& L = *layout;
  if (num_tokens < 0 || num_tokens > (1 << 30))
    return fail(PKVQK_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
  if (num_q_heads < 1 || num_q_heads + L.num_kv_heads > 4096)
    return fail(PKVQK_ERR_INVALID_ARG, "num_q_heads %d", num_q_heads);
  if (!(theta > 0.f) || !std::isfinite(theta)) return fail(PKVQK_ERR_INVALID_ARG, "theta must be > 0");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(PKVQK_ERR_INVALID_ARG, "eps must be >= 0");
  const int64_t st[6] = {q_stride_t, q_stride_h, k_stride_t, k_stride_h, v_stride_t, v_stride_h};
  for (int i = 0; i < 6; ++i)
    if (st[i] < 0 || (st[i] % 8) != 0)
      return fail(PKVQK_ERR_INVALID_ARG, "q/k/v strides must be non-negative multiples of 8");
  if (num_tokens == 0) return ok();
  PKVQK_TRY(check_device_ptr(q, "q"));
  PKVQK_TRY(check_device_ptr(k, "k"));
  PKVQK_TRY(check_device_ptr(v, "v"));
  PKVQK_TRY(check_device_ptr(positions, "positions"));
  PKVQK_TRY(check_device_ptr(slot_mapping, "slot_mapping"));
  PKVQK_TRY(check_device_ptr(gamma_q, "gamma_q"));
  PKVQK_TRY(check_device_ptr(gamma_k, "gamma_k"));
  PKVQK_TRY(check_device_ptr(k_cache, "k_cache"));
  PKVQK_TRY(check_device_ptr(v_cache, "v_cache"));
  if (status_flags != nullptr) PKVQK_TRY(check_device_ptr(status_flags, "status_flags"));
  const void* al[7] = {q, k, v, gamma_q, gamma_k, k_cache, v_cache};
  for (int i = 0; i < 7; ++i)
    if (!aligned16(al[i])) return fail(PKVQK_ERR_INVALID_ARG, "bf16 base pointer not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(positions) & 7u) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return fail(PKVQK_ERR_INVALID_ARG, "positions/slot_mapping not 8-byte aligned");
  if (table_positions > 0) {
    PKVQK_TRY(check_device_ptr(rope_table, "rope_table"));
    if (!aligned16(rope_table)) return fail(PKVQK_ERR_INVALID_ARG, "rope_table not 16-byte aligned");
  }

  pkvqk::NormRopeAppendArgs a;
  a.q = static_cast<__nv_bfloat16*>(q);
  a.q_stride_t = q_stride_t;
  a.q_stride_h = q_stride_h;
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.k_stride_t = k_stride_t;
  a.k_stride_h = k_stride_h;
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.v_stride_t = v_stride_t;
  a.v_stride_h = v_stride_h;
  a.positions = positions;
  a.slot_mapping = slot_mapping;
  a.gamma_q = static_cast<const __nv_bfloat16*>(gamma_q);
  a.gamma_k = static_cast<const __nv_bfloat16*>(gamma_k);
  a.eps = eps;
  rope_constants(theta, a.inv_freq, a.sincos_tab);
  a.num_tokens = num_tokens;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = L.num_kv_heads;
  a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  a.num_blocks = L.num_blocks;
  a.block_size = L.block_size;
  a.block_stride = L.block_stride;
  a.slot_stride = L.slot_stride;
  a.head_stride = L.head_stride;
  a.status_flags = status_flags;
  a.rope_table = table_positions > 0 ? static_cast<const float4*>(rope_table) : nullptr;
  a.table_positions = table_positions > 0 ? table_positions : 0;
  cudaError_t e = pkvqk::launch_norm_rope_append(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "norm_rope_append launch");
  return ok();
}

}  // namespace

pkvqk_status pkvqk_norm_rope_append(void* q, int64_t q_stride_t, int64_t q_stride_h,
                                    const void* k, int64_t k_stride_t, int64_t k_stride_h,
                                    const void* v, int64_t v_stride_t, int64_t v_stride_h,
                                    const int64_t* positions, const int64_t* slot_mapping,
                                    const void* gamma_q, const void* gamma_k, float theta,
                                    float eps, int32_t num_tokens, int32_t num_q_heads,
                                    void* k_cache, void* v_cache,
                                    const pkvqk_cache_layout* layout, int32_t* status_flags,
                                    pkvqk_stream_t stream) {
  return run_append(q, q_stride_t, q_stride_h, k, k_stride_t, k_stride_h, v, v_stride_t,
                    v_stride_h, positions, slot_mapping, gamma_q, gamma_k, theta, eps, num_tokens,
                    num_q_heads, k_cache, v_cache, layout, nullptr, 0, status_flags, stream);
}

pkvqk_status pkvqk_norm_rope_append_cached(
    void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k, int64_t k_stride_t,
    int64_t k_stride_h, const void* v, int64_t v_stride_t, int64_t v_stride_h,
    const int64_t* positions, const int64_t* slot_mapping, const void* gamma_q,
    const void* gamma_k, float theta, float eps, int32_t num_tokens, int32_t num_q_heads,
    void* k_cache, void* v_cache, const pkvqk_cache_layout* layout, const void* rope_table,
    int32_t table_positions, int32_t* status_flags, pkvqk_stream_t stream) {
  if (table_positions < 0 || table_positions > kRopeTableMaxPositions)
    return fail(PKVQK_ERR_INVALID_ARG, "table_positions %d (0..%d)", table_positions,
                kRopeTableMaxPositions);
  return run_append(q, q_stride_t, q_stride_h, k, k_stride_t, k_stride_h, v, v_stride_t,
                    v_stride_h, positions, slot_mapping, gamma_q, gamma_k, theta, eps, num_tokens,
                    num_q_heads, k_cache, v_cache, layout, rope_table, table_positions,
                    status_flags, stream);
}

size_t pkvqk_rope_table_bytes(int32_t max_positions) {
  if (max_positions <= 0 || max_positions > kRopeTableMaxPositions) return 0;
  return static_cast<size_t>(max_positions) * kRopeTableRowBytes;
}

pkvqk_status pkvqk_rope_table_build(void* table, int32_t max_positions, float theta,
                                    pkvqk_stream_t stream) {
  if (max_positions < 0 || max_positions > kRopeTableMaxPositions)
    return fail(PKVQK_ERR_INVALID_ARG, "max_positions %d (0..%d)", max_positions,
                kRopeTableMaxPositions);
  if (!(theta > 0.f) || !std::isfinite(theta)) return fail(PKVQK_ERR_INVALID_ARG, "theta must be > 0");
  if (max_positions == 0) return ok();
  PKVQK_TRY(check_device_ptr(table, "table"));
  if (!aligned16(table)) return fail(PKVQK_ERR_INVALID_ARG, "table not 16-byte aligned");
  double inv_freq[64];
  float tab[pkvqk::kSinCosKnots][4];
  rope_constants(theta, inv_freq, tab);
  const cudaError_t e = pkvqk::launch_rope_table_build(
      static_cast<float4*>(table), max_positions, inv_freq, tab,
      reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope table build launch");
  return ok();
}

int32_t pkvqk_choose_num_splits(int32_t batch, int32_t num_kv_heads, int32_t rows_per_kv_head,
                                int32_t max_seq_len, int64_t total_tokens, int32_t block_size,
                                int32_t sm_count) {
  if (batch <= 0 || num_kv_heads <= 0 || max_seq_len <= 0 || block_size <= 0) return 1;
  if (sm_count <= 0) sm_count = sm_count_current();
  // pkvqk_paged_decode runs more than 16 rows per kv head on the tensor-core
  // multi-query kernel: its own choice (rows = q_len * group with group 1)
  if (rows_per_kv_head > 16)
    return pkvqk_choose_prefill_splits(batch, num_kv_heads, rows_per_kv_head, 1, max_seq_len,
                                       sm_count);
  const pkvqk::DecodePlan plan = pkvqk::plan_decode(num_kv_heads, rows_per_kv_head);
  const int64_t groups = num_kv_heads / plan.heads_per_cta;
  const int64_t p_max = (max_seq_len + block_size - 1) / block_size;
  const int64_t tp = std::max<int64_t>((total_tokens + block_size - 1) / block_size, p_max);
  // Measured on GB300 (HBM-bound, dynamic CTA scheduling): the step is
  // fastest with ~0.84 x (resident CTA slots) CTAs in flight -- enough to
  // saturate HBM, one wave so no straggler wave -- and with the longest
  // sequence cut finely enough that its chunk is no larger than the average
  // CTA's share; chunks under 128 keys cost more in start-up than they gain,
  // except on short contexts (<= 2048 keys), where 64-key chunks spread the
  // few CTAs' work wider (1 x 512: 17.1 -> 15.0 us, 1 x 2048: 19.1 -> 17.1).
  const double target = 0.84 * sm_count * plan.ctas_per_sm;
  const int64_t s_fill = static_cast<int64_t>(target / static_cast<double>(groups * batch) + 0.5);
  // (a CTA covers one head group: tp * groups pages of work in all; to the
  // nearest count: the speculative-verify batch of mixed lengths, 32 x
  // U[2048, 8192] + 5, measured 111 us at 6 splits and 121 us at 7)
  const int64_t s_bal = static_cast<int64_t>(
      std::round(static_cast<double>(p_max) * target / (static_cast<double>(tp) * groups)));
  int64_t S = std::max<int64_t>(1, std::max(s_fill, s_bal));
  const int64_t min_chunk = p_max * block_size <= 2048 ? 64 : 128;
  const int64_t s_min_chunk =
      std::max<int64_t>(1, (p_max * block_size + min_chunk - 1) / min_chunk);
  S = std::min<int64_t>(S, std::min<int64_t>(s_min_chunk, std::min<int64_t>(p_max, 256)));
  // drop splits that the longest sequence leaves empty
  const int64_t chunk = (p_max + S - 1) / S;
  S = (p_max + chunk - 1) / chunk;
  // Strongly mixed lengths (the batch holds well under half of batch x
  // max_seq_len keys) on a large problem: the balanced schedule (0) measured
  // faster than any split count (GQA-8 serving batch, fill 0.24: 84 vs 91 us
  // at its best split); at milder mixes the split count above wins (verify
  // batch, fill 0.62: 111 us at 6 splits vs 115 balanced).  Its planning
  // prologue (~5 us) does not pay off on small problems.
  const double fill = static_cast<double>(total_tokens) /
                      (static_cast<double>(batch) * static_cast<double>(max_seq_len));
  const double kv_bytes = static_cast<double>(total_tokens) * num_kv_heads * 512.0;
  if (fill < 0.5 && kv_bytes >= 128.0 * (1 << 20) && batch * groups >= 8) return 0;
  return static_cast<int32_t>(std::max<int64_t>(1, S));
}

size_t pkvqk_decode_workspace_bytes(int32_t batch, int32_t q_len, int32_t num_q_heads,
                                    int32_t head_dim, int32_t num_splits) {
  if (batch <= 0 || q_len <= 0 || num_q_heads <= 0 || head_dim != 128 || num_splits == 1 ||
      num_splits < 0)
    return 0;
  if (num_splits == 0) {
    // bound over every kv-head count: slots (SMs + units) x rows per unit
    // <= (SMs + batch) x q_len x Hq, units <= batch x Hq
    const int64_t per = static_cast<int64_t>(q_len) * num_q_heads;
    return balanced_bytes((sm_count_current() + static_cast<int64_t>(batch)) * per,
                          static_cast<int64_t>(batch) * num_q_heads);
  }
  return partial_bytes(static_cast<int64_t>(batch) * q_len * num_q_heads, num_splits);
}

pkvqk_status pkvqk_paged_decode(const void* q, int64_t q_stride_t, int64_t q_stride_h,
                                const void* k_cache, const void* v_cache,
                                const pkvqk_cache_layout* layout, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                int32_t batch, int32_t q_len, int32_t num_q_heads,
                                int32_t num_splits, int32_t max_seq_len_hint, float scale,
                                void* out, float* lse_out, void* workspace,
                                size_t workspace_bytes_, int32_t* status_flags,
                                pkvqk_stream_t stream) {
  DecodeCall c{q,          q_stride_t,  q_stride_h,       k_cache,    v_cache,
               layout,     block_tables, max_blocks_per_seq, seq_lens, batch,
               q_len,      num_q_heads, num_splits,       max_seq_len_hint, scale,
               out,        lse_out,     workspace,        workspace_bytes_, status_flags,
               reinterpret_cast<cudaStream_t>(stream), false};
  return run_decode(c);
}

pkvqk_status pkvqk_paged_decode_partials(const void* q, int64_t q_stride_t, int64_t q_stride_h,
                                         const void* k_cache, const void* v_cache,
                                         const pkvqk_cache_layout* layout,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                         int32_t num_q_heads, int32_t num_splits,
                                         int32_t max_seq_len_hint, float scale, void* workspace,
                                         size_t workspace_bytes_, int32_t* status_flags,
                                         pkvqk_stream_t stream) {
  DecodeCall c{q,          q_stride_t,  q_stride_h,       k_cache,    v_cache,
               layout,     block_tables, max_blocks_per_seq, seq_lens, batch,
               q_len,      num_q_heads, num_splits,       max_seq_len_hint, scale,
               nullptr,    nullptr,     workspace,        workspace_bytes_, status_flags,
               reinterpret_cast<cudaStream_t>(stream), true};
  return run_decode(c);
}

pkvqk_status pkvqk_lse_combine(const float* ws_o, const float* ws_lse, int32_t rows,
                               int32_t head_dim, int32_t num_splits, void* out, float* lse_out,
                               pkvqk_stream_t stream) {
  if (head_dim != 128) return fail(PKVQK_ERR_UNSUPPORTED, "head_dim %d (only 128)", head_dim);
  if (rows < 0) return fail(PKVQK_ERR_INVALID_ARG, "rows %d", rows);
  if (num_splits < 1 || num_splits > 256)
    return fail(PKVQK_ERR_INVALID_ARG, "num_splits %d (1..256)", num_splits);
  if (rows == 0) return ok();
  PKVQK_TRY(check_device_ptr(ws_o, "ws_o"));
  PKVQK_TRY(check_device_ptr(ws_lse, "ws_lse"));
  PKVQK_TRY(check_device_ptr(out, "out"));
  if (lse_out != nullptr) PKVQK_TRY(check_device_ptr(lse_out, "lse_out"));
  if (!aligned16(ws_o) || !aligned16(out))
    return fail(PKVQK_ERR_INVALID_ARG, "ws_o/out not 16-byte aligned");
  cudaError_t e = pkvqk::launch_lse_combine(ws_o, ws_lse, rows, num_splits,
                                            static_cast<__nv_bfloat16*>(out), lse_out,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lse combine launch");
  return ok();
}

int32_t pkvqk_choose_prefill_splits(int32_t batch, int32_t num_kv_heads, int32_t q_len,
                                    int32_t group, int32_t max_seq_len, int32_t sm_count) {
  if (batch <= 0 || num_kv_heads <= 0 || q_len <= 0 || group <= 0 || max_seq_len <= 0) return 1;
  if (sm_count <= 0) sm_count = sm_count_current();
  const int64_t m_tiles = (static_cast<int64_t>(q_len) * group + pkvqk::kPrefillRowsPerCta - 1) /
                          pkvqk::kPrefillRowsPerCta;
  const int64_t ctas = static_cast<int64_t>(batch) * num_kv_heads * m_tiles;
  if (ctas >= sm_count) return 1;
  int64_t S = (sm_count + ctas - 1) / ctas;
  S = std::min<int64_t>(S, std::max<int64_t>(1, max_seq_len / 256));
  return static_cast<int32_t>(std::min<int64_t>(S, 256));
}

size_t pkvqk_prefill_workspace_bytes(int32_t batch, int32_t q_len, int32_t num_q_heads,
                                     int32_t head_dim, int32_t num_splits) {
  if (batch <= 0 || q_len <= 0 || num_q_heads <= 0 || head_dim != 128 || num_splits <= 1)
    return 0;
  return prefill_bytes(static_cast<int64_t>(batch) * q_len * num_q_heads, num_splits);
}

pkvqk_status pkvqk_paged_prefill(const void* q, int64_t q_stride_t, int64_t q_stride_h,
                                 const void* k_cache, const void* v_cache,
                                 const pkvqk_cache_layout* layout, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t batch, int32_t q_len, int32_t num_q_heads,
                                 int32_t num_splits, int32_t max_seq_len_hint, float scale,
                                 void* out, float* lse_out, void* workspace,
                                 size_t workspace_bytes_, int32_t* status_flags,
                                 pkvqk_stream_t stream) {
  DecodeCall c{q,          q_stride_t,  q_stride_h,       k_cache,    v_cache,
               layout,     block_tables, max_blocks_per_seq, seq_lens, batch,
               q_len,      num_q_heads, num_splits,       max_seq_len_hint, scale,
               out,        lse_out,     workspace,        workspace_bytes_, status_flags,
               reinterpret_cast<cudaStream_t>(stream), false};
  return run_prefill(c, nullptr, static_cast<int64_t>(batch) * q_len);
}

pkvqk_status pkvqk_paged_prefill_varlen(const void* q, int64_t q_stride_t, int64_t q_stride_h,
                                        const int32_t* cu_seqlens_q, int32_t max_q_len,
                                        int64_t total_q, const void* k_cache,
                                        const void* v_cache, const pkvqk_cache_layout* layout,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, int32_t batch,
                                        int32_t num_q_heads, int32_t num_splits,
                                        int32_t max_seq_len_hint, float scale, void* out,
                                        float* lse_out, void* workspace, size_t workspace_bytes_,
                                        int32_t* status_flags, pkvqk_stream_t stream) {
  if (cu_seqlens_q == nullptr) return fail(PKVQK_ERR_INVALID_ARG, "cu_seqlens_q is NULL");
  DecodeCall c{q,          q_stride_t,  q_stride_h,       k_cache,    v_cache,
               layout,     block_tables, max_blocks_per_seq, seq_lens, batch,
               max_q_len,  num_q_heads, num_splits,       max_seq_len_hint, scale,
               out,        lse_out,     workspace,        workspace_bytes_, status_flags,
               reinterpret_cast<cudaStream_t>(stream), false};
  return run_prefill(c, cu_seqlens_q, total_q);
}

}  // extern "C"
