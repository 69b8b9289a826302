// pkvqk_paged_decode_static_ws: split-KV paged decode whose scratch lives in
// a fixed array inside this library, for callers that cannot allocate.
//
// Who needs it: code that runs where no device allocation is allowed or
// possible — a plugin handed only input/output pointers by a host engine
// that owns all device memory, a caller whose allocator forbids allocation
// while a stream is being captured, or a foreign-language runtime with no
// handle on a CUDA allocator.  Such callers cannot size and pass the split
// workspace that pkvqk_paged_decode needs when num_splits > 1.
//
// The scratch is g_static_ws below: a file-scope __device__ array of
// kStaticWsBytes that every GPU which loads this library holds until the
// process exits.  Host code cannot use the array's name as a device address
// (it names a host-side shadow), so its device address is looked up with
// cudaGetSymbolAddress, with the device current.  The address belongs to the
// CUDA context that was current at the lookup, so it is cached per device
// together with that context's unique id (cuCtxGetId): a call made under
// another context of the same device (a driver context a host engine made
// current, or the primary context re-created after cudaDeviceReset) looks the
// address up again instead of passing the stale one to the kernel.
#include "pkvqk.h"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

namespace {

constexpr size_t kStaticWsBytes = size_t(16) << 20;   // 16 MiB of partials per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

struct CachedAddr {
  unsigned long long ctx_id;   // unique id of the context the lookup ran in
  void* addr;                  // g_static_ws in that context (nullptr: none yet)
};

std::mutex g_mu;
CachedAddr g_ws[kMaxDevices] = {};

// Driver entry points for the current context and its unique id, fetched
// once through the runtime (the library does not link libcuda).
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx_fns() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
}

// Unique id of the context current on this thread; false if there is none
// (the runtime has not made one current yet) or the query is unavailable.
bool current_ctx_id(unsigned long long* id) {
  load_ctx_fns();
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_static_ws in the current context of device `dev`.
cudaError_t static_ws_address(int dev, void** out) {
  unsigned long long id = 0;
  bool have_id = current_ctx_id(&id);
  std::lock_guard<std::mutex> lock(g_mu);
  CachedAddr& c = g_ws[dev];
  if (have_id && c.addr != nullptr && c.ctx_id == id) {
    *out = c.addr;
    return cudaSuccess;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
  if (e != cudaSuccess || p == nullptr) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
  // the lookup binds the device's primary context if none was current
  if (!have_id) have_id = current_ctx_id(&id);
  if (have_id) c = CachedAddr{id, p};      // without an id nothing is cached: look up every call
  *out = p;
  return cudaSuccess;
}

}  // namespace

namespace pkvqk {
void set_last_error(const char* msg);   // api.cu: the per-thread pkvqk_last_error() text
}

extern "C" PKVQK_API size_t pkvqk_static_workspace_capacity(void) { return kStaticWsBytes; }

extern "C" PKVQK_API pkvqk_status pkvqk_paged_decode_static_ws(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k_cache,
    const void* v_cache, const pkvqk_cache_layout* layout, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch, int32_t q_len,
    int32_t num_q_heads, int32_t num_splits, int32_t max_seq_len_hint, float scale, void* out,
    float* lse_out, int32_t* status_flags, pkvqk_stream_t stream) {
  // Arguments the shared validation rejects go straight to it, so that they
  // are reported as argument errors, never as a too-small static workspace.
  if (layout == nullptr || layout->num_kv_heads < 1 || layout->block_size < 1 ||
      layout->head_dim != 128 || num_q_heads < 1 || (num_q_heads % layout->num_kv_heads) != 0 ||
      q_len < 1 || q_len > 16 || batch < 0 || batch > 65535 || num_splits < 0 ||
      num_splits > 256 || max_blocks_per_seq < 1 || max_seq_len_hint < 0) {
    return pkvqk_paged_decode(q, q_stride_t, q_stride_h, k_cache, v_cache, layout, block_tables,
                              max_blocks_per_seq, seq_lens, batch, q_len, num_q_heads,
                              num_splits, max_seq_len_hint, scale, out, lse_out, nullptr, 0,
                              status_flags, stream);
  }
  // the split count the call will use (the documented num_splits == 0 rule)
  int S = num_splits;
  if (S == 0) {
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * layout->block_size;
    const int32_t hint = max_seq_len_hint > 0
                             ? max_seq_len_hint
                             : static_cast<int32_t>(cap < INT32_MAX ? cap : INT32_MAX);
    S = pkvqk_choose_num_splits(batch, layout->num_kv_heads,
                                q_len * (num_q_heads / layout->num_kv_heads), hint,
                                static_cast<int64_t>(hint) * batch, layout->block_size, 0);
    // The heuristic answers 0 (the balanced schedule, whose workspace this
    // call does not provide) only for batches of mixed lengths; the total
    // passed here is hint x batch, a uniform batch, so it never does.  The
    // clamp keeps this call on the split schedule should that rule change.
    if (S < 1) S = 1;
  }
  const size_t need =
      pkvqk_decode_workspace_bytes(batch, q_len, num_q_heads, layout->head_dim, S);
  if (need > kStaticWsBytes) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "pkvqk_paged_decode_static_ws: the static workspace holds %zu bytes but "
                  "batch %d x q_len %d x %d heads x %d splits needs %zu; use fewer splits or "
                  "pkvqk_paged_decode with a caller workspace",
                  kStaticWsBytes, batch, q_len, num_q_heads, S, need);
    pkvqk::set_last_error(msg);
    return PKVQK_ERR_WORKSPACE_TOO_SMALL;
  }

  void* ws = nullptr;
  if (need > 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
      pkvqk::set_last_error("pkvqk_paged_decode_static_ws: no usable current device");
      return PKVQK_ERR_CUDA;
    }
    e = static_ws_address(dev, &ws);
    if (e != cudaSuccess) {
      char msg[160];
      std::snprintf(msg, sizeof(msg), "pkvqk_paged_decode_static_ws: cudaGetSymbolAddress: %s",
                    cudaGetErrorName(e));
      pkvqk::set_last_error(msg);
      return PKVQK_ERR_CUDA;
    }
  }
  return pkvqk_paged_decode(q, q_stride_t, q_stride_h, k_cache, v_cache, layout, block_tables,
                            max_blocks_per_seq, seq_lens, batch, q_len, num_q_heads, S,
                            max_seq_len_hint, scale, out, lse_out, ws, need ? kStaticWsBytes : 0,
                            status_flags, stream);
}
