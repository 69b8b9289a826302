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
// (it names a host-side shadow), so its device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device.
#include "pkvqk.h"

#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

namespace {

constexpr size_t kStaticWsBytes = size_t(16) << 20;   // 16 MiB of partials per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {nullptr};

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
  if (layout == nullptr || layout->num_kv_heads < 1 || layout->block_size < 1 ||
      num_q_heads < 1 || q_len < 1 || batch < 0 || num_splits < 0 || max_blocks_per_seq < 1 ||
      max_seq_len_hint < 0) {
    // argument errors are reported by the shared validation below
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
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ws_addr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_ws);
      if (e != cudaSuccess || p == nullptr) {
        pkvqk::set_last_error("pkvqk_paged_decode_static_ws: cudaGetSymbolAddress failed");
        return PKVQK_ERR_CUDA;
      }
      g_ws_addr[dev] = p;
    }
    ws = g_ws_addr[dev];
  }
  return pkvqk_paged_decode(q, q_stride_t, q_stride_h, k_cache, v_cache, layout, block_tables,
                            max_blocks_per_seq, seq_lens, batch, q_len, num_q_heads, S,
                            max_seq_len_hint, scale, out, lse_out, ws, need ? kStaticWsBytes : 0,
                            status_flags, stream);
}
