// cb_paged_attention_noalloc: the attention step for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run a step: embedders whose device memory is owned by a custom
// allocator or a fixed arena that this library does not see (a plugin may not
// allocate behind its host's back), and real-time serving loops that forbid
// allocation because it can synchronise the device and has unbounded latency.
// For them this entry point takes its
// scratch -- split-K partial results, per-(request, KV head) arrival counters
// and the work-queue counter -- from one fixed array that lives in the
// library's own device memory, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable of CB_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host code
// must not use the variable's name as a device address (on the host it is only
// a stand-in), so the first call on each device looks the real address up with
// cudaGetSymbolAddress, with that device current, and caches it; make that
// first call before any stream capture.  All calls on a device share the array
// (it keeps the last call's contents), so calls that overlap on the GPU race.
#include <mutex>

#include "../../include/cbattn.h"
#include "cb_internal.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[CB_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_address() {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int cb_paged_attention_noalloc(const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                                          const int32_t* block_tables, int max_blocks_per_seq, int n_reqs,
                                          int n_tokens, int max_q_len, int max_kv_len, const void* k_cache,
                                          const void* v_cache, int num_blocks, void* out, float scale, int n_q_heads,
                                          int n_kv_heads, int head_dim, int block_size, void* stream) {
  // the step falls back to whole prefill pairs when the partials do not fit
  const size_t need = cb::workspace_min_bytes(n_reqs, n_tokens, max_q_len, max_kv_len, n_q_heads, n_kv_heads,
                                              head_dim, block_size);
  if (need == 0) return CB_EINVAL;
  if (need > (size_t)CB_NOALLOC_SCRATCH_BYTES) return CB_EWORKSPACE;   // sizes beyond the fixed scratch
  void* ws = scratch_address();
  if (!ws) return CB_ECUDA;
  // as much of the array as the size query asks for: the same plan as the
  // workspace entry point given that workspace, whenever it fits
  const size_t want = cb_paged_attention_workspace_size(n_reqs, n_tokens, max_q_len, max_kv_len, n_q_heads,
                                                        n_kv_heads, head_dim, block_size);
  const size_t use = want < (size_t)CB_NOALLOC_SCRATCH_BYTES ? want : (size_t)CB_NOALLOC_SCRATCH_BYTES;
  return cb_paged_attention(q, cu_q_lens, ctx_lens, block_tables, max_blocks_per_seq, n_reqs, n_tokens, max_q_len,
                            max_kv_len, k_cache, v_cache, num_blocks, out, scale, n_q_heads, n_kv_heads, head_dim,
                            block_size, ws, use, stream);
}
