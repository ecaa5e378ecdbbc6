// Slot-mapped KV append and the HBM copy probe.
//
// Append: [CB] Chunked prefill ("store the KV states") with the paged placement of
// [SM] PagedAttention 批处理: new token t's key/value rows for every KV head go to
// physical block slot/bs at in-block offset slot%bs.  Pure data movement: one
// 16-byte vector per thread, consecutive threads on consecutive 16-byte pieces of
// the same row, so reads of k_new and writes into the 256-byte (A=128) cache rows
// are both fully coalesced.  Bit-exact by construction.
#include <algorithm>

#include "cb_common.cuh"

namespace cb {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                                        const int64_t* __restrict__ slots, int n_tokens,
                                                        uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                        int64_t n_slots, int n_kv_heads, int chunks_per_row,
                                                        unsigned int* __restrict__ err) {
  append_pieces(k_new, v_new, slots, n_tokens, k_cache, v_cache, n_slots, n_kv_heads, chunks_per_row, err,
                blockIdx.x * (int64_t)blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int64_t* slots, int n_tokens, void* k_cache,
                             void* v_cache, int num_blocks, int n_kv_heads, int head_dim, unsigned int* err,
                             cudaStream_t stream) {
  if (n_tokens == 0) return cudaSuccess;
  const int chunks = head_dim / 8;
  const int64_t total = (int64_t)n_tokens * n_kv_heads * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  kv_append_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, n_tokens, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), (int64_t)num_blocks * kBlockSize, n_kv_heads, chunks, err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- block copies
// Copy-on-write of shared blocks ([KVB] 思想: blocks shared through the block
// table): cache block dst = block src, all KV heads, K and V.  grid.y = pair,
// grid.x CTAs stride over the block's 16-byte pieces.  Bit-exact.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t* __restrict__ pairs, uint4* __restrict__ k_cache,
                                                          uint4* __restrict__ v_cache, int num_blocks,
                                                          int64_t pieces_per_block, unsigned int* __restrict__ err) {
  const int src = __ldg(pairs + 2 * blockIdx.y), dst = __ldg(pairs + 2 * blockIdx.y + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, CB_DEVERR_BADBLOCK);
    return;
  }
  const uint4* ks = k_cache + (int64_t)src * pieces_per_block;
  const uint4* vs = v_cache + (int64_t)src * pieces_per_block;
  uint4* kd = k_cache + (int64_t)dst * pieces_per_block;
  uint4* vd = v_cache + (int64_t)dst * pieces_per_block;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < pieces_per_block;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 k = ks[i], v = vs[i];
    kd[i] = k;
    vd[i] = v;
  }
}

cudaError_t launch_copy_blocks(const int32_t* pairs, int n_pairs, void* k_cache, void* v_cache, int num_blocks,
                               int n_kv_heads, int head_dim, unsigned int* err, cudaStream_t stream) {
  if (n_pairs == 0) return cudaSuccess;
  const int64_t pieces = (int64_t)n_kv_heads * kBlockSize * head_dim / 8;
  const int ctas = (int)std::min<int64_t>(8, (pieces + 255) / 256);
  copy_blocks_kernel<<<dim3(ctas, n_pairs), 256, 0, stream>>>(pairs, static_cast<uint4*>(k_cache),
                                                             static_cast<uint4*>(v_cache), num_blocks, pieces, err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- HBM copy probe
// Streaming copy with four independent 16-byte loads in flight per thread.
__global__ void __launch_bounds__(512) hbm_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
          d = __ldcs(src + i + 3 * stride);
    __stcs(dst + i, a);
    __stcs(dst + i + stride, b);
    __stcs(dst + i + 2 * stride, c);
    __stcs(dst + i + 3 * stride, d);
  }
  for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

cudaError_t launch_hbm_copy(void* dst, const void* src, size_t bytes, int n_sms, cudaStream_t stream) {
  const size_t n = bytes / 16;
  if (n == 0) return cudaSuccess;
  hbm_copy_kernel<<<n_sms * 4, 512, 0, stream>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src), n);
  return cudaGetLastError();
}

}  // namespace cb
