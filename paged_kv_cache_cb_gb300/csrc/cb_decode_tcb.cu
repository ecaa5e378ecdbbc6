// Decode kernel for GQA steps with 8 KV heads and head_dim 128: the block-tile
// pipeline of cb_decode_tcb.cuh ([CB] KV cache, [KVN] MQA/GQA), with the
// requests ordered longest first.
#include "cb_decode_tcb.cuh"

namespace cb {

namespace {

using namespace tcb;

constexpr int kSmemLimit = 232448;

// Orders the requests longest first (keys (blocks, 2047 - r), descending: by
// rank counting for up to 256 requests, else a bitonic network in `keys`):
// order[i] = request at position i; then finish_plan.  Ends with
// __syncthreads().
template <int G>
__device__ void plan_sorted(const StepParams& P, Ctl<G>& C, unsigned long long* keys, int* order, int* bpre,
                            int* slot) {
  const int n = P.n_reqs, tid = threadIdx.x, T = blockDim.x;
  int npad = 1;
  while (npad < n) npad <<= 1;
  for (int i = tid; i < npad; i += T)
    keys[i] = i < n ? ((unsigned long long)decode_blocks(P, i, false) << 32) | (unsigned)(kMaxReqs - 1 - i) : 0ull;
  __syncthreads();
  if (n <= 256) {
    // few requests: each key's rank is the number of larger keys (keys are distinct)
    for (int i = tid; i < n; i += T) {
      const unsigned long long ki = keys[i];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += keys[j] > ki;
      order[rank] = kMaxReqs - 1 - (int)(ki & 0xffffffffu);
      bpre[rank] = (int)(ki >> 32);
    }
    npad = 0;                      // skip the sorting network
  }
  for (int k = 2; k <= npad; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < npad; i += T) {
        const int o = i ^ j;
        if (o > i) {
          const unsigned long long a = keys[i], b = keys[o];
          if (((i & k) == 0) ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[o] = a;
          }
        }
      }
      __syncthreads();
    }
  if (npad)
    for (int i = tid; i < n; i += T) {
      order[i] = kMaxReqs - 1 - (int)(keys[i] & 0xffffffffu);
      bpre[i] = (int)(keys[i] >> 32);
    }
  __syncthreads();
  finish_plan<G>(P, C, bpre, slot);
  fence_proxy_async_smem();        // `keys` is tile memory that TMA fills next
  __syncthreads();
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tcb_kernel(const StepParams P, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Tiles<G>& T = *reinterpret_cast<Tiles<G>*>(base);
  Ctl<G>& C = *reinterpret_cast<Ctl<G>*>(base + sizeof(Tiles<G>));
  int* order = reinterpret_cast<int*>(base + sizeof(Tiles<G>) + sizeof(Ctl<G>));
  int* bpre = order + P.n_reqs;
  int* slot = bpre + (P.n_reqs + 1);
  const int warp = threadIdx.x >> 5;

  zero_p<G>(T);                    // P's off-diagonal zeros
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    init_ctl<G>(C);
    fence_mbar_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&qmap);
  }
  if (warp == 5) {
    tmem_alloc(&C.tmem_base, Cfg<G>::TM);
    tmem_relinquish();
    tc_fence_before();
  }
  // the sort keys live in the K ring until the plan is made
  plan_sorted<G>(P, C, reinterpret_cast<unsigned long long*>(&T.k[0][0][0][0]), order, bpre, slot);
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  run_pipeline<G>(P, &kmap, &vmap, &qmap, T, C, order, bpre, slot, tmem);
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg<G>::TM);
  }
  merge_phase<G>(P, C, order, slot);
}

template <int G>
constexpr size_t smem_bytes(int n_reqs) {
  return 1024 + sizeof(Tiles<G>) + sizeof(Ctl<G>) + (size_t)(3 * n_reqs + 2) * 4;
}
static_assert(sizeof(Tiles<2>::k) >= kMaxReqs * 8, "sort keys fit in the K ring");
static_assert(smem_bytes<2>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(smem_bytes<4>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(smem_bytes<8>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");

template <int G>
cudaError_t launch_t(const StepParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                     int n_sms, cudaStream_t stream) {
  const size_t smem = smem_bytes<G>(p.n_reqs);
  if (smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_tcb_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // cooperative: the merge phase waits for every CTA
  StepParams pc = p;
  void* args[] = {&pc, const_cast<CUtensorMap*>(&kmap), const_cast<CUtensorMap*>(&vmap),
                  const_cast<CUtensorMap*>(&qmap)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(decode_tcb_kernel<G>), dim3(n_sms), dim3(kThreads),
                                     args, smem, stream);
}

}  // namespace

cudaError_t launch_decode_tcb(const StepParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              const CUtensorMap& qmap, int group, int n_sms, cudaStream_t stream) {
  switch (group) {
    case 2: return launch_t<2>(p, kmap, vmap, qmap, n_sms, stream);
    case 4: return launch_t<4>(p, kmap, vmap, qmap, n_sms, stream);
    case 8: return launch_t<8>(p, kmap, vmap, qmap, n_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cb
