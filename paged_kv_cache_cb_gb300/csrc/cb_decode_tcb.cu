// Decode kernel for head_dim 128 with 8 KV heads, or with 32 query heads on 2
// KV heads (GQA, G = 16) or on 1 (MQA): the block-tile pipeline of
// cb_decode_tcb.cuh ([CB] KV cache, [KVN] MQA/GQA).
#include "cb_decode_tcb.cuh"

namespace cb {

namespace {

using namespace tcb;

constexpr int kSmemLimit = 232448;

template <int G, int HKV>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tcb_kernel(const StepParams P, const AppendParams Ap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Tiles<G, HKV>& T = *reinterpret_cast<Tiles<G, HKV>*>(base);
  Ctl<G, HKV>& C = *reinterpret_cast<Ctl<G, HKV>*>(base + sizeof(Tiles<G, HKV>));
  int* bpre = reinterpret_cast<int*>(base + sizeof(Tiles<G, HKV>) + sizeof(Ctl<G, HKV>));
  int* slot = bpre + (P.n_reqs + 1);
  const int warp = threadIdx.x >> 5;

  zero_p<G, HKV>(T);                    // P's off-diagonal zeros
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    init_ctl<G, HKV>(C);
    fence_mbar_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&qmap);
  }
  if (warp == 5) {
    tmem_alloc(&C.tmem_base, Cfg<G, HKV>::TM);
    tmem_relinquish();
    tc_fence_before();
  }
  append_phase<HKV == 8>(P, Ap);             // the step's new rows, when this launch stores them
  for (int r = threadIdx.x; r < P.n_reqs; r += blockDim.x) bpre[r] = decode_blocks(P, r, false);
  __syncthreads();
  finish_plan<G, HKV>(P, C, bpre, slot);
  if (threadIdx.x == 0) C.per_request = per_request_merge<G, HKV>(P, false);
  append_wait<HKV == 8>(P, Ap);             // (its barrier publishes per_request too)
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  run_pipeline<G, HKV>(P, &kmap, &vmap, &qmap, T, C, bpre, slot, tmem, true);
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg<G, HKV>::TM);
  }
  merge_phase<G, HKV>(P, C, slot, reinterpret_cast<float*>(&T.k[0][0][0][0]), false);   // the K ring is free now
  release_counters(P);
}

template <int G, int HKV>
constexpr size_t smem_bytes(int n_reqs) {
  return 1024 + sizeof(Tiles<G, HKV>) + sizeof(Ctl<G, HKV>) + (size_t)(2 * n_reqs + 2) * 4;
}
static_assert(smem_bytes<2, 8>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(smem_bytes<4, 8>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(smem_bytes<8, 8>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(smem_bytes<16, 2>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(smem_bytes<32, 1>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");

template <int G, int HKV>
cudaError_t launch_t(const StepParams& p, const AppendParams& ap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     const CUtensorMap& qmap, int n_sms, cudaStream_t stream) {
  const size_t smem = smem_bytes<G, HKV>(p.n_reqs);
  if (smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(decode_tcb_kernel<G, HKV>), kSmemLimit);
  if (e != cudaSuccess) return e;
  // cooperative: the merge phase waits for every CTA
  StepParams pc = p;
  AppendParams apc = ap;
  void* args[] = {&pc, &apc, const_cast<CUtensorMap*>(&kmap), const_cast<CUtensorMap*>(&vmap),
                  const_cast<CUtensorMap*>(&qmap)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(decode_tcb_kernel<G, HKV>), dim3(n_sms), dim3(kThreads),
                                     args, smem, stream);
}

}  // namespace

cudaError_t launch_decode_tcb(const StepParams& p, const AppendParams& ap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& qmap, int group, int n_sms,
                              cudaStream_t stream) {
  if (p.n_kv_heads == 8) {
    switch (group) {
      case 2: return launch_t<2, 8>(p, ap, kmap, vmap, qmap, n_sms, stream);
      case 4: return launch_t<4, 8>(p, ap, kmap, vmap, qmap, n_sms, stream);
      case 8: return launch_t<8, 8>(p, ap, kmap, vmap, qmap, n_sms, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.n_kv_heads == 2 && group == 16) return launch_t<16, 2>(p, ap, kmap, vmap, qmap, n_sms, stream);
  if (p.n_kv_heads == 1 && group == 32) return launch_t<32, 1>(p, ap, kmap, vmap, qmap, n_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace cb
