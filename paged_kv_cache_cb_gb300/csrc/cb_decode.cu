// Decode-only step: every request has exactly one new token ([CB] KV cache;
// [KVB] Batch Decode).  A persistent grid (one CTA per SM) of NW warps; each
// warp pulls (request, KV head, split) items from a global counter and streams
// that split's K/V blocks through its own TMA ring (see cb_decode_item.cuh).
#include "cb_decode_item.cuh"

namespace cb {

namespace {

constexpr int kSmemLimit = 232448;   // opt-in dynamic shared memory per CTA on this part

// Shape (measured best among 7-10 warps x 2-3 stages): NST ring stages per
// warp, as many warps (<= 10) as shared memory holds, QK loop unrolled by 2
// (enough ILP, and registers for 10 warps).  An L2 prefetch of blocks beyond
// the ring was tried and only added traffic.
template <int A, int G>
struct DecodeCfg {
  static constexpr int NST = A == 128 ? 2 : 4;
  static constexpr int QKU = 2;
  using WS = DecWarpSmem<A, G, NST>;
  static constexpr int kPlanMax = (2 * (kMaxReqs + 1) + 96) * 4;
  static constexpr int NW_fit = (kSmemLimit - 1024 - kPlanMax) / (int)sizeof(WS);
  static constexpr int NW = NW_fit < 10 ? NW_fit : 10;
  static_assert(NW >= 4, "decode ring does not fit");
};

template <int A, int G>
__global__ void __launch_bounds__(DecodeCfg<A, G>::NW * 32, 1)
    decode_kernel(const StepParams P, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using C = DecodeCfg<A, G>;
  using WS = typename C::WS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  WS* rings = reinterpret_cast<WS*>(base);
  int* dec = reinterpret_cast<int*>(base + C::NW * sizeof(WS));
  int* spl = dec + (P.n_reqs + 1);
  int* scratch = spl + (P.n_reqs + 1);
  if (threadIdx.x == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  build_plan(P, 1, dec, spl, nullptr, scratch);
  decode_worker<A, G, C::NST, C::QKU>(P, &kmap, &vmap, rings[threadIdx.x >> 5], dec, spl);
}

template <int A, int G>
cudaError_t launch_decode_t(const StepParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int n_sms,
                            cudaStream_t stream) {
  using C = DecodeCfg<A, G>;
  const size_t smem = 1024 + C::NW * sizeof(typename C::WS) + (size_t)(2 * (p.n_reqs + 1) + 96) * 4;
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(decode_kernel<A, G>), kSmemLimit);
  if (e != cudaSuccess) return e;
  decode_kernel<A, G><<<n_sms, C::NW * 32, smem, stream>>>(p, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const StepParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int head_dim,
                          int group, int n_sms, cudaStream_t stream) {
#define CB_DEC_CASE(A_, G_) \
  if (head_dim == A_ && group == G_) return launch_decode_t<A_, G_>(p, kmap, vmap, n_sms, stream);
  CB_DEC_CASE(128, 1)
  CB_DEC_CASE(128, 2)
  CB_DEC_CASE(128, 4)
  CB_DEC_CASE(128, 8)
  CB_DEC_CASE(64, 1)
  CB_DEC_CASE(64, 2)
  CB_DEC_CASE(64, 4)
  CB_DEC_CASE(64, 8)
#undef CB_DEC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace cb
