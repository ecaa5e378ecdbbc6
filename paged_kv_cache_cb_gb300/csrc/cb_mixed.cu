// One launch for a mixed continuous-batching step ([CB] Continuous batching:
// prefill chunks and decode tokens in one ragged batch).
//
// Persistent grid, one CTA (6 warps) per SM.  Phase 1 runs this CTA's share of
// the prefill tiles (requests with more than one new token, [CB] Chunked
// prefill) on the tensor cores; phase 2 turns all six warps into decode
// workers that pull (request, KV head, split) items from a global counter, so
// CTAs that finish their prefill share early absorb more decode work.
//
// Prefill tile = (request r, KV head g, query tile): 128 rows = 128/G new tokens
// x the G query heads of group g (GQA heads packed into the M dimension, all
// sharing KV head g).  Row i is token i/G, head g*G + i%G, at absolute position
// ctx + token; it sees keys 0..ctx+token (the chunk's causal mask shifted by the
// stored prefix).  Keys stream in tiles of 128 (8 physical blocks of 16, each
// fetched through the block table by two 2-D TMA boxes of 16 rows x 64 columns,
// 128-byte swizzle, straight into the canonical K-major layout).
//
// Warp roles:  warps 0-3  softmax: thread i owns row i.  Reads S from tensor
//                         memory (TMEM), masks, keeps the running max m and sum
//                         l in base 2, writes P (bf16) to shared memory, rescales
//                         the O accumulator in TMEM when the max grows by more
//                         than 2^8 (lazy rescale: exact, the final O/l uses the
//                         same reference max), and finally writes O/l.
//              warp 4     TMA producer: Q tile, then K/V tiles into 2 stages.
//              warp 5     MMA issuer: S = Q K^T into one of two TMEM buffers
//                         (tcgen05.mma kind::f16, M=128 N=128 K=16 steps), and
//                         O += P V into the TMEM accumulator (V as MN-major
//                         operand); completion via tcgen05.commit -> mbarrier.
// S(j+1) is issued before O += P(j) V(j), so the tensor core computes the next
// score tile while the softmax warps work on the current one.
#include "cb_decode_item.cuh"

namespace cb {

namespace {

constexpr int kSmemLimit = 232448;
constexpr int kNumThreads = 192;
constexpr int kDecStages = 3;

template <int A>
struct PrefillTiles {
  static constexpr int kHalves = A / 64;
  static constexpr int kHalfBytes = 128 * 128;     // 128 rows x 128 bytes
  uint8_t q[kHalves][128][128];
  uint8_t k[2][kHalves][128][128];
  uint8_t v[2][kHalves][128][128];
  uint8_t p[2][128][128];                          // P: [key half][row][64 keys]
};

struct MixedCtl {
  uint64_t q_full, q_empty, k_full[2], v_full[2], kv_empty[2], s_full[2], s_free[2], p_full, o_done, o_free, drain;
  uint32_t tmem_base;
  volatile int abort;
  int scratch[96];
};

struct PreItem {
  int r, g, q0, ctx, tok_lo, tok_hi, kv_hi, nkt;
};

__device__ __forceinline__ PreItem pre_item(const StepParams& P, const int* pre, int item, int tok_per_tile) {
  PreItem I;
  I.r = find_request(pre, P.n_reqs, item);
  const int rem = item - pre[I.r];
  I.q0 = __ldg(P.cu_q_lens + I.r);
  const int q_len = __ldg(P.cu_q_lens + I.r + 1) - I.q0;
  I.ctx = __ldg(P.ctx_lens + I.r);
  const int n_qt = (q_len + tok_per_tile - 1) / tok_per_tile;
  const int qt = n_qt - 1 - rem / P.n_kv_heads;    // heaviest (last) query tiles first
  I.g = rem % P.n_kv_heads;
  I.tok_lo = qt * tok_per_tile;
  I.tok_hi = min(q_len, I.tok_lo + tok_per_tile);
  I.kv_hi = I.ctx + I.tok_hi;
  I.nkt = (I.kv_hi + kTileN - 1) / kTileN;
  return I;
}

// Bounded wait whose outcome is the same for all 32 lanes of the warp.
__device__ __forceinline__ bool warp_wait(const StepParams& P, uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  if (!ok) set_error(P.err, CB_DEVERR_TIMEOUT);
  return __all_sync(0xffffffffu, ok);
}

template <int A, int G>
__device__ void producer(const StepParams& P, const CUtensorMap* kmap, const CUtensorMap* vmap,
                         const CUtensorMap* qmap, PrefillTiles<A>& T, MixedCtl& C, const int* pre) {
  constexpr int TOK = kTileM / G;
  constexpr int H = A / 64;
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int n_pre = pre[P.n_reqs];
  const int Hkv = P.n_kv_heads;
  const int rows_total = P.num_blocks * Hkv * kBlockSize;
  uint32_t kv_it = 0, it = 0;
  for (int item = blockIdx.x; item < n_pre; item += gridDim.x, ++it) {
    if (C.abort) break;
    const PreItem I = pre_item(P, pre, item, TOK);
    int ok = 1;
    if (lane == 0) {
      ok = mbar_wait(&C.q_empty, (it & 1) ^ 1);
      if (ok) {
        mbar_arrive_expect_tx(&C.q_full, H * PrefillTiles<A>::kHalfBytes);
#pragma unroll
        for (int hf = 0; hf < H; ++hf) tma_load_3d(&T.q[hf][0][0], qmap, hf * 64, I.g * G, I.q0 + I.tok_lo, &C.q_full);
      }
    }
    if (!__shfl_sync(FULL, ok, 0)) {
      if (lane == 0) set_error(P.err, CB_DEVERR_TIMEOUT);
      C.abort = 1;
      break;
    }
    const int nblk_hi = (I.kv_hi + kBlockSize - 1) / kBlockSize;
    int y = rows_total;
    for (int j = 0; j < I.nkt; ++j, ++kv_it) {
      if ((j & 3) == 0) {          // table entries for this tile and the next three
        const int blk = j * 8 + lane;
        y = rows_total;
        if (blk < nblk_hi) {
          const int e = __ldg(P.block_tables + (size_t)I.r * P.max_blocks_per_seq + blk);
          if (e >= 0 && e < P.num_blocks)
            y = (e * Hkv + I.g) * kBlockSize;
          else
            set_error(P.err, CB_DEVERR_BADBLOCK);
        }
      }
      const int st = kv_it & 1;
      const uint32_t ph = (kv_it >> 1) & 1;
      ok = 1;
      if (lane == 0) ok = mbar_wait(&C.kv_empty[st], ph ^ 1);
      if (!__shfl_sync(FULL, ok, 0)) {
        if (lane == 0) set_error(P.err, CB_DEVERR_TIMEOUT);
        C.abort = 1;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&C.k_full[st], H * PrefillTiles<A>::kHalfBytes);
        mbar_arrive_expect_tx(&C.v_full[st], H * PrefillTiles<A>::kHalfBytes);
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int yb = __shfl_sync(FULL, y, (j & 3) * 8 + b);
        if (lane == 0) {
#pragma unroll
          for (int hf = 0; hf < H; ++hf) {
            tma_load_2d(&T.k[st][hf][b * kBlockSize][0], kmap, hf * 64, yb, &C.k_full[st]);
            tma_load_2d(&T.v[st][hf][b * kBlockSize][0], vmap, hf * 64, yb, &C.v_full[st]);
          }
        }
      }
    }
    if (C.abort) break;
  }
  // drain: every load issued above has landed before shared memory is reused
  if (lane == 0 && C.abort) {
    for (int s = 0; s < 2; ++s) {
      mbar_wait(&C.k_full[s], 0, 20000000ull);
      mbar_wait(&C.k_full[s], 1, 20000000ull);
      mbar_wait(&C.v_full[s], 0, 20000000ull);
      mbar_wait(&C.v_full[s], 1, 20000000ull);
    }
    mbar_wait(&C.q_full, 0, 20000000ull);
    mbar_wait(&C.q_full, 1, 20000000ull);
  }
}

template <int A, int G>
__device__ void mma_issuer(const StepParams& P, PrefillTiles<A>& T, MixedCtl& C, const int* pre, uint32_t tmem) {
  constexpr int TOK = kTileM / G;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, A, 1);
  const int n_pre = pre[P.n_reqs];
  const uint32_t q_s = smem_u32(&T.q[0][0][0]);
  const uint32_t p_s = smem_u32(&T.p[0][0][0]);
  const uint32_t tm_o = tmem + 256;
  uint32_t kv_it = 0, it = 0;
  bool ok = true;
  auto issue_s = [&](uint32_t kvj) -> bool {
    const int st = kvj & 1;
    const uint32_t ph = (kvj >> 1) & 1;
    if (!mbar_wait(&C.k_full[st], ph) || !mbar_wait(&C.s_free[st], ph ^ 1)) return false;
    tc_fence_after();
    const uint32_t k_s = smem_u32(&T.k[st][0][0][0]);
#pragma unroll
    for (int ks = 0; ks < A / 16; ++ks) {
      const uint32_t off = (ks >> 2) * PrefillTiles<A>::kHalfBytes + (ks & 3) * 32;
      tc_mma_f16(tmem + st * 128, smem_desc_sw128(q_s + off, 16, 1024), smem_desc_sw128(k_s + off, 16, 1024),
                 kIdescS, ks > 0);
    }
    tc_commit(&C.s_full[st]);
    return true;
  };
  for (int item = blockIdx.x; item < n_pre && ok; item += gridDim.x, ++it) {
    if (C.abort) break;
    const PreItem I = pre_item(P, pre, item, TOK);
    if (!mbar_wait(&C.q_full, it & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (!issue_s(kv_it)) {
      ok = false;
      break;
    }
    for (int j = 0; j < I.nkt; ++j) {
      const uint32_t kvj = kv_it + j;
      if (j + 1 < I.nkt) {
        if (!issue_s(kvj + 1)) {
          ok = false;
          break;
        }
      } else {
        tc_commit(&C.q_empty);    // the last S of this item has been issued: Q free once it completes
      }
      const int st = kvj & 1;
      const uint32_t ph = (kvj >> 1) & 1;
      if (!mbar_wait(&C.p_full, kvj & 1) || (j == 0 && !mbar_wait(&C.o_free, (it & 1) ^ 1)) ||
          !mbar_wait(&C.v_full[st], ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t v_s = smem_u32(&T.v[st][0][0][0]);
#pragma unroll
      for (int ks = 0; ks < kTileN / 16; ++ks) {
        const uint32_t poff = (ks >> 2) * PrefillTiles<A>::kHalfBytes + (ks & 3) * 32;
        tc_mma_f16(tm_o, smem_desc_sw128(p_s + poff, 16, 1024),
                   smem_desc_sw128(v_s + ks * 16 * 128, PrefillTiles<A>::kHalfBytes, 1024), kIdescPV,
                   (j > 0 || ks > 0) ? 1u : 0u);
      }
      tc_commit(&C.o_done);
      tc_commit(&C.kv_empty[st]);
    }
    kv_it += I.nkt;
  }
  if (!ok) {
    set_error(P.err, CB_DEVERR_TIMEOUT);
    C.abort = 1;
  }
  tc_commit(&C.drain);           // every MMA issued above is complete before TMEM is freed
  mbar_wait(&C.drain, 0, 20000000ull);
}

template <int A, int G>
__device__ void softmax_warps(const StepParams& P, PrefillTiles<A>& T, MixedCtl& C, const int* pre, uint32_t tmem) {
  constexpr int TOK = kTileM / G;
  constexpr int H = A / 64;
  const unsigned FULL = 0xffffffffu;
  const int row = threadIdx.x;               // 0..127
  const int warp = row >> 5;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const int n_pre = pre[P.n_reqs];
  const int Hq = P.n_q_heads;
  const float sl2 = P.scale_log2;
  uint32_t kv_it = 0, it = 0;
  for (int item = blockIdx.x; item < n_pre; item += gridDim.x, ++it) {
    if (C.abort) break;
    const PreItem I = pre_item(P, pre, item, TOK);
    const int tok_l = row / G, gq = row % G;
    const int ti = I.tok_lo + tok_l;
    const bool valid_row = ti < I.tok_hi;
    const int pos = I.ctx + min(ti, I.tok_hi - 1);     // last key this row may see
    float m = kNegInf, l = 0.f;
    bool ok = true;
    for (int j = 0; j < I.nkt; ++j) {
      const uint32_t kvj = kv_it + j;
      const int st = kvj & 1;
      const uint32_t ph = (kvj >> 1) & 1;
      if (!warp_wait(P, &C.s_full[st], ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + st * 128 + c * 32, s[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&C.s_free[st]);
      const int key0 = j * kTileN;
      float mt = kNegInf;
      if (key0 + kTileN - 1 <= pos) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            s[c][k] *= sl2;
            mt = fmaxf(mt, s[c][k]);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            s[c][k] = (key0 + c * 32 + k <= pos) ? s[c][k] * sl2 : kNegInf;
            mt = fmaxf(mt, s[c][k]);
          }
      }
      const float mn = fmaxf(m, mt);
      const bool need = mn > m + 8.f;
      if (j > 0) {
        if (!warp_wait(P, &C.o_done, (kvj - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      float alpha = 1.f;
      if (need) {
        alpha = ex2(m - mn);
        m = mn;
      }
      if (j > 0 && __any_sync(FULL, need)) {
#pragma unroll 1
        for (int c = 0; c < A / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + 256 + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(tmem + lane_base + 256 + c * 32, o);
        }
        tmem_wait_st();
      }
      float rs = 0.f;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const int c = h2 * 2 + (ch >> 2), k0 = (ch & 3) * 8;
          float pv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            pv[k] = ex2(s[c][k0 + k] - m);
            rs += pv[k];
          }
          uint4 w;
          w.x = pack_bf16(pv[0], pv[1]);
          w.y = pack_bf16(pv[2], pv[3]);
          w.z = pack_bf16(pv[4], pv[5]);
          w.w = pack_bf16(pv[6], pv[7]);
          *reinterpret_cast<uint4*>(&T.p[h2][row][(ch ^ (row & 7)) << 4]) = w;
        }
      l = l * alpha + rs;
      // rows past the last key of this tile's request part of the final block hold
      // whatever the cache had there: zero them so 0 * (non-finite) cannot reach O
      if (key0 + kTileN > I.kv_hi && (I.kv_hi & (kBlockSize - 1))) {
        if (!warp_wait(P, &C.v_full[st], ph)) {
          ok = false;
          break;
        }
        const int r0 = I.kv_hi - key0;
        const int r1 = min(kTileN, ((I.kv_hi + kBlockSize - 1) & ~(kBlockSize - 1)) - key0);
        const int total = (r1 - r0) * H * 8;
        for (int idx = row; idx < total; idx += 128) {
          const int rr = r0 + idx / (H * 8), rest = idx % (H * 8);
          *reinterpret_cast<uint4*>(&T.v[st][rest >> 3][rr][(rest & 7) << 4]) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&C.p_full);
    }
    if (!ok) {
      C.abort = 1;
      break;
    }
    const uint32_t kvl = kv_it + I.nkt - 1;
    if (!warp_wait(P, &C.o_done, kvl & 1)) {
      C.abort = 1;
      break;
    }
    tc_fence_after();
    const float inv = 1.f / l;
    uint16_t* orow = P.out + ((size_t)(I.q0 + ti) * Hq + (size_t)I.g * G + gq) * A;
#pragma unroll 1
    for (int c = 0; c < A / 32; ++c) {
      float o[32];
      tmem_ld32(tmem + lane_base + 256 + c * 32, o);
      tmem_wait_ld();
      if (valid_row) {
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          uint4 w;
          w.x = pack_bf16(o[k] * inv, o[k + 1] * inv);
          w.y = pack_bf16(o[k + 2] * inv, o[k + 3] * inv);
          w.z = pack_bf16(o[k + 4] * inv, o[k + 5] * inv);
          w.w = pack_bf16(o[k + 6] * inv, o[k + 7] * inv);
          *reinterpret_cast<uint4*>(orow + c * 32 + k) = w;
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&C.o_free);
    kv_it += I.nkt;
  }
}

template <int A, int G>
__global__ void __launch_bounds__(kNumThreads, 1)
    mixed_kernel(const StepParams P, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const __grid_constant__ CUtensorMap qmap) {
  constexpr int TOK = kTileM / G;
  using WS = DecWarpSmem<A, G, kDecStages>;
  static_assert(6 * sizeof(WS) <= sizeof(PrefillTiles<A>), "decode rings must fit in the tile region");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PrefillTiles<A>& T = *reinterpret_cast<PrefillTiles<A>*>(base);
  MixedCtl& C = *reinterpret_cast<MixedCtl*>(base + sizeof(PrefillTiles<A>));
  int* dec = reinterpret_cast<int*>(base + sizeof(PrefillTiles<A>) + sizeof(MixedCtl));
  int* spl = dec + (P.n_reqs + 1);
  int* pre = spl + (P.n_reqs + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&C.q_full, 1);
    mbar_init(&C.q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&C.k_full[s], 1);
      mbar_init(&C.v_full[s], 1);
      mbar_init(&C.kv_empty[s], 1);
      mbar_init(&C.s_full[s], 1);
      mbar_init(&C.s_free[s], 128);
    }
    mbar_init(&C.p_full, 128);
    mbar_init(&C.o_done, 1);
    mbar_init(&C.o_free, 128);
    mbar_init(&C.drain, 1);
    C.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&qmap);
  }
  if (warp == 5) {
    tmem_alloc(&C.tmem_base, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  build_plan(P, TOK, dec, spl, pre, C.scratch);     // ends with __syncthreads()
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;

  if (pre[P.n_reqs] > 0) {
    if (warp == 4) {
      producer<A, G>(P, &kmap, &vmap, &qmap, T, C, pre);
    } else if (warp == 5) {
      if (lane == 0) mma_issuer<A, G>(P, T, C, pre, tmem);
      __syncwarp();
    } else {
      softmax_warps<A, G>(P, T, C, pre, tmem);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (C.abort) return;
  decode_worker<A, G, kDecStages>(P, &kmap, &vmap, reinterpret_cast<WS*>(base)[warp], dec, spl);
}

template <int A, int G>
cudaError_t launch_mixed_t(const StepParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& qmap, int n_sms, cudaStream_t stream) {
  const size_t smem = 1024 + sizeof(PrefillTiles<A>) + sizeof(MixedCtl) + (size_t)3 * (p.n_reqs + 1) * 4;
  if (smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mixed_kernel<A, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  mixed_kernel<A, G><<<n_sms, kNumThreads, smem, stream>>>(p, kmap, vmap, qmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mixed(const StepParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const CUtensorMap& qmap, int head_dim, int group, int n_sms, cudaStream_t stream) {
#define CB_MIX_CASE(A_, G_) \
  if (head_dim == A_ && group == G_) return launch_mixed_t<A_, G_>(p, kmap, vmap, qmap, n_sms, stream);
  CB_MIX_CASE(128, 1)
  CB_MIX_CASE(128, 2)
  CB_MIX_CASE(128, 4)
  CB_MIX_CASE(128, 8)
  CB_MIX_CASE(64, 1)
  CB_MIX_CASE(64, 2)
  CB_MIX_CASE(64, 4)
  CB_MIX_CASE(64, 8)
#undef CB_MIX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace cb
