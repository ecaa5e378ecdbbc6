// Per-CTA work planning and the decode work item, shared by the decode-only
// kernel and the mixed (prefill + decode) kernel.
//
// Decode ([CB] KV cache: one new token attends over every stored key; [KVB]
// Batch Decode: scores scaled by 1/sqrt(head_dim), softmax, times V) is
// memory-bound: each (request, KV head) streams its K/V blocks once.  One warp
// owns one work item = (request r, KV head g, split s): the blocks
// [s*split_blocks, (s+1)*split_blocks) of r's table.  The warp serves all
// G = Hq/Hkv query heads of the group from one read of each K/V block (GQA).
//
// Data path: lane 0 issues 2-D TMA loads (128-byte swizzle) of whole
// (block, head) tiles -- 16 rows x head_dim -- into a private ring of NST stages
// in shared memory, completion tracked by one mbarrier per stage.  Compute per
// 16-token block:
//   QK: lane (t = lane&15, half = lane>>4) dots token t's keys over its half of
//       head_dim with the fp32 query rows (shared memory, broadcast reads; the
//       swizzle makes the 8 lanes of a quarter-warp hit distinct banks).
//   online softmax in base 2 (scores pre-multiplied by scale*log2 e), per head:
//       block max by xor-shuffles, running max m, running sum l, rescale alpha.
//   PV: lane owns head_dim/32 output dims and accumulates p_t * v_t over the
//       block's tokens (p via shared memory, V via swizzled reads).
// Splits write (m, l, unnormalised o) partials; the warp that finishes the last
// split of (r, g) -- found with an arrival counter -- merges them by
// log-sum-exp and writes the bf16 output.  A request with one split writes the
// output directly.
#pragma once
#include "cb_common.cuh"

namespace cb {

#define kNegInf (-__int_as_float(0x7f800000))

// ---------------------------------------------------------------- planning
// First block a decode with kv keys reads under a rolling window W: the block
// holding position kv - W, its first visible key (0 without a window).
__device__ __forceinline__ int window_first_block(long long kv, int window) {
  return window > 0 && kv > window ? (int)((kv - window) / kBlockSize) : 0;
}

// Work counts of request r.  Validates the metadata; a bad request gets no work
// and sets CB_DEVERR_BADLEN.
struct ReqWork {
  int dec_items, splits, pre_items;
};

__device__ __forceinline__ ReqWork request_work(const StepParams& P, int r, int tok_per_tile, bool allow_prefill) {
  ReqWork w{0, 0, 0};
  const int q0 = __ldg(P.cu_q_lens + r), q1 = __ldg(P.cu_q_lens + r + 1);
  const int ctx = __ldg(P.ctx_lens + r);
  const int q_len = q1 - q0;
  const long long kv = (long long)ctx + q_len;
  const long long nblk = (kv + kBlockSize - 1) / kBlockSize;
  if (q_len < 0 || ctx < 0 || q0 < 0 || q1 > P.n_tokens || nblk > P.max_blocks_per_seq ||
      kv > P.max_kv_len) {
    set_error(P.err, CB_DEVERR_BADLEN);
    return w;
  }
  if (q_len == 1) {
    const long long nb = nblk - window_first_block(kv, P.window);   // the blocks the window reaches
    w.splits = (int)((nb + P.split_blocks - 1) / P.split_blocks);
    w.dec_items = w.splits * P.n_kv_heads;
  } else if (q_len > 1) {
    if (!allow_prefill) {
      set_error(P.err, CB_DEVERR_BADLEN);
      return w;
    }
    w.pre_items = ((q_len + tok_per_tile - 1) / tok_per_tile) * P.n_kv_heads;
  }
  return w;
}

// Exclusive prefix sums over requests of decode items, decode splits and
// prefill tiles, into shared arrays of n_reqs + 1 entries (pre may be null).
// All threads of the block call it; ends with __syncthreads().
__device__ inline void build_plan(const StepParams& P, int tok_per_tile, int* dec, int* spl, int* pre, int* scratch) {
  const int n = P.n_reqs, T = blockDim.x, tid = threadIdx.x;
  const int seg = (n + T - 1) / T;
  const int lo = min(n, tid * seg), hi = min(n, lo + seg);
  const bool allow_prefill = pre != nullptr;
  int a = 0, b = 0, c = 0;
  for (int r = lo; r < hi; ++r) {
    const ReqWork w = request_work(P, r, tok_per_tile, allow_prefill);
    a += w.dec_items;
    b += w.splits;
    c += w.pre_items;
  }
  // inclusive scan of the per-thread sums: within warps, then across warps
  const int lane = tid & 31, wid = tid >> 5, nw = (T + 31) >> 5;
  int ia = a, ib = b, ic = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int xa = __shfl_up_sync(0xffffffffu, ia, off);
    const int xb = __shfl_up_sync(0xffffffffu, ib, off);
    const int xc = __shfl_up_sync(0xffffffffu, ic, off);
    if (lane >= off) {
      ia += xa;
      ib += xb;
      ic += xc;
    }
  }
  if (lane == 31) {
    scratch[wid] = ia;
    scratch[32 + wid] = ib;
    scratch[64 + wid] = ic;
  }
  __syncthreads();
  if (tid == 0) {
    int sa = 0, sb = 0, sc = 0;
    for (int w = 0; w < nw; ++w) {
      const int ta = scratch[w], tb = scratch[32 + w], tc = scratch[64 + w];
      scratch[w] = sa;
      scratch[32 + w] = sb;
      scratch[64 + w] = sc;
      sa += ta;
      sb += tb;
      sc += tc;
    }
    dec[n] = sa;
    spl[n] = sb;
    if (pre) pre[n] = sc;
  }
  __syncthreads();
  int ra = scratch[wid] + ia - a, rb = scratch[32 + wid] + ib - b, rc = scratch[64 + wid] + ic - c;
  for (int r = lo; r < hi; ++r) {
    const ReqWork w = request_work(P, r, tok_per_tile, allow_prefill);
    dec[r] = ra;
    spl[r] = rb;
    if (pre) pre[r] = rc;
    ra += w.dec_items;
    rb += w.splits;
    rc += w.pre_items;
  }
  __syncthreads();
}

// Largest r with prefix[r] <= item (prefix non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int find_request(const int* prefix, int n, int item) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------- decode warp
template <int A, int G, int NST>
struct alignas(1024) DecWarpSmem {
  static constexpr int kHalves = A / 64;
  static constexpr int kBoxBytes = kBlockSize * 128;                 // one 16-row x 64-col box
  static constexpr int kStageBytes = 2 * kHalves * kBoxBytes;        // K halves then V halves
  uint8_t kv[NST][2][kHalves][kBlockSize][128];
  float q[G][A];            // query rows of the group, times scale*log2 e
  float p[kBlockSize][G];   // this block's probabilities
  uint64_t full[NST];
};

// Runs one decode work item.  Returns false if a wait timed out (the warp must
// stop).  `parity` carries each stage's next mbarrier parity across items.
// QKU: unroll factor of the QK chunk loop (register pressure vs. ILP).
template <int A, int G, int NST, int QKU>
__device__ bool decode_item(const StepParams& P, const CUtensorMap* kmap, const CUtensorMap* vmap,
                            DecWarpSmem<A, G, NST>& S, uint32_t& parity, int r, int g, int split, int nsplit,
                            int split_slot0) {
  using WS = DecWarpSmem<A, G, NST>;
  constexpr int kHalves = WS::kHalves;
  constexpr int DPL = A / 32;     // output dims per lane
  constexpr int CPL = A / 16;     // 16-byte key chunks per lane in QK
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int Hq = P.n_q_heads, Hkv = P.n_kv_heads;
  const int t = __ldg(P.cu_q_lens + r);            // the request's single new token
  const int kv = __ldg(P.ctx_lens + r) + 1;
  const int nblk = (kv + kBlockSize - 1) / kBlockSize;
  const int b0 = window_first_block(kv, P.window) + split * P.split_blocks;
  const int nb = min(P.split_blocks, nblk - b0);
  const int key_lo = P.window > 0 ? kv - P.window : 0;     // first visible key (rolling window)

  // query rows of the group -> shared fp32, pre-scaled
  {
    const uint4* src = reinterpret_cast<const uint4*>(P.q + ((size_t)t * Hq + (size_t)g * G) * A);
    float* dst = &S.q[0][0];
    for (int i = lane; i < G * A / 8; i += 32) {
      const uint4 w = __ldg(src + i);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        dst[i * 8 + 2 * k] = bf16lo(ws[k]) * P.scale_log2;
        dst[i * 8 + 2 * k + 1] = bf16hi(ws[k]) * P.scale_log2;
      }
    }
  }
  // this split's physical blocks, one per lane
  int pblk = -1;
  if (lane < nb) {
    int e = __ldg(P.block_tables + (size_t)r * P.max_blocks_per_seq + b0 + lane);
    if (e < 0 || e >= P.num_blocks) {
      set_error(P.err, CB_DEVERR_BADBLOCK);
      e = -1;
    }
    pblk = e;
  }
  __syncwarp();
  const int rows_total = P.num_blocks * Hkv * kBlockSize;
  auto issue = [&](int ib, int st) {
    const int e = __shfl_sync(FULL, pblk, ib);
    if (lane == 0) {
      const int y = e >= 0 ? (e * Hkv + g) * kBlockSize : rows_total;   // beyond the extent: zero fill
      mbar_arrive_expect_tx(&S.full[st], WS::kStageBytes);
#pragma unroll
      for (int hf = 0; hf < kHalves; ++hf) tma_load_2d(&S.kv[st][0][hf][0][0], kmap, hf * 64, y, &S.full[st]);
#pragma unroll
      for (int hf = 0; hf < kHalves; ++hf) tma_load_2d(&S.kv[st][1][hf][0][0], vmap, hf * 64, y, &S.full[st]);
    }
  };
  const int npro = min(NST, nb);
  for (int i = 0; i < npro; ++i) issue(i, i);

  float m[G], lsum[G];
  uint64_t acc2[G][DPL / 2];     // unnormalised output columns (d0, d0+1), (d0+2, d0+3) as fp32 pairs
#pragma unroll
  for (int j = 0; j < G; ++j) {
    m[j] = kNegInf;
    lsum[j] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL / 2; ++k) acc2[j][k] = 0ull;
  }
  const int tq = lane & 15, hf_l = lane >> 4;
  const int d0 = lane * DPL;
  bool ok = true;
  int i = 0;
  for (; i < nb; ++i) {
    const int st = i % NST;
    if (!mbar_wait(&S.full[st], (parity >> st) & 1u)) {
      set_error(P.err, CB_DEVERR_TIMEOUT);
      ok = false;
      break;
    }
    parity ^= 1u << st;
    const int tokbase = (b0 + i) * kBlockSize;
    // ---- QK for token tq over half hf_l of head_dim: packed fp32x2 FMAs on
    // (even, odd) column pairs, two accumulators per head
    float s[G];
    {
      uint64_t part[G][2];
#pragma unroll
      for (int j = 0; j < G; ++j) part[j][0] = part[j][1] = 0ull;
#pragma unroll QKU
      for (int ci = 0; ci < CPL; ++ci) {
        const int cc = hf_l * CPL + ci;        // logical 16-byte chunk of the row
        const int half = cc >> 3, pos = cc & 7;
        const uint4 kw =
            *reinterpret_cast<const uint4*>(&S.kv[st][0][half][tq][(pos ^ (tq & 7)) << 4]);
        const uint64_t k01 = f2(bf16lo(kw.x), bf16hi(kw.x)), k23 = f2(bf16lo(kw.y), bf16hi(kw.y));
        const uint64_t k45 = f2(bf16lo(kw.z), bf16hi(kw.z)), k67 = f2(bf16lo(kw.w), bf16hi(kw.w));
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(&S.q[j][cc * 8]);
          const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(&S.q[j][cc * 8 + 4]);
          part[j][0] = ffma2(qa.x, k01, part[j][0]);
          part[j][1] = ffma2(qa.y, k23, part[j][1]);
          part[j][0] = ffma2(qb.x, k45, part[j][0]);
          part[j][1] = ffma2(qb.y, k67, part[j][1]);
        }
      }
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float a, b, c, d;
        f2split(part[j][0], a, b);
        f2split(part[j][1], c, d);
        s[j] = (a + b) + (c + d);
      }
    }
    const bool tvalid = tokbase + tq < kv && tokbase + tq >= key_lo;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      s[j] += __shfl_xor_sync(FULL, s[j], 16);
      s[j] = tvalid ? s[j] : kNegInf;
    }
    // ---- online softmax, base 2
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float mb = s[j];
      mb = fmaxf(mb, __shfl_xor_sync(FULL, mb, 1));
      mb = fmaxf(mb, __shfl_xor_sync(FULL, mb, 2));
      mb = fmaxf(mb, __shfl_xor_sync(FULL, mb, 4));
      mb = fmaxf(mb, __shfl_xor_sync(FULL, mb, 8));
      const float mn = fmaxf(m[j], mb);
      const float alpha = ex2(m[j] - mn);
      const float pj = ex2(s[j] - mn);
      lsum[j] = lsum[j] * alpha + (hf_l == 0 ? pj : 0.f);
      const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
      for (int k = 0; k < DPL / 2; ++k) acc2[j][k] = fmul2(acc2[j][k], a2);
      m[j] = mn;
      if (hf_l == 0) S.p[tq][j] = pj;
    }
    __syncwarp();
    // ---- PV: this lane's DPL dims.  Always 16 unrolled token steps (the loads
    // of all steps can be in flight together); a token past the request's last
    // key contributes exactly zero (its V is replaced by 0, its p is already 0).
    {
      const int cc = d0 >> 3, half = cc >> 3, pos = cc & 7, boff = (d0 & 7) * 2;
      const int nvalid = kv - tokbase;
#pragma unroll
      for (int tt = 0; tt < kBlockSize; ++tt) {
        const uint8_t* vrow = &S.kv[st][1][half][tt][((pos ^ (tt & 7)) << 4) + boff];
        float vf[DPL];
        if constexpr (DPL == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(vrow);
          vf[0] = bf16lo(w.x);
          vf[1] = bf16hi(w.x);
          vf[2] = bf16lo(w.y);
          vf[3] = bf16hi(w.y);
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow);
          vf[0] = bf16lo(w);
          vf[1] = bf16hi(w);
        }
        if (tt >= nvalid) {
#pragma unroll
          for (int k = 0; k < DPL; ++k) vf[k] = 0.f;
        }
        float pj[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int j = 0; j < G; j += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(&S.p[tt][j]);
            pj[j] = p4.x;
            pj[j + 1] = p4.y;
            pj[j + 2] = p4.z;
            pj[j + 3] = p4.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < G; ++j) pj[j] = S.p[tt][j];
        }
        const uint64_t v01 = f2(vf[0], vf[1]);
        uint64_t v23 = 0ull;
        if constexpr (DPL == 4) v23 = f2(vf[2], vf[3]);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const uint64_t pp = f2(pj[j], pj[j]);
          acc2[j][0] = ffma2(pp, v01, acc2[j][0]);
          if constexpr (DPL == 4) acc2[j][1] = ffma2(pp, v23, acc2[j][1]);
        }
      }
    }
    __syncwarp();
    if (i + NST < nb) issue(i + NST, st);
  }
  if (!ok) {
    // drain this item's copies still in flight (short bound), then stop
    for (int k = i; k < min(i + NST, nb); ++k) {
      const int st = k % NST;
      mbar_wait(&S.full[st], (parity >> st) & 1u, 20000000ull);
      parity ^= 1u << st;
    }
    return false;
  }

  // ---- totals and output
  float acc[G][DPL];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int k = 0; k < DPL / 2; ++k) f2split(acc2[j][k], acc[j][2 * k], acc[j][2 * k + 1]);
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float l = lsum[j];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(FULL, l, off);
    lsum[j] = l;
  }
  if (nsplit == 1) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float inv = 1.f / lsum[j];
      uint16_t* o = P.out + ((size_t)t * Hq + (size_t)g * G + j) * A + d0;
      if constexpr (DPL == 4) {
        uint2 w;
        w.x = pack_bf16(acc[j][0] * inv, acc[j][1] * inv);
        w.y = pack_bf16(acc[j][2] * inv, acc[j][3] * inv);
        *reinterpret_cast<uint2*>(o) = w;
      } else {
        *reinterpret_cast<uint32_t*>(o) = pack_bf16(acc[j][0] * inv, acc[j][1] * inv);
      }
    }
    return true;
  }
  const int slot = split_slot0 + split;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const size_t base = (size_t)slot * Hq + (size_t)g * G + j;
    float* pa = P.part_acc + base * A + d0;
#pragma unroll
    for (int k = 0; k < DPL; ++k) pa[k] = acc[j][k];
    if (lane == 0) {
      P.part_ml[base * 2] = m[j];
      P.part_ml[base * 2 + 1] = lsum[j];
    }
  }
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(P.counters + (size_t)r * Hkv + g, 1) == nsplit - 1;
  last = __shfl_sync(FULL, last, 0);
  if (!last) return true;
  __threadfence();
  // merge the splits of (r, g): o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
#pragma unroll 1
  for (int j = 0; j < G; ++j) {
    const size_t h = (size_t)g * G + j;
    float M = kNegInf;
    for (int s2 = lane; s2 < nsplit; s2 += 32) M = fmaxf(M, __ldcg(P.part_ml + ((size_t)(split_slot0 + s2) * Hq + h) * 2));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
    float o[DPL], L = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[k] = 0.f;
#pragma unroll 1
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const size_t base = (size_t)(split_slot0 + s2) * Hq + h;
      const float w = ex2(__ldcg(P.part_ml + base * 2) - M);
      L += w * __ldcg(P.part_ml + base * 2 + 1);
      const float* pa = P.part_acc + base * A + d0;
#pragma unroll
      for (int k = 0; k < DPL; ++k) o[k] += w * __ldcg(pa + k);
    }
    const float inv = 1.f / L;
    uint16_t* out = P.out + ((size_t)t * Hq + h) * A + d0;
    if constexpr (DPL == 4) {
      uint2 w;
      w.x = pack_bf16(o[0] * inv, o[1] * inv);
      w.y = pack_bf16(o[2] * inv, o[3] * inv);
      *reinterpret_cast<uint2*>(out) = w;
    } else {
      *reinterpret_cast<uint32_t*>(out) = pack_bf16(o[0] * inv, o[1] * inv);
    }
  }
  if (lane == 0) P.counters[(size_t)r * Hkv + g] = 0;
  return true;
}

// Pull decode items from the global queue until none is left.  `dec` and
// `spl` are the plan's prefix arrays.
template <int A, int G, int NST, int QKU = A / 16>
__device__ void decode_worker(const StepParams& P, const CUtensorMap* kmap, const CUtensorMap* vmap,
                              DecWarpSmem<A, G, NST>& S, const int* dec, const int* spl) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int total = dec[P.n_reqs];
  uint32_t parity = 0;
  while (true) {
    int item = 0;
    if (lane == 0) item = atomicAdd(P.queue, 1);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (item >= total) break;
    const int r = find_request(dec, P.n_reqs, item);
    const int nsplit = spl[r + 1] - spl[r];
    const int rem = item - dec[r];
    const int split = rem / P.n_kv_heads, g = rem - split * P.n_kv_heads;
    if (!decode_item<A, G, NST, QKU>(P, kmap, vmap, S, parity, r, g, split, nsplit, spl[r])) break;
  }
}

}  // namespace cb
