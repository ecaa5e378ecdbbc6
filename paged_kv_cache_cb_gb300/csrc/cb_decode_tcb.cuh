// The block-tile decode pipeline (head_dim 128; 8 KV heads, or MQA / GQA with
// 1 or 2 KV heads and 32 query heads), shared by the decode kernel
// (cb_decode_tcb.cu) and the decode phase of the mixed kernel (cb_mixed.cu).
//
// [CB] KV cache: each request's new token attends over all its stored keys;
// [KVN] MQA/GQA: query head h reads KV head h / G.  In the cache layout
// [block][KV head][16 tokens][128], one block of all HKV KV heads is 16 * HKV
// contiguous rows, so a 128-row tile is BPT = 8 / HKV consecutive blocks of the
// request's table: one block of 8 heads, or 8 blocks of the single MQA head.
// Each block is fetched as two 16*HKV-row x 64-column TMA boxes; a tile is
// exactly an M = 128 MMA operand.  Row i of a tile is (block i / (16 HKV) of
// the tile, KV head (i / 16) % HKV, token i % 16).
//     S[rows, q heads]   = K_tile . q^T                 (M=128, N=Hq, K=128 dims)
//     O^T[dims, q heads] += V_tile^T . P^T              (M=128, N=Hq, K=128 rows)
// P[h, row] is non-zero only where row's KV head is h/G (the GQA head mapping
// written as a block-structured matrix): the zeros are written once and the
// softmax threads rewrite only the entries of their rows' heads.  With 8 KV
// heads each head's rows of a tile are the 16 rows of one half-warp; with 1 or
// 2 KV heads a head's rows span all four softmax warps, so its tile maximum
// and its row sums are reduced across the warps (a transpose-reduce inside each
// warp leaves lane l with q head l, then shared memory).
//
// Work: the decode requests' blocks, laid end to end in request order and cut
// into equal chunks of W blocks (whole tiles, up to 32 tiles' worth, chosen to
// fill the grid in the fewest rounds, at most three with 8 KV heads and four
// otherwise); one CTA (12 warps) per SM, persistent, takes
// chunks from a global counter (the decode kernel's CTA b starts with chunk b).  A chunk is one or more segments (request r, blocks [b0, b0+nb));
// a request cut into several segments leaves split partials, merged by the
// whole grid once every chunk is done.  Equal chunks keep the CTAs' finishing
// times together.  The chunk boundaries depend only on the step's lengths, so
// results are bitwise reproducible.
//   warps 0-3  thread = tile row (scores for its G query heads) and = output
//              dimension (O).  Per tile: max over the 16 tokens of a KV head by
//              half-warp shuffles, base-2 running max with lazy rescale
//              (> 2^8; the factors reach the O threads through shared memory),
//              P to shared memory, per-thread partial sums; at a segment's
//              end, its row sums and maxima go to the epilogue warps.
//   warp 4     K producer: claims chunks, publishes segments, loads the
//              request's Hq query rows (one TMA box) and streams K tiles.
//   warp 6     V producer: streams the published segments' V tiles, so a full
//              V ring never holds up K loads (and the reverse).
//   warp 5     S issuer (one lane), event driven: S(n) once K(n) lands.
//   warp 11    PV issuer (one lane): O += P(n) V(n) once P(n) and V(n) are
//              ready (two issuing threads: one thread's MMA and commit issue
//              costs had bounded one SM's decode stream near 54 GB/s).  With
//              one KV head warp 5 issues both streams from one event loop
//              and warp 11 idles.
//   warps 7-10 epilogue: per segment, read O (double-buffered in TMEM) once its
//              last PV lands and write O/l or the split partial, while the
//              softmax warps go on with the next segment.
// After the pipeline, when some request was cut into splits, a grid-wide
// barrier and a merge phase in which the grid merges (request, head) pairs of
// those requests (a warp per pair, or a CTA per pair when pairs are fewer than
// CTAs).  A launch given the step's new K/V rows stores them first (every
// thread of the grid a share) and meets at a grid-wide counter before any
// cache read.
// Every wait is bounded; the softmax warps take every stop decision at a
// barrier that reduces it over all four warps, so none is left at a barrier.
#pragma once
#include "cb_decode_item.cuh"

namespace cb {
namespace tcb {

constexpr int kThreads = 384;
constexpr int kMergeTid0 = 224;   // epilogue warps 7-10
// most rounds of chunks per CTA: with 8 KV heads 3 measured ~1 % faster than 4
// on the mixed step, the 48-decode step and the trace (fewer splits to merge),
// with 1 KV head 4 stayed ~1 % faster; 2 and 6 were slower
template <int HKV>
constexpr int kChunksPerCta = HKV == 8 ? 3 : 4;
// blocks per CTA per round before a step takes another round: small steps make
// one round of longer chunks (fewer splits to merge); the 256-request trace
// measured 8: 1.449, 12: 1.429, 16: 1.426, 24: 1.416, 32: 1.408, 48: 1.443 ms
// per iteration (same box), the steps of 48 and more decodes unchanged up to 32
constexpr int kRoundBlocks = 24;
constexpr int kMinChunk = 4;       // blocks

// Shapes: HKV KV heads (8, 2 or 1), G query heads per KV head; Hq = HKV * G.
template <int G, int HKV = 8>
struct Cfg {
  static_assert(HKV == 8 || HKV == 2 || HKV == 1, "KV heads");
  static_assert(HKV == 8 || HKV * G == 32, "with fewer than 8 KV heads: 32 query heads");
  static constexpr int Hq = HKV * G;
  static constexpr int BPT = 8 / HKV;                 // physical blocks per 128-row tile
  static constexpr int KS = Hq == 64 ? 2 : 3;         // K ring stages (32 KB each)
  static constexpr int VS = 2;                        // V ring stages
  static constexpr int TM = Hq <= 16 ? 128 : Hq <= 32 ? 256 : 512;   // TMEM columns: S x3, O x2, Hq each
  static constexpr int MaxW = 32 * BPT;               // most blocks in a chunk (32 tiles' worth of table entries / lanes)
};

template <int G, int HKV = 8>
struct Tiles {
  static constexpr int Hq = Cfg<G, HKV>::Hq;
  uint8_t k[Cfg<G, HKV>::KS][2][128][128];   // [stage][dim half][row][128 B]
  uint8_t v[Cfg<G, HKV>::VS][2][128][128];
  uint8_t q[2][2][Hq][128];            // [buffer][dim half][q head][128 B]
  uint8_t p[2][2][Hq][128];            // [buffer][row half][q head][128 B]: K-major B of O^T += V^T P^T
};

// One segment: request r (query token t, kv keys), split `split` of nsplit
// (partials at slot0 + split), blocks [b0, b0 + nb) of its table, in nt tiles
// of BPT blocks (the last one possibly partial).
struct BItem {
  int r, split, nsplit, slot0, t, kv, b0, nb, nt;
};

// 16-byte aligned (its size too), so that xr's float4 reads are aligned
// wherever a kernel places it after another 16-byte aligned region.
template <int G, int HKV = 8>
struct alignas(16) Ctl {
  static constexpr int Hq = Cfg<G, HKV>::Hq;
  uint64_t item_full[2], item_empty[2], q_full[2], q_empty[2];
  uint64_t k_full[Cfg<G, HKV>::KS], k_empty[Cfg<G, HKV>::KS], v_full[Cfg<G, HKV>::VS];
  uint64_t s_full[3], p_full[2], o_done[2], drain, drain2;
  BItem item[2];               // the segment published in each slot (r < 0: no more work)
  int rows[2][Cfg<G, HKV>::MaxW];   // its blocks' first cache rows
  struct {
    int cu, ctx, pad[2];
    int bt[Cfg<G, HKV>::MaxW];
  } raw[2];                    // an item's metadata as copied from global memory
  float alpha[2][Hq];          // per-tile rescale factors of O, per q head
  alignas(16) float xr[4][32];   // fewer than 8 KV heads: per-warp maxima / sums, lane = q head (float4 reads)
  struct {
    BItem I;                   // r < 0: no more segments
    uint32_t last_pv;
    float lsum[Hq], mmax[Hq];  // row sums / maxima per q head
  } ep[2];                     // finished segments handed to the epilogue warps
  uint64_t ep_full[2], ep_empty[2], o_full[2], o_free[2];
  int merge_ok;                // every CTA reached the merge barrier in time
  int split_any;               // some request is cut into several splits (merge phase needed)
  int W, NC, total;             // chunk size (blocks), number of chunks, blocks in all
  int pv_issued;               // PV MMAs issued so far (the PV issuer writes, the S issuer reads)
  uint32_t tmem_base;
  volatile int abort;
  int scratch[96];
  int merge_ready;             // the current merge task's splits are all written (CTA-wide tasks)
  int per_request;             // splits are counted per request and each merge waits for its own (no grid barrier)
};

// Single-thread bounded wait: on time-out records the error and raises abort.
template <class C>
__device__ __forceinline__ bool lwait(const StepParams& P, C& c, uint64_t* bar, uint32_t parity) {
  if (mbar_wait(bar, parity)) return true;
  set_error(P.err, CB_DEVERR_TIMEOUT);
  c.abort = 1;
  return false;
}
// Warp-wide bounded wait (result uniform over the warp).
template <class C>
__device__ __forceinline__ bool wwait(const StepParams& P, C& c, uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  if (!ok) {
    set_error(P.err, CB_DEVERR_TIMEOUT);
    c.abort = 1;
  }
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- plan (all threads)
// Blocks of decode request r: 0 for a request with no new token and, when
// prefill requests are allowed, for one with several; metadata that cannot be
// right gives 0 and CB_DEVERR_BADLEN.
__device__ __forceinline__ int decode_blocks(const StepParams& P, int r, bool allow_prefill) {
  const int q0 = __ldg(P.cu_q_lens + r), q1 = __ldg(P.cu_q_lens + r + 1);
  const int ctx = __ldg(P.ctx_lens + r);
  const long long kv = (long long)ctx + 1, nblk = (kv + kBlockSize - 1) / kBlockSize;
  if (q0 >= 0 && q1 <= P.n_tokens && (q1 - q0 == 0 || (allow_prefill && q1 - q0 > 1))) return 0;
  if (q1 - q0 != 1 || ctx < 0 || q0 < 0 || q1 > P.n_tokens || nblk > P.max_blocks_per_seq || kv > P.max_kv_len) {
    set_error(P.err, CB_DEVERR_BADLEN);
    return 0;
  }
  return (int)nblk - window_first_block(kv, P.window);   // the blocks its rolling window reaches
}

// Exclusive prefix sum of a[0..n) in place, a[n] = total (returned).  All
// threads of the block call it; scratch holds >= 33 ints.
__device__ inline int block_scan_excl(int* a, int n, int* scratch) {
  const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = (T + 31) >> 5;
  const int seg = (n + T - 1) / T, lo = min(n, tid * seg), hi = min(n, lo + seg);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += a[i];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) scratch[wid] = incl;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const int v = scratch[w];
      scratch[w] = run;
      run += v;
    }
    scratch[32] = run;
    a[n] = run;
  }
  __syncthreads();
  int run = scratch[wid] + incl - local;
  for (int i = lo; i < hi; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  const int total = scratch[32];
  __syncthreads();
  return total;
}

// Inclusive prefix sum over a warp's lanes.
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += u;
  }
  return v;
}

// Given bpre[r] = decode blocks of request r (r < n), makes bpre the exclusive
// prefix of blocks, picks the chunk size W and makes slot the prefix of splits
// (a request spanning chunks f..l has l - f + 1).  W fills the grid in the
// fewest rounds: R = ceil(total / (kRoundBlocks * grid)) rounds, at most
// kChunksPerCta (more rounds balance larger steps dynamically), then
// W = ceil(total / (R * grid)) in [kMinChunk, 32], raised if the partial
// buffers could not hold the splits (n + chunks).  Each thread owns a run of
// consecutive requests; both prefix sums are warp scans whose warp totals
// every thread adds up itself, so the plan costs three barriers.  All threads
// call it (a whole number of warps, at most 32); every CTA computes the same
// plan.  Ends with __syncthreads().
template <int G, int HKV>
__device__ void finish_plan(const StepParams& P, Ctl<G, HKV>& C, int* bpre, int* slot) {
  const int n = P.n_reqs, tid = threadIdx.x, T = blockDim.x, lane = tid & 31, wid = tid >> 5, nw = T >> 5;
  const int seg = (n + T - 1) / T, lo = min(n, tid * seg), hi = min(n, lo + seg);
  int own = 0;                     // this thread's blocks
  for (int i = lo; i < hi; ++i) own += bpre[i];
  const int incl = warp_incl_scan(own);
  if (lane == 31) C.scratch[wid] = incl;
  __syncthreads();
  int total = 0, run = incl - own;
  for (int w = 0; w < nw; ++w) {
    const int v = C.scratch[w];
    total += v;
    run += w < wid ? v : 0;
  }
  constexpr int BPT = Cfg<G, HKV>::BPT;
  const int grid = gridDim.x;
  // a round is kRoundBlocks 8-head blocks' worth of K/V per CTA: BPT blocks of fewer heads each
  const int rg = kRoundBlocks * BPT * grid;
  const int R = max(1, min(kChunksPerCta<HKV>, (total + rg - 1) / rg));
  int want = (total + R * grid - 1) / (R * grid);
  const int cap = max(1, P.max_splits_total - n);   // chunks the partial buffers can take
  want = max(want, (total + cap - 1) / cap);
  want = (want + BPT - 1) / BPT * BPT;           // whole tiles
  const int W = max(kMinChunk, min(Cfg<G, HKV>::MaxW, want));
  int splits_own = 0, many = 0;
  for (int i = lo; i < hi; ++i) {
    const int blk = bpre[i];
    const int sp = blk > 0 ? (run + blk - 1) / W - run / W + 1 : 0;
    bpre[i] = run;
    slot[i] = sp;
    splits_own += sp;
    many |= sp > 1;
    run += blk;
  }
  const int sincl = warp_incl_scan(splits_own);
  if (lane == 31) C.scratch[32 + wid] = sincl;
  many = __syncthreads_or(many);
  int splits = 0, srun = sincl - splits_own;
  for (int w = 0; w < nw; ++w) {
    const int v = C.scratch[32 + w];
    splits += v;
    srun += w < wid ? v : 0;
  }
  for (int i = lo; i < hi; ++i) {
    const int sp = slot[i];
    slot[i] = srun;
    srun += sp;
  }
  if (tid == 0) {
    bpre[n] = total;
    slot[n] = splits;
    if (many) C.split_any = 1;
    C.W = W;
    C.total = total;
    C.NC = (total + W - 1) / W;
    if (splits > P.max_splits_total) {   // cannot happen when the workspace is sized by the library
      set_error(P.err, CB_DEVERR_BADLEN);
      C.NC = 0;
    }
  }
  __syncthreads();
}

// Barrier set-up (one thread) and P's off-diagonal zeros (all threads; the
// caller fences and synchronises before the pipeline starts).
template <int G, int HKV>
__device__ void init_ctl(Ctl<G, HKV>& C) {
  for (int s = 0; s < 2; ++s) {
    mbar_init(&C.item_full[s], 1);
    mbar_init(&C.item_empty[s], 2 + 128 + 1);   // both MMA issuers, softmax threads, V producer
    mbar_init(&C.q_full[s], 1);
    mbar_init(&C.q_empty[s], 1);
    mbar_init(&C.p_full[s], 128);
    mbar_init(&C.o_done[s], 1);
    mbar_init(&C.ep_full[s], 128);
    mbar_init(&C.ep_empty[s], 128);
    mbar_init(&C.o_full[s], 1);
    mbar_init(&C.o_free[s], 128);
  }
  for (int s = 0; s < Cfg<G, HKV>::KS; ++s) {
    mbar_init(&C.k_full[s], 1);
    mbar_init(&C.k_empty[s], 1);
  }
  for (int s = 0; s < Cfg<G, HKV>::VS; ++s) {
    mbar_init(&C.v_full[s], 1);
  }
  for (int s = 0; s < 3; ++s) mbar_init(&C.s_full[s], 1);
  mbar_init(&C.drain, 1);
  mbar_init(&C.drain2, 1);
  C.pv_issued = 0;
  C.abort = 0;
  C.split_any = 0;
}
template <int G, int HKV>
__device__ void zero_p(Tiles<G, HKV>& T) {
  for (int i = threadIdx.x; i < (int)sizeof(T.p) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(&T.p[0][0][0][0])[i] = make_uint4(0, 0, 0, 0);
}

// v[k] for a k that is the same in every lane (a select chain: an indexed
// register array would live in local memory).
template <int N>
__device__ __forceinline__ int pick(const int (&v)[N], int k) {
  int r = v[0];
#pragma unroll
  for (int i = 1; i < N; ++i) r = k == i ? v[i] : r;
  return r;
}

// ---------------------------------------------------------------- K producer (warp 4)
// Walks the segments of the chunks it claims.  The next segment's request
// lengths and block-table entries are copied into shared memory (cp.async) a
// tile or two before the current segment's last tile is issued, and the next
// chunk is claimed (an atomic) a few tiles before that, so neither round trip
// stalls the stream; claiming no earlier keeps the dynamic balance.
template <int G, int HKV>
__device__ void b_producer(const StepParams& P, const CUtensorMap* kmap, const CUtensorMap* qmap, Tiles<G, HKV>& T,
                           Ctl<G, HKV>& C, const int* bpre, const int* slot, bool static_first) {
  constexpr int Hq = Cfg<G, HKV>::Hq, KS = Cfg<G, HKV>::KS, BPT = Cfg<G, HKV>::BPT;
  constexpr uint32_t kTileBytes = 2 * 128 * 128;
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int n = P.n_reqs, W = C.W, NC = C.NC, total = C.total;
  const int rows_total = P.num_blocks * HKV * kBlockSize;
  auto find_pos = [&](int x) {     // the request whose blocks hold linear block x
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (bpre[mid] <= x)
        lo = mid;
      else
        hi = mid - 1;
    }
    return lo;
  };
  auto fetch = [&](int i, int x, int buf) {
    const int r = i;
    int b0 = x - bpre[i];          // the request's blocks start at its window's first block
    if (P.window > 0) b0 += window_first_block((long long)__ldg(P.ctx_lens + r) + 1, P.window);
    if (lane == 0) {
      cp_async4(&C.raw[buf].cu, P.cu_q_lens + r);
      cp_async4(&C.raw[buf].ctx, P.ctx_lens + r);
    }
    for (int b = lane; b < W && b0 + b < P.max_blocks_per_seq; b += 32)
      cp_async4(&C.raw[buf].bt[b], P.block_tables + (size_t)r * P.max_blocks_per_seq + b0 + b);
    cp_async_commit();
  };
  // With static_first, CTA b starts on chunk b and the counter hands out the
  // chunks from gridDim.x on (no atomic round trip before the first load).
  const int claim0 = static_first ? (int)gridDim.x : 0;
  auto claim = [&]() {
    int v = 0;
    if (lane == 0) v = claim0 + atomicAdd(P.queue, 1);
    return v;                      // valid in lane 0
  };
  // segment cursor: chunk c (-1: none left), next linear block x, chunk end, request i
  int c = static_first ? (int)blockIdx.x : __shfl_sync(FULL, claim(), 0), x = 0, end = 0, i = 0;
  if (c >= NC) c = -1;
  if (c >= 0) {
    x = c * W;
    end = min(x + W, total);
    i = find_pos(x);
    fetch(i, x, 0);
  }
  uint32_t it = 0, kt = 0, qt = 0;   // segments, K and q tiles issued
  bool ok = true;
  while (ok) {
    const int sl = it & 1;
    BItem I;
    I.r = -1;
    // this segment's physical blocks as cache rows: block lane + 32 k in yv[k]
    // (past the segment or the cache: beyond the extent, which TMA fills with zeros)
    int yv[BPT];
#pragma unroll
    for (int k = 0; k < BPT; ++k) yv[k] = rows_total;
    int seg_end = 0;
    if (c >= 0) {
      cp_async_wait_all();
      __syncwarp();
      seg_end = min(end, bpre[i + 1]);
      I.r = i;
      I.b0 = x - bpre[i] + window_first_block((long long)C.raw[sl].ctx + 1, P.window);
      I.nb = seg_end - x;
      I.nt = (I.nb + BPT - 1) / BPT;
      I.split = c - bpre[i] / W;
      I.nsplit = slot[i + 1] - slot[i];
      I.slot0 = slot[i];
      I.t = C.raw[sl].cu;
      I.kv = C.raw[sl].ctx + 1;
#pragma unroll
      for (int k = 0; k < BPT; ++k) {
        if (lane + 32 * k < I.nb) {
          const int e = C.raw[sl].bt[lane + 32 * k];
          if (e >= 0 && e < P.num_blocks)
            yv[k] = e * HKV * kBlockSize;
          else
            set_error(P.err, CB_DEVERR_BADBLOCK);   // rows past the cache read as zeros
        }
      }
      __syncwarp();                // raw[sl] is refilled two segments from now
    }
    int good = 1;
    if (lane == 0) {
      good = lwait(P, C, &C.item_empty[sl], ((it >> 1) & 1) ^ 1);
    }
    good = __shfl_sync(FULL, good, 0);
    if (good) {
#pragma unroll
      for (int k = 0; k < BPT; ++k) C.rows[sl][lane + 32 * k] = yv[k];
    }
    __syncwarp();
    if (lane == 0) {
      if (good) {
        C.item[sl] = I;
        mbar_arrive(&C.item_full[sl]);
      }
      if (good && I.r >= 0) good = lwait(P, C, &C.q_empty[sl], ((it >> 1) & 1) ^ 1);
      if (good && I.r >= 0) {
        mbar_arrive_expect_tx(&C.q_full[sl], 2 * Hq * 128);
        tma_load_3d(&T.q[sl][0][0][0], qmap, 0, 0, I.t, &C.q_full[sl]);
        tma_load_3d(&T.q[sl][1][0][0], qmap, 64, 0, I.t, &C.q_full[sl]);
        ++qt;
      }
    }
    if (!__shfl_sync(FULL, good, 0)) {
      ok = false;
      break;
    }
    if (I.r < 0) break;
    // the next segment: the rest of this chunk, else the first of a new chunk
    const bool chunk_done = seg_end >= end;
    const int claim_at = chunk_done ? max(0, I.nt - 4) : -1, fetch_at = max(0, I.nt - 2);
    // (requests with no decode token have no blocks and are skipped)
    int nc = c, nx = seg_end, ni = seg_end < end ? find_pos(seg_end) : i, nend = end, nraw = 0;
    for (int j = 0; j < I.nt && ok; ++j) {
      if (j == claim_at) nraw = claim();
      if (j == fetch_at) {
        if (chunk_done) {
          nc = __shfl_sync(FULL, nraw, 0);
          if (nc >= NC) nc = -1;
          if (nc >= 0) {
            nx = nc * W;
            nend = min(nx + W, total);
            ni = find_pos(nx);
          }
        }
        if (nc >= 0) fetch(ni, nx, sl ^ 1);
      }
      // tile j: blocks j*BPT .. j*BPT + BPT - 1 of the segment; lane L < 2 BPT
      // loads half L % 2 of block L / 2 (all in one 32-block group of yv)
      const int blk = j * BPT + ((lane >> 1) & (BPT - 1));
      const int yb = __shfl_sync(FULL, pick<BPT>(yv, (j * BPT) >> 5), blk & 31);
      const int ks = kt % KS;
      if (lane == 0) {
        // the stage is free once S of the tile that used it has completed
        good = lwait(P, C, KS == 3 ? &C.s_full[ks] : &C.k_empty[ks], ((kt / KS) & 1) ^ 1);
        if (good) mbar_arrive_expect_tx(&C.k_full[ks], kTileBytes);
      }
      ok = __shfl_sync(FULL, good, 0);
      if (ok && lane < 2 * BPT)
        tma_load_2d(&T.k[ks][lane & 1][(lane >> 1) * 16 * HKV][0], kmap, (lane & 1) * 64, yb, &C.k_full[ks]);
      if (ok) ++kt;
    }
    c = nc;
    x = nx;
    i = ni;
    end = nend;
    ++it;
  }
  cp_async_wait_all();             // a metadata copy still in flight lands before the CTA exits
  if (lane == 0 && !ok) {
    // let the tile copies already issued land before the CTA exits: at most the
    // last KS K tiles and two q tiles can still be in flight
    for (uint32_t k = kt > (uint32_t)KS ? kt - KS : 0; k < kt; ++k)
      mbar_wait(&C.k_full[k % KS], (k / KS) & 1, 20000000ull);
    for (uint32_t k = qt > 2u ? qt - 2 : 0; k < qt; ++k) mbar_wait(&C.q_full[k & 1], (k >> 1) & 1, 20000000ull);
  }
}

// ---------------------------------------------------------------- V producer (warp 6)
template <int G, int HKV>
__device__ void v_producer(const StepParams& P, const CUtensorMap* vmap, Tiles<G, HKV>& T, Ctl<G, HKV>& C) {
  constexpr int VS = Cfg<G, HKV>::VS, BPT = Cfg<G, HKV>::BPT;
  constexpr uint32_t kTileBytes = 2 * 128 * 128;
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  uint32_t it = 0, vt = 0;
  bool ok = true;
  while (ok) {
    const int sl = it & 1;
    int good = 1;
    if (lane == 0) good = lwait(P, C, &C.item_full[sl], (it >> 1) & 1);
    if (!__shfl_sync(FULL, good, 0)) {
      ok = false;
      break;
    }
    const int r = C.item[sl].r, nt = C.item[sl].nt;
    int yv[BPT];
#pragma unroll
    for (int k = 0; k < BPT; ++k) yv[k] = C.rows[sl][lane + 32 * k];
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.item_empty[sl]);
    if (r < 0) break;
    for (int j = 0; j < nt && ok; ++j) {
      const int blk = j * BPT + ((lane >> 1) & (BPT - 1));
      const int yb = __shfl_sync(FULL, pick<BPT>(yv, (j * BPT) >> 5), blk & 31);
      const int vs = vt % VS;
      if (lane == 0) {
        good = lwait(P, C, &C.o_done[vs], ((vt / VS) & 1) ^ 1);   // free once PV of its tile completed
        if (good) mbar_arrive_expect_tx(&C.v_full[vs], kTileBytes);
      }
      ok = __shfl_sync(FULL, good, 0);
      if (ok && lane < 2 * BPT)
        tma_load_2d(&T.v[vs][lane & 1][(lane >> 1) * 16 * HKV][0], vmap, (lane & 1) * 64, yb, &C.v_full[vs]);
      if (ok) ++vt;
    }
    ++it;
  }
  if (lane == 0 && !ok)   // the last VS V tiles may still be in flight
    for (uint32_t k = vt > (uint32_t)VS ? vt - VS : 0; k < vt; ++k)
      mbar_wait(&C.v_full[k % VS], (k / VS) & 1, 20000000ull);
}

// ---------------------------------------------------------------- MMA issuers (warps 5 and 11, one lane each)
// Two threads in different warps issue the MMAs, so their issue costs overlap:
// the S issuer (warp 5) issues S(n) = K(n) q^T as soon as K(n) has landed and
// one of the three TMEM score buffers is free (S runs at most two tiles ahead
// of PV: S(n) waits until PV(n-3) was issued, which means the softmax has read
// S(n-3) and written P(n-3)); the PV issuer (warp 11) issues O += P(n) V(n) as
// soon as P(n) and V(n) are ready.  A late V tile then holds up only its own
// PV, not the K stream behind it.  A tcgen05.commit covers the MMAs of the
// issuing thread only, so each stream commits its own barriers: S(n) completes
// s_full[n % 3] (with three K stages it also frees K stage n % 3: the K
// producer waits on it), PV(n) completes o_done[n & 1], which also frees V
// stage n & 1 and P buffer n & 1.  None of these waits can alias a later
// phase: the next completion of the same barrier needs the waiter's own
// progress first (the next K or V load, the next P).
template <int G, int HKV>
__device__ void b_mma_s(const StepParams& P, Tiles<G, HKV>& T, Ctl<G, HKV>& C, uint32_t tmem) {
  constexpr int Hq = Cfg<G, HKV>::Hq, KS = Cfg<G, HKV>::KS;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, Hq, 0, 0);
  constexpr uint32_t kStage = (2 * 128 * 128) >> 4;              // one K/V stage, descriptor units
  constexpr uint32_t kQP = (2 * Hq * 128) >> 4;                  // one q / P buffer
  // K, q: K-major, 8-row atoms 1024 B apart
  const uint64_t kd0 = smem_desc_sw128(smem_u32(&T.k[0][0][0][0]), 16, 1024);
  const uint64_t qd0 = smem_desc_sw128(smem_u32(&T.q[0][0][0][0]), 16, 1024);
  uint32_t ns = 0;                 // tiles whose S has been issued
  int s_it = 0, s_j = 0, s_nb = -1;   // segment, tile in it, its length in tiles (-1: not read yet)
  bool ok = true;
  uint64_t idle_since = 0;
  for (;;) {
    bool progress = false;
    if (s_nb < 0 && mbar_ready(&C.item_full[s_it & 1], (s_it >> 1) & 1)) {
      const int r = C.item[s_it & 1].r, nt = C.item[s_it & 1].nt;
      mbar_arrive(&C.item_empty[s_it & 1]);
      if (r < 0) break;
      s_nb = nt;
      s_j = 0;
      progress = true;
    }
    if (s_nb > 0 && (int)ns < *(volatile int*)&C.pv_issued + 3) {
      const int sl = s_it & 1, ks = ns % KS;
      if ((s_j > 0 || mbar_ready(&C.q_full[sl], (s_it >> 1) & 1)) && mbar_ready(&C.k_full[ks], (ns / KS) & 1)) {
        tc_fence_after();
        const uint32_t d = tmem + (ns % 3) * Hq;
        const uint64_t kd = kd0 + ks * kStage, qd = qd0 + sl * kQP;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offk = ((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4;
          const uint32_t offq = ((kk >> 2) * Hq * 128 + (kk & 3) * 32) >> 4;
          tc_mma_f16(d, kd + offk, qd + offq, kIdescS, kk > 0);
        }
        tc_commit(&C.s_full[ns % 3]);
        if constexpr (KS != 3) tc_commit(&C.k_empty[ks]);   // with three stages s_full frees the K stage
        ++ns;
        if (++s_j == s_nb) {
          tc_commit(&C.q_empty[sl]);   // every S of this segment issued: q is free once they complete
          ++s_it;
          s_nb = -1;
        }
        progress = true;
      }
    }
    if (progress) {
      idle_since = 0;
    } else {
      const uint64_t now = globaltimer_ns();
      if (!idle_since) {
        idle_since = now;
      } else if (now - idle_since > kWaitLimitNs || C.abort) {
        set_error(P.err, CB_DEVERR_TIMEOUT);
        ok = false;
        break;
      }
    }
  }
  if (!ok) C.abort = 1;
  tc_commit(&C.drain);          // every MMA this thread issued has completed before TMEM is freed
  mbar_wait(&C.drain, 0, 20000000ull);
}

template <int G, int HKV>
__device__ void b_mma_pv(const StepParams& P, Tiles<G, HKV>& T, Ctl<G, HKV>& C, uint32_t tmem) {
  constexpr int Hq = Cfg<G, HKV>::Hq, VS = Cfg<G, HKV>::VS;
  static_assert(VS == 2, "o_done[n & 1] frees V stage n % VS");
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, Hq, 0, 1);   // A = V^T: MN-major
  constexpr uint32_t kStage = (2 * 128 * 128) >> 4;
  constexpr uint32_t kQP = (2 * Hq * 128) >> 4;
  // V^T: MN-major, rows (the reduction index) 128 B apart in 1024 B atoms, the
  // two 64-dim halves 16 KB apart.  P: K-major.
  const uint64_t vd0 = smem_desc_sw128(smem_u32(&T.v[0][0][0][0]), 128 * 128, 1024);
  const uint64_t pd0 = smem_desc_sw128(smem_u32(&T.p[0][0][0][0]), 16, 1024);
  uint32_t np = 0;                 // tiles whose PV has been issued
  int p_it = 0, p_j = 0, p_nb = -1;   // segment, tile in it, its length in tiles
  bool ok = true;
  uint64_t idle_since = 0;
  for (;;) {
    bool progress = false;
    if (p_nb < 0 && mbar_ready(&C.item_full[p_it & 1], (p_it >> 1) & 1)) {
      const int r = C.item[p_it & 1].r, nt = C.item[p_it & 1].nt;
      mbar_arrive(&C.item_empty[p_it & 1]);
      if (r < 0) break;
      p_nb = nt;
      p_j = 0;
      progress = true;
    }
    if (p_nb > 0) {
      const int pb = np & 1, vs = np % VS;
      if (mbar_ready(&C.p_full[pb], (np >> 1) & 1) && mbar_ready(&C.v_full[vs], (np / VS) & 1) &&
          (p_j > 0 || mbar_ready(&C.o_free[p_it & 1], ((p_it >> 1) & 1) ^ 1))) {
        tc_fence_after();
        const uint64_t vd = vd0 + vs * kStage, pd = pd0 + pb * kQP;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offv = (kk * 16 * 128) >> 4;
          const uint32_t offp = ((kk >> 2) * Hq * 128 + (kk & 3) * 32) >> 4;
          tc_mma_f16(tmem + (3 + (p_it & 1)) * Hq, vd + offv, pd + offp, kIdescPV, (p_j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&C.o_done[np & 1]);   // also frees V stage np % 2 and P buffer np & 1
        ++np;
        *(volatile int*)&C.pv_issued = (int)np;   // the S issuer may reuse S buffer (np - 1) % 3
        if (++p_j == p_nb) {
          tc_commit(&C.o_full[p_it & 1]);   // the segment's O is complete once this lands
          ++p_it;
          p_nb = -1;
        }
        progress = true;
      }
    }
    if (progress) {
      idle_since = 0;
    } else {
      const uint64_t now = globaltimer_ns();
      if (!idle_since) {
        idle_since = now;
      } else if (now - idle_since > kWaitLimitNs || C.abort) {
        set_error(P.err, CB_DEVERR_TIMEOUT);
        ok = false;
        break;
      }
    }
  }
  if (!ok) C.abort = 1;
  tc_commit(&C.drain2);
  mbar_wait(&C.drain2, 0, 20000000ull);
}

// One thread issuing both streams (the S issuer's and the PV issuer's steps in
// one event loop, the same barriers and commits): used with 1 KV head (MQA),
// where a tile's 8 rows per block are 16 TMA boxes and the softmax of 32 heads
// per row, not MMA issue, bound the stream, and a second polling thread only
// takes issue slots from the softmax warps (MQA decode 292 -> 241 us measured;
// with 2 KV heads the split issuers stay 2% faster).
template <int G, int HKV>
__device__ void b_mma_both(const StepParams& P, Tiles<G, HKV>& T, Ctl<G, HKV>& C, uint32_t tmem) {
  constexpr int Hq = Cfg<G, HKV>::Hq, KS = Cfg<G, HKV>::KS, VS = Cfg<G, HKV>::VS;
  static_assert(VS == 2, "o_done[n & 1] frees V stage n % VS");
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, Hq, 0, 0);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, Hq, 0, 1);
  constexpr uint32_t kStage = (2 * 128 * 128) >> 4;
  constexpr uint32_t kQP = (2 * Hq * 128) >> 4;
  const uint64_t kd0 = smem_desc_sw128(smem_u32(&T.k[0][0][0][0]), 16, 1024);
  const uint64_t qd0 = smem_desc_sw128(smem_u32(&T.q[0][0][0][0]), 16, 1024);
  const uint64_t vd0 = smem_desc_sw128(smem_u32(&T.v[0][0][0][0]), 128 * 128, 1024);
  const uint64_t pd0 = smem_desc_sw128(smem_u32(&T.p[0][0][0][0]), 16, 1024);
  uint32_t ns = 0, np = 0;
  int s_it = 0, s_j = 0, s_nb = -1;   // S cursor: segment, tile in it, its length in tiles
  int p_it = 0, p_j = 0, p_nb = -1;   // PV cursor
  bool s_done = false, ok = true;
  uint64_t idle_since = 0;
  for (;;) {
    bool progress = false;
    if (!s_done && s_nb < 0 && mbar_ready(&C.item_full[s_it & 1], (s_it >> 1) & 1)) {
      const int r = C.item[s_it & 1].r, nt = C.item[s_it & 1].nt;
      s_done = r < 0;
      s_nb = s_done ? 0 : nt;         // the last item's nt is not set
      s_j = 0;
      progress = true;
    }
    if (s_nb > 0 && !s_done && ns < np + 3) {
      const int sl = s_it & 1, ks = ns % KS;
      if ((s_j > 0 || mbar_ready(&C.q_full[sl], (s_it >> 1) & 1)) && mbar_ready(&C.k_full[ks], (ns / KS) & 1)) {
        tc_fence_after();
        const uint32_t d = tmem + (ns % 3) * Hq;
        const uint64_t kd = kd0 + ks * kStage, qd = qd0 + sl * kQP;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offk = ((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4;
          const uint32_t offq = ((kk >> 2) * Hq * 128 + (kk & 3) * 32) >> 4;
          tc_mma_f16(d, kd + offk, qd + offq, kIdescS, kk > 0);
        }
        tc_commit(&C.s_full[ns % 3]);
        if constexpr (KS != 3) tc_commit(&C.k_empty[ks]);
        ++ns;
        if (++s_j == s_nb) {
          tc_commit(&C.q_empty[sl]);
          ++s_it;
          s_nb = -1;
        }
        progress = true;
      }
    }
    // the PV cursor reads each segment's item after the S cursor: both arrive on item_empty
    if (p_nb < 0 && p_it < s_it + (s_nb >= 0 ? 1 : 0)) {
      const int r = C.item[p_it & 1].r, nt = C.item[p_it & 1].nt;
      mbar_arrive(&C.item_empty[p_it & 1]);
      mbar_arrive(&C.item_empty[p_it & 1]);   // both issuer arrivals (this thread stands for the two)
      p_nb = r < 0 ? -2 : nt;                 // -2: no more segments
      p_j = 0;
      progress = true;
    }
    if (p_nb > 0 && np < ns) {
      const int pb = np & 1, vs = np % VS;
      if (mbar_ready(&C.p_full[pb], (np >> 1) & 1) && mbar_ready(&C.v_full[vs], (np / VS) & 1) &&
          (p_j > 0 || mbar_ready(&C.o_free[p_it & 1], ((p_it >> 1) & 1) ^ 1))) {
        tc_fence_after();
        const uint64_t vd = vd0 + vs * kStage, pd = pd0 + pb * kQP;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offv = (kk * 16 * 128) >> 4;
          const uint32_t offp = ((kk >> 2) * Hq * 128 + (kk & 3) * 32) >> 4;
          tc_mma_f16(tmem + (3 + (p_it & 1)) * Hq, vd + offv, pd + offp, kIdescPV, (p_j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&C.o_done[np & 1]);
        ++np;
        if (++p_j == p_nb) {
          tc_commit(&C.o_full[p_it & 1]);
          ++p_it;
          p_nb = -1;
        }
        progress = true;
      }
    }
    if (s_done && p_nb == -2) break;
    if (progress) {
      idle_since = 0;
    } else {
      const uint64_t now = globaltimer_ns();
      if (!idle_since) {
        idle_since = now;
      } else if (now - idle_since > kWaitLimitNs || C.abort) {
        set_error(P.err, CB_DEVERR_TIMEOUT);
        ok = false;
        break;
      }
    }
  }
  if (!ok) C.abort = 1;
  tc_commit(&C.drain);
  mbar_wait(&C.drain, 0, 20000000ull);
}

// n (8, 16, 32 or 64) consecutive TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float* v) {
  if constexpr (N == 8) {
    float t[8];
    tmem_ld8(taddr, t);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = t[i];
  } else if constexpr (N == 16) {
    float t[8], u[8];
    tmem_ld8(taddr, t);
    tmem_ld8(taddr + 8, u);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = t[i];
      v[8 + i] = u[i];
    }
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
      float t[32];
      tmem_ld32(taddr + c * 32, t);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[c * 32 + i] = t[i];
    }
  }
}

// Transpose-reduce over groups of N consecutive lanes (N = 16 or 32), each
// holding N values: afterwards v[0] of lane l is the maximum (MAX) or the sum
// of value l % N over the group's lanes.  At the step with offset o a lane
// keeps the half of its live values selected by bit o of its lane index and
// swaps the other half with lane ^ o: N - 1 shuffles in all.
template <int N, bool MAX>
__device__ __forceinline__ void xreduce(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = N / 2; o >= 1; o >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float keep = up ? v[i + o] : v[i];
      const float send = up ? v[i] : v[i + o];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
}

// ---------------------------------------------------------------- softmax (warps 0-3)
template <int G, int HKV>
__device__ void b_softmax(const StepParams& P, Tiles<G, HKV>& T, Ctl<G, HKV>& C, uint32_t tmem) {
  constexpr int Hq = Cfg<G, HKV>::Hq, VS = Cfg<G, HKV>::VS, BPT = Cfg<G, HKV>::BPT;
  const int tid = threadIdx.x;                 // tile row; output dimension
  const int warp = tid >> 5, lane = tid & 31;
  // tile row = (block bi of the tile, KV head g, token tok)
  const int bi = tid / (16 * HKV), g = (tid >> 4) % HKV, tok = tid & 15;
  const bool hi = (lane >> 4) & 1;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const float sl2 = P.scale_log2;
  const int h0 = g * G;                        // this row's query heads h0 .. h0+G-1
  uint32_t it = 0, sc = 0;                     // items and tiles seen
  for (;;) {
    const int slot = it & 1;
    bool good = wwait(P, C, &C.item_full[slot], (it >> 1) & 1);
    BItem I;
    I.r = -1;
    if (good) {
      I = C.item[slot];
      mbar_arrive(&C.item_empty[slot]);
    }
    if (named_bar_or(1, 128, !good || C.abort) || I.r < 0) break;
    float m[G], lp[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      m[i] = kNegInf;
      lp[i] = 0.f;
    }
    bool stop = false;
    for (int j = 0; j < I.nt; ++j, ++sc) {
      const int sb = sc & 1;
      const int bseg = j * BPT + bi;             // this row's block within the segment
      const int pos = (I.b0 + bseg) * kBlockSize + tok;
      const bool valid = bseg < I.nb && pos < I.kv && (P.window <= 0 || pos >= I.kv - P.window);
      bool need_any = false;
      const int sbuf = sc % 3;    // TMEM score buffer (sb: P buffer)
      good = wwait(P, C, &C.s_full[sbuf], (sc / 3) & 1);
      float x[G];                 // scores of this row's G query heads, times scale * log2 e
      if (good) {
        tc_fence_after();
        if constexpr (HKV == 8) {
          // this warp's two KV heads own columns [2*warp*G, 2*warp*G + 2G); each half-warp keeps its G
          float sv[2 * G];
          if constexpr (G == 2) {
            float t8[8];
            tmem_ld8(tmem + lane_base + sbuf * Hq + ((4 * warp) & ~7), t8);
            tmem_wait_ld();
            const bool upper = warp & 1;   // columns 4..7 of the 8 loaded
#pragma unroll
            for (int i = 0; i < 4; ++i) sv[i] = upper ? t8[4 + i] : t8[i];
          } else {
            tmem_ld_n<2 * G>(tmem + lane_base + sbuf * Hq + 2 * warp * G, sv);
            tmem_wait_ld();
          }
#pragma unroll
          for (int i = 0; i < G; ++i) x[i] = valid ? (hi ? sv[G + i] : sv[i]) * sl2 : kNegInf;
        } else {
          // Hq = 32 columns: the half-warps' KV heads (2 heads: columns [16 hw, 16 hw + 16); 1 head: all)
          float sv[32];
          tmem_ld_n<32>(tmem + lane_base + sbuf * Hq, sv);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < G; ++i) x[i] = valid ? (HKV == 2 && hi ? sv[G + i] : sv[i]) * sl2 : kNegInf;
        }
      } else {
#pragma unroll
        for (int i = 0; i < G; ++i) x[i] = kNegInf;
      }
      // With 1 or 2 KV heads a KV head's rows span the four warps.  The exact
      // tile maximum matters only where it would move the reference (lazy
      // rescale: more than 2^8 above it), so the cross-warp exchange runs only
      // when some row of the tile has such a score -- the first tile of a
      // segment, and rarely after; otherwise the reference stays.
      bool exch = false;
      if constexpr (HKV != 8) {
        bool grow = false;
#pragma unroll
        for (int i = 0; i < G; ++i) grow |= x[i] > m[i] + 8.f;
        exch = named_bar_or(1, 128, grow);
        if (exch) {
          float v[G];
#pragma unroll
          for (int i = 0; i < G; ++i) v[i] = x[i];
          xreduce<G, true>(v);                     // lane l: the warp's maximum of q head l
          C.xr[warp][lane] = v[0];
          named_bar(1, 128);
        }
      }
      if (good) {
        // per q head: the tile maximum over the rows of its KV head, the
        // running maximum (lazy rescale) and its factor, p (kept as packed
        // bf16 pairs until the P buffer is free) and the row sum.  The
        // factors' buffer sb was last read by these threads two tiles ago.
        uint32_t pk[(G + 1) / 2];
#pragma unroll
        for (int i0 = 0; i0 < G; i0 += (G >= 4 ? 4 : G)) {
          constexpr int U = G >= 4 ? 4 : G;
          float mxs[U];
          if constexpr (HKV == 8) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
              float mx = x[i0 + u];
#pragma unroll
              for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
              mxs[u] = mx;
            }
          } else {
            static_assert(HKV == 8 || U == 4, "four heads per step");
            if (exch) {
              const float4 a = *reinterpret_cast<const float4*>(&C.xr[0][g * G + i0]);
              const float4 b = *reinterpret_cast<const float4*>(&C.xr[1][g * G + i0]);
              const float4 cc = *reinterpret_cast<const float4*>(&C.xr[2][g * G + i0]);
              const float4 d = *reinterpret_cast<const float4*>(&C.xr[3][g * G + i0]);
              mxs[0] = fmaxf(fmaxf(a.x, b.x), fmaxf(cc.x, d.x));
              mxs[1] = fmaxf(fmaxf(a.y, b.y), fmaxf(cc.y, d.y));
              mxs[2] = fmaxf(fmaxf(a.z, b.z), fmaxf(cc.z, d.z));
              mxs[3] = fmaxf(fmaxf(a.w, b.w), fmaxf(cc.w, d.w));
            } else {
#pragma unroll
              for (int u = 0; u < U; ++u) mxs[u] = m[i0 + u];
            }
          }
          float pv[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = i0 + u;
            // every tile of a segment holds at least one valid key, so mxs is finite
            const bool need = mxs[u] > m[i] + 8.f;
            const float alpha = need ? ex2(m[i] - mxs[u]) : 1.f;
            m[i] = need ? mxs[u] : m[i];
            need_any |= need;
            pv[u] = ex2(x[i] - m[i]);
            lp[i] = lp[i] * alpha + pv[u];
            if (tok == 0) C.alpha[sb][h0 + i] = alpha;
          }
#pragma unroll
          for (int u = 0; u < U; u += 2) pk[(i0 + u) / 2] = pack_bf16(pv[u], U > 1 ? pv[u + 1] : 0.f);
        }
        // the P buffer is free once PV(sc - 2) has completed
        good = wwait(P, C, &C.o_done[sb], ((sc >> 1) & 1) ^ 1);
        if (good) {
          const int half = tid >> 6, c = tid & 63, chunk = c >> 3, within = (c & 7) * 2;
#pragma unroll
          for (int i = 0; i < G; ++i) {
            const int h = h0 + i;
            const uint16_t hv = (uint16_t)((i & 1) ? (pk[i / 2] >> 16) : (pk[i / 2] & 0xFFFFu));
            *reinterpret_cast<uint16_t*>(&T.p[sb][half][h][((chunk ^ (h & 7)) << 4) + within]) = hv;
          }
        }
      }
      if (named_bar_or(1, 128, need_any || !good || C.abort)) {
        if (named_bar_or(1, 128, !good || C.abort)) {
          stop = true;
          break;
        }
        if (j > 0) {   // rescale O once O += P(j-1) V(j-1) has landed
          const uint32_t n = sc - 1;
          if (wwait(P, C, &C.o_done[n & 1], (n >> 1) & 1)) {
            tc_fence_after();
            float o[Hq];
            tmem_ld_n<Hq>(tmem + lane_base + (3 + (it & 1)) * Hq, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < Hq / 8; ++c) {
              float t8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) t8[i] = o[c * 8 + i] * C.alpha[sb][c * 8 + i];
              tmem_st8(tmem + lane_base + (3 + (it & 1)) * Hq + c * 8, t8);
            }
            tmem_wait_st();
          }
        }
      }
      // value rows of tokens past the request's last key hold whatever the cache
      // had there: each such row's thread zeroes it (0 * non-finite must not reach O)
      if (!valid) {
        const int vs = sc % VS;
        if (mbar_wait(&C.v_full[vs], (sc / VS) & 1)) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(&T.v[vs][hf][tid][c << 4]) = make_uint4(0, 0, 0, 0);
        } else {
          set_error(P.err, CB_DEVERR_TIMEOUT);
          C.abort = 1;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&C.p_full[sb]);
    }
    if (stop) break;
    // ---- the segment's row sums and maxima per q head (16 rows of its KV head) go to
    // the epilogue warps, which read O when its last PV lands; this warp group
    // goes straight on to the next segment (its PVs use the other O buffer)
    const int e = it & 1;
    good = wwait(P, C, &C.ep_empty[e], ((it >> 1) & 1) ^ 1);
    if constexpr (HKV == 8) {
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float l = lp[i];
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (good && tok == 0) {
          C.ep[e].lsum[h0 + i] = l;
          C.ep[e].mmax[h0 + i] = m[i];
        }
      }
    } else {
      // row sums over the four warps: lane l of each warp holds q head l's share
      xreduce<G, false>(lp);
      C.xr[warp][lane] = lp[0];
      named_bar(1, 128);
      if (good && tid < 32) C.ep[e].lsum[tid] = (C.xr[0][tid] + C.xr[1][tid]) + (C.xr[2][tid] + C.xr[3][tid]);
      if (good && tok == 0) {
#pragma unroll
        for (int i = 0; i < G; ++i) C.ep[e].mmax[h0 + i] = m[i];
      }
    }
    if (good && tid == 0) {
      C.ep[e].I = I;
      C.ep[e].last_pv = sc - 1;
    }
    if (good) mbar_arrive(&C.ep_full[e]);
    if (named_bar_or(1, 128, !good || C.abort)) break;
    ++it;
  }
  // end mark for the epilogue warps
  if (wwait(P, C, &C.ep_empty[it & 1], ((it >> 1) & 1) ^ 1)) {
    if (tid == 0) C.ep[it & 1].I.r = -1;
    mbar_arrive(&C.ep_full[it & 1]);
  }
}

// ---------------------------------------------------------------- epilogue (warps 7-10)
// Per segment: wait until its last PV has landed in its O buffer, read O^T
// (thread = output dimension: TMEM lane 32 * (warp % 4) + lane), free the
// buffer, then write O/l -- or, for one split of several, the partial
// (O, m, l) for the merge phase.
template <int G, int HKV>
__device__ void b_epilogue(const StepParams& P, Ctl<G, HKV>& C, uint32_t tmem) {
  constexpr int Hq = Cfg<G, HKV>::Hq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x - kMergeTid0;
  const int d = 32 * (warp & 3) + lane;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  uint32_t k = 0;
  for (;;) {
    const int e = k & 1;
    bool good = wwait(P, C, &C.ep_full[e], (k >> 1) & 1);
    BItem I;
    I.r = -1;
    if (good) I = C.ep[e].I;
    float o[Hq];
    if (good && I.r >= 0) {
      good = wwait(P, C, &C.o_full[e], (k >> 1) & 1);
      if (good) {
        tc_fence_after();
        tmem_ld_n<Hq>(tmem + lane_base + (3 + e) * Hq, o);
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive(&C.o_free[e]);
    }
    if (named_bar_or(2, 128, !good || C.abort) || I.r < 0) break;
    if (I.nsplit == 1) {
#pragma unroll
      for (int h = 0; h < Hq; ++h)
        P.out[((size_t)I.t * Hq + h) * 128 + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o[h] / C.ep[e].lsum[h]));
    } else {
      const size_t base = (size_t)(I.slot0 + I.split) * Hq;
#pragma unroll
      for (int h = 0; h < Hq; ++h) P.part_acc[(base + h) * 128 + d] = o[h];
      if (tid < Hq) {
        P.part_ml[(base + tid) * 2] = C.ep[e].mmax[tid];
        P.part_ml[(base + tid) * 2 + 1] = C.ep[e].lsum[tid];
      }
      if constexpr (HKV == 8)
        if (C.per_request) __threadfence();   // this thread's share of the partial before the request's count
    }
    named_bar(2, 128);             // every thread is done with ep[e]
    if constexpr (HKV == 8)
      if (C.per_request && I.nsplit > 1 && tid == 0) atomicAdd(P.counters + I.r, 1);   // one more split written
    mbar_arrive(&C.ep_empty[e]);
    ++k;
  }
}

// Whether a launch merges each request as soon as its own splits are written
// instead of after a grid-wide barrier: with 8 KV heads, unless other partial
// results need the barrier (grid_sync).  With 1 or 2 KV heads the barrier
// stays (the waits' code alone cost the MQA kernel registers and 7 %).  The
// same in every CTA.
template <int G, int HKV>
__device__ __forceinline__ bool per_request_merge(const StepParams& P, bool grid_sync) {
  (void)P;
  return HKV == 8 && !grid_sync;   // compiled in only there: its registers cost the 1- and 2-head kernels
}

// ---------------------------------------------------------------- split merge (all warps of the grid)
__device__ __forceinline__ unsigned ld_acquire_gpu(const int* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------- fused KV append (all threads)
// A launch given the step's new K/V rows (Ap.n_tokens > 0) stores them before
// anything reads the cache: every thread of the grid copies its share of the
// 16-byte pieces (append_pieces), and once the CTA has built its plans it
// fences the stores and arrives on the grid-wide counter P.queue[2].  The launch is cooperative, so all CTAs are resident and the
// counter reaches gridDim.x.  The stores are made visible to the async proxy
// (the TMA loads of the producers) on both sides of the counter.  Not inlined:
// the copy loop's registers stay out of the pipeline's allocation.
static __device__ __noinline__ void append_store(const AppendParams& Ap, int64_t n_slots, int n_kv_heads,
                                                 unsigned int* err) {
  const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i0 >= (int64_t)Ap.n_tokens * n_kv_heads * 16) return;    // no piece for this thread: nothing to fence
  append_pieces(Ap.k_new, Ap.v_new, Ap.slots, Ap.n_tokens, Ap.k_cache, Ap.v_cache, n_slots, n_kv_heads, 16, err, i0,
                (int64_t)gridDim.x * blockDim.x);
  fence_proxy_async_global();
  __threadfence();
}
// With COUNT (launches whose merge may wait per request) it also zeroes its
// share of the per-request split counters P.counters[0, n_reqs) before its
// CTA arrives, and the launch meets at the counter even with no rows to store,
// so the counters are zero wherever the pipeline counts.
template <bool COUNT>
__device__ __forceinline__ void append_phase(const StepParams& P, const AppendParams& Ap) {
  if constexpr (COUNT) {
    const int g0 = blockIdx.x * blockDim.x + threadIdx.x;
    if (g0 < P.n_reqs) {
      for (int r = g0; r < P.n_reqs; r += gridDim.x * blockDim.x) P.counters[r] = 0;
      __threadfence();
    }
  } else if (Ap.n_tokens == 0) {
    return;
  }
  if (Ap.n_tokens != 0) append_store(Ap, (int64_t)P.num_blocks * kBlockSize, P.n_kv_heads, P.err);
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(P.queue + 2, 1);
}
// Bounded wait until every CTA has arrived after its append stores; a time-out
// records CB_DEVERR_TIMEOUT and goes on (the step's result is then unreliable,
// and the host is told).  All threads of the CTA call it.
template <bool COUNT>
__device__ __forceinline__ void append_wait(const StepParams& P, const AppendParams& Ap) {
  if (!COUNT && Ap.n_tokens == 0) return;
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(P.queue + 2) < gridDim.x) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        set_error(P.err, CB_DEVERR_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  fence_proxy_async_global();
}

// The launch's counters P.queue[0..3] are left at zero for the next launch on
// the stream: each CTA counts its exit in P.queue[3] once it is done with all
// of them, and the last one resets them.  All threads of the CTA call it last.
__device__ __forceinline__ void release_counters(const StepParams& P) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(P.queue + 3, 1) == (int)gridDim.x - 1) {
      P.queue[0] = 0;
      P.queue[1] = 0;
      P.queue[2] = 0;
      __threadfence();
      P.queue[3] = 0;
    }
  }
}

// After the pipeline, when some request was cut into several splits (every CTA
// made the same plan, so all take the same branch): a grid-wide barrier (the
// launch is cooperative, so every CTA is resident; the wait is bounded; the
// last CTA to arrive does not wait), then every warp of the grid merges one
// (request, q head) of the requests cut into several splits at a time, by
// log-sum-exp over the splits' partials (m: running max, l: sum, acc: O):
//   out = sum_s 2^(m_s - M) acc_s / L,  M = max_s m_s,  L = sum_s 2^(m_s - M) l_s.
// Lane = 4 output dimensions; eight splits' loads in flight.  All threads of
// the CTA call it; red: nw * 128 floats of shared memory that nothing else
// uses any more (the tile rings).
template <int G, int HKV>
__device__ void merge_phase(const StepParams& P, Ctl<G, HKV>& C, const int* slot, float* red, bool grid_sync) {
  constexpr int Hq = Cfg<G, HKV>::Hq;
  const unsigned FULL = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!C.split_any) return;        // every output was written by its only split
  const int nw = blockDim.x >> 5;
  const int n_task = P.n_reqs * Hq;
  bool per_request = false;
  if constexpr (HKV == 8) per_request = C.per_request;   // per_request_merge(P, grid_sync), set with the plan
  (void)grid_sync;
  __syncthreads();
  if (per_request) {
    if (threadIdx.x == 0) C.merge_ok = 1;
  } else if (threadIdx.x == 0) {
    C.merge_ok = 1;
    __threadfence();               // this CTA's partials before its arrival
    if (atomicAdd(P.queue + 1, 1) + 1 < gridDim.x) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(P.queue + 1) < gridDim.x) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          set_error(P.err, CB_DEVERR_TIMEOUT);
          C.merge_ok = 0;
          break;
        }
        __nanosleep(32);
      }
    } else {
      __threadfence();             // last to arrive: the others' partials are released before their arrivals
    }
  }
  __syncthreads();
  if (!C.merge_ok) return;
  // Few tasks: a CTA per (request, head), its warps sharing the splits and
  // adding their sums in shared memory (red: nw * 128 floats); else a warp per task.
  const bool cta_mode = n_task <= (int)gridDim.x;
  const int g = cta_mode ? nw : 1, sub = cta_mode ? warp : 0;
  const int task0 = cta_mode ? (int)blockIdx.x : (int)blockIdx.x * nw + warp;
  const int tstride = cta_mode ? (int)gridDim.x : (int)gridDim.x * nw;
  for (int task = task0; task < n_task; task += tstride) {
    const int i = task / Hq, h = task - i * Hq;
    const int slot0 = slot[i], ns = slot[i + 1] - slot0;
    if (ns <= 1) continue;         // the same for every warp of the task
    if (HKV == 8 && per_request) {
      // without the grid-wide barrier: wait (bounded) until every split of
      // request i has written its partial, so a request's merge overlaps the
      // other requests' streams
      int ready = 1;
      if (cta_mode ? threadIdx.x == 0 : lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while ((int)ld_acquire_gpu(P.counters + i) < ns) {
          if (globaltimer_ns() - t0 > kWaitLimitNs || C.abort) {
            set_error(P.err, CB_DEVERR_TIMEOUT);
            ready = 0;
            break;
          }
          __nanosleep(32);
        }
        if (cta_mode) C.merge_ready = ready;
      }
      if (cta_mode) {
        __syncthreads();
        ready = C.merge_ready;
        __syncthreads();           // merge_ready is read by every thread before the next task sets it
      } else {
        ready = __shfl_sync(FULL, ready, 0);
      }
      if (!ready) continue;
      (void)ld_acquire_gpu(P.counters + i);   // this thread's reads of the partials come after the count
    }
    // (m, l) of splits lane + 32k, k < 4, stay in registers; splits past 128 are re-read
    const float2* ml = reinterpret_cast<const float2*>(P.part_ml) + (size_t)slot0 * Hq + h;
    float2 v[4];
    float M = kNegInf;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int sp = lane + 32 * k;
      v[k] = sp < ns ? __ldcg(ml + (size_t)sp * Hq) : make_float2(kNegInf, 0.f);
      M = fmaxf(M, v[k].x);
    }
    for (int sp = lane + 128; sp < ns; sp += 32) M = fmaxf(M, __ldcg(ml + (size_t)sp * Hq).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
    float L = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (lane + 32 * k < ns) L += ex2(v[k].x - M) * v[k].y;
    for (int sp = lane + 128; sp < ns; sp += 32) {
      const float2 t = __ldcg(ml + (size_t)sp * Hq);
      L += ex2(t.x - M) * t.y;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(FULL, L, off);
    const float inv = 1.f / L;
    float wk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) wk[k] = lane + 32 * k < ns ? ex2(v[k].x - M) * inv : 0.f;
    // this warp's splits sub, sub + g, ...: eight loads in flight
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* src = reinterpret_cast<const float4*>(P.part_acc + ((size_t)slot0 * Hq + h) * 128) + lane;
    for (int s0 = sub; s0 < ns; s0 += 8 * g) {
      float4 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int sp = s0 + u * g;
        x[u] = sp < ns ? __ldcg(src + (size_t)sp * Hq * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int sp = s0 + u * g;   // the same in every lane
        if (sp >= ns) break;
        float w;
        if (sp < 128) {
          const int k = sp >> 5;
          w = __shfl_sync(FULL, k == 0 ? wk[0] : k == 1 ? wk[1] : k == 2 ? wk[2] : wk[3], sp & 31);
        } else {
          w = ex2(__ldcg(ml + (size_t)sp * Hq).x - M) * inv;
        }
        acc.x += w * x[u].x;
        acc.y += w * x[u].y;
        acc.z += w * x[u].z;
        acc.w += w * x[u].w;
      }
    }
    const int t = __ldg(P.cu_q_lens + i);
    uint2* dst = reinterpret_cast<uint2*>(P.out + ((size_t)t * Hq + h) * 128 + lane * 4);
    if (cta_mode) {
      float4* r4 = reinterpret_cast<float4*>(red);
      r4[warp * 32 + lane] = acc;
      __syncthreads();
      if (warp == 0) {
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < nw; ++w) {
          const float4 y = r4[w * 32 + lane];
          sum.x += y.x;
          sum.y += y.y;
          sum.z += y.z;
          sum.w += y.w;
        }
        *dst = make_uint2(pack_bf16(sum.x, sum.y), pack_bf16(sum.z, sum.w));
      }
      __syncthreads();             // red is reused by the next task
    } else {
      *dst = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
    }
  }
}

// The decode pipeline on all kThreads threads (warp roles above) over the plan
// (bpre, slot of finish_plan).  static_first: the CTAs enter together, so CTA b
// takes chunk b without the counter (the mixed launch's CTAs enter after
// prefill shares of different lengths and claim every chunk).
// TMEM columns [tmem, tmem + 5 Hq) must be allocated to the CTA.
template <int G, int HKV>
__device__ void run_pipeline(const StepParams& P, const CUtensorMap* kmap, const CUtensorMap* vmap,
                             const CUtensorMap* qmap, Tiles<G, HKV>& T, Ctl<G, HKV>& C, const int* bpre, const int* slot,
                             uint32_t tmem, bool static_first) {
  const int warp = threadIdx.x >> 5;
  if (warp == 4) {
    b_producer<G, HKV>(P, kmap, qmap, T, C, bpre, slot, static_first);
  } else if (warp == 6) {
    v_producer<G, HKV>(P, vmap, T, C);
  } else if (warp >= 7 && warp <= 10) {
    b_epilogue<G, HKV>(P, C, tmem);
  } else if (warp == 5) {
    if ((threadIdx.x & 31) == 0) {
      if constexpr (HKV != 1)
        b_mma_s<G, HKV>(P, T, C, tmem);
      else
        b_mma_both<G, HKV>(P, T, C, tmem);
    }
    __syncwarp();
  } else if (warp == 11) {
    if constexpr (HKV != 1)
      if ((threadIdx.x & 31) == 0) b_mma_pv<G, HKV>(P, T, C, tmem);
    __syncwarp();
  } else {
    b_softmax<G, HKV>(P, T, C, tmem);
  }
}

}  // namespace tcb
}  // namespace cb
