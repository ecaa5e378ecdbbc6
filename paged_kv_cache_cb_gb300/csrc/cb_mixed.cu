// One launch for a mixed continuous-batching step ([CB] Continuous batching:
// prefill chunks and decode tokens in one ragged batch).
//
// Persistent grid, one CTA per SM.  Phase 1 runs this CTA's share of the
// prefill work (requests with more than one new token, [CB] Chunked prefill) on
// the tensor cores; phase 2 serves the decode tokens from a global counter, so
// CTAs that finish their prefill share early absorb more decode work.  Phase 2
// is the block-tile pipeline of cb_decode_tcb.cuh (12 warps; whole blocks of
// every KV head per MMA tile) when head_dim is 128, there are 8 KV heads and G >= 2
// (or 32 query heads on 1 or 2 KV heads)
// (a cooperative launch, which may also store the step's new K/V rows first),
// else 8 warps of the CUDA-core decode workers (10 warps in all).  The share of
// phase 1 is whole items round robin; with fewer items than CTAs beside a long
// decode stream, whole items packed two to a CTA on half as many CTAs (the
// others stream decodes from the start, pack_items); or, on the cooperative
// launch with more items than CTAs, an equal range of the items' key tiles
// (PieceIter): items cut at CTA boundaries leave partial results that the CTA
// which ran their first tiles merges after the grid-wide barrier
// (prefill_merge).
//
// Prefill item = (request r, KV head g, pair of query tiles A and B).  A query
// tile is 128 rows = 128/G new tokens x the G query heads of group g (GQA heads
// packed into the MMA's M dimension, all sharing KV head g); tile B holds the
// next 128/G tokens.  Row i of a tile is token i/G, head g*G + i%G, at absolute
// position ctx + token; it sees keys 0..ctx+token (the chunk's causal mask
// shifted by the stored prefix).  Keys stream in tiles of 128 (8 physical
// blocks of 16, each fetched through the block table as two 2-D TMA boxes of 16
// rows x 64 columns, 128-byte swizzle, straight into the canonical K-major
// layout); both query tiles use every K and V tile.
//
// Tensor memory (512 columns): S_A|P_A [0,128), S_B|P_B [128,256), O_A, O_B.
// P (bf16) is written over the first half of its own S columns and consumed as
// the A operand of O += P V straight from tensor memory.
//
// Warp roles:  warps 0-3  softmax of tile A, warps 4-7 softmax of tile B:
//                         thread = row.  Reads S from TMEM, masks, keeps the
//                         running max m (base 2, scale folded in) and sum l,
//                         writes P, rescales O in TMEM only when the max grows
//                         by more than 2^8 (lazy rescale: exact, the final O/l
//                         uses the same reference max), finally writes O/l.
//              warp 8     TMA producer: Q pair, K tiles and V tiles into
//                         separate 2-stage rings; 16 lanes issue the boxes.
//              warp 9     MMA issuer (one lane): polls both tiles' chains
//                         S(j), PV(j), S(j+1), ... and issues whichever MMA
//                         is ready, so one tile's softmax overlaps the other
//                         tile's MMAs.
// Every wait is bounded.
#include "cb_decode_tcb.cuh"

namespace cb {

namespace {

constexpr int kSmemLimit = 232448;
constexpr int kNumThreads = 320;
constexpr int kDecWarps = 8;
constexpr int kDecStages = 2;

template <int A>
struct PrefillTiles {
  static constexpr int kHalves = A / 64;
  static constexpr int kHalfBytes = 128 * 128;                 // 128 rows x 128 bytes
  static constexpr int kTileBytes = kHalves * kHalfBytes;     // one 128-row tile of Q, K or V
  uint8_t q[2][kHalves][128][128];                             // query tiles A, B
  uint8_t k[2][kHalves][128][128];                             // key ring
  uint8_t v[2][kHalves][128][128];                             // value ring
};

constexpr int kMaxOwnItems = 2;    // whole prefill items one CTA may be dealt

struct alignas(16) MixedCtl {     // 16-byte multiple: the decode phase's control block follows it
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];        // per query tile (A, B)
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort;
  int scratch[96];
  // this CTA's prefill work (PieceIter): balanced: units [pc_u0, pc_u0 + pc_len)
  // starting at tile pc_j0 of item pc_item; else whole items from pc_item on
  int pc_balanced, pc_item, pc_j0, pc_len, pc_L;
  long long pc_u0;
  // packed (pc_nown >= 0): the whole items pc_own[0 .. pc_nown), longest first
  int pc_own[kMaxOwnItems], pc_nown;
  // the item whose first piece this CTA ran and which goes on in later CTAs
  int own_item, own_slot;
  long long own_u;
  long long scan[12];
};

// Key tiles [jlo, nkt) of the pair: jlo > 0 only under a rolling window, whose
// earliest row (position ctx + tok_lo) sees keys from ctx + tok_lo - W + 1 on.
struct PreItem {
  int r, g, q0, ctx, tok_lo, tok_hi, kv_hi, nkt, jlo;
};

__device__ __forceinline__ int first_key_tile(int ctx, int tok_lo, int window) {
  return window > 0 ? max(0, ctx + tok_lo - window + 1) / kTileN : 0;
}

// Item -> (request, KV head, token range of the tile pair).  Pairs of the same
// request are numbered from its last tokens (most keys) down.
__device__ __forceinline__ PreItem pre_item(const StepParams& P, const int* pre, int item, int tok_per_pair) {
  PreItem I;
  I.r = find_request(pre, P.n_reqs, item);
  const int rem = item - pre[I.r];
  I.q0 = __ldg(P.cu_q_lens + I.r);
  const int q_len = __ldg(P.cu_q_lens + I.r + 1) - I.q0;
  I.ctx = __ldg(P.ctx_lens + I.r);
  const int n_pairs = (q_len + tok_per_pair - 1) / tok_per_pair;
  const int pr = n_pairs - 1 - rem / P.n_kv_heads;
  I.g = rem % P.n_kv_heads;
  I.tok_lo = pr * tok_per_pair;
  I.tok_hi = min(q_len, I.tok_lo + tok_per_pair);
  I.kv_hi = I.ctx + I.tok_hi;
  I.nkt = (I.kv_hi + kTileN - 1) / kTileN;
  I.jlo = first_key_tile(I.ctx, I.tok_lo, P.window);
  return I;
}

// Key tiles of tile pair pr of a request with ctx stored and q_len new tokens.
__device__ __forceinline__ int pair_tiles(int ctx, int q_len, int pr, int tok_per_pair, int window) {
  const int tok_hi = min(q_len, (pr + 1) * tok_per_pair);
  return (ctx + tok_hi + kTileN - 1) / kTileN - first_key_tile(ctx, pr * tok_per_pair, window);
}
// Key tiles of all of request r's prefill items (every KV head).
__device__ __forceinline__ long long request_tiles(const StepParams& P, int r, int tok_per_pair) {
  const int q0 = __ldg(P.cu_q_lens + r), q_len = __ldg(P.cu_q_lens + r + 1) - q0, ctx = __ldg(P.ctx_lens + r);
  if (q_len <= 1 || ctx < 0) return 0;
  long long t = 0;
  for (int pr = 0, n = (q_len + tok_per_pair - 1) / tok_per_pair; pr < n; ++pr)
    t += pair_tiles(ctx, q_len, pr, tok_per_pair, P.window);
  return t * P.n_kv_heads;
}

// A CTA's prefill pieces (item, key tiles [j0, j1)) in order.  Round robin:
// whole items blockIdx.x, blockIdx.x + gridDim.x, ...  Packed: the whole items
// the plan dealt to this CTA.  Balanced (the cooperative launch with room for
// partial results): the concatenation of all items' key tiles, in item order,
// cut into gridDim.x equal ranges of pc_L units; the CTA's range may start and
// end inside items.
struct PieceIter {
  int item, j0, left, balanced, k, nown;
  const int* own;                  // packed (nown >= 0): the CTA's items, in shared memory
  long long u;                     // balanced: unit at which the next piece starts
  __device__ explicit PieceIter(const MixedCtl& C)
      : item(C.pc_item), j0(C.pc_j0), left(C.pc_len), balanced(C.pc_balanced), k(-1), nown(C.pc_nown),
        own(C.pc_own), u(C.pc_u0) {}
  // next piece into I, [a, b); piece number k (0 first); ustart: its first unit
  __device__ bool next(const StepParams& P, const int* pre, int n_pre, int tok_per_pair, PreItem& I, int& a, int& b,
                       long long& ustart) {
    if (!balanced && nown >= 0) {
      if (k + 1 >= nown) return false;
      item = own[k + 1];
    }
    if (item >= n_pre || (balanced && left <= 0)) return false;
    I = pre_item(P, pre, item, tok_per_pair);
    ++k;
    if (balanced) {
      a = I.jlo + j0;
      b = min(I.nkt, a + left);
      ustart = u;
      u += b - a;
      left -= b - a;
      ++item;
      j0 = 0;
    } else {
      a = I.jlo;
      b = I.nkt;
      ustart = 0;
      if (nown < 0) item += gridDim.x;
    }
    return true;
  }
};

// Measured on GB300: one key tile of a tile pair (two 128-row query tiles
// against 128 keys, S and PV) takes about 2.6 us of a CTA inside a full grid
// (the long-context chunk, 1.07 TFLOP in 1.07 ms on 152 CTAs), and the decode
// stream of a mixed step moves about 6 bytes per ns.
constexpr long long kPairTileNs = 2600;
constexpr long long kDecodeBytesPerNs = 6000;

// Fewer items than CTAs: deal them to fewer CTAs when the step's decode stream
// is long enough to hide it, so that more CTAs stream K/V from the start
// instead of waiting for their one short item.  The items, longest first
// (ties by index), go to CTAs 0 .. Np-1, then back from Np-1 to 0 (a long one
// meets a short one); Np = ceil(n_pre / k) for the largest k <= kMaxOwnItems
// (two: a third short item per CTA measured slower than none) whose
// largest CTA load, at kPairTileNs per key tile with a 30 % margin, ends
// within the decode bytes' time at kDecodeBytesPerNs.  Whole items only: no
// partial results.  work: 2 kMaxDecodeGrid + 4 ints of free shared memory.
// All threads call it; every CTA takes the same decision.  Ends with
// __syncthreads().
template <int TOK2>
__device__ void pack_items(const StepParams& P, MixedCtl& C, const int* pre, int n_pre, long long dec_bytes,
                           int* work) {
  const int T = blockDim.x, tid = threadIdx.x;
  int* len = work;                 // key tiles of item i
  int* order = work + kMaxDecodeGrid;   // items, longest first
  int* mx = work + 2 * kMaxDecodeGrid;  // largest CTA load with k = 2 .. kMaxOwnItems
  for (int i = tid; i < n_pre; i += T) {
    const PreItem I = pre_item(P, pre, i, TOK2);
    len[i] = I.nkt - I.jlo;
  }
  if (tid < kMaxOwnItems - 1) mx[tid] = 0;
  __syncthreads();
  for (int i = tid; i < n_pre; i += T) {
    const int li = len[i];
    int rank = 0;
    for (int j = 0; j < n_pre; ++j) {
      const int lj = len[j];
      rank += lj > li || (lj == li && j < i);
    }
    order[rank] = i;
  }
  __syncthreads();
  for (int k = 2; k <= kMaxOwnItems; ++k) {
    const int np = (n_pre + k - 1) / k;
    for (int c = tid; c < np; c += T) {
      int load = 0;
      for (int q = 0; q < k; ++q) {
        const int r = q * np + ((q & 1) ? np - 1 - c : c);
        if (r < n_pre) load += len[order[r]];
      }
      atomicMax(&mx[k - 2], load);
    }
  }
  __syncthreads();
  int kk = 1;
  for (int k = kMaxOwnItems; k >= 2 && kk == 1; --k)
    if ((long long)mx[k - 2] * kPairTileNs * 13 <= dec_bytes / kDecodeBytesPerNs * 10) kk = k;
  if (kk > 1 && tid == 0) {
    const int np = (n_pre + kk - 1) / kk, c = blockIdx.x;
    int no = 0;
    for (int q = 0; q < kk && c < np; ++q) {
      const int r = q * np + ((q & 1) ? np - 1 - c : c);
      if (r < n_pre) C.pc_own[no++] = order[r];
    }
    C.pc_nown = no;
  }
  __syncthreads();
}

// Plan of the balanced prefill (all threads; ends with __syncthreads()).  U =
// all items' key tiles; CTA b runs units [b L, b L + L), L = ceil(U / grid).
// Balanced only with room for the partials, more items than CTAs and L >= 4;
// otherwise round robin, or the items packed onto fewer CTAs (pack_items).
// Every CTA takes the same decision.  dec_bytes: the step's decode K/V bytes;
// work: shared memory free until the prefill starts (pack_items).
template <int TOK2>
__device__ void prefill_plan(const StepParams& P, const PrefillSplit& S, MixedCtl& C, const int* pre,
                             long long dec_bytes, int* work) {
  const int n = P.n_reqs, T = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n_pre = pre[n];
  if (tid == 0) {
    C.pc_balanced = 0;
    C.pc_item = blockIdx.x;
    C.pc_nown = -1;
    C.pc_j0 = 0;
    C.pc_len = 0;
    C.pc_L = 0;
    C.pc_u0 = 0;
    C.own_item = -1;
  }
  if (S.part == nullptr || S.slots < 2 * (int)gridDim.x || n_pre <= (int)gridDim.x) {
    __syncthreads();
    if (n_pre > 1 && n_pre <= (int)gridDim.x && (int)gridDim.x <= kMaxDecodeGrid)
      pack_items<TOK2>(P, C, pre, n_pre, dec_bytes, work);
    return;
  }
  // exclusive scan of the tiles over contiguous request segments
  const int seg = (n + T - 1) / T, lo = min(n, tid * seg), hi = min(n, lo + seg);
  long long local = 0;
  for (int r = lo; r < hi; ++r) local += request_tiles(P, r, TOK2);
  long long incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) C.scan[wid] = incl;
  __syncthreads();
  long long before = 0, U = 0;
  for (int w = 0; w < (T + 31) / 32; ++w) {
    if (w < wid) before += C.scan[w];
    U += C.scan[w];
  }
  const long long excl = before + incl - local;
  const long long L = (U + gridDim.x - 1) / gridDim.x;
  if (L >= 4 && U < (1LL << 40)) {                  // uniform: every thread of every CTA sees the same U
    const long long u0 = (long long)blockIdx.x * L;
    const long long len = max(0LL, min(U, u0 + L) - u0);
    if (tid == 0) {
      C.pc_balanced = 1;
      C.pc_L = (int)L;
      C.pc_u0 = u0;
      C.pc_len = (int)len;
      C.pc_item = n_pre;                            // past the end unless a start is found below
    }
    __syncthreads();
    if (len > 0 && u0 >= excl && u0 < excl + local) {
      long long acc = excl;
      for (int r = lo; r < hi; ++r) {
        const long long t = request_tiles(P, r, TOK2);
        if (u0 < acc + t) {                         // r's items: pairs from the last down, KV heads inside
          const int q0 = __ldg(P.cu_q_lens + r), q_len = __ldg(P.cu_q_lens + r + 1) - q0;
          const int ctx = __ldg(P.ctx_lens + r), n_pairs = (q_len + TOK2 - 1) / TOK2;
          long long off = u0 - acc;
          for (int rem = 0; rem < n_pairs * P.n_kv_heads; ++rem) {
            const int nkt = pair_tiles(ctx, q_len, n_pairs - 1 - rem / P.n_kv_heads, TOK2, P.window);
            if (off < nkt) {
              C.pc_item = pre[r] + rem;
              C.pc_j0 = (int)off;
              break;
            }
            off -= nkt;
          }
          break;
        }
        acc += t;
      }
    }
  }
  __syncthreads();
}

// Bounded wait whose outcome is the same for all 32 lanes of the warp.
__device__ __forceinline__ bool warp_wait(const StepParams& P, uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  if (!ok) set_error(P.err, CB_DEVERR_TIMEOUT);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait of a single thread; a timeout records the error and aborts the CTA.
__device__ __forceinline__ bool lane_wait(const StepParams& P, MixedCtl& C, uint64_t* bar, uint32_t parity) {
  if (mbar_wait(bar, parity)) return true;
  set_error(P.err, CB_DEVERR_TIMEOUT);
  C.abort = 1;
  return false;
}

// ---------------------------------------------------------------- producer (warp 8)
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
  // lane -> (block b, half hf) among the 8 x H boxes of one key/value tile
  const int my_b = (lane / H) & 7, my_hf = lane % H;
  const bool issuer = lane < 8 * H;
  uint32_t kt = 0, it = 0;
  PieceIter pieces(C);
  PreItem I;
  int j0, j1;
  long long u_start;
  for (; pieces.next(P, pre, n_pre, 2 * TOK, I, j0, j1, u_start); ++it) {
    if (C.abort) break;
    int ok = 1;
    if (lane == 0) {
      ok = lane_wait(P, C, &C.q_empty, (it & 1) ^ 1);
      if (ok) {
        mbar_arrive_expect_tx(&C.q_full, 2 * PrefillTiles<A>::kTileBytes);
#pragma unroll
        for (int side = 0; side < 2; ++side)
#pragma unroll
          for (int hf = 0; hf < H; ++hf)
            tma_load_3d(&T.q[side][hf][0][0], qmap, hf * 64, I.g * G, I.q0 + I.tok_lo + side * TOK, &C.q_full);
      }
    }
    if (!__shfl_sync(FULL, ok, 0)) break;
    const int nblk_hi = (I.kv_hi + kBlockSize - 1) / kBlockSize;
    // under a rolling window, blocks wholly before the earliest row's window
    // are seen by no row of the pair: they are not read (their table entries
    // may already have been released) and their rows load as zeros
    const int nblk_lo = P.window > 0 ? max(0, I.ctx + I.tok_lo - P.window + 1) / kBlockSize : 0;
    int y = rows_total;
    for (int j = j0; j < j1; ++j, ++kt) {
      if (((j - j0) & 3) == 0) {   // table entries for this tile and the next three
        const int blk = j * 8 + lane;
        y = rows_total;            // past the extent: TMA fills zeros
        if (blk < nblk_hi && blk >= nblk_lo) {
          const int e = __ldg(P.block_tables + (size_t)I.r * P.max_blocks_per_seq + blk);
          if (e >= 0 && e < P.num_blocks)
            y = (e * Hkv + I.g) * kBlockSize;
          else
            set_error(P.err, CB_DEVERR_BADBLOCK);
        }
      }
      const int yb = __shfl_sync(FULL, y, ((j - j0) & 3) * 8 + my_b);
      const int st = kt & 1;
      const uint32_t ph = (kt >> 1) & 1;
      ok = 1;
      if (lane == 0) {
        ok = lane_wait(P, C, &C.k_empty[st], ph ^ 1);
        if (ok) mbar_arrive_expect_tx(&C.k_full[st], PrefillTiles<A>::kTileBytes);
      }
      if (!__shfl_sync(FULL, ok, 0)) break;
      if (issuer) tma_load_2d(&T.k[st][my_hf][my_b * kBlockSize][0], kmap, my_hf * 64, yb, &C.k_full[st]);
      if (lane == 0) {
        ok = lane_wait(P, C, &C.v_empty[st], ph ^ 1);
        if (ok) mbar_arrive_expect_tx(&C.v_full[st], PrefillTiles<A>::kTileBytes);
      }
      if (!__shfl_sync(FULL, ok, 0)) break;
      if (issuer) tma_load_2d(&T.v[st][my_hf][my_b * kBlockSize][0], vmap, my_hf * 64, yb, &C.v_full[st]);
    }
    if (C.abort) break;
  }
  if (lane == 0 && C.abort) {      // let copies already issued land before shared memory is reused
    for (int s = 0; s < 2; ++s)
      for (int par = 0; par < 2; ++par) {
        mbar_wait(&C.k_full[s], par, 20000000ull);
        mbar_wait(&C.v_full[s], par, 20000000ull);
      }
    mbar_wait(&C.q_full, 0, 20000000ull);
    mbar_wait(&C.q_full, 1, 20000000ull);
  }
}

// ---------------------------------------------------------------- MMA issuer (warp 9, one lane)
// Each query tile is an independent chain  S(0) P(0) PV(0) S(1) P(1) PV(1) ...
// S(j+1) overwrites the columns PV(j) reads P from; both are issued by this one
// thread, and tcgen05.mma operations of one thread execute in issue order, so
// S(j+1) may be queued right behind PV(j).  The issuer polls both chains and
// issues whichever next MMA is ready, so the two tiles drift half a period
// apart: while one tile's softmax runs, the tensor core works on the other
// tile's MMAs.
template <int A>
struct MmaIssuer {
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, A, 1);
  const StepParams& P;
  PrefillTiles<A>& T;
  MixedCtl& C;
  uint32_t tmem;
  uint32_t pv_cnt0 = 0, pv_cnt1 = 0;   // O += P V issued per side (= o_done phases)
  uint32_t p_cnt0 = 0, p_cnt1 = 0;     // P tiles consumed per side (= p_full phases)
  // Shared-memory descriptors of the tile bases, built once.  The start-address
  // field is the low 14 bits (address >> 4), so a K step of an operand is an
  // add of a compile-time constant: the issuing thread spends a few cycles per
  // MMA instead of rebuilding 64-bit descriptors in a serial chain.
  uint64_t qd[2], kd[2], vd[2];

  __device__ MmaIssuer(const StepParams& p, PrefillTiles<A>& t, MixedCtl& c, uint32_t tm)
      : P(p), T(t), C(c), tmem(tm) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      qd[i] = smem_desc_sw128(smem_u32(&T.q[i][0][0][0]), 16, 1024);
      kd[i] = smem_desc_sw128(smem_u32(&T.k[i][0][0][0]), 16, 1024);
      vd[i] = smem_desc_sw128(smem_u32(&T.v[i][0][0][0]), PrefillTiles<A>::kHalfBytes, 1024);
    }
  }

  // S_side = Q_side K(kj)^T, if its inputs are ready
  template <int SIDE>
  __device__ bool try_s(uint32_t kj) {
    const int st = kj & 1;
    if (!mbar_ready(&C.k_full[st], (kj >> 1) & 1)) return false;
    tc_fence_after();
    const uint64_t q0 = qd[SIDE], k0 = st ? kd[1] : kd[0];   // (a select: an indexed array would live in local memory)
#pragma unroll
    for (int ks = 0; ks < A / 16; ++ks) {
      const uint64_t off = ((ks >> 2) * PrefillTiles<A>::kHalfBytes + (ks & 3) * 32) >> 4;
      tc_mma_f16(tmem + SIDE * 128, q0 + off, k0 + off, kIdescS, ks > 0);
    }
    tc_commit(&C.s_full[SIDE]);
    return true;
  }

  // O_side (+)= P_side V(kj) with P read from tensor memory, if ready
  template <int SIDE>
  __device__ bool try_pv(int j, uint32_t kj, uint32_t it) {
    const int st = kj & 1;
    uint32_t& pc = SIDE == 0 ? p_cnt0 : p_cnt1;
    if (!mbar_ready(&C.p_full[SIDE], pc & 1)) return false;
    if (!mbar_ready(&C.v_full[st], (kj >> 1) & 1)) return false;
    if (j == 0 && !mbar_ready(&C.o_free[SIDE], (it & 1) ^ 1)) return false;
    ++pc;
    tc_fence_after();
    const uint64_t v0 = st ? vd[1] : vd[0];
    const uint32_t p_t = tmem + SIDE * 128;
    const uint32_t o_t = tmem + 256 + SIDE * A;
#pragma unroll
    for (int ks = 0; ks < kTileN / 16; ++ks)
      tc_mma_f16_ts(o_t, p_t + ks * 8, v0 + ((ks * 16 * 128) >> 4), kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
    tc_commit(&C.o_done[SIDE]);
    if (SIDE == 0)
      ++pv_cnt0;
    else
      ++pv_cnt1;
    return true;
  }
};

template <int A, int G>
__device__ void mma_issuer(const StepParams& P, PrefillTiles<A>& T, MixedCtl& C, const int* pre, uint32_t tmem) {
  constexpr int TOK = kTileM / G;
  const int n_pre = pre[P.n_reqs];
  MmaIssuer<A> M(P, T, C, tmem);
  uint32_t kt = 0, it = 0;
  bool ok = true;
  PieceIter pieces(C);
  PreItem I;
  int j0, j1;
  long long u_start;
  for (; ok && pieces.next(P, pre, n_pre, 2 * TOK, I, j0, j1, u_start); ++it) {
    if (C.abort) break;
    if (!lane_wait(P, C, &C.q_full, it & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const int n = j1 - j0;          // this piece's key tiles
    int ns0 = 0, ns1 = 0, np0 = 0, np1 = 0;     // next S / next PV per side
    bool q_released = false;
    uint64_t t_last = globaltimer_ns();
    while (np0 < n || np1 < n) {
      bool prog = false;
      // side A: its next S, or its next PV followed at once by the S after it,
      // so this tile's scores never queue behind the other tile's MMAs
      if (np0 < ns0 && M.template try_pv<0>(np0, kt + np0, it)) {
        ++np0;
        if (np1 >= np0) tc_commit(&C.v_empty[(kt + np0 - 1) & 1]);      // both sides read V(np0-1)
        prog = true;
      }
      if (ns0 == np0 && ns0 < n && M.template try_s<0>(kt + ns0)) {
        ++ns0;
        if (ns1 >= ns0) tc_commit(&C.k_empty[(kt + ns0 - 1) & 1]);      // both sides read K(ns0-1)
        prog = true;
      }
      // side B, the same
      if (np1 < ns1 && M.template try_pv<1>(np1, kt + np1, it)) {
        ++np1;
        if (np0 >= np1) tc_commit(&C.v_empty[(kt + np1 - 1) & 1]);
        prog = true;
      }
      if (ns1 == np1 && ns1 < n && M.template try_s<1>(kt + ns1)) {
        ++ns1;
        if (ns0 >= ns1) tc_commit(&C.k_empty[(kt + ns1 - 1) & 1]);
        prog = true;
      }
      if (!q_released && ns0 == n && ns1 == n) {
        tc_commit(&C.q_empty);   // every S of this item is issued: Q is free once they complete
        q_released = true;
      }
      if (prog) {
        t_last = globaltimer_ns();
      } else {
        // nothing ready: yield the issue slot to the softmax warps of this
        // sub-partition instead of spinning
        __nanosleep(64);
        if (globaltimer_ns() - t_last > kWaitLimitNs || C.abort) {
          set_error(P.err, CB_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
    kt += n;
  }
  if (!ok) C.abort = 1;
  tc_commit(&C.drain);           // every MMA issued above completes before TMEM is freed
  mbar_wait(&C.drain, 0, 20000000ull);
}

// ---------------------------------------------------------------- softmax (warps 0-7)
template <int A, int G>
__device__ void softmax_side(const StepParams& P, const PrefillSplit& S, PrefillTiles<A>& T, MixedCtl& C,
                             const int* pre, uint32_t tmem, int side) {
  constexpr int TOK = kTileM / G;
  constexpr int H = A / 64;
  const unsigned FULL = 0xffffffffu;
  const int row = threadIdx.x & 127;
  const int warp_q = (threadIdx.x >> 5) & 3;                // TMEM lane quarter of this warp
  const uint32_t lane_base = (uint32_t)(warp_q * 32) << 16;
  const uint32_t s_col = side * 128;
  const uint32_t o_col = 256 + side * A;
  const int n_pre = pre[P.n_reqs];
  const int Hq = P.n_q_heads;
  const float sl2 = P.scale_log2;
  uint32_t sc = 0;                                           // S tiles consumed (= global key tiles)
  PieceIter pieces(C);
  PreItem I;
  int j0, j1;
  long long u_start;
  while (pieces.next(P, pre, n_pre, 2 * TOK, I, j0, j1, u_start)) {
    if (C.abort) break;
    const int tok_l = row / G, gq = row % G;
    const int ti = I.tok_lo + side * TOK + tok_l;
    const bool valid_row = ti < I.tok_hi;
    const int pos = I.ctx + min(ti, I.tok_hi - 1);            // last key this row may see
    // first key it may see (rolling window); key k is visible iff k - lo <= pos - lo as unsigned
    const int lo = P.window > 0 ? max(0, pos - P.window + 1) : 0;
    const unsigned span = (unsigned)(pos - lo);
    float m = kNegInf, l = 0.f;                               // m: running max, times scale*log2 e
    bool ok = true;
    for (int j = j0; j < j1; ++j, ++sc) {
      if (!warp_wait(P, &C.s_full[side], sc & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = j * kTileN;
      const bool masked_tile = key0 + kTileN - 1 > pos || key0 < lo;
      // pass 1: row max over the visible keys (two 64-column loads)
      float mt;
      {
        float a[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float sv[64];
          tmem_ld64(tmem + lane_base + s_col + h * 64, sv);
          tmem_wait_ld();
          if (!masked_tile) {
#pragma unroll
            for (int k = 0; k < 64; k += 2) a[(k >> 1) & 3] = max3(a[(k >> 1) & 3], sv[k], sv[k + 1]);
          } else {
#pragma unroll
            for (int k = 0; k < 64; k += 2) {
              const int key = key0 + h * 64 + k;
              a[(k >> 1) & 3] = max3(a[(k >> 1) & 3], (unsigned)(key - lo) > span ? kNegInf : sv[k],
                                     (unsigned)(key + 1 - lo) > span ? kNegInf : sv[k + 1]);
            }
          }
        }
        mt = max3(a[0], a[1], fmaxf(a[2], a[3])) * sl2;
      }
      const float mn = fmaxf(m, mt);
      const bool need = mn > m + 8.f;
      float alpha = 1.f;
      if (need) {
        alpha = ex2(m - mn);
        m = mn;
      }
      if (j > j0 && __any_sync(FULL, need)) {
        // rescale O: the previous O += P V of this side must be complete
        if (!warp_wait(P, &C.o_done[side], (sc - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < A / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + o_col + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(tmem + lane_base + o_col + c * 32, o);
        }
      }
      // pass 2: p = 2^(s*scale*log2 e - m), packed to bf16 pairs over the S columns
      // (64 columns per load), the exponent arguments with packed fp32x2 FMAs.
      const uint64_t sl2x2 = f2(sl2, sl2), nmx2 = f2(-m, -m);
      uint64_t rs2[2] = {0ull, 0ull};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float sv[64];
        tmem_ld64(tmem + lane_base + s_col + h * 64, sv);
        tmem_wait_ld();
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const uint64_t t = ffma2(f2(sv[2 * k], sv[2 * k + 1]), sl2x2, nmx2);
          float t0, t1;
          f2split(t, t0, t1);
          float p0 = ex2(t0), p1 = ex2(t1);
          if (masked_tile) {
            const int key = key0 + h * 64 + 2 * k;
            p0 = (unsigned)(key - lo) > span ? 0.f : p0;
            p1 = (unsigned)(key + 1 - lo) > span ? 0.f : p1;
          }
          rs2[k & 1] = fadd2(rs2[k & 1], f2(p0, p1));
          pk[k] = pack_bf16(p0, p1);
        }
        // P of columns [64h, 64h+64) goes to columns [32h, 32h+32): S there was read above
        tmem_st32u(tmem + lane_base + s_col + h * 32, pk);
      }
      float rs[4];
      f2split(rs2[0], rs[0], rs[1]);
      f2split(rs2[1], rs[2], rs[3]);
      l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
      // zero the value rows past the pair's last key in its final block: they hold
      // whatever the cache had there, and 0 * non-finite must not reach O.  Both
      // sides write the same zeros, since either side's O += P V may run first.
      if (key0 + kTileN > I.kv_hi && (I.kv_hi & (kBlockSize - 1))) {
        const int st = sc & 1;
        if (!warp_wait(P, &C.v_full[st], (sc >> 1) & 1)) {
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
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&C.p_full[side]);
    }
    if (!ok) {
      C.abort = 1;
      break;
    }
    if (!warp_wait(P, &C.o_done[side], (sc - 1) & 1)) {
      C.abort = 1;
      break;
    }
    tc_fence_after();
    if (j0 > I.jlo || j1 < I.nkt) {
      // a piece of an item cut at a CTA boundary: its unnormalised O and (m, l)
      // go to this CTA's slot (2b: first piece, 2b + 1: last); the CTA that ran
      // the item's first tiles merges the pieces after the grid-wide barrier
      const int slot = 2 * (int)blockIdx.x + (pieces.k == 0 ? 0 : 1);
      if (slot < S.slots) {
        float* base = S.part + (size_t)slot * kPreRows * (A + 2);
        float* orow_p = base + (size_t)(side * kTileM + row) * A;
#pragma unroll 1
        for (int c = 0; c < A / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + o_col + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(orow_p + c * 32 + k) = make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
        }
        *reinterpret_cast<float2*>(base + (size_t)kPreRows * A + (side * kTileM + row) * 2) = make_float2(m, l);
        if (j0 == I.jlo && side == 0 && row == 0) {
          C.own_item = pieces.item - 1;
          C.own_slot = slot;
          C.own_u = u_start;
        }
      } else {
        set_error(P.err, CB_DEVERR_BADLEN);
      }
      tc_fence_before();
      mbar_arrive(&C.o_free[side]);
      continue;
    }
    const float inv = 1.f / l;
    uint16_t* orow = P.out + ((size_t)(I.q0 + ti) * Hq + (size_t)I.g * G + gq) * A;
#pragma unroll 1
    for (int c = 0; c < A / 32; ++c) {
      float o[32];
      tmem_ld32(tmem + lane_base + o_col + c * 32, o);
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
    mbar_arrive(&C.o_free[side]);
  }
}

// After the grid-wide barrier, the CTA that ran the first tiles of an item cut
// at CTA boundaries merges the item's pieces by log-sum-exp over their
// partials (as the decode's split merge): per row, M = max_k m_k,
// L = sum_k 2^(m_k - M) l_k, out = sum_k 2^(m_k - M) O_k / L.  The item's
// pieces are in CTAs b .. (item end - 1) / L: this CTA's own slot, then slot
// 2c (the first piece) of each later CTA c.  All threads of the CTA call it.
template <int A, int G>
__device__ void prefill_merge(const StepParams& P, const PrefillSplit& S, const MixedCtl& C, const int* pre) {
  constexpr int TOK = kTileM / G, Q = A / 4;
  if (!C.pc_balanced || C.own_item < 0) return;
  const PreItem I = pre_item(P, pre, C.own_item, 2 * TOK);
  const int c0 = blockIdx.x, c1 = (int)((C.own_u + (I.nkt - I.jlo) - 1) / C.pc_L);
  const size_t slot_floats = (size_t)kPreRows * (A + 2);
  for (int task = threadIdx.x; task < kPreRows * Q; task += blockDim.x) {
    const int row = task / Q, ch = task - row * Q;
    const int side = row / kTileM, i = row - side * kTileM;
    const int ti = I.tok_lo + side * TOK + i / G;
    if (ti >= I.tok_hi) continue;
    float M = kNegInf;
    for (int c = c0; c <= c1; ++c) {
      const int slot = c == c0 ? C.own_slot : 2 * c;
      if (slot < S.slots) M = fmaxf(M, __ldcg(S.part + slot * slot_floats + (size_t)kPreRows * A + row * 2));
    }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = c0; c <= c1; ++c) {
      const int slot = c == c0 ? C.own_slot : 2 * c;
      if (slot >= S.slots) continue;
      const float* base = S.part + slot * slot_floats;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(base + (size_t)kPreRows * A) + row);
      const float w = ex2(ml.x - M);             // 0 for a piece in which the row saw no key
      const float4 o = __ldcg(reinterpret_cast<const float4*>(base + (size_t)row * A) + ch);
      L += w * ml.y;
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
    const float inv = 1.f / L;
    uint16_t* orow = P.out + ((size_t)(I.q0 + ti) * P.n_q_heads + (size_t)I.g * G + i % G) * A + ch * 4;
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
  }
}

// Shared memory of the mixed kernel: the tile region (prefill tiles, or the
// decode pipeline's rings in phase 2), the control blocks and the plan arrays.
template <int A, int G, bool BT, int HKV>
struct MixedLayout {
  static constexpr size_t kRegion = sizeof(PrefillTiles<A>);
  static constexpr size_t kCtl2 = 0;
};
template <int G, int HKV>
struct MixedLayout<128, G, true, HKV> {
  static constexpr size_t kRegion = sizeof(PrefillTiles<128>) > sizeof(tcb::Tiles<G, HKV>)
                                        ? sizeof(PrefillTiles<128>)
                                        : sizeof(tcb::Tiles<G, HKV>);
  static constexpr size_t kCtl2 = sizeof(tcb::Ctl<G, HKV>);
};
template <int A, int G, bool BT, int HKV>
constexpr size_t mixed_smem(int n_reqs) {
  return 1024 + MixedLayout<A, G, BT, HKV>::kRegion + sizeof(MixedCtl) + MixedLayout<A, G, BT, HKV>::kCtl2 +
         (size_t)3 * (n_reqs + 1) * 4;
}

// BT: the decode phase is the block-tile pipeline, for HKV KV heads (a
// template parameter of that pipeline; the prefill phase reads P.n_kv_heads).
template <int A, int G, bool BT, int HKV>
__global__ void __launch_bounds__(BT ? tcb::kThreads : kNumThreads, 1)
    mixed_kernel(const StepParams P, const AppendParams Ap, const PrefillSplit Sp, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap,
                 const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap_b,
                 const __grid_constant__ CUtensorMap vmap_b, const __grid_constant__ CUtensorMap qmap_d) {
  constexpr int TOK = kTileM / G;
  using WS = DecWarpSmem<A, (BT ? 1 : G), kDecStages>;   // CUDA-core decode rings (unused with BT)
  using L = MixedLayout<A, G, BT, HKV>;
  static_assert(kDecWarps * sizeof(WS) <= sizeof(PrefillTiles<A>), "decode rings must fit in the tile region");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PrefillTiles<A>& T = *reinterpret_cast<PrefillTiles<A>*>(base);
  MixedCtl& C = *reinterpret_cast<MixedCtl*>(base + L::kRegion);
  // plan arrays: CUDA-core decode: dec, spl, pre; block-tile decode: pre, bpre, slot
  int* a0 = reinterpret_cast<int*>(base + L::kRegion + sizeof(MixedCtl) + L::kCtl2);
  int* a1 = a0 + (P.n_reqs + 1);
  int* a2 = a1 + (P.n_reqs + 1);
  int* pre = BT ? a0 : a2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&C.q_full, 1);
    mbar_init(&C.q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&C.k_full[s], 1);
      mbar_init(&C.k_empty[s], 1);
      mbar_init(&C.v_full[s], 1);
      mbar_init(&C.v_empty[s], 1);
      mbar_init(&C.s_full[s], 1);
      mbar_init(&C.p_full[s], 128);
      mbar_init(&C.o_done[s], 1);
      mbar_init(&C.o_free[s], 128);
    }
    mbar_init(&C.drain, 1);
    C.abort = 0;
    C.pc_balanced = 0;             // prefill pieces: whole items round robin unless the plan balances them
    C.pc_item = blockIdx.x;
    C.pc_nown = -1;
    C.pc_j0 = 0;
    C.pc_len = 0;
    C.pc_L = 0;
    C.pc_u0 = 0;
    C.own_item = -1;
    if constexpr (BT) {
      tcb::init_ctl<G, HKV>(*reinterpret_cast<tcb::Ctl<G, HKV>*>(base + L::kRegion + sizeof(MixedCtl)));
      prefetch_tmap(&kmap_b);
      prefetch_tmap(&vmap_b);
      prefetch_tmap(&qmap_d);
    }
    fence_mbar_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&qmap);
  }
  if (warp == 9) {
    tmem_alloc(&C.tmem_base, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  if constexpr (BT) {
    // prefill items per request and decode blocks per request, both in request order
    tcb::Ctl<G, HKV>& C2 = *reinterpret_cast<tcb::Ctl<G, HKV>*>(base + L::kRegion + sizeof(MixedCtl));
    tcb::append_phase<HKV == 8>(P, Ap);      // the step's new rows, when this launch stores them
    for (int r = threadIdx.x; r < P.n_reqs; r += blockDim.x) {
      pre[r] = request_work(P, r, 2 * TOK, true).pre_items;
      a1[r] = tcb::decode_blocks(P, r, true);
    }
    __syncthreads();
    tcb::block_scan_excl(pre, P.n_reqs, C2.scratch);
    tcb::finish_plan<G, HKV>(P, C2, a1, a2);
    prefill_plan<2 * TOK>(P, Sp, C, pre, (long long)C2.total * (2 * HKV * kBlockSize * A * 2),
                          reinterpret_cast<int*>(&T.q[0][0][0][0]));   // the tiles are free until the prefill
    if (threadIdx.x == 0 && C.pc_balanced) C2.split_any = 1;   // the pieces' merge needs the grid-wide barrier
    if (threadIdx.x == 0) C2.per_request = tcb::per_request_merge<G, HKV>(P, C.pc_balanced != 0);
    tcb::append_wait<HKV == 8>(P, Ap);       // before the first TMA load of the cache
  } else {
    build_plan(P, 2 * TOK, a0, a1, a2, C.scratch);   // ends with __syncthreads()
  }
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;

  if (pre[P.n_reqs] > 0) {
    if (warp == 8) {
      producer<A, G>(P, &kmap, &vmap, &qmap, T, C, pre);
    } else if (warp == 9) {
      if (lane == 0) mma_issuer<A, G>(P, T, C, pre, tmem);
      __syncwarp();
    } else if (warp < 8) {
      softmax_side<A, G>(P, Sp, T, C, pre, tmem, warp >> 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (BT) {
    // phase 2: the tile region becomes the decode pipeline's rings
    tcb::Tiles<G, HKV>& T2 = *reinterpret_cast<tcb::Tiles<G, HKV>*>(base);
    tcb::Ctl<G, HKV>& C2 = *reinterpret_cast<tcb::Ctl<G, HKV>*>(base + L::kRegion + sizeof(MixedCtl));
    tcb::zero_p<G, HKV>(T2);
    fence_proxy_async_smem();
    __syncthreads();
    tc_fence_after();
    if (!C.abort) tcb::run_pipeline<G, HKV>(P, &kmap_b, &vmap_b, &qmap_d, T2, C2, a1, a2, tmem, false);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    // the balanced prefill's pieces are merged after a grid-wide barrier; without
    // them each request's merge waits only for its own splits
    tcb::merge_phase<G, HKV>(P, C2, a2, reinterpret_cast<float*>(&T2.k[0][0][0][0]), C.pc_balanced != 0);
    if (C.pc_balanced && C2.merge_ok) prefill_merge<A, G>(P, Sp, C, pre);
    tcb::release_counters(P);
  } else {
    if (warp == 9) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    if (C.abort || warp >= kDecWarps) return;
    decode_worker<A, G, kDecStages, 2>(P, &kmap, &vmap, reinterpret_cast<WS*>(base)[warp], a0, a1);
  }
}
static_assert(sizeof(PrefillTiles<128>) % 16 == 0 && sizeof(MixedCtl) % 16 == 0, "control blocks 16-byte aligned");
static_assert(mixed_smem<128, 2, true, 8>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(mixed_smem<128, 4, true, 8>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(mixed_smem<128, 8, true, 8>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(mixed_smem<128, 16, true, 2>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");
static_assert(mixed_smem<128, 32, true, 1>(kMaxReqs) <= (size_t)kSmemLimit, "shared memory");

template <int A, int G, bool BT, int HKV>
cudaError_t launch_mixed_t(const StepParams& p, const AppendParams& ap, const PrefillSplit& ps, const CUtensorMap* maps,
                           int n_sms, cudaStream_t stream) {
  const size_t smem = mixed_smem<A, G, BT, HKV>(p.n_reqs);
  if (smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;
  if (!BT && ap.n_tokens != 0) return cudaErrorInvalidValue;   // only the cooperative launch stores rows
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(mixed_kernel<A, G, BT, HKV>), kSmemLimit);
  if (e != cudaSuccess) return e;
  if constexpr (BT) {   // cooperative: the decode merge phase waits for every CTA
    StepParams pc = p;
    AppendParams apc = ap;
    PrefillSplit psc = ps;
    void* args[] = {&pc, &apc, &psc, const_cast<CUtensorMap*>(&maps[0]), const_cast<CUtensorMap*>(&maps[1]),
                    const_cast<CUtensorMap*>(&maps[2]), const_cast<CUtensorMap*>(&maps[3]),
                    const_cast<CUtensorMap*>(&maps[4]), const_cast<CUtensorMap*>(&maps[5])};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(mixed_kernel<A, G, BT, HKV>), dim3(n_sms),
                                       dim3(tcb::kThreads), args, smem, stream);
  } else {
    mixed_kernel<A, G, BT, HKV><<<n_sms, kNumThreads, smem, stream>>>(p, ap, PrefillSplit{}, maps[0], maps[1], maps[2],
                                                                   maps[3], maps[4], maps[5]);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_mixed(const StepParams& p, const AppendParams& ap, const PrefillSplit& ps, const CUtensorMap* maps,
                         bool block_tiles, int head_dim, int group, int n_sms, cudaStream_t stream) {
#define CB_MIX_CASE(A_, G_, BT_, HKV_)                                                      \
  if (head_dim == A_ && group == G_ && block_tiles == BT_ && (!BT_ || p.n_kv_heads == HKV_)) \
    return launch_mixed_t<A_, G_, BT_, HKV_>(p, ap, ps, maps, n_sms, stream);
  CB_MIX_CASE(128, 2, true, 8)
  CB_MIX_CASE(128, 4, true, 8)
  CB_MIX_CASE(128, 8, true, 8)
  CB_MIX_CASE(128, 16, true, 2)
  CB_MIX_CASE(128, 32, true, 1)
  CB_MIX_CASE(128, 1, false, 0)
  CB_MIX_CASE(128, 2, false, 0)
  CB_MIX_CASE(128, 4, false, 0)
  CB_MIX_CASE(128, 8, false, 0)
  CB_MIX_CASE(64, 1, false, 0)
  CB_MIX_CASE(64, 2, false, 0)
  CB_MIX_CASE(64, 4, false, 0)
  CB_MIX_CASE(64, 8, false, 0)
#undef CB_MIX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace cb
