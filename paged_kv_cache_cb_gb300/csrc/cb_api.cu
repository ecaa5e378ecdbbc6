// C-ABI entry points of include/cbattn.h: argument checks, workspace carving,
// TMA tensor-map encoding and kernel dispatch.  Host code only (plus the
// library's per-stream device state).
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <new>
#include <set>

#include "../../include/cbattn.h"
#include "cb_internal.h"

namespace cb {

// Library state of one (device, stream): the block-tile launches' four work
// counters (chunk claims, merge barrier, append barrier, exits) and the error
// word that every kernel launched on that stream ORs its CB_DEVERR_* bits into.
// Zero at load; every block-tile launch leaves its counters at zero (its last
// CTA resets them), so no launch needs a memset first; cb_last_error(stream)
// reads and clears the stream's error word.
struct StreamSlot {
  int queue[4];
  unsigned int err;
  unsigned int pad[3];
};
constexpr int kStreamSlots = 4096;
__device__ StreamSlot g_stream_slots[kStreamSlots];

namespace {

constexpr int kMaxDevices = 64;
thread_local int g_last_launches = 0;

struct DeviceInfo {
  int n_sms = 0;
};

bool device_info(DeviceInfo* out) {
  static DeviceInfo cache[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = cache[dev];
  if (d.n_sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    d.n_sms = sms;
  }
  *out = d;
  return true;
}

// The slot of (current device, stream), handed out in order of first use
// (create = false: only look it up).  Returns nullptr on a CUDA error, when a
// device has used up its kStreamSlots slots (*full = true), or, without
// create, when the stream has none yet.
StreamSlot* stream_slot(cudaStream_t stream, bool create, bool* full = nullptr) {
  static void* base[kMaxDevices] = {};
  static int next[kMaxDevices] = {};
  static std::map<std::pair<int, uintptr_t>, int> slot_of;
  static std::mutex mu;
  if (full) *full = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!base[dev] && cudaGetSymbolAddress(&base[dev], g_stream_slots) != cudaSuccess) return nullptr;
  const auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(stream));
  auto it = slot_of.find(key);
  if (it == slot_of.end()) {
    if (!create) return nullptr;
    if (next[dev] >= kStreamSlots) {
      if (full) *full = true;
      return nullptr;
    }
    it = slot_of.emplace(key, next[dev]++).first;
  }
  return static_cast<StreamSlot*>(base[dev]) + it->second;
}

// Error word of `stream`'s slot for a launch (nullptr: see stream_slot); rc
// receives the code to return when there is none.
unsigned int* launch_err(cudaStream_t stream, int* rc) {
  bool full = false;
  StreamSlot* sl = stream_slot(stream, true, &full);
  *rc = full ? CB_ESTATE : CB_ECUDA;
  return sl ? &sl->err : nullptr;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Cache viewed as rows of head_dim values: [num_blocks * Hkv * block_size][A];
// box = `box_rows` rows x 64 columns, 128-byte swizzle: 16 rows is one (block,
// head), 16 * Hkv rows one block of every head.
bool encode_cache_map(CUtensorMap* m, const void* cache, int num_blocks, int n_kv_heads, int head_dim,
                      int box_rows = kBlockSize) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)num_blocks * n_kv_heads * kBlockSize};
  const cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q viewed as [n_tokens][Hq][A]; box = box_tokens tokens x box_heads heads x 64
// columns.  Prefill: 128/G tokens x the G heads of one group, a 128-row query
// tile (row = token * G + head); decode: 1 token x all Hq heads.
bool encode_q_map(CUtensorMap* m, const void* q, int n_tokens, int n_q_heads, int head_dim, int box_heads,
                  int box_tokens) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_q_heads, (cuuint64_t)n_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_q_heads * head_dim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

// Smallest decode split the launcher may choose; the workspace is sized for it.
constexpr int kMinSplitBlocks = 8;

// The dynamic shared-memory opt-in of a kernel, once per (device, kernel): the
// attribute belongs to the current device's context.
cudaError_t opt_in_smem(const void* kernel, int bytes) {
  static std::set<std::pair<int, const void*>> done;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, kernel})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({dev, kernel});
  return e;
}

namespace {

// Offsets for a given capacity of split partials (and pre_slots prefill slots).
WorkspaceLayout layout_for_splits(long long splits, int n_reqs, int n_q_heads, int n_kv_heads, int head_dim,
                                  int pre_slots) {
  WorkspaceLayout L{};
  L.max_splits_total = (int)splits;
  L.pre_slots = pre_slots;
  size_t off = 0;
  L.counters = off;
  off = align_up(off + (size_t)n_reqs * n_kv_heads * 4, 16);
  L.queue = off;
  off = align_up(off + 16, 256);
  L.pre_part = off;
  off = align_up(off + (size_t)pre_slots * kPreRows * (head_dim + 2) * 4, 256);
  L.part_ml = off;
  off = align_up(off + (size_t)splits * n_q_heads * 2 * 4, 256);
  L.part_acc = off;
  off = align_up(off + (size_t)splits * n_q_heads * head_dim * 4, 256);
  L.total = off;
  return L;
}

// Shapes of the block-tile decode (128-row tiles of whole blocks): head_dim 128
// with 8 KV heads and G >= 2, or 32 query heads on 2 KV heads (G = 16) or on 1
// (MQA, G = 32).
bool block_tile_shape(int n_q_heads, int n_kv_heads, int head_dim) {
  if (head_dim != 128 || n_q_heads % n_kv_heads) return false;
  return (n_kv_heads == 8 && n_q_heads / n_kv_heads >= 2) || (n_q_heads == 32 && (n_kv_heads == 2 || n_kv_heads == 1));
}

}  // namespace

WorkspaceLayout workspace_layout(int n_reqs, int max_kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                                 int split_blocks, bool prefill_split) {
  const long long nblk = (max_kv_len + kBlockSize - 1) / kBlockSize;
  // a request's blocks are cut into pieces of >= split_blocks blocks at
  // boundaries that need not start at its first block: one piece more at most
  long long splits = (long long)n_reqs * ((nblk + split_blocks - 1) / split_blocks + 1);
  // the block-tile decode cuts small steps into shorter chunks: at most
  // 4 rounds of one chunk per CTA beyond that
  if (block_tile_shape(n_q_heads, n_kv_heads, head_dim)) splits += 4LL * kMaxDecodeGrid + 8;
  const int pre_slots = prefill_split && block_tile_shape(n_q_heads, n_kv_heads, head_dim) ? 2 * kMaxDecodeGrid : 0;
  return layout_for_splits(splits, n_reqs, n_q_heads, n_kv_heads, head_dim, pre_slots);
}

// The same offsets with as many split partials as `bytes` can hold (at least
// L's): a larger workspace than the size query asked for lets the decode cut
// a step into more, shorter pieces.
WorkspaceLayout workspace_layout_for_bytes(const WorkspaceLayout& L, size_t bytes, int n_reqs, int n_q_heads,
                                           int n_kv_heads, int head_dim) {
  const size_t per_split = (size_t)n_q_heads * (2 + head_dim) * 4;
  if (bytes <= L.part_ml + 512) return L;
  const long long fit = std::min<long long>((long long)((bytes - L.part_ml - 512) / per_split), 1LL << 24);
  if (fit <= L.max_splits_total) return L;
  return layout_for_splits(fit, n_reqs, n_q_heads, n_kv_heads, head_dim, L.pre_slots);
}

int choose_split_blocks(int n_reqs, int max_kv_len, int n_kv_heads, int n_sms) {
  const long long nblk = (max_kv_len + kBlockSize - 1) / kBlockSize;
  const long long want = 4LL * n_sms * 8;           // items per decode warp slot, a few each
  for (int sb = kMaxSplitBlocks; sb > kMinSplitBlocks; sb >>= 1)
    if ((long long)n_reqs * n_kv_heads * ((nblk + sb - 1) / sb) >= want) return sb;
  return kMinSplitBlocks;
}

}  // namespace cb

using namespace cb;

namespace {

bool shape_ok(int n_q_heads, int n_kv_heads, int head_dim, int block_size) {
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  if (block_size != kBlockSize) return false;
  const int g = n_q_heads / n_kv_heads;
  if (g == 1 || g == 2 || g == 4 || g == 8) return true;
  return block_tile_shape(n_q_heads, n_kv_heads, head_dim);    // G = 16, 32
}

}  // namespace

extern "C" {

int cb_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int n_tokens, void* k_cache,
                 void* v_cache, int num_blocks, int n_kv_heads, int head_dim, int block_size, void* stream) {
  if (n_tokens < 0 || num_blocks <= 0 || n_kv_heads <= 0 || (head_dim != 64 && head_dim != 128) ||
      block_size != kBlockSize)
    return CB_EINVAL;
  if (n_tokens == 0) {
    g_last_launches = 0;
    return CB_OK;
  }
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return CB_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache)) return CB_EINVAL;
  int rc = CB_OK;
  unsigned int* err = launch_err(static_cast<cudaStream_t>(stream), &rc);
  if (!err) return rc;
  cudaError_t e = launch_kv_append(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_blocks, n_kv_heads,
                                   head_dim, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return CB_ECUDA;
  g_last_launches = 1;
  return CB_OK;
}

int cb_copy_blocks(const int32_t* pairs, int n_pairs, void* k_cache, void* v_cache, int num_blocks, int n_kv_heads,
                   int head_dim, int block_size, void* stream) {
  if (n_pairs < 0 || n_pairs > 65535 || num_blocks <= 0 || n_kv_heads <= 0 || (head_dim != 64 && head_dim != 128) ||
      block_size != kBlockSize)
    return CB_EINVAL;
  if (n_pairs == 0) {
    g_last_launches = 0;
    return CB_OK;
  }
  if (!pairs || !k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache)) return CB_EINVAL;
  int rc = CB_OK;
  unsigned int* err = launch_err(static_cast<cudaStream_t>(stream), &rc);
  if (!err) return rc;
  if (launch_copy_blocks(pairs, n_pairs, k_cache, v_cache, num_blocks, n_kv_heads, head_dim, err,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CB_ECUDA;
  g_last_launches = 1;
  return CB_OK;
}

}  // extern "C"

namespace cb {
// Smallest workspace a step accepts (without the balanced prefill's partials).
size_t workspace_min_bytes(int n_reqs, int n_tokens, int max_q_len, int max_kv_len, int n_q_heads, int n_kv_heads,
                           int head_dim, int block_size) {
  if (n_reqs < 0 || n_reqs > CB_MAX_REQS || n_tokens < 0 || max_q_len < 1 || max_kv_len < 1 ||
      !shape_ok(n_q_heads, n_kv_heads, head_dim, block_size))
    return 0;
  return workspace_layout(n_reqs, max_kv_len, n_q_heads, n_kv_heads, head_dim, kMinSplitBlocks, false).total;
}
}  // namespace cb

extern "C" {

size_t cb_paged_attention_workspace_size(int n_reqs, int n_tokens, int max_q_len, int max_kv_len, int n_q_heads,
                                         int n_kv_heads, int head_dim, int block_size) {
  if (n_reqs < 0 || n_reqs > CB_MAX_REQS || n_tokens < 0 || max_q_len < 1 || max_kv_len < 1 ||
      !shape_ok(n_q_heads, n_kv_heads, head_dim, block_size))
    return 0;
  return workspace_layout(n_reqs, max_kv_len, n_q_heads, n_kv_heads, head_dim, kMinSplitBlocks, max_q_len > 1).total;
}

}  // extern "C"

namespace {

// The step's new K/V rows, for the entry point that stores them too.
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int64_t* slots;
};

// Attention step, optionally preceded by the append of the step's new rows
// (app != nullptr): inside the attention launch where it is cooperative (the
// block-tile paths), else as a cb_kv_append launch before it.
int attention_step(const AppendArgs* app, const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                   const int32_t* block_tables, int max_blocks_per_seq, int n_reqs, int n_tokens, int max_q_len,
                   int max_kv_len, const void* k_cache, const void* v_cache, int num_blocks, void* out, float scale,
                   int n_q_heads, int n_kv_heads, int head_dim, int block_size, int window, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (!shape_ok(n_q_heads, n_kv_heads, head_dim, block_size) || window < 0) return CB_EINVAL;
  if (n_reqs < 0 || n_reqs > CB_MAX_REQS || n_tokens < 0 || max_q_len < 1 || max_kv_len < 1 ||
      max_blocks_per_seq < 1 || num_blocks <= 0 || !(scale > 0.f) || max_q_len > max_kv_len)
    return CB_EINVAL;
  if ((long long)num_blocks * n_kv_heads * kBlockSize >= (1LL << 31) - kBlockSize) return CB_EINVAL;
  if (n_reqs == 0 || n_tokens == 0) {
    g_last_launches = 0;
    return CB_OK;
  }
  if (!q || !cu_q_lens || !ctx_lens || !block_tables || !k_cache || !v_cache || !out || !workspace) return CB_EINVAL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace))
    return CB_EINVAL;
  if (app && (!app->k_new || !app->v_new || !app->slots || !aligned16(app->k_new) || !aligned16(app->v_new)))
    return CB_EINVAL;
  // the balanced prefill's partial results when the workspace has room for them
  WorkspaceLayout L0 =
      workspace_layout(n_reqs, max_kv_len, n_q_heads, n_kv_heads, head_dim, kMinSplitBlocks, max_q_len > 1);
  if (workspace_bytes < L0.total)
    L0 = workspace_layout(n_reqs, max_kv_len, n_q_heads, n_kv_heads, head_dim, kMinSplitBlocks, false);
  if (workspace_bytes < L0.total) return CB_EWORKSPACE;
  const WorkspaceLayout L = workspace_layout_for_bytes(L0, workspace_bytes, n_reqs, n_q_heads, n_kv_heads, head_dim);
  DeviceInfo di;
  if (!device_info(&di)) return CB_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool slots_full = false;
  StreamSlot* slot = stream_slot(s, true, &slots_full);
  if (!slot) return slots_full ? CB_ESTATE : CB_ECUDA;

  StepParams p{};
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.q = static_cast<const uint16_t*>(q);
  p.cu_q_lens = cu_q_lens;
  p.ctx_lens = ctx_lens;
  p.block_tables = block_tables;
  p.out = static_cast<uint16_t*>(out);
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_kv_len = max_kv_len;
  p.n_reqs = n_reqs;
  p.n_tokens = n_tokens;
  p.num_blocks = num_blocks;
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = n_kv_heads;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = window;
  p.split_blocks = choose_split_blocks(n_reqs, max_kv_len, n_kv_heads, di.n_sms);
  p.max_splits_total = L.max_splits_total;
  p.counters = reinterpret_cast<int*>(ws + L.counters);
  p.queue = reinterpret_cast<int*>(ws + L.queue);
  p.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
  p.part_acc = reinterpret_cast<float*>(ws + L.part_acc);
  p.err = &slot->err;

  const int group = n_q_heads / n_kv_heads;
  // GQA with 8 KV heads and head_dim 128: decode tokens run the block-tile
  // pipeline (one block of all heads is one 128-row MMA tile)
  const bool block_tiles = block_tile_shape(n_q_heads, n_kv_heads, head_dim);
  // maps: [0, 1] K, V with 16-row boxes; [2] prefill q; [3, 4] K, V with
  // 128-row boxes; [5] decode q (one token, all heads)
  CUtensorMap maps[6];
  if (max_q_len > 1 || !block_tiles) {
    if (!encode_cache_map(&maps[0], k_cache, num_blocks, n_kv_heads, head_dim, kBlockSize) ||
        !encode_cache_map(&maps[1], v_cache, num_blocks, n_kv_heads, head_dim, kBlockSize))
      return CB_ECUDA;
  }
  if (max_q_len > 1 && !encode_q_map(&maps[2], q, n_tokens, n_q_heads, head_dim, group, kTileM / group))
    return CB_ECUDA;
  if (block_tiles) {
    if (!encode_cache_map(&maps[3], k_cache, num_blocks, n_kv_heads, head_dim, n_kv_heads * kBlockSize) ||
        !encode_cache_map(&maps[4], v_cache, num_blocks, n_kv_heads, head_dim, n_kv_heads * kBlockSize) ||
        !encode_q_map(&maps[5], q, n_tokens, n_q_heads, head_dim, n_q_heads, 1))
      return CB_ECUDA;
  }
  // the append goes into the launch where that launch is cooperative
  AppendParams ap{};
  int launches = 1;
  if (app && block_tiles) {
    ap.k_new = static_cast<const uint4*>(app->k_new);
    ap.v_new = static_cast<const uint4*>(app->v_new);
    ap.slots = app->slots;
    ap.k_cache = static_cast<uint4*>(const_cast<void*>(k_cache));
    ap.v_cache = static_cast<uint4*>(const_cast<void*>(v_cache));
    ap.n_tokens = n_tokens;
  } else if (app) {
    if (launch_kv_append(app->k_new, app->v_new, app->slots, n_tokens, const_cast<void*>(k_cache),
                         const_cast<void*>(v_cache), num_blocks, n_kv_heads, head_dim, p.err, s) != cudaSuccess)
      return CB_ECUDA;
    launches = 2;
  }
  if (block_tiles) {
    // library counters that every block-tile launch leaves at zero: no memset
    p.queue = slot->queue;
  } else if (cudaMemsetAsync(ws + L.counters, 0, L.pre_part - L.counters, s) != cudaSuccess) {
    return CB_ECUDA;                          // split arrival counters and the work queue start at zero
  }
  cudaError_t e;
  if (max_q_len == 1 && block_tiles) {
    e = launch_decode_tcb(p, ap, maps[3], maps[4], maps[5], group, std::min(di.n_sms, kMaxDecodeGrid), s);
  } else if (max_q_len == 1) {
    e = launch_decode(p, maps[0], maps[1], head_dim, group, di.n_sms, s);
  } else {
    if (!block_tiles) maps[3] = maps[4] = maps[5] = maps[0];   // unused by the kernel
    PrefillSplit ps{};
    if (L.pre_slots > 0) {
      ps.part = reinterpret_cast<float*>(ws + L.pre_part);
      ps.slots = L.pre_slots;
    }
    e = launch_mixed(p, ap, ps, maps, block_tiles, head_dim, group, block_tiles ? std::min(di.n_sms, kMaxDecodeGrid) : di.n_sms,
                     s);
  }
  if (e != cudaSuccess) return CB_ECUDA;
  g_last_launches = launches;
  return CB_OK;
}

}  // namespace

extern "C" {

int cb_paged_attention(const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens, const int32_t* block_tables,
                       int max_blocks_per_seq, int n_reqs, int n_tokens, int max_q_len, int max_kv_len,
                       const void* k_cache, const void* v_cache, int num_blocks, void* out, float scale,
                       int n_q_heads, int n_kv_heads, int head_dim, int block_size, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return attention_step(nullptr, q, cu_q_lens, ctx_lens, block_tables, max_blocks_per_seq, n_reqs, n_tokens,
                        max_q_len, max_kv_len, k_cache, v_cache, num_blocks, out, scale, n_q_heads, n_kv_heads,
                        head_dim, block_size, 0, workspace, workspace_bytes, stream);
}

int cb_paged_attention_window(const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                              const int32_t* block_tables, int max_blocks_per_seq, int n_reqs, int n_tokens,
                              int max_q_len, int max_kv_len, const void* k_cache, const void* v_cache, int num_blocks,
                              void* out, float scale, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                              int window, void* workspace, size_t workspace_bytes, void* stream) {
  return attention_step(nullptr, q, cu_q_lens, ctx_lens, block_tables, max_blocks_per_seq, n_reqs, n_tokens,
                        max_q_len, max_kv_len, k_cache, v_cache, num_blocks, out, scale, n_q_heads, n_kv_heads,
                        head_dim, block_size, window, workspace, workspace_bytes, stream);
}

int cb_kv_append_paged_attention(const void* k_new, const void* v_new, const int64_t* slot_mapping, const void* q,
                                 const int32_t* cu_q_lens, const int32_t* ctx_lens, const int32_t* block_tables,
                                 int max_blocks_per_seq, int n_reqs, int n_tokens, int max_q_len, int max_kv_len,
                                 void* k_cache, void* v_cache, int num_blocks, void* out, float scale, int n_q_heads,
                                 int n_kv_heads, int head_dim, int block_size, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  const AppendArgs app{k_new, v_new, slot_mapping};
  return attention_step(&app, q, cu_q_lens, ctx_lens, block_tables, max_blocks_per_seq, n_reqs, n_tokens, max_q_len,
                        max_kv_len, k_cache, v_cache, num_blocks, out, scale, n_q_heads, n_kv_heads, head_dim,
                        block_size, 0, workspace, workspace_bytes, stream);
}

int cb_kv_append_paged_attention_window(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                        const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                                        const int32_t* block_tables, int max_blocks_per_seq, int n_reqs, int n_tokens,
                                        int max_q_len, int max_kv_len, void* k_cache, void* v_cache, int num_blocks,
                                        void* out, float scale, int n_q_heads, int n_kv_heads, int head_dim,
                                        int block_size, int window, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  const AppendArgs app{k_new, v_new, slot_mapping};
  return attention_step(&app, q, cu_q_lens, ctx_lens, block_tables, max_blocks_per_seq, n_reqs, n_tokens, max_q_len,
                        max_kv_len, k_cache, v_cache, num_blocks, out, scale, n_q_heads, n_kv_heads, head_dim,
                        block_size, window, workspace, workspace_bytes, stream);
}

int cb_last_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CB_ECUDA;
  StreamSlot* slot = stream_slot(s, false);
  if (!slot) return CB_OK;                       // nothing was launched on this stream
  unsigned int bits = 0;
  if (cudaMemcpy(&bits, &slot->err, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) return CB_ECUDA;
  if (bits) {
    const unsigned int zero = 0;
    if (cudaMemcpy(&slot->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return CB_ECUDA;
  }
  if (bits & CB_DEVERR_TIMEOUT) return CB_ETIMEOUT;
  if (bits) return CB_EDEVICE;
  return CB_OK;
}

const char* cb_strerror(int code) {
  switch (code) {
    case CB_OK: return "ok";
    case CB_EINVAL: return "invalid argument (size, shape, null or misaligned pointer)";
    case CB_ECUDA: return "CUDA runtime or launch error";
    case CB_EWORKSPACE: return "workspace too small";
    case CB_EDEVICE: return "kernel found bad metadata (block id, slot or length out of range)";
    case CB_ETIMEOUT: return "kernel wait timed out";
    case CB_ESTATE: return "state error or capacity exceeded (scheduler, or streams per device)";
    default: return "unknown error";
  }
}

int cb_hbm_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (!dst || !src || (bytes & 15) || !aligned16(dst) || !aligned16(src)) return CB_EINVAL;
  DeviceInfo di;
  if (!device_info(&di)) return CB_ECUDA;
  if (launch_hbm_copy(dst, src, bytes, di.n_sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) return CB_ECUDA;
  g_last_launches = 1;
  return CB_OK;
}

int cb_last_launch_count(void) { return g_last_launches; }

// ---------------------------------------------------------------- graphs
struct cb_graph {
  cudaGraphExec_t exec = nullptr;
  int device = -1;
};

cb_graph* cb_graph_create(void) { return new (std::nothrow) cb_graph(); }

void cb_graph_destroy(cb_graph* g) {
  if (!g) return;
  if (g->exec) (void)cudaGraphExecDestroy(g->exec);
  delete g;
}

int cb_graph_begin(cb_graph* g, void* stream) {
  if (!g || !stream) return CB_EINVAL;
  if (cudaStreamBeginCapture(static_cast<cudaStream_t>(stream), cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    (void)cudaGetLastError();
    return CB_ECUDA;
  }
  return CB_OK;
}

int cb_graph_end(cb_graph* g, void* stream) {
  if (!g || !stream) return CB_EINVAL;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGraph_t graph = nullptr;
  if (cudaStreamEndCapture(s, &graph) != cudaSuccess || !graph) {
    (void)cudaGetLastError();
    if (graph) (void)cudaGraphDestroy(graph);
    return CB_ECUDA;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGraphDestroy(graph);
    return CB_ECUDA;
  }
  if (g->exec && g->device == dev) {
    // the same kernels in the same order: new parameters in place, no instantiation
    cudaGraphExecUpdateResultInfo info;
    if (cudaGraphExecUpdate(g->exec, graph, &info) != cudaSuccess) {
      (void)cudaGetLastError();
      (void)cudaGraphExecDestroy(g->exec);
      g->exec = nullptr;
    }
  } else if (g->exec) {
    (void)cudaGraphExecDestroy(g->exec);
    g->exec = nullptr;
  }
  if (!g->exec) {
    if (cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) {
      (void)cudaGetLastError();
      g->exec = nullptr;
      (void)cudaGraphDestroy(graph);
      return CB_ECUDA;
    }
    g->device = dev;
  }
  (void)cudaGraphDestroy(graph);
  if (cudaGraphLaunch(g->exec, s) != cudaSuccess) {
    (void)cudaGetLastError();
    return CB_ECUDA;
  }
  return CB_OK;
}

}  // extern "C"
