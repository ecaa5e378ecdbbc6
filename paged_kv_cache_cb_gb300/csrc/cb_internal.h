// Internal constants and launch interfaces shared by the library's translation
// units.  Not part of the public C ABI (that is include/cbattn.h).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace cb {

// Device error-word bits.
constexpr unsigned CB_DEVERR_TIMEOUT = 1u;   // a bounded mbarrier wait ran out
constexpr unsigned CB_DEVERR_BADBLOCK = 2u;  // block-table entry outside [0, num_blocks)
constexpr unsigned CB_DEVERR_BADSLOT = 4u;   // slot outside the cache
constexpr unsigned CB_DEVERR_BADLEN = 8u;    // lengths inconsistent with the table / launch

// Longest a kernel waits on one mbarrier phase before giving up (wall clock).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

constexpr int kBlockSize = 16;     // tokens per physical KV block
constexpr int kTileM = 128;        // query rows per tensor-core tile
constexpr int kTileN = 128;        // keys per tensor-core tile
constexpr int kMaxReqs = 2048;     // requests per step (plan arrays live in shared memory)
constexpr int kMaxSplitBlocks = 32;  // decode split size limit (one warp-wide table load)
constexpr int kMaxDecodeGrid = 160;  // CTAs of the block-tile decode launches (at most one per SM)

// Everything a step's attention kernels read besides the tensor maps.
struct StepParams {
  const uint16_t* q;            // bf16 [n_tokens][Hq][A]
  const int32_t* cu_q_lens;     // [n_reqs + 1]
  const int32_t* ctx_lens;      // [n_reqs]
  const int32_t* block_tables;  // [n_reqs][max_blocks_per_seq]
  uint16_t* out;                // bf16 [n_tokens][Hq][A]
  int max_blocks_per_seq;
  int max_kv_len;               // caller's bound on ctx + q_len (sizes the partial buffers)
  int n_reqs;
  int n_tokens;
  int num_blocks;
  int n_q_heads;
  int n_kv_heads;
  float scale_log2;             // scale * log2(e): scores kept in the base-2 domain
  int window;                   // rolling window W: a query at position p sees keys p-W+1..p (0: no window)
  int split_blocks;             // decode split size (blocks)
  int max_splits_total;         // capacity of the partial buffers (splits)
  // workspace
  int* counters;                // [n_reqs * Hkv] split arrival counters (zeroed per call)
  int* queue;                   // [4] work counters (zeroed per call)
  float* part_ml;               // [max_splits_total * Hq * 2] (max, sum) per split and head
  float* part_acc;              // [max_splits_total * Hq * A] unnormalised outputs per split
  unsigned int* err;            // the launching stream's error word
};

// The step's new K/V rows when the block-tile launches store them themselves
// (n_tokens == 0: they do not): the launch first stores token t's rows at
// slots[t], then waits for every CTA's stores (StepParams::queue[2]) before its
// first cache read.
struct AppendParams {
  const uint4* k_new;           // bf16 [n_tokens][Hkv][A] as 16-byte pieces
  const uint4* v_new;
  const int64_t* slots;         // [n_tokens]
  uint4* k_cache;               // the caches that the tensor maps read
  uint4* v_cache;
  int n_tokens;
};

// Partial results of prefill tile pairs cut at CTA boundaries (the mixed
// launch's balanced prefill; part == nullptr: whole pairs round robin).  Slot
// 2b holds CTA b's first piece, 2b + 1 its last: [2 * 128 rows][A] unnormalised
// O, then [2 * 128 rows][2] (running max in base 2 with the scale, row sum).
struct PrefillSplit {
  float* part;
  int slots;                    // capacity (slots)
};
constexpr int kPreRows = 2 * kTileM;   // rows of a tile pair

// Workspace carving (byte offsets), shared by the size query and the launcher.
struct WorkspaceLayout {
  size_t counters, queue, pre_part, part_ml, part_acc, total;
  int max_splits_total;
  int pre_slots;                // prefill partial slots (0: none)
};
// prefill_split: room for the balanced prefill's partial results.
WorkspaceLayout workspace_layout(int n_reqs, int max_kv_len, int n_q_heads, int n_kv_heads, int head_dim,
                                 int split_blocks, bool prefill_split = false);
size_t workspace_min_bytes(int n_reqs, int n_tokens, int max_q_len, int max_kv_len, int n_q_heads, int n_kv_heads,
                           int head_dim, int block_size);
// L with as many split partials as `bytes` of workspace hold (never fewer).
WorkspaceLayout workspace_layout_for_bytes(const WorkspaceLayout& L, size_t bytes, int n_reqs, int n_q_heads,
                                           int n_kv_heads, int head_dim);
int choose_split_blocks(int n_reqs, int max_kv_len, int n_kv_heads, int n_sms);
// Dynamic shared-memory opt-in of `kernel` on the current device (set once per
// device and kernel).
cudaError_t opt_in_smem(const void* kernel, int bytes);

// Kernel launchers (defined in the .cu files); return a cudaError_t.
cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int64_t* slots, int n_tokens,
                             void* k_cache, void* v_cache, int num_blocks, int n_kv_heads, int head_dim,
                             unsigned int* err, cudaStream_t stream);
cudaError_t launch_decode(const StepParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int head_dim,
                          int group, int n_sms, cudaStream_t stream);
// Decode with 128-row tensor-core tiles of whole blocks (8 KV heads: one block;
// 2 or 1 KV heads with 32 query heads: 4 or 8 blocks); the cache maps must have
// boxes of one block (16 x Hkv rows) and the q map a box of one token's Hq heads.  It
// cuts the work into equal pieces itself (p.split_blocks is not used); the
// partial buffers must hold n_reqs * (ceil(max blocks / 8) + 1) splits.
cudaError_t launch_decode_tcb(const StepParams& p, const AppendParams& ap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& qmap, int group, int n_sms,
                              cudaStream_t stream);
// Mixed prefill + decode step.  maps: K, V with 16-row boxes, the prefill q
// map, then (block_tiles: the block-tile decode phase) K, V with 128-row boxes
// and the decode q map.
cudaError_t launch_mixed(const StepParams& p, const AppendParams& ap, const PrefillSplit& ps, const CUtensorMap* maps,
                         bool block_tiles, int head_dim, int group, int n_sms, cudaStream_t stream);
cudaError_t launch_copy_blocks(const int32_t* pairs, int n_pairs, void* k_cache, void* v_cache, int num_blocks,
                               int n_kv_heads, int head_dim, unsigned int* err, cudaStream_t stream);
cudaError_t launch_hbm_copy(void* dst, const void* src, size_t bytes, int n_sms, cudaStream_t stream);

}  // namespace cb
