/*
 * cbattn -- one continuous-batching attention step over a paged KV cache,
 * for NVIDIA GB300 (sm_103a).  Plain C ABI: pointers and sizes only.
 *
 * Sources (pages on KV caching and continuous batching):
 *  [CB]  "Continuous batching from first principles" (Chinese translation,
 *        news.myit.tw): sections Attention, KV cache, Chunked prefill,
 *        Continuous batching.
 *  [SM]  "AWS SageMaker 推理方案" (clvsit.github.io): section PagedAttention 批处理.
 *  [KVN] "KV Cache与Continuous Batching" notes (huajishe.fun): sections
 *        MQA/GQA, Continuous Batching原理, 调度策略.
 *  [KVB] "kv_cache" blog (klklkl10086.github.io): sections Batch Decode, 思想.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Element type of q, k_new, v_new, caches and out is bf16 (IEEE bfloat16,
 *    passed as void*).  Accumulation is fp32.
 *  - "device" pointers must point to memory of the current CUDA device; "host"
 *    pointers to ordinary (or pinned) host memory.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every GPU entry
 *    point only enqueues work and returns; nothing here synchronises except
 *    cb_last_error().
 *  - The caller owns every buffer.  Nothing allocates device memory per call.
 *  - KV cache layout (both K and V): [num_blocks][n_kv_heads][block_size][head_dim],
 *    row-major, so one (block, kv head) is block_size*head_dim contiguous values.
 *    Token position p of a request lives in physical block
 *    block_tables[r][p / block_size] at offset p % block_size ([SM] PagedAttention:
 *    logical blocks mapped to physical blocks by a block table).
 *  - Ragged batch ([CB] Continuous batching): requests are concatenated with no
 *    batch dimension; request r owns query rows cu_q_lens[r] .. cu_q_lens[r+1]-1.
 *    q and out are [n_tokens][n_q_heads][head_dim]; k_new and v_new are
 *    [n_tokens][n_kv_heads][head_dim].
 *  - GQA / MQA ([KVN] MQA/GQA): n_q_heads % n_kv_heads == 0 and query head h
 *    reads KV head h / (n_q_heads / n_kv_heads).
 *  - Supported shapes: head_dim 64 or 128; block_size 16;
 *    n_q_heads / n_kv_heads in {1, 2, 4, 8}; with head_dim 128 also 32 query
 *    heads on 2 KV heads (16 per group) or on 1 (MQA); n_reqs <= CB_MAX_REQS.
 *  - Return value: CB_OK (0) on success, a negative CB_E* code otherwise.  Size
 *    and pointer checks happen on the host before anything is enqueued; a
 *    rejected call enqueues nothing.
 *  - Per-stream state: the library keeps, in its own device memory, one slot
 *    per (device, stream) used -- an error word that the kernels launched on
 *    that stream report bad metadata or timeouts into (read and cleared by
 *    cb_last_error(stream)), and the block-tile launches' work counters.  Slots
 *    are handed out in order of first use, at most 4096 per device; a call on a
 *    further stream returns CB_ESTATE.  The first call on a device looks up the
 *    slots' device address (cudaGetSymbolAddress): make it before any stream
 *    capture.  Addresses are cached per device, so cudaDeviceReset is not
 *    supported while the library is in use.
 */
#ifndef CBATTN_H
#define CBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CB_OK 0
#define CB_EINVAL (-1)     /* bad size, unsupported shape, null pointer, misaligned pointer */
#define CB_ECUDA (-2)      /* a CUDA runtime/driver call or kernel launch failed */
#define CB_EWORKSPACE (-3) /* workspace too small (see cb_paged_attention_workspace_size) */
#define CB_EDEVICE (-4)    /* a kernel found bad metadata (block id or slot out of range) */
#define CB_ETIMEOUT (-5)   /* a kernel's bounded wait ran out; its outputs are undefined */
#define CB_ESTATE (-6)     /* scheduler: bad request id / state, or capacity exceeded */

#define CB_MAX_REQS 2048

/* ---------------------------------------------------------------- KV append
 * [CB] Chunked prefill ("store the KV states") and [SM] PagedAttention (new
 * tokens' KV written into the request's physical blocks): for every new token
 * t with slot_mapping[t] >= 0, for every KV head g,
 *     k_cache[slot / block_size][g][slot % block_size][:] = k_new[t][g][:]
 * and the same for v.  A negative slot skips the token.  The copy is bit-exact.
 *
 *  k_new, v_new   device, bf16 [n_tokens][n_kv_heads][head_dim]
 *  slot_mapping   device, int64 [n_tokens]
 *  k_cache,v_cache device, bf16 [num_blocks][n_kv_heads][block_size][head_dim]
 * Errors: CB_EINVAL (sizes, null pointers, pointers not 16-byte aligned),
 * CB_ECUDA (launch).  A slot >= num_blocks*block_size is not written; it sets
 * the device error word (cb_last_error then returns CB_EDEVICE).
 * Ordering: run it before cb_paged_attention of the same step on the same
 * stream, so that attention sees the new keys.
 */
int cb_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int n_tokens,
                 void* k_cache, void* v_cache, int num_blocks, int n_kv_heads, int head_dim,
                 int block_size, void* stream);

/* Copy whole KV blocks: for each pair i, block pairs[2i+1] of both caches
 * becomes a copy of block pairs[2i] (every KV head, K and V) -- the
 * copy-on-write of shared blocks that cb_sched_step_copies lists ([KVB] 思想:
 * blocks shared through the block table).  Run it on the step's stream before
 * the step's append, once per layer's caches.
 *  pairs    device, int32 [n_pairs][2] (src, dst); the dsts are distinct and
 *           none is a src of another pair (the pairs may be copied in any order)
 *  n_pairs  0 .. 65535
 *  k_cache, v_cache  device, bf16 cache layout above, 16-byte aligned
 * Bit-exact.  A block id outside [0, num_blocks) skips its pair and sets the
 * device error word (cb_last_error -> CB_EDEVICE).  Returns CB_OK, CB_EINVAL or
 * CB_ECUDA. */
int cb_copy_blocks(const int32_t* pairs, int n_pairs, void* k_cache, void* v_cache, int num_blocks,
                   int n_kv_heads, int head_dim, int block_size, void* stream);

/* ---------------------------------------------------------------- attention
 * One attention step ([CB] Attention, Chunked prefill, Continuous batching):
 * for request r with ctx = ctx_lens[r] stored tokens and q_len new tokens, new
 * token i (absolute position ctx + i) of query head h attends to keys
 * 0 .. ctx + i of KV head g = h / (n_q_heads / n_kv_heads), read through
 * block_tables[r]:
 *     out[t][h] = softmax_j(scale * q[t][h] . K[j]) . V[j],   j <= ctx + i.
 * The new tokens' keys must already be in the cache (cb_kv_append).  Requests
 * never see each other's keys (the block-diagonal ragged mask).
 * Requests with q_len > 1 run as 128-row tiles on the tensor cores.  Decode
 * requests (q_len == 1) are split over their KV blocks and the splits merged by
 * log-sum-exp: with head_dim 128 and 8 KV heads (or 32 query heads on 1 or 2)
 * on the tensor cores (128-row MMA tiles of whole physical blocks of every KV
 * head: one block of 8 heads, 4 of 2, 8 of 1; the merge runs on the whole grid
 * after a grid-wide barrier, so that launch is cooperative and fails with
 * CB_ECUDA if the device cannot hold one CTA on every SM at once), otherwise on
 * CUDA cores.  Everything is one kernel launch (plus, except on the block-tile
 * paths, a memset of the workspace's counters).  The block-tile launches keep
 * four work counters in the stream's library slot instead (see "Per-stream
 * state" above) and leave them at zero: calls on one stream are ordered; calls
 * that overlap on the GPU (unordered streams, concurrent replays of one
 * captured graph) must come from different streams.
 *
 *  q              device, bf16 [n_tokens][n_q_heads][head_dim]
 *  cu_q_lens      device, int32 [n_reqs + 1], cu_q_lens[0] = 0, non-decreasing,
 *                 cu_q_lens[n_reqs] = n_tokens
 *  ctx_lens       device, int32 [n_reqs], >= 0
 *  block_tables   device, int32 [n_reqs][max_blocks_per_seq]; entries past
 *                 ceil((ctx + q_len) / block_size) are never read
 *  max_q_len      host int, >= every q_len (1 selects the decode-only kernel)
 *  max_kv_len     host int, >= every ctx + q_len; sizes the split-K workspace
 *  k_cache,v_cache device, bf16 cache layout above
 *  out            device, bf16 [n_tokens][n_q_heads][head_dim]
 *  scale          multiplies q.k before the softmax (1/sqrt(head_dim) in the
 *                 [KVB] Batch Decode listing)
 *  workspace      device, >= cb_paged_attention_workspace_size(...) bytes,
 *                 16-byte aligned; contents need no initialisation
 * Errors: CB_EINVAL, CB_EWORKSPACE, CB_ECUDA.  Device-side metadata checks
 * (block ids >= num_blocks, lengths beyond the table) skip the bad access and
 * set the error word (cb_last_error -> CB_EDEVICE).
 */
int cb_paged_attention(const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                       const int32_t* block_tables, int max_blocks_per_seq, int n_reqs, int n_tokens,
                       int max_q_len, int max_kv_len, const void* k_cache, const void* v_cache,
                       int num_blocks, void* out, float scale, int n_q_heads, int n_kv_heads,
                       int head_dim, int block_size, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Bytes of workspace cb_paged_attention needs for these sizes (0 on invalid
 * sizes).  Pure host function.  With max_q_len > 1 on the block-tile shapes (8
 * KV heads, head_dim 128, G >= 2) it includes ~43 MB for the partial results of
 * prefill tile pairs that the launch cuts at CTA boundaries to balance its CTAs.
 * A workspace that is smaller by up to that region is still accepted; the launch
 * then keeps every tile pair whole. */
size_t cb_paged_attention_workspace_size(int n_reqs, int n_tokens, int max_q_len, int max_kv_len,
                                         int n_q_heads, int n_kv_heads, int head_dim, int block_size);

/* ---------------------------------------------------------------- append + attention
 * One whole step of a layer ([CB] Chunked prefill: the chunk's K/V states are
 * stored, then its queries attend to the cached prefix and to themselves):
 * the same result as cb_kv_append(k_new, v_new, slot_mapping, n_tokens, ...)
 * followed by cb_paged_attention(q, ...) on `stream`, with the arguments of
 * both (n_tokens, the cache, num_blocks and the shape are shared; k_cache and
 * v_cache are written).  Token t's new rows go to slot_mapping[t] before any
 * request reads the cache, so every new token attends to its own key.
 * Where the attention launch is cooperative (8 KV heads, head_dim 128, G >= 2)
 * its CTAs store the rows themselves and meet at a grid-wide counter in the
 * workspace before the first cache read: one kernel launch for the step.
 * Other shapes run the two kernels back to back.
 *  k_new, v_new   device, bf16 [n_tokens][n_kv_heads][head_dim], 16-byte aligned
 *  slot_mapping   device, int64 [n_tokens]; < 0 skips the token
 *  workspace      cb_paged_attention_workspace_size(...) bytes, as for
 *                 cb_paged_attention
 * Errors: those of the two calls; a slot >= num_blocks * block_size is skipped
 * and reported like a bad block id (cb_last_error -> CB_EDEVICE).
 */
int cb_kv_append_paged_attention(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                 const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                                 const int32_t* block_tables, int max_blocks_per_seq, int n_reqs,
                                 int n_tokens, int max_q_len, int max_kv_len, void* k_cache,
                                 void* v_cache, int num_blocks, void* out, float scale, int n_q_heads,
                                 int n_kv_heads, int head_dim, int block_size, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- rolling window
 * [KVB] "Rolling KV Cache" (a heading whose body is missing from the page).
 * Reading: a rolling cache keeps each request's W most recent keys, so new
 * token i of request r (absolute position p = ctx + i) attends to the keys at
 * positions max(0, p - W + 1) .. p only:
 *     out[t][h] = softmax_j(scale * q[t][h] . K[j]) . V[j],   p - W < j <= p.
 * Same arguments, layouts, workspace and errors as cb_paged_attention (and
 * cb_kv_append_paged_attention), plus
 *  window   W >= 1 (0: no window, the same as the calls without it; < 0:
 *           CB_EINVAL).
 * Decodes read only the blocks from the one holding position ctx + 1 - W on;
 * prefill tiles skip key tiles that no query of the tile can see.  Block-table
 * entries before a request's window are never read, so a caller may already
 * have released those blocks (cb_sched_set_window does) and left any value
 * there.  The workspace size query is the same. */
int cb_paged_attention_window(const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                              const int32_t* block_tables, int max_blocks_per_seq, int n_reqs, int n_tokens,
                              int max_q_len, int max_kv_len, const void* k_cache, const void* v_cache, int num_blocks,
                              void* out, float scale, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                              int window, void* workspace, size_t workspace_bytes, void* stream);

int cb_kv_append_paged_attention_window(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                        const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                                        const int32_t* block_tables, int max_blocks_per_seq, int n_reqs, int n_tokens,
                                        int max_q_len, int max_kv_len, void* k_cache, void* v_cache, int num_blocks,
                                        void* out, float scale, int n_q_heads, int n_kv_heads, int head_dim,
                                        int block_size, int window, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* ---------------------------------------------------------------- no-allocation variant
 * The pages have no counterpart: this exists for callers that cannot allocate
 * device memory when they run a step -- hosts whose device memory is owned by
 * an arena or custom allocator that this library cannot see (a plugin may not
 * call cudaMalloc behind its host's back), and latency-bound serving loops that
 * forbid allocation because it can synchronise the device and has unbounded
 * latency.
 *
 * Same arguments, semantics and errors as cb_paged_attention, minus the
 * workspace: the scratch (split-K partials and counters) comes from one
 * library-owned device array of CB_NOALLOC_SCRATCH_BYTES, held on every GPU that
 * loads the library until the process exits.  Nothing is allocated per call.
 *  - Sizes whose smallest accepted workspace exceeds CB_NOALLOC_SCRATCH_BYTES
 *    are rejected with CB_EWORKSPACE before anything is enqueued.
 *  - It uses as much of the array as cb_paged_attention_workspace_size asks
 *    for, so a step whose full workspace fits is planned exactly as
 *    cb_paged_attention plans it with that workspace (the same outputs, bit
 *    for bit).  A larger step is run with the array alone: without room for
 *    the balanced prefill's partial results the launch keeps prefill tile
 *    pairs whole, and its outputs then differ within rounding.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make that
 *    first call before any stream capture.
 *  - The counters that must start at zero are cleared by every call (an async
 *    memset on `stream`) or, on the block-tile paths, kept at zero in the
 *    library's per-stream slots; the partial results are fully rewritten.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents: calls that may overlap on the GPU (different streams without
 *    ordering between them) race and give undefined results.  Serialise them,
 *    e.g. by issuing them on one stream.
 */
#define CB_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

int cb_paged_attention_noalloc(const void* q, const int32_t* cu_q_lens, const int32_t* ctx_lens,
                               const int32_t* block_tables, int max_blocks_per_seq, int n_reqs, int n_tokens,
                               int max_q_len, int max_kv_len, const void* k_cache, const void* v_cache,
                               int num_blocks, void* out, float scale, int n_q_heads, int n_kv_heads,
                               int head_dim, int block_size, void* stream);

/* Synchronise `stream`, then read and clear that stream's error word: the bad
 * metadata or timeouts reported by kernels this library launched on `stream`
 * (never another stream's).
 * Returns CB_OK, CB_EDEVICE, CB_ETIMEOUT or CB_ECUDA. */
int cb_last_error(void* stream);

/* Static description of an error code (never NULL). */
const char* cb_strerror(int code);

/* ---------------------------------------------------------------- measurement
 * Device-to-device copy of `bytes` (multiple of 16, both pointers 16-byte
 * aligned) with a plain streaming kernel: the HBM copy roofline probe. */
int cb_hbm_copy(void* dst, const void* src, size_t bytes, void* stream);

/* Number of kernels the calling thread's last successful GPU call of this
 * library enqueued (for launch accounting in benchmarks). */
int cb_last_launch_count(void);

/* ---------------------------------------------------------------- graphs
 * A serving loop's launches (for instance the attention step of every layer of
 * one iteration) recorded and replayed as one CUDA graph.  Kernels of a graph
 * follow one another ~0.8 us after their predecessor ends, against ~2.8 us
 * for separate stream launches (measured on GB300 with these launches'
 * shapes), which matters for short steps.
 *   cb_graph_begin(g, stream)  starts capturing `stream` (thread-local capture
 *                              mode): every call of this library on `stream`
 *                              from this thread until cb_graph_end is recorded,
 *                              not run.  `stream` must not be NULL (the legacy
 *                              default stream cannot be captured).
 *   cb_graph_end(g, stream)    ends the capture and launches the recorded
 *                              work on `stream`.  The graph object keeps one
 *                              instantiated graph: it is updated in place when
 *                              the new recording has the same shape of work
 *                              (the same kernels in the same order, parameters
 *                              free to change), otherwise instantiated anew.
 * Arguments are captured by value; the buffers they point to are read when the
 * graph runs.  A shape's first call on a device must run outside a capture
 * (it sets up the library's per-device state); cb_last_error synchronises and
 * must not be called while `stream` is being captured.  Errors of the
 * recorded kernels reach cb_last_error(stream) as for direct calls.  A graph
 * object may be reused for any number of begin/end pairs, on one thread at a
 * time.
 * cb_graph_create returns NULL when out of memory.  begin/end return CB_OK,
 * CB_EINVAL (NULL graph or stream) or CB_ECUDA (the capture, update,
 * instantiation or launch failed; a failed capture is ended and discarded). */
typedef struct cb_graph cb_graph;
cb_graph* cb_graph_create(void);
void cb_graph_destroy(cb_graph* g);
int cb_graph_begin(cb_graph* g, void* stream);
int cb_graph_end(cb_graph* g, void* stream);

/* ---------------------------------------------------------------- host metadata
 * Slot mapping of a step, on the host ([SM] PagedAttention: block table lookup):
 * for request r and new token i, slot = table[r][(ctx+i) / bs] * bs + (ctx+i) % bs.
 *  q_lens, ctx_lens  host int32 [n_reqs]; block_tables host int32
 *  [n_reqs][max_blocks_per_seq]; slot_mapping_out host int64 [sum q_lens].
 * Returns CB_OK or CB_EINVAL (a needed table entry is negative or the table is
 * too short). */
int cb_build_slot_mapping(const int32_t* q_lens, const int32_t* ctx_lens, const int32_t* block_tables,
                          int max_blocks_per_seq, int n_reqs, int block_size, int64_t* slot_mapping_out);

/* ---------------------------------------------------------------- scheduler
 * FCFS iteration-level continuous-batching scheduler with a paged block
 * allocator and recompute preemption ([KVN] Continuous Batching原理 and 调度策略;
 * [CB] Chunked prefill; [SM] PagedAttention: a block is taken only when the
 * request's last block is full).  Host only; it produces the metadata of each
 * step and never touches the GPU.  Rules, per step:
 *   arrivals join the waiting queue; running decodes (one position left) get 1
 *   token each in arrival order, preempting the latest-arrived unscheduled
 *   running request when no block is free; running prefills get
 *   min(remaining, budget left) tokens, preempting only later-arrived
 *   unscheduled requests and otherwise cutting the chunk to what fits; waiting
 *   requests are admitted in arrival order while budget remains, stopping at the
 *   first that gets no token or was preempted in this step.  A preempted request
 *   frees all blocks, keeps its produced tokens and later recomputes them.
 *   The free list is FIFO, seeded by `free_order`.
 * The opaque handle is owned by the caller and freed by cb_sched_destroy.
 */
typedef struct cb_sched cb_sched;

/* free_order: host int32 [num_blocks], a permutation of 0..num_blocks-1 (the
 * initial free-list order).  max_batch: capacity of one step's batch (requests). */
cb_sched* cb_sched_create(int num_blocks, int block_size, int token_budget, int max_batch,
                          const int32_t* free_order);
void cb_sched_destroy(cb_sched* s);

/* Padded batching instead of continuous batching -- the baselines of [CB]
 * Continuous batching (batched generation: prompts padded on the left to the
 * batch's longest, the batch run until its longest generation ends) and [SM]
 * 动态批处理 (dynamic batching: the requests that arrive within a waiting window,
 * or until the batch is full, run as one batch).  From then on cb_sched_step
 * plans padded batches:
 *  - a batch forms only when none is running, from the waiting requests in
 *    arrival order, at most batch_size of them, once batch_size are waiting,
 *    no further request will arrive, or (max_wait >= 0, dynamic batching) the
 *    oldest has waited max_wait steps since its arrival; max_wait -1: static
 *    batching, which waits for a full batch; the batch is cut from its end
 *    until its padded length fits the pool;
 *  - its first step is the padded prefill: every request processes n_max
 *    positions (the longest prompt; the first n_max - prompt_len are pads) at
 *    ctx 0; then one position per request per step (ctx n_max, n_max + 1, ...)
 *    until the longest output is done, finished requests decoding pads;
 *  - blocks are taken on demand and all return when the batch ends; prefix
 *    groups, preemption and the rolling window do not apply.
 * The token budget given to cb_sched_create is then only the capacity of the
 * step's slot_mapping array (a padded prefill needs batch_size x the longest
 * prompt); a step that does not fit returns CB_ESTATE.
 * batch_size 1 .. max_batch.  Call before the first cb_sched_step.  Returns
 * CB_OK or CB_EINVAL. */
int cb_sched_set_batching(cb_sched* s, int batch_size, int max_wait);

/* Real (not pad) tokens of the last cb_sched_step: all of them under
 * continuous batching; under padded batching the prompt tokens of a padded
 * prefill and, in a decode step, one per request still generating. */
long long cb_sched_last_real_tokens(const cb_sched* s);

/* Rolling KV cache ([KVB] "Rolling KV Cache"; reading: a query at position p
 * sees keys p - window + 1 .. p, as in cb_paged_attention_window): at the end
 * of every step each running request lets go of the blocks that its next
 * query can no longer see (all positions before stored - window + 1); their
 * block-table entries become -1, which the windowed attention calls never
 * read.  A request publishes its shared prefix only while it holds all of it.
 * window 0 (the default): no window.  Call before the first cb_sched_step.
 * Returns CB_OK or CB_EINVAL (null handle, window < 0, or steps already run). */
int cb_sched_set_window(cb_sched* s, int window);

/* Register a request (ids are assigned 0, 1, 2, ... in call order; calls must
 * come in non-decreasing arrival_step order).  Returns the id or CB_EINVAL. */
int cb_sched_add_request(cb_sched* s, int arrival_step, int prompt_len, int output_len);

/* The same for a request whose first prefix_len prompt tokens are those of
 * every request of prefix group `group` (a shared system prompt, [KVN]
 * 与Prefix Caching的结合): their K/V are computed once and the blocks holding
 * them are shared ([KVB] 思想: block tables point at the same blocks).
 * group >= 0 with 1 <= prefix_len < prompt_len, one prefix_len per group;
 * group -1 with prefix_len 0 is a request with no shared prefix.
 * Scheduling with prefixes (applied within the rules above):
 *  - after a step, the first request of a group whose stored tokens cover the
 *    prefix publishes it (its blocks over positions [0, prefix_len) gain a
 *    reference; blocks return to the free list when no request or published
 *    prefix holds them);
 *  - a request of the group admitted with nothing stored starts with the
 *    published positions stored: whole blocks shared, a partial last block
 *    copied first into a block of its own (copy-on-write); with no block free
 *    for that copy it waits, like any request that finds no room;
 *  - a running request that needs a block when none is free first drops
 *    published prefixes, oldest first, and only then preempts.
 * Returns the id or CB_EINVAL. */
int cb_sched_add_request_prefix(cb_sched* s, int arrival_step, int prompt_len, int output_len, int group,
                                int prefix_len);

/* Run one scheduling step and write its metadata into caller-owned host arrays:
 *  req_ids [max_batch], q_lens [max_batch], ctx_lens [max_batch],
 *  cu_q_lens [max_batch + 1], block_tables [max_batch][max_blocks_per_seq]
 *  (unused entries -1), slot_mapping [token_budget] int64.
 * *n_reqs_out / *n_tokens_out receive the batch size and token count.  Then
 * advances every scheduled request as if the forward pass had run.  Returns the
 * number of requests preempted in this step (>= 0), or CB_ESTATE when the batch
 * does not fit the arrays. */
int cb_sched_step(cb_sched* s, int32_t* req_ids, int32_t* q_lens, int32_t* ctx_lens, int32_t* cu_q_lens,
                  int32_t* block_tables, int max_blocks_per_seq, int64_t* slot_mapping, int* n_reqs_out,
                  int* n_tokens_out);

/* The block copies (copy-on-write of shared partial blocks) of the last
 * cb_sched_step: pairs (src, dst) of block ids into host int32 [2 * max_pairs].
 * They must run on the device (cb_copy_blocks, every layer's cache) before that
 * step's append.  Returns the number of pairs, CB_ESTATE if more than
 * max_pairs, or CB_EINVAL. */
int cb_sched_step_copies(const cb_sched* s, int32_t* pairs, int max_pairs);

/* 1 when no request is pending, waiting or running. */
int cb_sched_done(const cb_sched* s);
/* Free blocks right now. */
int cb_sched_free_blocks(const cb_sched* s);
/* Per-request state: produced tokens, stored tokens, preemption count, and
 * state (0 pending, 1 waiting, 2 running, 3 finished, 4 rejected). */
int cb_sched_request_info(const cb_sched* s, int req_id, int* produced, int* stored, int* preemptions,
                          int* state);

/* KV-cache memory right now (after the last step), against a contiguous cache
 * that reserves max_seq_len positions per request for its whole life ([KVB]
 * 连续内存分配: TraditionalKVCache) where the paged pool takes a block only when
 * the last one is full ([SM] PagedAttention 批处理).  out (host int64 [4]):
 *  out[0] running requests,
 *  out[1] tokens whose K/V the running requests have stored and still hold
 *         (a rolling window lets go of whole blocks),
 *  out[2] token slots in the blocks taken from the pool (held blocks x block_size),
 *  out[3] token slots a contiguous cache would reserve (out[0] x max_seq_len).
 * Paged waste = 1 - out[1] / out[2]; contiguous waste = 1 - out[1] / out[3].
 * Returns CB_OK, or CB_EINVAL (null handle or out, max_seq_len < 1). */
int cb_sched_kv_memory(const cb_sched* s, int max_seq_len, int64_t* out);

#ifdef __cplusplus
}
#endif
#endif /* CBATTN_H */
