// FCFS iteration-level continuous-batching scheduler with a paged block
// allocator and recompute preemption.  Host only; produces each step's
// attention metadata (request order, new tokens, stored tokens, block tables,
// slot mapping).
//
// [KVN] Continuous Batching原理: every iteration retires finished requests,
// admits new ones and steps every running request.  [KVN] 调度策略: FCFS order,
// preemption when memory runs out.  [CB] Chunked prefill / Continuous batching:
// prompts may run in chunks, and prefill and decode tokens share one ragged
// batch bounded by a token budget.  [SM] PagedAttention: a request takes a new
// block only when its last block is full.
//
// The per-step rules (the pages print no algorithm; this is the plain FCFS
// reading):
//  a. arrivals join the waiting queue (kept in arrival order);
//  b. running requests with one position left (decoding) get 1 token each in
//     arrival order; with no free block, the latest-arrived running request with
//     nothing scheduled this step is preempted (possibly the request itself);
//  c. running requests still prefilling get min(remaining, budget left) tokens,
//     preempting only later-arrived unscheduled requests, else cut to what fits;
//  d. waiting requests are admitted in order while budget is left, stopping at
//     the first one that gets no token or was preempted in this step.
// A preempted request frees all blocks, keeps its produced tokens and re-runs
// prompt + produced tokens as a prefill later.  Free blocks are FIFO.
//
// Shared prompt prefixes ([KVN] 与Prefix Caching的结合: requests that share a
// system prompt compute its K/V once; [KVB] 思想: blocks are shared by pointing
// several block tables at them).  Blocks carry reference counts (requests and
// published prefixes holding them) and return to the free list at zero.
//  e. after a step, the first request of a prefix group whose stored tokens
//     cover the group's prefix publishes it: the blocks holding positions
//     [0, prefix) gain a reference;
//  f. a request of the group admitted with nothing stored takes the published
//     blocks: whole blocks by reference; a last, partial block is copied into a
//     block of its own first (copy-on-write: the request will write its own
//     tokens into that block), the copy listed for the caller to run before the
//     step's append (with no block free for the copy it is not admitted yet,
//     like any request that finds no room).  It starts with the shared
//     positions stored;
//  g. when a running request needs a block and none is free, published
//     prefixes are dropped (oldest first) before a request is preempted.
//  h. with a rolling window W (cb_sched_set_window), at the end of each step a
//     running request lets go of the blocks whose positions all lie before
//     stored - W + 1 (its next query cannot see them); their table entries
//     become -1.  A request publishes its prefix only while it holds all of it.
// The request that published a prefix keeps writing its own positions into
// the shared partial block; those slots lie past the prefix, and every other
// holder reads them from its own copy.
#include <algorithm>
#include <deque>
#include <map>
#include <vector>

#include "../../include/cbattn.h"

namespace {

enum State { kPending = 0, kWaiting = 1, kRunning = 2, kFinished = 3, kRejected = 4 };

struct Req {
  int rid, arrival, prompt, output;
  int group = -1, prefix = 0;          // shared prompt prefix: group and its length (0: none)
  int produced = 0, stored = 0, state = kPending, preemptions = 0;
  std::vector<int> blocks;
  int remaining() const { return prompt + produced - stored; }
};

// A published prefix: the blocks holding positions [0, tokens) of its group.
struct Prefix {
  std::vector<int> blocks;
  int tokens = 0;
  int order = 0;                       // publication order (the oldest is dropped first)
};

struct Sched {
  int num_blocks, bs, budget, max_batch;
  int window = 0;                      // rolling window (0: none)
  // padded batching (cb_sched_set_batching): batch size (0: continuous
  // batching), max wait in steps (-1: static), the running batch (arrival
  // order), its longest prompt and output, the steps it has run
  int pad_b = 0, pad_wait = -1;
  std::vector<int> batch;
  int n_max = 0, o_max = 0, k = 0;
  long long last_real = 0;             // real (not pad) tokens of the last step
  std::deque<int> free_list;
  std::vector<int> ref;                // holders of each block
  std::map<int, Prefix> prefixes;      // group -> published prefix
  std::vector<int> copies;             // this step's copy-on-write pairs (src, dst)
  std::map<int, int> group_prefix;     // prefix length of each group seen
  int n_published = 0;
  std::vector<Req> reqs;
  size_t next_pending = 0;
  std::vector<int> waiting;   // request ids, ascending
  std::vector<int> running;   // request ids, ascending
  int now = 0;

  int blocks_for(long long n) const { return (int)((n + bs - 1) / bs); }

  int take() {
    const int b = free_list.front();
    free_list.pop_front();
    ref[b] = 1;
    return b;
  }
  void drop(int b) {
    if (--ref[b] == 0) free_list.push_back(b);
  }
  void grow(Req& r, long long n_tokens) {
    const int need = blocks_for(n_tokens) - (int)r.blocks.size();
    for (int i = 0; i < need; ++i) r.blocks.push_back(take());
  }
  void release(Req& r) {
    for (int b : r.blocks)
      if (b >= 0) drop(b);
    r.blocks.clear();
  }
  // h. rolling window: let go of the blocks r's next query cannot see
  void slide(Req& r) {
    if (window <= 0) return;
    const long long first_seen = (long long)r.stored - window + 1;
    const int n = (int)std::min<long long>((long long)r.blocks.size(), std::max(0LL, first_seen) / bs);
    for (int i = 0; i < n; ++i)
      if (r.blocks[i] >= 0) {
        drop(r.blocks[i]);
        r.blocks[i] = -1;
      }
  }
  // g. drop the oldest published prefix; false when there is none
  bool evict_prefix() {
    auto oldest = prefixes.end();
    for (auto it = prefixes.begin(); it != prefixes.end(); ++it)
      if (oldest == prefixes.end() || it->second.order < oldest->second.order) oldest = it;
    if (oldest == prefixes.end()) return false;
    for (int b : oldest->second.blocks) drop(b);
    prefixes.erase(oldest);
    return true;
  }
  // e. publish r's prefix if its group has none and r has stored it
  void publish(const Req& r) {
    if (r.group < 0 || r.prefix <= 0 || r.stored < r.prefix || prefixes.count(r.group)) return;
    for (int i = 0; i < blocks_for(r.prefix); ++i)
      if (r.blocks[i] < 0) return;       // part of it already left the window
    Prefix px;
    px.tokens = r.prefix;
    px.order = n_published++;
    for (int i = 0; i < blocks_for(r.prefix); ++i) {
      px.blocks.push_back(r.blocks[i]);
      ref[r.blocks[i]]++;
    }
    prefixes[r.group] = px;
  }
  // f. attach `share` positions of prefix px to r (nothing stored yet); cow:
  // the last shared block is partial and a free block is there for its copy
  void attach(Req& r, const Prefix& px, int share, bool cow) {
    const int whole = share / bs;
    for (int i = 0; i < whole; ++i) {
      r.blocks.push_back(px.blocks[i]);
      ref[px.blocks[i]]++;
    }
    if (cow) {
      const int b = take();
      copies.push_back(px.blocks[whole]);
      copies.push_back(b);
      r.blocks.push_back(b);
    }
    r.stored = share;
  }
  static void insert_sorted(std::vector<int>& v, int rid) { v.insert(std::lower_bound(v.begin(), v.end(), rid), rid); }
  static void erase(std::vector<int>& v, int rid) {
    auto it = std::lower_bound(v.begin(), v.end(), rid);
    if (it != v.end() && *it == rid) v.erase(it);
  }
  void preempt(int rid) {
    Req& r = reqs[rid];
    release(r);
    r.stored = 0;
    r.state = kWaiting;
    r.preemptions++;
    erase(running, rid);
    insert_sorted(waiting, rid);
  }
};

}  // namespace

struct cb_sched {
  Sched s;
};

extern "C" {

cb_sched* cb_sched_create(int num_blocks, int block_size, int token_budget, int max_batch, const int32_t* free_order) {
  if (num_blocks <= 0 || block_size <= 0 || token_budget <= 0 || max_batch <= 0 || !free_order) return nullptr;
  std::vector<char> seen(num_blocks, 0);
  for (int i = 0; i < num_blocks; ++i) {
    const int b = free_order[i];
    if (b < 0 || b >= num_blocks || seen[b]) return nullptr;
    seen[b] = 1;
  }
  cb_sched* h = new cb_sched();
  h->s.num_blocks = num_blocks;
  h->s.bs = block_size;
  h->s.budget = token_budget;
  h->s.max_batch = max_batch;
  h->s.ref.assign(num_blocks, 0);
  for (int i = 0; i < num_blocks; ++i) h->s.free_list.push_back(free_order[i]);
  return h;
}

void cb_sched_destroy(cb_sched* h) { delete h; }

int cb_sched_set_batching(cb_sched* h, int batch_size, int max_wait) {
  if (!h || batch_size < 1 || batch_size > h->s.max_batch || max_wait < -1 || h->s.now != 0) return CB_EINVAL;
  h->s.pad_b = batch_size;
  h->s.pad_wait = max_wait;
  return CB_OK;
}

long long cb_sched_last_real_tokens(const cb_sched* h) { return h ? h->s.last_real : 0; }

int cb_sched_set_window(cb_sched* h, int window) {
  if (!h || window < 0 || h->s.now != 0) return CB_EINVAL;
  h->s.window = window;
  return CB_OK;
}

int cb_sched_add_request_prefix(cb_sched* h, int arrival_step, int prompt_len, int output_len, int group,
                                int prefix_len) {
  if (!h || arrival_step < 0 || prompt_len < 1 || output_len < 1) return CB_EINVAL;
  if (group < -1 || (group >= 0 && (prefix_len < 1 || prefix_len >= prompt_len)) || (group < 0 && prefix_len != 0))
    return CB_EINVAL;
  Sched& s = h->s;
  if (!s.reqs.empty() && arrival_step < s.reqs.back().arrival) return CB_EINVAL;
  if (group >= 0) {                    // one prefix length per group
    auto it = s.group_prefix.find(group);
    if (it != s.group_prefix.end() && it->second != prefix_len) return CB_EINVAL;
    s.group_prefix[group] = prefix_len;
  }
  Req r;
  r.rid = (int)s.reqs.size();
  r.arrival = arrival_step;
  r.prompt = prompt_len;
  r.output = output_len;
  r.group = group;
  r.prefix = group >= 0 ? prefix_len : 0;
  s.reqs.push_back(r);
  return r.rid;
}

int cb_sched_add_request(cb_sched* h, int arrival_step, int prompt_len, int output_len) {
  return cb_sched_add_request_prefix(h, arrival_step, prompt_len, output_len, -1, 0);
}

int cb_sched_step_copies(const cb_sched* h, int32_t* pairs, int max_pairs) {
  if (!h || max_pairs < 0 || (max_pairs > 0 && !pairs)) return CB_EINVAL;
  const int n = (int)h->s.copies.size() / 2;
  if (n > max_pairs) return CB_ESTATE;
  for (int i = 0; i < 2 * n; ++i) pairs[i] = h->s.copies[i];
  return n;
}

int cb_sched_done(const cb_sched* h) {
  if (!h) return 1;
  const Sched& s = h->s;
  return s.next_pending == s.reqs.size() && s.waiting.empty() && s.running.empty();
}

int cb_sched_free_blocks(const cb_sched* h) { return h ? (int)h->s.free_list.size() : 0; }

int cb_sched_request_info(const cb_sched* h, int req_id, int* produced, int* stored, int* preemptions, int* state) {
  if (!h || req_id < 0 || req_id >= (int)h->s.reqs.size()) return CB_ESTATE;
  const Req& r = h->s.reqs[req_id];
  if (produced) *produced = r.produced;
  if (stored) *stored = r.stored;
  if (preemptions) *preemptions = r.preemptions;
  if (state) *state = r.state;
  return CB_OK;
}

int cb_sched_kv_memory(const cb_sched* h, int max_seq_len, int64_t* out) {
  if (!h || !out || max_seq_len < 1) return CB_EINVAL;
  const Sched& s = h->s;
  long long stored = 0;                // tokens whose K/V the running requests still hold
  for (int rid : s.running) {
    const Req& r = s.reqs[rid];
    stored += r.stored;
    for (int b : r.blocks)
      if (b < 0) stored -= s.bs;
  }
  out[0] = (int64_t)s.running.size();
  out[1] = stored;
  out[2] = (int64_t)(s.num_blocks - (int)s.free_list.size()) * s.bs;
  out[3] = (int64_t)s.running.size() * max_seq_len;
  return CB_OK;
}

}  // extern "C"

namespace {

// One step of padded batching ([CB] Continuous batching: batched generation
// with left padding; [SM] 动态批处理): a batch forms, when none runs, from the
// waiting requests in arrival order -- at most pad_b of them, once pad_b are
// waiting, no further request will arrive or (dynamic batching) the oldest has
// waited pad_wait steps -- cut from its end until its padded length fits the
// pool.  Its first step is the padded prefill (n_max positions per request);
// then it decodes one position per request per step until the longest output
// is done; finished requests keep decoding pads.  Blocks are taken on demand
// and all return when the batch ends.
int padded_step(Sched& s, int32_t* req_ids, int32_t* q_lens, int32_t* ctx_lens, int32_t* cu_q_lens,
                int32_t* block_tables, int max_blocks_per_seq, int64_t* slot_mapping, int* n_reqs_out,
                int* n_tokens_out) {
  while (s.next_pending < s.reqs.size() && s.reqs[s.next_pending].arrival <= s.now) {
    Req& r = s.reqs[s.next_pending++];
    if (s.blocks_for((long long)r.prompt + r.output - 1) > s.num_blocks) {
      r.state = kRejected;
      continue;
    }
    r.state = kWaiting;
    s.waiting.push_back(r.rid);
  }
  if (s.batch.empty() && !s.waiting.empty()) {
    const bool full = (int)s.waiting.size() >= s.pad_b;
    const bool last = s.next_pending == s.reqs.size();
    const bool timed_out = s.pad_wait >= 0 && s.now - s.reqs[s.waiting.front()].arrival >= s.pad_wait;
    if (full || last || timed_out) {
      int b = std::min((int)s.waiting.size(), s.pad_b);
      for (; b > 0; --b) {
        int np = 0, no = 0;
        for (int i = 0; i < b; ++i) {
          np = std::max(np, s.reqs[s.waiting[i]].prompt);
          no = std::max(no, s.reqs[s.waiting[i]].output);
        }
        if ((long long)b * s.blocks_for((long long)np + no - 1) <= s.num_blocks) {
          s.n_max = np;
          s.o_max = no;
          break;
        }
      }
      s.batch.assign(s.waiting.begin(), s.waiting.begin() + b);
      s.waiting.erase(s.waiting.begin(), s.waiting.begin() + b);
      s.k = 0;
      for (int rid : s.batch) {
        s.reqs[rid].state = kRunning;
        s.running.push_back(rid);
      }
    }
  }
  int rc = 0, tok = 0;
  long long real = 0;
  const int nb = (int)s.batch.size();
  // the caller's arrays hold max_batch requests and `budget` tokens
  if (nb > s.max_batch || (long long)nb * (s.k == 0 ? s.n_max : 1) > s.budget) return CB_ESTATE;
  cu_q_lens[0] = 0;
  for (int i = 0; i < nb; ++i) {
    Req& r = s.reqs[s.batch[i]];
    const int n = s.k == 0 ? s.n_max : 1, c = s.k == 0 ? 0 : s.n_max + s.k - 1;
    real += s.k == 0 ? r.prompt : (s.k < r.output ? 1 : 0);
    s.grow(r, (long long)c + n);
    req_ids[i] = r.rid;
    q_lens[i] = n;
    ctx_lens[i] = c;
    cu_q_lens[i + 1] = cu_q_lens[i] + n;
    int32_t* row = block_tables + (size_t)i * max_blocks_per_seq;
    if ((int)r.blocks.size() > max_blocks_per_seq) rc = CB_ESTATE;
    for (int b = 0; b < max_blocks_per_seq; ++b) row[b] = b < (int)r.blocks.size() ? r.blocks[b] : -1;
    for (int p = c; p < c + n; ++p) slot_mapping[tok++] = (int64_t)r.blocks[p / s.bs] * s.bs + p % s.bs;
    r.stored += n;
    if (s.k < r.output) r.produced = std::min(r.output, s.k + 1);
  }
  *n_reqs_out = nb;
  *n_tokens_out = tok;
  s.last_real = real;
  if (nb > 0 && ++s.k == s.o_max) {                // the longest generation is done
    for (int rid : s.batch) {
      Req& r = s.reqs[rid];
      s.release(r);
      r.state = kFinished;
      Sched::erase(s.running, rid);
    }
    s.batch.clear();
  }
  s.now++;
  return rc;
}

}  // namespace

extern "C" {

int cb_sched_step(cb_sched* h, int32_t* req_ids, int32_t* q_lens, int32_t* ctx_lens, int32_t* cu_q_lens,
                  int32_t* block_tables, int max_blocks_per_seq, int64_t* slot_mapping, int* n_reqs_out,
                  int* n_tokens_out) {
  if (!h || !req_ids || !q_lens || !ctx_lens || !cu_q_lens || !block_tables || !slot_mapping || !n_reqs_out ||
      !n_tokens_out || max_blocks_per_seq < 1)
    return CB_EINVAL;
  Sched& s = h->s;
  s.copies.clear();
  if (s.pad_b > 0)
    return padded_step(s, req_ids, q_lens, ctx_lens, cu_q_lens, block_tables, max_blocks_per_seq, slot_mapping,
                       n_reqs_out, n_tokens_out);
  // a. arrivals
  while (s.next_pending < s.reqs.size() && s.reqs[s.next_pending].arrival <= s.now) {
    Req& r = s.reqs[s.next_pending++];
    if (s.blocks_for((long long)r.prompt + r.output - 1) > s.num_blocks) {
      r.state = kRejected;
      continue;
    }
    r.state = kWaiting;
    s.waiting.push_back(r.rid);
  }
  struct Item {
    int rid, n, c;
  };
  std::vector<Item> sched;
  std::vector<int> preempted;
  std::vector<char> scheduled(s.reqs.size(), 0);
  int budget = s.budget;
  auto victim = [&](int after_rid) -> int {
    for (auto it = s.running.rbegin(); it != s.running.rend(); ++it)
      if (*it > after_rid && !scheduled[*it]) return *it;
      else if (*it <= after_rid) break;
    return -1;
  };
  auto full = [&] { return (int)sched.size() >= s.max_batch; };

  // b. running decodes, arrival order
  {
    const std::vector<int> snap = s.running;
    for (int rid : snap) {
      if (budget == 0 || full()) break;
      Req& r = s.reqs[rid];
      if (r.state != kRunning || r.remaining() != 1) continue;
      while (s.blocks_for((long long)r.stored + 1) - (int)r.blocks.size() > (int)s.free_list.size()) {
        if (s.evict_prefix()) continue;
        const int v = victim(rid - 1);           // includes rid itself
        s.preempt(v);
        preempted.push_back(v);
        if (v == rid) break;
      }
      if (r.state != kRunning) continue;
      s.grow(r, (long long)r.stored + 1);
      sched.push_back({rid, 1, r.stored});
      scheduled[rid] = 1;
      budget -= 1;
    }
  }
  // c. running prefills, arrival order
  {
    const std::vector<int> snap = s.running;
    for (int rid : snap) {
      if (budget == 0 || full()) break;
      Req& r = s.reqs[rid];
      if (r.state != kRunning || scheduled[rid] || r.remaining() <= 1) continue;
      const int want = std::min(r.remaining(), budget);
      while (s.blocks_for((long long)r.stored + want) - (int)r.blocks.size() > (int)s.free_list.size()) {
        if (s.evict_prefix()) continue;
        const int v = victim(rid);
        if (v < 0) break;
        s.preempt(v);
        preempted.push_back(v);
      }
      const long long fit = (long long)(r.blocks.size() + s.free_list.size()) * s.bs - r.stored;
      const int n = (int)std::min<long long>(want, fit);
      if (n <= 0) continue;
      s.grow(r, (long long)r.stored + n);
      sched.push_back({rid, n, r.stored});
      scheduled[rid] = 1;
      budget -= n;
    }
  }
  // d. admissions, queue order
  while (!s.waiting.empty() && budget > 0 && !full()) {
    const int rid = s.waiting.front();
    if (std::find(preempted.begin(), preempted.end(), rid) != preempted.end()) break;
    Req& r = s.reqs[rid];
    // f. a published prefix of its group: whole blocks shared, a partial last one copied
    const Prefix* px = nullptr;
    if (r.stored == 0 && r.group >= 0) {
      auto it = s.prefixes.find(r.group);
      if (it != s.prefixes.end()) px = &it->second;
    }
    const int share = px ? px->tokens : 0;
    const bool cow = share % s.bs != 0;   // with no block free for the copy, fit <= 0: it waits
    const long long fit =
        (long long)((int)s.free_list.size() - (cow ? 1 : 0)) * s.bs + (cow ? s.bs - share % s.bs : 0);
    const int n = (int)std::min<long long>(std::min(r.prompt + r.produced - share, budget), fit);
    if (n <= 0) break;
    if (px && share > 0) s.attach(r, *px, share, cow);
    s.waiting.erase(s.waiting.begin());
    r.state = kRunning;
    Sched::insert_sorted(s.running, rid);
    s.grow(r, (long long)r.stored + n);
    sched.push_back({rid, n, r.stored});
    scheduled[rid] = 1;
    budget -= n;
  }

  // metadata
  int rc = (int)preempted.size();
  const int nb = (int)sched.size();
  int tok = 0;
  cu_q_lens[0] = 0;
  for (int i = 0; i < nb; ++i) {
    const Req& r = s.reqs[sched[i].rid];
    req_ids[i] = sched[i].rid;
    q_lens[i] = sched[i].n;
    ctx_lens[i] = sched[i].c;
    cu_q_lens[i + 1] = cu_q_lens[i] + sched[i].n;
    int32_t* row = block_tables + (size_t)i * max_blocks_per_seq;
    if ((int)r.blocks.size() > max_blocks_per_seq) rc = CB_ESTATE;
    for (int b = 0; b < max_blocks_per_seq; ++b) row[b] = b < (int)r.blocks.size() ? r.blocks[b] : -1;
    for (int p = sched[i].c; p < sched[i].c + sched[i].n; ++p)
      slot_mapping[tok++] = (int64_t)r.blocks[p / s.bs] * s.bs + p % s.bs;
  }
  *n_reqs_out = nb;
  *n_tokens_out = tok;
  s.last_real = tok;                             // no pads in continuous batching

  // the forward pass runs here; every scheduled request advances
  for (const Item& it : sched) {
    Req& r = s.reqs[it.rid];
    r.stored += it.n;
    s.publish(r);                                // e.
    if (r.stored == r.prompt + r.produced) r.produced++;
    if (r.produced == r.output) {
      r.state = kFinished;
      s.release(r);
      Sched::erase(s.running, it.rid);
    } else {
      s.slide(r);                                // h.
    }
  }
  s.now++;
  return rc;
}

int cb_build_slot_mapping(const int32_t* q_lens, const int32_t* ctx_lens, const int32_t* block_tables,
                          int max_blocks_per_seq, int n_reqs, int block_size, int64_t* slot_mapping_out) {
  if (!q_lens || !ctx_lens || !block_tables || !slot_mapping_out || n_reqs < 0 || block_size <= 0 ||
      max_blocks_per_seq < 1)
    return CB_EINVAL;
  long long t = 0;
  for (int r = 0; r < n_reqs; ++r) {
    if (q_lens[r] < 0 || ctx_lens[r] < 0) return CB_EINVAL;
    for (int i = 0; i < q_lens[r]; ++i) {
      const long long p = (long long)ctx_lens[r] + i;
      const long long lb = p / block_size;
      if (lb >= max_blocks_per_seq) return CB_EINVAL;
      const int e = block_tables[(size_t)r * max_blocks_per_seq + lb];
      if (e < 0) return CB_EINVAL;
      slot_mapping_out[t++] = (int64_t)e * block_size + p % block_size;
    }
  }
  return CB_OK;
}

}  // extern "C"
