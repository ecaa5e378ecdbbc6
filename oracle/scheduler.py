"""FCFS continuous-batching scheduler oracle (test infrastructure only).

An event simulator of the iteration-level scheduler that decides, step by step,
which tokens of which requests run, and that owns the paged KV block pool.  It
produces the per-step metadata of the attention step (request order, new tokens,
stored tokens, block tables, slot mapping) and nothing else: no attention is
computed here.

Sources:
* [KVN] §Continuous Batching原理: each iteration retires finished requests, admits
  new ones and runs one step for every running request.
* [KVN] §调度策略: first-come-first-served order; preemption when GPU memory
  runs out.
* [CB] §Chunked prefill / §Continuous batching: a prompt may be processed in
  chunks; prefill and decode tokens share one ragged batch whose size is bounded
  by a token budget m.
* [SM] §PagedAttention 批处理: a new physical block is taken only once the
  request's current block is full.

Readings (the algorithm figure of [CB] §Continuous batching is missing; the
pages leave these points open):
1. Per request: P prompt tokens, O output tokens, g produced so far, c tokens
   whose KV is stored.  The known tokens are the P prompt tokens followed by the
   g produced ones; a step processes positions c .. c+n-1 of them, and when it
   reaches the last known token (c + n == P + g) it produces one more token.
   A request with exactly one position left to process is "decoding".  It is
   finished when g == O, so it processes P + O - 1 positions in all.
2. Each step, in this order:
   a. arrivals (arrival step <= now) join the waiting queue in arrival order;
   b. running decoding requests, in arrival order, get 1 token each; when one
      needs a block and none is free, the latest-arrived running request that
      has nothing scheduled in this step is preempted (this may be the request
      itself);
   c. running requests still prefilling, in arrival order, get
      min(remaining, budget left) tokens; to find blocks they may preempt only
      later-arrived running requests with nothing scheduled; the chunk is cut to
      the tokens that fit;
   d. waiting requests are admitted in queue order while budget is left; the
      first chunk is min(remaining, budget left, tokens that fit in free blocks);
      admission stops at the first request that gets no token or that was
      preempted in this same step (no preemption, no skipping ahead).
   Then every scheduled request advances, and finished ones return their blocks.
3. Preemption is by recompute (swapping is not described): the victim returns
   all its blocks, keeps its produced tokens and goes back to the waiting queue
   with c = 0, so its next prefill covers P + g positions.  The waiting queue is
   kept in arrival order (ties in arrival step broken by request id), so a
   preempted request is served before every request that arrived after it.
   "Latest-arrived" likewise means the largest request id.
4. The free list is FIFO: blocks are taken from its front and returned to its
   back in block-table order; its initial order is an input (a seeded
   permutation of the pool, so blocks are scattered).
5. A request needing more blocks than the whole pool can ever hold
   (ceil((P + O - 1) / block_size) > num_blocks) is rejected on arrival.
6. Optional ``max_batch`` caps the number of requests in one step (each pass
   stops once the batch holds that many); by default only the token budget
   bounds the batch.
7. Shared prompt prefixes ([KVN] §与Prefix Caching的结合: requests sharing a
   system prompt compute its KV once; [KVB] §思想: sharing blocks is a matter of
   pointing block tables at the same blocks).  A request may belong to a prefix
   group whose first L prompt tokens it shares (1 <= L < prompt).  Blocks count
   their holders (requests and published prefixes) and go back to the free list
   when none is left:
   - at the end of a step, the first request of a group whose stored tokens
     reach L publishes the blocks covering positions [0, L) (one more holder
     each);
   - admitting a request of the group with nothing stored: it holds the
     published whole blocks, and a partial last block is copied into a fresh
     block of its own (copy-on-write, listed in the step's metadata for the
     device to run before the append).  It starts with the shared positions
     stored.  Its first chunk is min(prompt + produced - shared, budget left,
     positions that fit: the free blocks after the copy plus the room left in
     the copy), so with no free block for the copy it is not admitted yet, like
     any request that finds no room;
   - a running request needing a block when none is free first drops the
     oldest published prefix (repeatedly) and only then preempts; admission
     neither drops prefixes nor preempts.
8. Rolling window ([KVB] §Rolling KV Cache, a heading with no body; reading: a
   query at position p sees keys p - W + 1 .. p).  With a window W > 0, at the
   end of every step each running request lets go of the blocks that its next
   query (at position ``stored``) can no longer see, i.e. whose positions all
   lie before stored - W + 1; their table entries become -1 and they are never
   read again.  A request publishes its prefix only while it still holds every
   block of it.
"""
from collections import deque
from dataclasses import dataclass, field

import numpy as np


@dataclass
class Request:
    rid: int
    arrival: int
    prompt_len: int
    output_len: int
    produced: int = 0          # g
    stored: int = 0            # c
    blocks: list = field(default_factory=list)
    state: str = "pending"     # pending, waiting, running, finished, rejected
    preemptions: int = 0
    group: int = -1            # prefix group (-1: none)
    prefix_len: int = 0        # shared prompt positions of the group

    @property
    def remaining(self):
        return self.prompt_len + self.produced - self.stored


@dataclass
class StepMetadata:
    step: int
    req_ids: np.ndarray       # int32 [B], batch order
    q_lens: np.ndarray        # int32 [B]
    ctx_lens: np.ndarray      # int32 [B] tokens stored before this step
    block_tables: list        # list of int lists: valid entries only
    slot_mapping: np.ndarray  # int64 [sum(q_lens)]
    preempted: list           # request ids preempted during this step
    finished: list            # request ids that finished at the end of this step
    copies: list = field(default_factory=list)   # (src, dst) block copies to run before the append


def _blocks_for(n_tokens, block_size):
    return -(-n_tokens // block_size)


class FCFSScheduler:
    def __init__(self, requests, token_budget, block_size, num_blocks, free_order, max_batch=None, window=0):
        """requests: iterable of (arrival_step, prompt_len, output_len[, group,
        prefix_len]), ids = index, sorted by arrival.  free_order: the initial
        free-list order (a permutation of range(num_blocks)).  window: rolling
        window W (0: none; reading 8)."""
        self.reqs = []
        for i, t in enumerate(requests):
            a, p, o = (int(x) for x in t[:3])
            g, pl = (int(t[3]), int(t[4])) if len(t) > 3 else (-1, 0)
            assert g < 0 or 1 <= pl < p, "a shared prefix leaves at least one prompt token"
            self.reqs.append(Request(i, a, p, o, group=g, prefix_len=pl if g >= 0 else 0))
        arrivals = [r.arrival for r in self.reqs]
        assert arrivals == sorted(arrivals), "requests must be given in arrival order"
        assert sorted(int(b) for b in free_order) == list(range(num_blocks))
        self.budget = int(token_budget)
        self.max_batch = int(max_batch) if max_batch is not None else None
        self.window = int(window)
        self.bs = int(block_size)
        self.num_blocks = int(num_blocks)
        self.free = deque(int(b) for b in free_order)
        self.holders = [0] * self.num_blocks
        self.published = {}        # group -> (blocks, positions, publication number)
        self.n_published = 0
        self.pending = deque(self.reqs)
        self.waiting = []          # kept in arrival (id) order, head first
        self.running = []          # kept in arrival (id) order
        self.now = 0

    # --- allocator -------------------------------------------------------
    def _take(self):
        b = self.free.popleft()
        self.holders[b] = 1
        return b

    def _let_go(self, b):
        self.holders[b] -= 1
        if self.holders[b] == 0:
            self.free.append(b)

    def _grow(self, req, n_tokens):
        need = _blocks_for(n_tokens, self.bs) - len(req.blocks)
        for _ in range(need):
            req.blocks.append(self._take())

    def _release(self, req):
        for b in req.blocks:
            if b >= 0:
                self._let_go(b)
        req.blocks = []

    def _slide(self, req):
        """Rolling window: let go of the blocks the next query cannot see."""
        if self.window <= 0:
            return
        first_seen = req.stored - self.window + 1
        for i in range(min(len(req.blocks), max(0, first_seen) // self.bs)):
            if req.blocks[i] >= 0:
                self._let_go(req.blocks[i])
                req.blocks[i] = -1

    def _drop_oldest_prefix(self):
        if not self.published:
            return False
        g = min(self.published, key=lambda k: self.published[k][2])
        blocks, _, _ = self.published.pop(g)
        for b in blocks:
            self._let_go(b)
        return True

    def _maybe_publish(self, req):
        if req.group < 0 or req.group in self.published or req.stored < req.prefix_len:
            return
        blocks = req.blocks[:_blocks_for(req.prefix_len, self.bs)]
        if any(b < 0 for b in blocks):
            return                                  # part of it already left the window
        for b in blocks:
            self.holders[b] += 1
        self.published[req.group] = (list(blocks), req.prefix_len, self.n_published)
        self.n_published += 1

    def _preempt(self, req):
        self._release(req)
        req.stored = 0
        req.state = "waiting"
        req.preemptions += 1
        self.running.remove(req)
        self.waiting.append(req)
        self.waiting.sort(key=lambda r: r.rid)

    # --- memory accounting ----------------------------------------------
    def kv_memory(self, max_seq_len):
        """KV memory after the last step, in token slots: running requests, tokens
        they have stored, slots in the blocks taken from the pool, and the slots a
        contiguous cache reserving max_seq_len positions per request would hold
        ([KVB] 连续内存分配: the TraditionalKVCache reservation; [SM] PagedAttention
        批处理: a block is taken only when the last one is full)."""
        running = len(self.running)
        # tokens whose K/V the running requests still hold (a rolling window
        # lets go of whole blocks of stored tokens)
        stored = sum(r.stored - self.bs * sum(1 for b in r.blocks if b < 0) for r in self.running)
        paged = (self.num_blocks - len(self.free)) * self.bs
        return dict(running=running, stored=stored, paged=paged, contiguous=running * int(max_seq_len))

    # --- one iteration ---------------------------------------------------
    def done(self):
        return not self.pending and not self.waiting and not self.running

    def step(self):
        while self.pending and self.pending[0].arrival <= self.now:
            r = self.pending.popleft()
            if _blocks_for(r.prompt_len + r.output_len - 1, self.bs) > self.num_blocks:
                r.state = "rejected"
                continue
            r.state = "waiting"
            self.waiting.append(r)

        budget = self.budget
        copies = []                # copy-on-write (src, dst) of this step
        sched = []                 # (req, n_tokens, stored_before)
        scheduled_ids = set()
        preempted = []

        def full():
            return self.max_batch is not None and len(sched) >= self.max_batch

        def victim(after_rid):
            cands = [r for r in self.running
                     if r.rid not in scheduled_ids and r.rid > after_rid]
            return max(cands, key=lambda r: r.rid) if cands else None

        # b. running decodes
        for req in list(self.running):
            if budget == 0 or full():
                break
            if req.state != "running" or req.remaining != 1:
                continue
            while _blocks_for(req.stored + 1, self.bs) - len(req.blocks) > len(self.free):
                if self._drop_oldest_prefix():
                    continue
                v = victim(req.rid - 1)              # candidates include req itself
                self._preempt(v)
                preempted.append(v.rid)
                if v is req:
                    break
            if req.state != "running":
                continue
            self._grow(req, req.stored + 1)
            sched.append((req, 1, req.stored))
            scheduled_ids.add(req.rid)
            budget -= 1

        # c. running prefills
        for req in list(self.running):
            if budget == 0 or full():
                break
            if req.state != "running" or req.rid in scheduled_ids or req.remaining <= 1:
                continue
            want = min(req.remaining, budget)
            while _blocks_for(req.stored + want, self.bs) - len(req.blocks) > len(self.free):
                if self._drop_oldest_prefix():
                    continue
                v = victim(req.rid)
                if v is None:
                    break
                self._preempt(v)
                preempted.append(v.rid)
            fit = (len(req.blocks) + len(self.free)) * self.bs - req.stored
            n = min(want, fit)
            if n <= 0:
                continue
            self._grow(req, req.stored + n)
            sched.append((req, n, req.stored))
            scheduled_ids.add(req.rid)
            budget -= n

        # d. admissions
        while self.waiting and budget > 0 and not full():
            req = self.waiting[0]
            if req.rid in preempted:
                break
            pub = self.published.get(req.group) if req.stored == 0 and req.group >= 0 else None
            shared = pub[1] if pub else 0
            tail = shared % self.bs                 # positions in a partial last shared block
            room = (len(self.free) - (1 if tail else 0)) * self.bs + (self.bs - tail if tail else 0)
            n = min(req.prompt_len + req.produced - shared, budget, room)
            if n <= 0:
                break
            if shared:
                whole = shared // self.bs
                for b in pub[0][:whole]:
                    self.holders[b] += 1
                    req.blocks.append(b)
                if tail:
                    mine = self._take()
                    copies.append((pub[0][whole], mine))
                    req.blocks.append(mine)
                req.stored = shared
            self.waiting.pop(0)
            req.state = "running"
            self.running.append(req)
            self.running.sort(key=lambda r: r.rid)
            self._grow(req, req.stored + n)
            sched.append((req, n, req.stored))
            scheduled_ids.add(req.rid)
            budget -= n

        # metadata
        slots = []
        for req, n, c in sched:
            for p in range(c, c + n):
                slots.append(req.blocks[p // self.bs] * self.bs + p % self.bs)
        meta = StepMetadata(
            step=self.now,
            req_ids=np.array([r.rid for r, _, _ in sched], dtype=np.int32),
            q_lens=np.array([n for _, n, _ in sched], dtype=np.int32),
            ctx_lens=np.array([c for _, _, c in sched], dtype=np.int32),
            block_tables=[list(r.blocks) for r, _, _ in sched],
            slot_mapping=np.array(slots, dtype=np.int64),
            preempted=preempted,
            finished=[],
            copies=copies,
        )

        # the forward pass happens here; then every scheduled request advances
        for req, n, _ in sched:
            req.stored += n
            self._maybe_publish(req)
            if req.stored == req.prompt_len + req.produced:
                req.produced += 1
            if req.produced == req.output_len:
                req.state = "finished"
                self._release(req)
                self.running.remove(req)
                meta.finished.append(req.rid)
            else:
                self._slide(req)
        self.now += 1
        return meta

    def run(self, max_steps=1_000_000):
        out = []
        while not self.done() and self.now < max_steps:
            out.append(self.step())
        return out


class PaddedBatcher:
    """Static and dynamic batching with padding, the baselines that continuous
    batching is measured against.

    Sources: [CB] §Continuous batching (batched generation: every prompt of the
    batch is padded on the left to the batch's longest prompt, and the batch runs
    until its longest generation ends); [SM] §动态批处理 (dynamic batching: the
    requests that arrive within a waiting window, or until the batch is full, run
    together as one batch) and §连续批处理 (continuous batching, for comparison).

    Readings (the pages describe the policies, not their parameters):
    1. A batch forms only when no batch is running, from the waiting requests in
       arrival order, at most ``batch_size`` of them.  Static batching
       (max_wait None) waits until batch_size requests are waiting or no further
       request will arrive; dynamic batching also starts a batch once its oldest
       waiting request has waited max_wait steps since its arrival.
    2. The batch's first step is its padded prefill: every request processes
       n_max positions (n_max = the longest prompt; the first n_max - P positions
       are pads), all in one step, and produces its first token.  Then the batch
       decodes one position per request per step until the longest output is
       done: o_max - 1 decode steps; a request that has finished keeps decoding
       pad positions.  So each request processes n_max + o_max - 1 positions.
    3. Pad positions are computed and stored like real ones; the real tokens of
       a request are its P prompt tokens and its O - 1 decoded positions.
    4. Blocks are taken on demand from the FIFO free list (a block when the last
       is full, as in FCFSScheduler) and all return when the batch ends.  A
       request whose padded length cannot fit the pool is rejected on arrival;
       a batch is cut short, from its end, until its padded length fits the
       pool.
    """

    def __init__(self, requests, batch_size, block_size, num_blocks, free_order, max_wait=None):
        self.reqs = [Request(i, int(a), int(p), int(o)) for i, (a, p, o) in enumerate(t[:3] for t in requests)]
        arrivals = [r.arrival for r in self.reqs]
        assert arrivals == sorted(arrivals), "requests must be given in arrival order"
        assert sorted(int(b) for b in free_order) == list(range(num_blocks))
        self.B = int(batch_size)
        self.max_wait = None if max_wait is None else int(max_wait)
        self.bs = int(block_size)
        self.num_blocks = int(num_blocks)
        self.free = deque(int(b) for b in free_order)
        self.pending = deque(self.reqs)
        self.waiting = []
        self.batch = []            # running batch, arrival order
        self.n_max = self.o_max = 0
        self.k = 0                 # steps the batch has run
        self.now = 0

    def done(self):
        return not self.pending and not self.waiting and not self.batch

    def _blocks(self, n):
        return -(-n // self.bs)

    def _form_batch(self):
        if self.batch or not self.waiting:
            return
        full = len(self.waiting) >= self.B
        last = not self.pending
        timed_out = self.max_wait is not None and self.now - self.waiting[0].arrival >= self.max_wait
        if not (full or last or timed_out):
            return
        b = self.waiting[:self.B]
        while b:
            n_max = max(r.prompt_len for r in b)
            o_max = max(r.output_len for r in b)
            if len(b) * self._blocks(n_max + o_max - 1) <= self.num_blocks:
                break
            b = b[:-1]
        self.batch = b
        del self.waiting[:len(b)]
        self.n_max = max(r.prompt_len for r in b)
        self.o_max = max(r.output_len for r in b)
        self.k = 0
        for r in b:
            r.state = "running"

    def step(self):
        """One step; returns (StepMetadata, real tokens of the step)."""
        while self.pending and self.pending[0].arrival <= self.now:
            r = self.pending.popleft()
            if self._blocks(r.prompt_len + r.output_len - 1) > self.num_blocks:
                r.state = "rejected"
                continue
            r.state = "waiting"
            self.waiting.append(r)
        self._form_batch()
        sched = []
        real = 0
        if self.batch:
            for r in self.batch:
                if self.k == 0:
                    n, c = self.n_max, 0
                    real += r.prompt_len
                else:
                    n, c = 1, self.n_max + self.k - 1
                    real += 1 if self.k < r.output_len else 0
                need = self._blocks(c + n) - len(r.blocks)
                for _ in range(need):
                    r.blocks.append(self.free.popleft())
                sched.append((r, n, c))
        slots = []
        for r, n, c in sched:
            for p in range(c, c + n):
                slots.append(r.blocks[p // self.bs] * self.bs + p % self.bs)
        meta = StepMetadata(step=self.now, req_ids=np.array([r.rid for r, _, _ in sched], dtype=np.int32),
                            q_lens=np.array([n for _, n, _ in sched], dtype=np.int32),
                            ctx_lens=np.array([c for _, _, c in sched], dtype=np.int32),
                            block_tables=[list(r.blocks) for r, _, _ in sched],
                            slot_mapping=np.array(slots, dtype=np.int64), preempted=[], finished=[])
        if self.batch:
            for r, n, _ in sched:
                r.stored += n
                if self.k < r.output_len:
                    r.produced = min(r.output_len, self.k + 1)
            self.k += 1
            if self.k == self.o_max:                     # the longest generation is done
                for r in self.batch:
                    for b in r.blocks:
                        self.free.append(b)
                    r.blocks = []
                    r.state = "finished"
                    meta.finished.append(r.rid)
                self.batch = []
        self.now += 1
        return meta, real
