"""Pins of the FCFS scheduler oracle: the pages' worked examples and invariants
that any correct paged, chunked, preempting FCFS scheduler must keep."""
import json
import os

import numpy as np
import pytest

import workloads as wl
from oracle import paged as op
from oracle.scheduler import FCFSScheduler


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_chunked_prefill_worked_example(golden_dir):
    """[CB] §Chunked prefill: a 7-token prompt with room for 4 tokens per pass runs
    as a 4-token chunk and then a 3-token chunk after 4 stored tokens."""
    g = _load(golden_dir, "chunking_n7_m4.json")
    s = FCFSScheduler([(0, g["n"], 1)], token_budget=g["m"], block_size=16, num_blocks=4,
                      free_order=range(4))
    steps = s.run()
    assert [m.q_lens.tolist() for m in steps] == [[q] for q in g["chunk_sizes"]]
    assert [m.ctx_lens.tolist() for m in steps] == [[c] for c in g["chunk_ctx"]]
    assert s.reqs[0].state == "finished" and s.reqs[0].produced == 1


def test_iteration_level_example(golden_dir):
    """[KVN] §Iteration-level调度详解: req3 finishes and req5 joins the next step."""
    g = _load(golden_dir, "iteration_example.json")
    reqs = [(0, 1, 50), (0, 1, 50), (0, 1, 2), (0, 1, 50), (2, 1, 50)]
    s = FCFSScheduler(reqs, token_budget=64, block_size=16, num_blocks=64, free_order=range(64))
    s.step()                        # step 0: the four prompts are prefilled
    t = s.step()                    # step t: four decodes; req3 produces its last token
    t1 = s.step()                   # step t+1
    assert (t.req_ids + 1).tolist() == g["batch_t"]
    assert t.finished == [2]
    assert (t1.req_ids + 1).tolist() == g["batch_t_plus_1"]


def test_decode_takes_a_block_only_when_the_last_is_full():
    """[SM] §PagedAttention 批处理: a new block only once the current one is full."""
    s = FCFSScheduler([(0, 15, 4)], token_budget=64, block_size=16, num_blocks=8, free_order=range(8))
    m0 = s.step()                   # prefill 15 tokens -> 1 block
    assert m0.block_tables == [[0]]
    m1 = s.step()                   # decode position 15 -> still block 0
    assert m1.block_tables == [[0]] and m1.slot_mapping.tolist() == [15]
    m2 = s.step()                   # decode position 16 -> second block
    assert m2.block_tables == [[0, 1]] and m2.slot_mapping.tolist() == [16]


def test_preemption_by_recompute_small_case():
    """Pool of 2 blocks (32 tokens): two 16-token prompts fill it; when the first
    needs a third block the later request is preempted and later recomputed."""
    s = FCFSScheduler([(0, 16, 3), (0, 16, 3)], token_budget=64, block_size=16,
                      num_blocks=2, free_order=[1, 0])
    m0 = s.step()
    assert m0.q_lens.tolist() == [16, 16] and m0.block_tables == [[1], [0]]
    m1 = s.step()                   # request 0 decodes position 16 -> needs a block
    assert m1.preempted == [1]
    assert m1.req_ids.tolist() == [0] and m1.block_tables == [[1, 0]]
    steps = [m0, m1] + s.run()
    r1 = s.reqs[1]
    assert r1.state == "finished" and r1.preemptions == 1
    # request 1 recomputes its prompt plus the one token it had produced (16 + 1)
    rec = [m for m in steps if 1 in m.req_ids.tolist() and m.ctx_lens[m.req_ids.tolist().index(1)] == 0]
    assert [int(m.q_lens[m.req_ids.tolist().index(1)]) for m in rec] == [16, 17]


def _check_trace(tr, max_steps=100000):
    s = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks,
                      wl.free_order(tr.num_blocks, tr.seed))
    steps = s.run(max_steps)
    assert s.done(), "trace did not finish"
    first_admit = []
    last = {}
    for m in steps:
        ids = m.req_ids.tolist()
        assert len(set(ids)) == len(ids)
        assert int(m.q_lens.sum()) <= tr.token_budget
        assert all(q >= 1 for q in m.q_lens.tolist())
        seen = set()
        for r, q, c, tab in zip(ids, m.q_lens.tolist(), m.ctx_lens.tolist(), m.block_tables):
            assert len(tab) == -(-(c + q) // tr.block_size)
            assert not (set(tab) & seen)
            seen |= set(tab)
            if r not in first_admit:
                first_admit.append(r)
            prev = last.get(r)
            assert c == 0 or (prev is not None and c == prev), (r, c, prev)
            last[r] = c + q
        if m.preempted:
            for r in m.preempted:
                last[r] = 0
        want = op.slot_mapping(m.block_tables, m.q_lens.tolist(), m.ctx_lens.tolist(), tr.block_size)
        assert np.array_equal(m.slot_mapping, want)
    assert first_admit == sorted(first_admit), "admission must follow arrival order"
    for r in s.reqs:
        if r.state == "rejected":
            continue
        assert r.state == "finished"
        assert r.produced == r.output_len
        assert r.stored == r.prompt_len + r.output_len - 1
        assert r.blocks == []
    assert sorted(s.free) == list(range(tr.num_blocks))
    return s, steps


@pytest.mark.parametrize("seed", range(12))
def test_invariants_on_tight_small_traces(seed):
    tr = wl.small_trace(seed)
    s, steps = _check_trace(tr)
    if seed < 4:
        assert s.now > 0


def test_tight_traces_do_preempt():
    total = 0
    for seed in range(12):
        s, _ = _check_trace(wl.small_trace(seed))
        total += sum(r.preemptions for r in s.reqs)
    assert total > 0


def test_block_ownership_is_exclusive_every_step():
    tr = wl.small_trace(3, n_requests=30, num_blocks=24)
    s = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks,
                      wl.free_order(tr.num_blocks, tr.seed))
    while not s.done():
        s.step()
        owned = [b for r in s.reqs for b in r.blocks]
        assert len(owned) == len(set(owned))
        assert sorted(owned + list(s.free)) == list(range(tr.num_blocks))


def test_kv_memory_closed_form_single_request():
    """[SM] §PagedAttention 批处理: blocks are taken only when the last one is full;
    [KVB] §连续内存分配: a contiguous cache reserves max_seq_len slots per request.
    A 20-token prompt with 5 outputs (24 positions in all) in blocks of 16."""
    s = FCFSScheduler([(0, 20, 5)], token_budget=64, block_size=16, num_blocks=8, free_order=range(8))
    s.step()                                     # the prompt: 20 stored, 2 blocks
    assert s.kv_memory(24) == dict(running=1, stored=20, paged=32, contiguous=24)
    for _ in range(3):
        s.step()                                 # decodes at positions 20, 21, 22
    assert s.kv_memory(24) == dict(running=1, stored=23, paged=32, contiguous=24)
    s.step()                                     # position 23 is the last: finished, blocks returned
    assert s.kv_memory(24) == dict(running=0, stored=0, paged=0, contiguous=0)


@pytest.mark.parametrize("seed", range(4))
def test_kv_memory_paged_waste_is_below_one_block_per_request(seed):
    """Paged: each running request wastes only the tail of its last block
    (< block_size slots); contiguous: max_seq_len minus what is stored."""
    tr = wl.small_trace(seed)
    s = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks,
                      wl.free_order(tr.num_blocks, tr.seed))
    maxlen = max(p + o - 1 for _, p, o in tr.requests)
    while not s.done():
        s.step()
        m = s.kv_memory(maxlen)
        per_req = sum(-(-r.stored // tr.block_size) * tr.block_size for r in s.running)
        assert m["paged"] == per_req
        assert 0 <= m["paged"] - m["stored"] <= m["running"] * (tr.block_size - 1)
        assert m["stored"] <= m["contiguous"]


def test_prefix_sharing_worked_example():
    """[KVN] §与Prefix Caching的结合 with [KVB] §思想 (blocks shared through the block
    table): two requests share a 20-token system prompt in blocks of 16.  The
    first stores it (blocks a, b; b holds positions 16..19 of it and then its own
    tokens) and publishes it; the second holds block a, gets a copy of b in a
    block of its own (copy-on-write: it will write its own tokens there) and
    starts with 20 positions stored."""
    reqs = [(0, 30, 3, 0, 20), (1, 25, 2, 0, 20)]
    s = FCFSScheduler(reqs, token_budget=64, block_size=16, num_blocks=8, free_order=range(8))
    m0 = s.step()
    assert m0.q_lens.tolist() == [30] and m0.copies == []
    a, b = s.reqs[0].blocks
    assert s.published[0][:2] == ([a, b], 20)
    m1 = s.step()                                    # request 0 decodes, request 1 is admitted
    assert m1.req_ids.tolist() == [0, 1] and m1.q_lens.tolist() == [1, 5] and m1.ctx_lens.tolist() == [30, 20]
    (src, dst), = m1.copies
    assert src == b and dst not in (a, b)
    assert m1.block_tables[1] == [a, dst]
    assert s.holders[a] == 3 and s.holders[b] == 2 and s.holders[dst] == 1
    # request 1's own positions 20..24 go to its copy, never into the shared blocks
    assert m1.slot_mapping[1:].tolist() == [dst * 16 + p % 16 for p in range(20, 25)]


def _held(s):
    h = [0] * s.num_blocks
    for r in s.running:
        for b in r.blocks:
            h[b] += 1
    for blocks, _, _ in s.published.values():
        for b in blocks:
            h[b] += 1
    return h


@pytest.mark.parametrize("seed", range(6))
def test_prefix_sharing_invariants(seed):
    """Every block's holder count equals the running requests and published
    prefixes that hold it; free blocks have none; no step writes a position a
    published prefix shares; a request admitted onto a prefix starts with its
    positions stored and the prefix's whole blocks first in its table."""
    tr = wl.with_prefixes(wl.small_trace(seed, num_blocks=26), 3, 18 + 5 * seed, seed=seed)
    s = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks,
                      wl.free_order(tr.num_blocks, tr.seed))
    shares = 0
    while not s.done():
        before = {g: (list(p[0]), p[1]) for g, p in s.published.items()}
        m = s.step()
        held = _held(s)
        assert held == s.holders
        assert all(s.holders[b] == 0 for b in s.free)
        assert len(s.free) + sum(1 for h in held if h) == s.num_blocks
        protected = set()                  # prefixes published through the whole step (none dropped)
        for g, (blocks, n) in before.items():
            if g in s.published and s.published[g][0] == blocks:
                for p in range(n):
                    protected.add(blocks[p // tr.block_size] * tr.block_size + p % tr.block_size)
        assert not protected.intersection(m.slot_mapping.tolist())
        for i, rid in enumerate(m.req_ids.tolist()):
            r = s.reqs[rid]
            if r.group in before and m.ctx_lens[i] > 0 and any(dst == m.block_tables[i][-1] or dst in m.block_tables[i]
                                                               for _, dst in m.copies):
                blocks, n = before[r.group]
                whole = n // tr.block_size
                assert m.block_tables[i][:whole] == blocks[:whole]
                assert m.ctx_lens[i] == n
                shares += 1
    assert shares > 0 or all(p[1] % tr.block_size == 0 for p in before.values())


def test_max_batch_caps_every_pass():
    """The optional per-step request cap: four 4-token prompts with 3 outputs
    each arrive together, the token budget (64) would take them all, and a cap
    of 2 runs them two at a time -- requests 0 and 1 for their prefill and both
    decodes, then requests 2 and 3.  Admitting max_batch + 1 (or one fewer)
    changes the first step's batch."""
    s = FCFSScheduler([(0, 4, 3)] * 4, token_budget=64, block_size=16, num_blocks=8, free_order=range(8),
                      max_batch=2)
    batches = [m.req_ids.tolist() for m in s.run()]
    assert batches == [[0, 1]] * 3 + [[2, 3]] * 3
    # without the cap the same requests run together
    s = FCFSScheduler([(0, 4, 3)] * 4, token_budget=64, block_size=16, num_blocks=8, free_order=range(8))
    assert [m.req_ids.tolist() for m in s.run()] == [[0, 1, 2, 3]] * 3


def _two_prefixes_then_pressure():
    """Blocks of 4, a pool of 6.  Request 0 (group 0) and request 1 (group 1)
    each store a 4-token prefix in one block, publish it and finish, so that
    only the published prefixes hold blocks 0 and 2.  Request 2 (no group)
    then takes the four free blocks with a 16-token prompt, and its first
    decode (position 16) needs a fifth block while none is free."""
    reqs = [(0, 5, 1, 0, 4), (1, 5, 1, 1, 4), (2, 16, 2), (4, 6, 1, 1, 4)]
    return FCFSScheduler(reqs, token_budget=64, block_size=4, num_blocks=6, free_order=range(6))


def test_prefix_drop_takes_the_oldest_first():
    """A running request short of a block first drops published prefixes,
    oldest publication first ([KVN] §与Prefix Caching的结合 gives the sharing;
    the order is this scheduler's reading).  Group 0's prefix (block 0,
    published first) goes; group 1's (block 2) stays and is shared by the
    group-1 request that arrives later.  Dropping the newest would hand block 2
    to request 2 instead; preempting instead of dropping would stop request 2."""
    s = _two_prefixes_then_pressure()
    m0, m1, m2 = s.step(), s.step(), s.step()
    assert m0.block_tables == [[0, 1]] and m1.block_tables == [[2, 3]]
    assert sorted(s.published) == [0, 1] and s.published[0][0] == [0] and s.published[1][0] == [2]
    assert m2.block_tables == [[4, 5, 1, 3]] and len(s.free) == 0
    m3 = s.step()                                  # request 2 decodes position 16
    assert m3.req_ids.tolist() == [2] and m3.preempted == []
    assert m3.block_tables == [[4, 5, 1, 3, 0]]    # block 0: group 0's prefix, dropped
    assert list(s.published) == [1] and s.published[1][0] == [2]
    m4 = s.step()                                  # request 3 (group 1) joins the surviving prefix
    assert m4.req_ids.tolist() == [3] and m4.ctx_lens.tolist() == [4] and m4.q_lens.tolist() == [2]
    assert m4.block_tables[0][0] == 2 and m4.copies == []


def test_partial_prefix_block_waits_for_a_free_block():
    """Copy-on-write needs a block for the copy: a request joining a prefix
    whose last block is partial is not admitted while no block is free (no
    copy is listed and nothing is shared yet), and is admitted with the copy as
    soon as one is.  Blocks of 4, a pool of 4: requests 0 and 1 (7-token
    prompts, 2 outputs: 8 positions, two blocks each) fill the pool; request 0
    publishes its 6-token prefix (blocks 0 and 1, block 1 partial).  Request 2
    of the same group arrives at step 1, while no block is free."""
    reqs = [(0, 7, 2, 0, 6), (0, 7, 2), (1, 7, 1, 0, 6)]
    s = FCFSScheduler(reqs, token_budget=64, block_size=4, num_blocks=4, free_order=range(4))
    m0 = s.step()
    assert m0.req_ids.tolist() == [0, 1] and m0.block_tables == [[0, 1], [2, 3]] and len(s.free) == 0
    assert s.published[0][:2] == ([0, 1], 6)
    m1 = s.step()                  # both decode their last token; request 2 cannot be admitted
    assert m1.req_ids.tolist() == [0, 1] and m1.copies == [] and m1.preempted == []
    assert s.reqs[2].state == "waiting" and s.reqs[2].blocks == []
    assert s.holders[:2] == [1, 1] and sorted(s.free) == [2, 3]   # the prefix alone holds blocks 0, 1
    m2 = s.step()                  # block 2 is free: whole block 0 shared, partial block 1 copied into 2
    assert m2.req_ids.tolist() == [2] and m2.copies == [(1, 2)]
    assert m2.block_tables == [[0, 2]] and m2.ctx_lens.tolist() == [6] and m2.q_lens.tolist() == [1]
    assert m2.slot_mapping.tolist() == [2 * 4 + 6 % 4]


# ----------------------------------------------------------------- rolling window
def test_rolling_window_lets_go_of_unseen_blocks_by_hand():
    """[KVB] §Rolling KV Cache (heading only; reading: position p sees keys
    p - W + 1 .. p).  A 40-token prompt with W = 20 in blocks of 16: after the
    prefill the next query (position 40) sees keys 21.., so block 0 (0..15) is
    let go (-1) and returned to the pool; block 1 (16..31) goes once the next
    query sees keys 32.. only (after position 50 is stored)."""
    s = FCFSScheduler([(0, 40, 20)], token_budget=64, block_size=16, num_blocks=8, free_order=range(8), window=20)
    m0 = s.step()
    assert m0.block_tables == [[0, 1, 2]]
    assert s.reqs[0].blocks == [-1, 1, 2] and list(s.free) == [3, 4, 5, 6, 7, 0]
    assert s.kv_memory(64)["stored"] == 40 - 16
    m1 = s.step()                                  # decode position 40 into block 2
    assert m1.block_tables == [[-1, 1, 2]] and m1.slot_mapping.tolist() == [2 * 16 + 8]
    for _ in range(7):                             # positions 41..47
        s.step()
    m = s.step()                                   # position 48 opens a block: the front of the free list
    assert m.block_tables == [[-1, 1, 2, 3]] and m.slot_mapping.tolist() == [3 * 16]
    assert s.reqs[0].blocks == [-1, 1, 2, 3]       # stored 49: next query sees 30.., block 1 still needed
    s.step()                                       # position 49
    s.step()                                       # position 50: stored 51, next query sees 32..
    assert s.reqs[0].blocks == [-1, -1, 2, 3] and list(s.free)[-1] == 1


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("window", [1, 17, 40])
def test_rolling_window_invariants(seed, window):
    """Every step: a running request holds exactly the blocks that hold a
    position its next query can see (and -1 before them); free + held = pool;
    the trace completes with every request's full output."""
    tr = wl.small_trace(seed, num_blocks=12)
    s = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks,
                      wl.free_order(tr.num_blocks, tr.seed), window=window)
    bs = tr.block_size
    while not s.done():
        s.step()
        held = []
        for r in s.running:
            first_seen = r.stored - window + 1
            for i, b in enumerate(r.blocks):
                if (i + 1) * bs <= first_seen:
                    assert b == -1, (r.rid, i)
                else:
                    assert b >= 0, (r.rid, i)
                    held.append(b)
        assert len(held) == len(set(held))
        assert sorted(held + list(s.free)) == list(range(tr.num_blocks))
        assert s.kv_memory(1)["stored"] == sum(min(r.stored, r.stored - (max(0, r.stored - window + 1) // bs) * bs)
                                               for r in s.running)
    for r in s.reqs:
        assert r.state in ("finished", "rejected")
        if r.state == "finished":
            assert r.produced == r.output_len


# ----------------------------------------------------------------- padded batching
from oracle.scheduler import PaddedBatcher  # noqa: E402
from oracle import sizes as osz  # noqa: E402


def test_static_batch_by_hand():
    """[CB] §Continuous batching (batched generation, left padding) and [SM]
    §动态批处理: batches of 2.  Requests (arrival, prompt, output): (0,3,2),
    (0,5,1) run first -- a padded prefill of 5 positions each (3 + 5 real
    tokens) and one decode step (real for request 0 only).  Request 2 (arrives
    at 1) waits for a second request, which arrives at 5; their batch pads to 4
    positions and decodes 2 steps for request 2's 3 outputs."""
    pb = PaddedBatcher([(0, 3, 2), (0, 5, 1), (1, 2, 3), (5, 4, 1)], batch_size=2, block_size=4, num_blocks=8,
                       free_order=range(8))
    steps = []
    while not pb.done():
        m, real = pb.step()
        steps.append((m.req_ids.tolist(), m.q_lens.tolist(), m.ctx_lens.tolist(), real))
    assert steps == [([0, 1], [5, 5], [0, 0], 8), ([0, 1], [1, 1], [5, 5], 1),
                     ([], [], [], 0), ([], [], [], 0), ([], [], [], 0),
                     ([2, 3], [4, 4], [0, 0], 6), ([2, 3], [1, 1], [4, 4], 1), ([2, 3], [1, 1], [5, 5], 1)]
    assert sum(s[3] for s in steps) == sum(p + o - 1 for _, p, o in [(0, 3, 2), (0, 5, 1), (1, 2, 3), (5, 4, 1)])


def test_dynamic_batch_starts_after_max_wait():
    """Dynamic batching starts a partial batch once its oldest request has
    waited max_wait steps: request 2 (arrival 1) runs alone at step 3."""
    pb = PaddedBatcher([(0, 3, 2), (0, 5, 1), (1, 2, 3), (5, 4, 1)], batch_size=2, block_size=4, num_blocks=8,
                       free_order=range(8), max_wait=2)
    ids = []
    while not pb.done():
        m, _ = pb.step()
        ids.append(m.req_ids.tolist())
    assert ids == [[0, 1], [0, 1], [], [2], [2], [2], [3]]


@pytest.mark.parametrize("seed", range(4))
def test_padded_prefill_pads_equal_the_left_padded_batch(seed):
    """The padded prefill's pad positions are those of the left-padded batch
    built by hand (oracle.sizes.left_padded_batch); every request processes
    n_max + o_max - 1 positions; real tokens are each request's P + O - 1."""
    tr = wl.small_trace(seed, num_blocks=60)
    pb = PaddedBatcher(tr.requests, batch_size=4, block_size=tr.block_size, num_blocks=tr.num_blocks,
                       free_order=wl.free_order(tr.num_blocks, tr.seed))
    total_real = 0
    while not pb.done():
        batch = list(pb.batch)
        m, real = pb.step()
        total_real += real
        if len(m.q_lens) and m.ctx_lens[0] == 0:            # a padded prefill
            lens = [pb.reqs[r].prompt_len for r in m.req_ids.tolist()]
            rows = osz.left_padded_batch(lens)
            assert int(m.q_lens.sum()) - real == sum(row.count("pad") for row in rows)
    done = [r for r in pb.reqs if r.state == "finished"]
    assert total_real == sum(r.prompt_len + r.output_len - 1 for r in done)
    assert all(r.state in ("finished", "rejected") for r in pb.reqs)
