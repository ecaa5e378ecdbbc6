"""The C++ scheduler (cb_sched_*) against the FCFS scheduler oracle: identical
metadata, step by step, on tight traces that preempt, on the pages' worked
examples and on the full-size continuous-batching trace."""
import numpy as np
import pytest

import workloads as wl
from oracle.scheduler import FCFSScheduler


def _L():
    from paged_kv_cache_cb_gb300 import _lib as L
    import os
    if not os.path.exists(L.LIB_PATH):
        from paged_kv_cache_cb_gb300 import build
        build.build()
    return L


def _compare(tr, max_batch=None, max_steps=200000, free=None, window=0):
    L = _L()
    free = wl.free_order(tr.num_blocks, tr.seed) if free is None else free
    o = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks, free, max_batch=max_batch,
                      window=window)
    maxblk = max(-(-(t[1] + t[2] - 1) // tr.block_size) for t in tr.requests)
    mb = max_batch or tr.token_budget
    maxlen = max(t[1] + t[2] - 1 for t in tr.requests)
    s = L.Scheduler(tr.num_blocks, tr.block_size, tr.token_budget, mb, free, maxblk, window=window)
    for t in tr.requests:
        s.add_request(*t)
    n = 0
    total_pre = 0
    total_copies = 0
    while not o.done():
        assert not s.done()
        m = o.step()
        g = s.step()
        assert np.array_equal(g["req_ids"], m.req_ids), n
        assert np.array_equal(g["q_lens"], m.q_lens), n
        assert np.array_equal(g["ctx_lens"], m.ctx_lens), n
        assert np.array_equal(g["cu_q_lens"], np.concatenate([[0], np.cumsum(m.q_lens)]).astype(np.int32))
        assert np.array_equal(g["slot_mapping"], m.slot_mapping), n
        for i, tab in enumerate(m.block_tables):
            row = g["block_tables"][i]
            assert row[:len(tab)].tolist() == tab
            assert np.all(row[len(tab):] == -1)
        assert g["n_preempted"] == len(m.preempted)
        total_pre += g["n_preempted"]
        assert s.free_blocks() == len(o.free)
        assert s.kv_memory(maxlen) == o.kv_memory(maxlen), n
        assert s.step_copies().tolist() == [list(c) for c in m.copies], n
        total_copies += len(m.copies)
        n += 1
        assert n < max_steps
    assert s.done()
    for r in o.reqs:
        info = s.request_info(r.rid)
        assert info["state"] == r.state and info["produced"] == r.produced
        assert info["preemptions"] == r.preemptions
    _compare.copies = total_copies
    return n, total_pre


@pytest.mark.parametrize("seed", range(10))
def test_cpp_scheduler_equals_oracle_on_tight_traces(seed):
    _compare(wl.small_trace(seed))


def test_cpp_scheduler_preempts_like_the_oracle():
    total = sum(_compare(wl.small_trace(seed, num_blocks=16))[1] for seed in range(6))
    assert total > 0


@pytest.mark.parametrize("max_batch", [2, 5])
def test_cpp_scheduler_batch_cap(max_batch):
    _compare(wl.small_trace(3), max_batch=max_batch)


class _Hand:
    def __init__(self, requests, token_budget, block_size, num_blocks):
        self.requests, self.token_budget, self.block_size, self.num_blocks = requests, token_budget, block_size, num_blocks
        self.seed = 0


@pytest.mark.parametrize("case", ["batch_cap", "oldest_prefix_dropped", "copy_waits_for_a_block"])
def test_cpp_scheduler_on_the_hand_worked_cases(case):
    """The hand-worked scheduler cases of the oracle's pins (request cap, oldest
    prefix dropped first, a copy-on-write admission waiting for a free block),
    with their explicit free-list order."""
    if case == "batch_cap":
        _compare(_Hand([(0, 4, 3)] * 4, 64, 16, 8), max_batch=2, free=list(range(8)))
    elif case == "oldest_prefix_dropped":
        _compare(_Hand([(0, 5, 1, 0, 4), (1, 5, 1, 1, 4), (2, 16, 2), (4, 6, 1, 1, 4)], 64, 4, 6),
                 free=list(range(6)))
    else:
        _compare(_Hand([(0, 7, 2, 0, 6), (0, 7, 2), (1, 7, 1, 0, 6)], 64, 4, 4), free=list(range(4)))


def test_cpp_scheduler_full_trace_prefix():
    """The first 150 steps of the 256-request trace (60 GB pool, 2048-token budget)."""
    tr = wl.trace(seed=0)
    L = _L()
    free = wl.free_order(tr.num_blocks, tr.seed)
    o = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks, free)
    maxblk = max(-(-(p + out - 1) // tr.block_size) for _, p, out in tr.requests)
    s = L.Scheduler(tr.num_blocks, tr.block_size, tr.token_budget, tr.token_budget, free, maxblk)
    for a, p, out in tr.requests:
        s.add_request(a, p, out)
    for n in range(150):
        m, g = o.step(), s.step()
        assert np.array_equal(g["req_ids"], m.req_ids) and np.array_equal(g["slot_mapping"], m.slot_mapping)
        assert int(m.q_lens.sum()) <= tr.token_budget


def test_cpp_scheduler_rejects_bad_free_list():
    L = _L()
    with pytest.raises(L.CBError):
        L.Scheduler(4, 16, 8, 8, [0, 1, 1, 3], 4)


@pytest.mark.parametrize("seed", range(8))
def test_cpp_scheduler_shares_prefixes_like_the_oracle(seed):
    """Prefix groups: shared blocks, copy-on-write pairs, dropped prefixes and
    preemptions, identical to the oracle step by step."""
    tr = wl.with_prefixes(wl.small_trace(seed, num_blocks=24 + 4 * (seed % 3)), 3, 20 + seed, seed=seed)
    _compare(tr)
    assert _compare.copies > 0 or (20 + seed) % 16 == 0


def test_cpp_scheduler_prefix_trace_prefix():
    """The first 300 steps of the 256-request trace with 8 shared 1000-token system prompts."""
    _compare_steps(wl.with_prefixes(wl.trace(seed=0), 8, 1000, seed=0), 300)


def _compare_steps(tr, steps):
    L = _L()
    free = wl.free_order(tr.num_blocks, tr.seed)
    o = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks, free)
    maxblk = max(-(-(t[1] + t[2] - 1) // tr.block_size) for t in tr.requests)
    s = L.Scheduler(tr.num_blocks, tr.block_size, tr.token_budget, tr.token_budget, free, maxblk)
    for t in tr.requests:
        s.add_request(*t)
    for n in range(steps):
        m, g = o.step(), s.step()
        assert np.array_equal(g["req_ids"], m.req_ids) and np.array_equal(g["slot_mapping"], m.slot_mapping), n
        assert np.array_equal(g["ctx_lens"], m.ctx_lens), n
        assert s.step_copies().tolist() == [list(c) for c in m.copies], n


def test_cpp_scheduler_rejects_bad_prefix():
    L = _L()
    s = L.Scheduler(8, 16, 32, 8, list(range(8)), 4)
    with pytest.raises(L.CBError):
        s.add_request(0, 10, 2, 0, 10)          # the prefix must leave a prompt token
    s.add_request(0, 20, 2, 1, 5)
    with pytest.raises(L.CBError):
        s.add_request(0, 20, 2, 1, 6)           # one prefix length per group


def test_scheduler_memory_and_copies_argument_checks():
    import ctypes
    L = _L()
    lib = L.lib()
    s = L.Scheduler(8, 16, 32, 4, list(range(8)), 4)
    out = np.zeros(4, np.int64)
    assert lib.cb_sched_kv_memory(s._h, 0, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))) == L.CB_EINVAL
    assert lib.cb_sched_kv_memory(None, 10, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))) == L.CB_EINVAL
    assert lib.cb_sched_step_copies(s._h, None, -1) == L.CB_EINVAL
    assert lib.cb_sched_step_copies(s._h, None, 0) == 0          # no step yet: no copies
    s.add_request(0, 20, 2, 0, 18)
    s.add_request(1, 20, 2, 0, 18)
    s.step()
    s.step()                                                      # the second request takes a copy of the partial block
    assert s.step_copies().shape == (1, 2)
    assert lib.cb_sched_step_copies(s._h, None, 0) == L.CB_ESTATE   # one pair does not fit in zero


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("window", [1, 17, 40])
def test_cpp_scheduler_rolling_window(seed, window):
    """The rolling window's block release (tables with -1 before the window)
    step by step, on tight traces, with and without shared prefixes."""
    _compare(wl.small_trace(seed, num_blocks=12), window=window)
    _compare(wl.with_prefixes(wl.small_trace(seed, num_blocks=20), 3, 9 + seed, seed=seed), window=window)


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("max_wait", [-1, 0, 3])
def test_cpp_padded_batching_equals_oracle(seed, max_wait):
    """Static (max_wait -1) and dynamic batching with padding: the C++ planner
    equals oracle.scheduler.PaddedBatcher step by step, real tokens included."""
    from oracle.scheduler import PaddedBatcher
    L = _L()
    tr = wl.small_trace(seed, num_blocks=40)
    free = wl.free_order(tr.num_blocks, tr.seed)
    B = 4
    o = PaddedBatcher(tr.requests, B, tr.block_size, tr.num_blocks, free, max_wait=None if max_wait < 0 else max_wait)
    maxp = max(t[1] for t in tr.requests)
    maxblk = max(-(-(t[1] + t[2] - 1) // tr.block_size) for t in tr.requests) + -(-maxp // tr.block_size)
    s = L.Scheduler(tr.num_blocks, tr.block_size, B * maxp, B, free, maxblk, padded_batch=B, max_wait=max_wait)
    for t in tr.requests:
        s.add_request(*t)
    n = 0
    while not o.done():
        assert not s.done()
        m, real = o.step()
        g = s.step()
        assert np.array_equal(g["req_ids"], m.req_ids), n
        assert np.array_equal(g["q_lens"], m.q_lens), n
        assert np.array_equal(g["ctx_lens"], m.ctx_lens), n
        assert np.array_equal(g["slot_mapping"], m.slot_mapping), n
        for i, tab in enumerate(m.block_tables):
            assert g["block_tables"][i][:len(tab)].tolist() == tab
        assert g["real_tokens"] == real, n
        assert s.free_blocks() == len(o.free)
        n += 1
    assert s.done()
