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


def _compare(tr, max_batch=None, max_steps=200000):
    L = _L()
    free = wl.free_order(tr.num_blocks, tr.seed)
    o = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks, free, max_batch=max_batch)
    maxblk = max(-(-(p + out - 1) // tr.block_size) for _, p, out in tr.requests)
    mb = max_batch or tr.token_budget
    maxlen = max(p + out - 1 for _, p, out in tr.requests)
    s = L.Scheduler(tr.num_blocks, tr.block_size, tr.token_budget, mb, free, maxblk)
    for a, p, out in tr.requests:
        s.add_request(a, p, out)
    n = 0
    total_pre = 0
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
        n += 1
        assert n < max_steps
    assert s.done()
    for r in o.reqs:
        info = s.request_info(r.rid)
        assert info["state"] == r.state and info["produced"] == r.produced
        assert info["preemptions"] == r.preemptions
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
