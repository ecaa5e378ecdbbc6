"""Continuous batching end to end on the GPU: the C++ FCFS scheduler picks each
iteration's batch (chunked prefills, decodes, preemption by recompute on a
tight block pool), the library appends the new rows through the scheduler's slot
mapping and runs attention through its block tables.  A host shadow records
every (layer, request, position) row written; the fp64 oracle, fed from that
shadow in the pages' contiguous layout, must agree with the GPU outputs."""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import L, assert_close
from oracle import attention as oa

pytestmark = pytest.mark.gpu


def _bf16(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("seed,num_blocks,head_dim,hq,hk", [(1, 16, 64, 8, 2), (2, 20, 128, 8, 2), (3, 18, 128, 32, 8)])
def test_scheduled_trace_matches_oracle(seed, num_blocks, head_dim, hq, hk):
    _scheduled_trace(seed, num_blocks, head_dim, hq, hk)


@pytest.mark.parametrize("seed,num_blocks,hq,hk,window", [(4, 12, 8, 2, 24), (5, 12, 32, 8, 40), (6, 12, 32, 1, 17)])
def test_scheduled_trace_rolling_window(seed, num_blocks, hq, hk, window):
    """The rolling cache end to end: the scheduler lets go of blocks that left
    every window (their table entries become -1) and hands them to other
    requests, which overwrite them; the windowed attention never reads them."""
    _scheduled_trace(seed, num_blocks, 128, hq, hk, window=window)


@pytest.mark.parametrize("max_wait", [-1, 4], ids=["static", "dynamic"])
def test_scheduled_trace_padded_batching(max_wait):
    """Padded static / dynamic batching on the same kernels: padded prefills of
    a whole batch and lock-step decodes, against the oracle over every position
    (pads included: they are computed and stored like real tokens)."""
    _scheduled_trace(7, 60, 128, 32, 8, padded=4, max_wait=max_wait)


@pytest.mark.parametrize("seed,num_blocks,window", [(0, 40, 0), (3, 16, 0), (4, 40, 24)],
                         ids=["ample", "tight_preempting", "window"])
def test_scheduled_trace_recorded_as_graphs(seed, num_blocks, window):
    _scheduled_trace(seed, num_blocks, 128, 32, 8, window=window, graphs=True)


def _scheduled_trace(seed, num_blocks, head_dim, hq, hk, window=0, padded=0, max_wait=-1, graphs=False):
    """A small scheduled trace through the library, every third step (and every
    step that preempts) checked against the oracle.  graphs: each step's layer
    calls recorded and launched as one CUDA graph (cb_graph_begin / cb_graph_end)
    on a stream of their own, one graph object per kind of step, a kind's first
    step run directly -- the serving loop of the benchmark's trace."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = L()
    stream = torch.cuda.Stream() if graphs else torch.cuda.current_stream()
    recorders, seen, recorded = {}, set(), 0
    tr = wl.small_trace(seed, num_blocks=num_blocks)
    a, bs, nl = head_dim, tr.block_size, 2
    max_seq = max(p + o - 1 for _, p, o in tr.requests)
    budget, max_reqs = tr.token_budget, tr.token_budget
    if padded:
        max_seq = max(p for _, p, _ in tr.requests) + max(o for _, _, o in tr.requests) - 1
        budget, max_reqs = padded * max(p for _, p, _ in tr.requests), padded
    maxblk = -(-max_seq // bs)
    sched = lib.Scheduler(tr.num_blocks, bs, budget, max_reqs, wl.free_order(tr.num_blocks, tr.seed), maxblk,
                          window=window, padded_batch=padded, max_wait=max_wait)
    for arr, p, o in tr.requests:
        sched.add_request(arr, p, o)
    kc = [torch.zeros(tr.num_blocks, hk, bs, a, dtype=torch.bfloat16, device="cuda") for _ in range(nl)]
    vc = [torch.zeros_like(kc[0]) for _ in range(nl)]
    ws = torch.empty(lib.cb_paged_attention_workspace_size(max_reqs, budget, budget, max_seq, hq, hk, a, bs),
                     dtype=torch.uint8, device="cuda")
    shadow = [dict() for _ in range(nl)]          # (rid, pos) -> (k row, v row), float64
    rng = np.random.default_rng(seed)
    steps = checked = preempted = released = 0
    torch.cuda.synchronize()                      # the caches and workspace above, before `stream` uses them
    while not sched.done() and steps < 2000:
        with torch.cuda.stream(stream):
            m = sched.step()
            steps += 1
            preempted += m["n_preempted"]
            b = len(m["req_ids"])
            if b == 0:
                continue
            t = int(m["cu_q_lens"][-1])
            cu = torch.from_numpy(m["cu_q_lens"]).cuda()
            ctx = torch.from_numpy(m["ctx_lens"]).cuda()
            bt = torch.from_numpy(np.ascontiguousarray(m["block_tables"])).cuda()
            sl = torch.from_numpy(m["slot_mapping"]).cuda()
            q_lens, ctx_lens = m["q_lens"].tolist(), m["ctx_lens"].tolist()
            released += int((m["block_tables"] == -1).sum()) - sum(
                max(0, maxblk - -(-(c + n) // bs)) for c, n in zip(ctx_lens, q_lens))
            check = steps % 3 == 0 or m["n_preempted"] > 0
            host = [(_bf16(rng, (t, hq, a)), _bf16(rng, (t, hk, a)), _bf16(rng, (t, hk, a))) for _ in range(nl)]
            dev = [(q.cuda(), k.cuda(), v.cuda(), torch.empty(t, hq, a, dtype=torch.bfloat16, device="cuda"))
                   for q, k, v in host]
            kind = max(q_lens) > 1
            rec = None
            if graphs and kind in seen:
                stream.synchronize()                   # the copies above are done before the recording starts
                rec = recorders.setdefault(kind, lib.Graph())
                rec.begin(stream)
                recorded += 1
            for layer in range(nl):
                dq, dk, dv, out = dev[layer]
                lib.cb_kv_append(dk, dv, sl, kc[layer], vc[layer])
                lib.cb_paged_attention_window(dq, cu, ctx, bt, kc[layer], vc[layer], out, 1 / math.sqrt(a), ws,
                                              max(q_lens), max(c + n for c, n in zip(ctx_lens, q_lens)), window)
            if rec is not None:
                rec.end(stream)
            seen.add(kind)
            for layer in range(nl):
                q, k, v = host[layer]
                out = dev[layer][3]
                kd, vd = k.double().numpy(), v.double().numpy()
                tok = 0
                for rid, n, c in zip(m["req_ids"].tolist(), q_lens, ctx_lens):
                    for i in range(n):
                        shadow[layer][(rid, c + i)] = (kd[tok], vd[tok])
                        tok += 1
                if check:
                    ks, vs = [], []
                    for rid, n, c in zip(m["req_ids"].tolist(), q_lens, ctx_lens):
                        ks.append(np.stack([shadow[layer][(rid, p)][0] for p in range(c + n)]))
                        vs.append(np.stack([shadow[layer][(rid, p)][1] for p in range(c + n)]))
                    ref = oa.attention_step(q.double().numpy(), q_lens, ctx_lens, ks, vs, 1 / math.sqrt(a), hq, hk,
                                            window=window)
                    assert_close(out.double().cpu().numpy(), ref, f"step {steps} layer {layer}")
                    checked += 1
            assert lib.cb_last_error() == 0
    assert sched.done()
    assert checked > 20
    if graphs:
        assert recorded > 20, "most steps are meant to run as graphs"
    if num_blocks == 16:
        assert preempted > 0, "the tight pool is meant to exercise preemption"
    if window:
        assert released > 0, "the window is meant to release blocks"


def test_full_size_trace_sampled():
    """The full continuous-batching trace (256 requests, 32 layers of GQA 32/8 x
    128, FCFS with a 2048-token budget, 60 GB pool) through the library; sampled
    (iteration, layer, request) outputs against the oracle.  Each layer's new
    rows come from one fixed seeded buffer indexed by the token's place in its
    step, so a map (request, position) -> that index rebuilds any request's keys
    and values on the host."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = L()
    tr = wl.trace(seed=0)
    nl, hq, hk, a, bs, budget, nb = tr.n_layers, tr.n_q_heads, tr.n_kv_heads, tr.head_dim, tr.block_size, \
        tr.token_budget, tr.num_blocks
    dev = torch.device("cuda")
    kc = [torch.zeros((nb, hk, bs, a), dtype=torch.bfloat16, device=dev) for _ in range(nl)]
    vc = [torch.zeros_like(kc[0]) for _ in range(nl)]
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    qn = [torch.randn((budget, hq, a), generator=g, device=dev, dtype=torch.bfloat16) for _ in range(nl)]
    kn = [torch.randn((budget, hk, a), generator=g, device=dev, dtype=torch.bfloat16) for _ in range(nl)]
    vn = [torch.randn((budget, hk, a), generator=g, device=dev, dtype=torch.bfloat16) for _ in range(nl)]
    out = torch.empty((budget, hq, a), dtype=torch.bfloat16, device=dev)
    maxblk = max(-(-(p + o - 1) // bs) for _, p, o in tr.requests)
    max_seq = max(p + o - 1 for _, p, o in tr.requests)
    sched = lib.Scheduler(nb, bs, budget, min(budget, lib.CB_MAX_REQS), wl.free_order(nb, tr.seed), maxblk)
    for arr, p, o in tr.requests:
        sched.add_request(arr, p, o)
    ws = torch.empty(lib.cb_paged_attention_workspace_size(min(budget, lib.CB_MAX_REQS), budget, budget, max_seq, hq,
                                                           hk, a, bs), dtype=torch.uint8, device=dev)
    check_layers = (0, 13, nl - 1)
    host = {l: (kn[l].double().cpu().numpy(), vn[l].double().cpu().numpy()) for l in check_layers}
    tok_of = {}                    # (rid, pos) -> index of the row in its step's new-row buffers
    rng = np.random.default_rng(11)
    steps = checked = 0
    while not sched.done():
        m = sched.step()
        steps += 1
        b = len(m["req_ids"])
        if b == 0:
            continue
        t = int(m["cu_q_lens"][-1])
        cu = torch.from_numpy(m["cu_q_lens"]).to(dev)
        ctx = torch.from_numpy(m["ctx_lens"]).to(dev)
        bt = torch.from_numpy(np.ascontiguousarray(m["block_tables"])).to(dev)
        sl = torch.from_numpy(m["slot_mapping"]).to(dev)
        q_lens, ctx_lens, rids = m["q_lens"].tolist(), m["ctx_lens"].tolist(), m["req_ids"].tolist()
        max_q, max_kv = max(q_lens), max(c + n for c, n in zip(ctx_lens, q_lens))
        tok = 0
        for rid, n, c in zip(rids, q_lens, ctx_lens):
            for i in range(n):
                tok_of[(rid, c + i)] = tok
                tok += 1
        check = steps % 150 == 1 or (max_q > 1 and steps % 37 == 0)
        for layer in range(nl):
            lib.cb_kv_append(kn[layer][:t], vn[layer][:t], sl, kc[layer], vc[layer])
            lib.cb_paged_attention(qn[layer][:t], cu, ctx, bt, kc[layer], vc[layer], out[:t], 1 / math.sqrt(a), ws,
                                   max_q, max_kv)
            if check and layer in check_layers:
                got = out[:t].double().cpu().numpy()
                qd = qn[layer][:t].double().cpu().numpy()
                kd, vd = host[layer]
                cu_h = m["cu_q_lens"]
                picks = sorted(set([0, b - 1] + rng.choice(b, size=min(2, b), replace=False).tolist()))
                for j in picks:
                    rid, n, c = rids[j], q_lens[j], ctx_lens[j]
                    idx = [tok_of[(rid, p)] for p in range(c + n)]
                    # a long chunk: its first and last rows and a few in between
                    rows = sorted(set([0, n - 1] + rng.choice(n, size=min(n, 4), replace=False).tolist()))
                    ref = oa.attention_rows(qd[cu_h[j] + np.array(rows)], kd[idx], vd[idx], [c + i for i in rows],
                                            1 / math.sqrt(a), hq, hk)
                    assert_close(got[cu_h[j] + np.array(rows)], ref, f"step {steps} layer {layer} request {rid}")
                    checked += 1
        assert lib.cb_last_error() == 0, f"step {steps}"
    assert steps > 1000 and checked > 60
    del kc, vc
    torch.cuda.empty_cache()
