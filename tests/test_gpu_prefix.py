"""GPU parity of shared prompt prefixes ([KVN] §与Prefix Caching的结合; [KVB] §思想:
blocks shared by pointing block tables at them).

The scheduler lets requests of a prefix group hold the blocks another request
filled with the group's prefix, and copies a partial last block before a
request writes its own tokens into it (copy-on-write, cb_copy_blocks).  Here
each step of such traces runs on the GPU: copies, then the one-call append +
attention.  Key/value rows depend only on (group, position) for the shared
positions and on (request, position) otherwise, so every request's output must
equal the oracle's attention over its own contiguous keys -- the result a run
without sharing gives."""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import L, assert_close
from oracle import attention as oa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L().lib()


def test_copy_blocks_is_bit_exact():
    lib = L()
    g = torch.Generator().manual_seed(3)
    kc = torch.randn(40, 8, 16, 128, generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn(40, 8, 16, 128, generator=g).to(torch.bfloat16).cuda()
    want_k, want_v = kc.clone(), vc.clone()
    pairs = [(3, 17), (3, 20), (39, 0), (5, 6)]
    for s_, d_ in pairs:
        want_k[d_], want_v[d_] = want_k[s_], want_v[s_]
    lib.cb_copy_blocks(torch.tensor(pairs, dtype=torch.int32).cuda(), kc, vc)
    assert lib.cb_last_error() == 0
    assert torch.equal(kc.view(torch.int16), want_k.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), want_v.view(torch.int16))
    lib.cb_copy_blocks(torch.tensor([(2, 40)], dtype=torch.int32).cuda(), kc, vc)   # outside the pool: skipped
    assert lib.cb_last_error() == lib.CB_EDEVICE
    assert torch.equal(kc.view(torch.int16), want_k.view(torch.int16))


def _rows(n_contents, max_len, heads, a, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n_contents, max_len, heads, a)).astype(np.float32)


@pytest.mark.parametrize("hq,hk,a,prefix,seed", [(32, 8, 128, 20, 0), (32, 8, 128, 37, 1), (16, 8, 128, 32, 2),
                                                 (4, 4, 64, 23, 3)])
def test_prefix_trace_matches_unshared_oracle(hq, hk, a, prefix, seed):
    lib = L()
    base = wl.small_trace(seed, num_blocks=28)
    tr = wl.with_prefixes(base, 3, prefix, seed=seed)
    bs = tr.block_size
    max_len = max(p + o for _, p, o, _, _ in tr.requests)
    n_req = len(tr.requests)
    # content ids: groups 0..2, then 3 + request id
    K = _rows(3 + n_req, max_len, hk, a, seed)
    V = _rows(3 + n_req, max_len, hk, a, seed + 1)
    Q = _rows(n_req, max_len, hq, a, seed + 2)
    bf = lambda x: torch.from_numpy(x).to(torch.bfloat16)
    Kb, Vb, Qb = bf(K), bf(V), bf(Q)                 # what the device sees
    K64, V64, Q64 = (t.to(torch.float64).numpy() for t in (Kb, Vb, Qb))

    def content(rid, p):
        _, _, _, g, pl = tr.requests[rid]
        return g if g >= 0 and p < pl else 3 + rid

    maxblk = max(-(-(p + o - 1) // bs) for _, p, o, _, _ in tr.requests)
    sched = lib.Scheduler(tr.num_blocks, bs, tr.token_budget, tr.token_budget, wl.free_order(tr.num_blocks, tr.seed),
                          maxblk)
    for t in tr.requests:
        sched.add_request(*t)
    kc = torch.zeros(tr.num_blocks, hk, bs, a, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    scale = 1.0 / math.sqrt(a)
    ws = torch.empty(lib.cb_paged_attention_workspace_size(tr.token_budget, tr.token_budget, tr.token_budget,
                                                           max_len, hq, hk, a, bs), dtype=torch.uint8, device="cuda")
    copies = shared_steps = 0
    while not sched.done():
        m = sched.step()
        pairs = sched.step_copies()
        if len(pairs):
            lib.cb_copy_blocks(torch.from_numpy(pairs).cuda(), kc, vc)
            copies += len(pairs)
        b = len(m["req_ids"])
        if b == 0:
            continue
        rows = [(int(r), p) for r, c, n in zip(m["req_ids"], m["ctx_lens"], m["q_lens"]) for p in range(c, c + n)]
        k_new = torch.stack([Kb[content(r, p), p] for r, p in rows]).cuda()
        v_new = torch.stack([Vb[content(r, p), p] for r, p in rows]).cuda()
        q = torch.stack([Qb[r, p] for r, p in rows]).cuda()
        out = torch.empty_like(q)
        q_lens, ctx = m["q_lens"].astype(np.int32), m["ctx_lens"].astype(np.int32)
        lib.cb_kv_append_paged_attention(
            k_new, v_new, torch.from_numpy(m["slot_mapping"][:len(rows)]).cuda(), q,
            torch.from_numpy(m["cu_q_lens"][:b + 1].astype(np.int32)).cuda(), torch.from_numpy(ctx).cuda(),
            torch.from_numpy(np.ascontiguousarray(m["block_tables"][:b])).cuda(), kc, vc, out, scale, ws,
            int(q_lens.max()), int((q_lens + ctx).max()))
        status = lib.cb_last_error()
        assert status == 0, lib.cb_strerror(status)
        ks = [np.stack([K64[content(int(r), p), p] for p in range(c + n)]) for r, c, n in zip(m["req_ids"], ctx, q_lens)]
        vs = [np.stack([V64[content(int(r), p), p] for p in range(c + n)]) for r, c, n in zip(m["req_ids"], ctx, q_lens)]
        qs = np.stack([Q64[r, p] for r, p in rows])
        ref = oa.attention_step(qs, q_lens.tolist(), ctx.tolist(), ks, vs, scale, hq, hk)
        assert_close(out.to(torch.float64).cpu().numpy(), ref, f"step {m['step'] if 'step' in m else ''}")
        shared_steps += any(tr.requests[int(r)][3] >= 0 and c > 0 for r, c in zip(m["req_ids"], ctx))
    assert shared_steps > 0
    assert copies > 0 or prefix % bs == 0
