"""cb_paged_attention_noalloc: the attention step for callers that cannot
allocate device memory when they run it (a plugin whose host owns all device
memory through its own arena, a serving loop that forbids allocation because
cudaMalloc may synchronise and has unbounded latency).  Its scratch is a fixed
array inside the library, so the caller passes only inputs and outputs.

Checked here through the C ABI against cb_paged_attention (the entry point that
takes a caller-owned workspace), on two calls in a row, within the parity
tolerance of the other GPU tests.  This file is collected last on purpose."""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import ATOL, L, cu_of

pytestmark = pytest.mark.gpu


def _step_buffers(shape):
    lib = L()
    inp = wl.step_inputs_cpu(shape)
    dev = "cuda"
    slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    kc, vc = inp["k_pool"].to(dev), inp["v_pool"].to(dev)
    lib.cb_kv_append(inp["k_new"].to(dev), inp["v_new"].to(dev), torch.from_numpy(slots).to(dev), kc, vc)
    meta = dict(q=inp["q"].to(dev), cu=torch.from_numpy(cu_of(shape.q_lens)).to(dev),
                ctx=torch.tensor(shape.ctx_lens, dtype=torch.int32, device=dev),
                bt=torch.from_numpy(inp["block_tables"]).to(dev), kc=kc, vc=vc,
                max_q=max(shape.q_lens), max_kv=max(c + n for c, n in zip(shape.ctx_lens, shape.q_lens)),
                scale=1.0 / math.sqrt(shape.head_dim))
    return meta


def _with_workspace(shape, m):
    lib = L()
    wsb = lib.cb_paged_attention_workspace_size(shape.n_reqs, shape.n_tokens, m["max_q"], m["max_kv"],
                                                shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.block_size)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(m["q"])
    lib.cb_paged_attention(m["q"], m["cu"], m["ctx"], m["bt"], m["kc"], m["vc"], out, m["scale"], ws,
                           m["max_q"], m["max_kv"])
    assert lib.cb_last_error() == 0
    return out


def _no_alloc(m):
    lib = L()
    out = torch.full_like(m["q"], float("nan"))
    lib.cb_paged_attention_noalloc(m["q"], m["cu"], m["ctx"], m["bt"], m["kc"], m["vc"], out, m["scale"],
                                   m["max_q"], m["max_kv"])
    assert lib.cb_last_error() == 0
    return out


@pytest.mark.parametrize("shape", [
    wl.tiny(),                                                              # mixed: decodes, a chunk, a prefill
    wl.random_step(21, n_reqs=12, max_ctx=2500, max_q=1, n_q_heads=8, n_kv_heads=2, head_dim=128, p_decode=1.0),
    wl.random_step(22, n_reqs=9, max_ctx=900, max_q=200, n_q_heads=16, n_kv_heads=4, head_dim=128),
    # 8 KV heads: the block-tile decode (its own launch, and the mixed launch's decode phase)
    wl.random_step(23, n_reqs=12, max_ctx=2500, max_q=1, n_q_heads=32, n_kv_heads=8, head_dim=128, p_decode=1.0),
    wl.random_step(24, n_reqs=9, max_ctx=900, max_q=200, n_q_heads=32, n_kv_heads=8, head_dim=128),
], ids=lambda s: f"{s.name}_h{s.n_q_heads}_{s.n_kv_heads}")
def test_no_alloc_matches_workspace_entry_point_twice(shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m = _step_buffers(shape)
    ref_t = _with_workspace(shape, m)
    ref = ref_t.float().cpu().numpy()
    lib = L()
    fits = lib.cb_paged_attention_workspace_size(shape.n_reqs, shape.n_tokens, m["max_q"], m["max_kv"], shape.n_q_heads,
                                                 shape.n_kv_heads, shape.head_dim,
                                                 shape.block_size) <= lib.CB_NOALLOC_SCRATCH_BYTES
    for call in range(2):          # the shared scratch keeps the previous call's contents
        got_t = _no_alloc(m)
        got = got_t.float().cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        err = float(np.abs(got - ref).max())
        assert err <= ATOL, f"call {call}: max abs difference {err}"
        if fits:                   # the same plan as the workspace entry point: the same bits
            assert torch.equal(got_t, ref_t), f"call {call}: planned differently"


def test_no_alloc_rejects_steps_larger_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = L()
    n_reqs, max_kv = 2048, 32768
    need = lib.cb_paged_attention_workspace_size(n_reqs, n_reqs, 1, max_kv, 32, 8, 128, 16)
    assert need > lib.CB_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(n_reqs, 32, 128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.CBError) as e:
        lib.cb_paged_attention_noalloc(q, torch.arange(n_reqs + 1, dtype=torch.int32, device="cuda"),
                                       torch.zeros(n_reqs, dtype=torch.int32, device="cuda"),
                                       torch.zeros(n_reqs, 1, dtype=torch.int32, device="cuda"), cache, cache, q,
                                       0.1, 1, max_kv)
    assert e.value.code == lib.CB_EWORKSPACE
