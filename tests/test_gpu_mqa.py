"""MQA and wide GQA on the GPU ([KVN] MQA/GQA: one KV head serves every query
head; GQA groups of 16): 32 query heads on 1 KV head (G = 32) and on 2 (G = 16),
head_dim 128.  Decode runs the block-tile pipeline with 128-row tiles of 8 (or
4) physical blocks of those heads; prefill chunks run 128-row query tiles of 4
(or 8) tokens x 32 (or 16) heads.  Against the fp64 oracle, with the parity
bounds of the other GPU tests."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import L, assert_close, device_step, f64, oracle_step, sampled_request_oracle

pytestmark = pytest.mark.gpu

SHAPES = [(32, 1), (32, 2)]
IDS = ["mqa32x1", "gqa32x2"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L().lib()


def _parity(shape, scale=None, fused=False):
    inp = wl.step_inputs_cpu(shape)
    out, _, _, _ = device_step(shape, inp, scale=scale, fused=fused)
    return assert_close(f64(out), oracle_step(shape, inp, scale=scale), shape.name)


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
def test_decode_edges(hq, hkv):
    """One key, block and tile boundaries (16, 128 keys), tails, and contexts of
    several chunks (merged splits)."""
    base = wl.random_step(200 + hkv, n_reqs=14, max_ctx=3000, max_q=1, n_q_heads=hq, n_kv_heads=hkv, head_dim=128,
                          p_decode=1.0)
    ctx = list(base.ctx_lens)
    ctx[:9] = [0, 15, 16, 127, 128, 129, 4095, 8190, 12000]
    _parity(wl.scaled(base, ctx_lens=ctx, num_blocks=base.num_blocks + 2000))


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
@pytest.mark.parametrize("n_reqs", [1, 2, 5, 300])
def test_decode_step_sizes(hq, hkv, n_reqs):
    """From one request (cut into many short chunks over the grid) to 300."""
    shape = wl.random_step(210 + n_reqs + hkv, n_reqs=n_reqs, max_ctx=6000, max_q=1, n_q_heads=hq, n_kv_heads=hkv,
                           head_dim=128, p_decode=1.0)
    _parity(shape)


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
def test_decode_running_max_rescales(hq, hkv):
    shape = wl.random_step(230 + hkv, n_reqs=6, max_ctx=2500, max_q=1, n_q_heads=hq, n_kv_heads=hkv, head_dim=128,
                           p_decode=1.0)
    _parity(shape, scale=0.6)


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
def test_mixed_decodes_and_chunks(hq, hkv):
    """Decodes and prefill chunks in one launch: chunks of several query tiles
    after stored prefixes of 0, mid-block and long lengths."""
    shape = wl.StepShape(f"mixed_{hq}x{hkv}", hq, hkv, 128, 16, 900,
                         q_lens=(1, 300, 1, 129, 2, 1, 77, 1), ctx_lens=(500, 200, 33, 0, 333, 4000, 1000, 16),
                         seed=240 + hkv)
    _parity(shape)


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
def test_unwritten_cache_slots_do_not_leak(hq, hkv):
    """Every slot no request owns holds NaN: outputs stay finite and correct."""
    shape = wl.random_step(250 + hkv, n_reqs=11, max_ctx=1200, max_q=150, n_q_heads=hq, n_kv_heads=hkv,
                           head_dim=128, p_decode=0.6)
    inp = wl.step_inputs_cpu(shape)
    keep = torch.zeros(shape.num_blocks, shape.block_size, dtype=torch.bool)
    for r, c in enumerate(shape.ctx_lens):
        for p in range(c):
            keep[int(inp["block_tables"][r, p // shape.block_size]), p % shape.block_size] = True
    poison = ~keep[:, None, :, None]
    for name in ("k_pool", "v_pool"):
        inp[name] = inp[name].masked_fill(poison, float("nan"))
    out, _, _, _ = device_step(shape, inp)
    assert torch.isfinite(out).all()
    assert_close(f64(out), oracle_step(shape, inp), shape.name)


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
def test_one_call_equals_two_calls(hq, hkv):
    """cb_kv_append_paged_attention (the append inside the cooperative launch)
    gives the same bits and the same cache as cb_kv_append + cb_paged_attention."""
    shape = wl.random_step(260 + hkv, n_reqs=9, max_ctx=2000, max_q=90, n_q_heads=hq, n_kv_heads=hkv, head_dim=128,
                           p_decode=0.5)
    inp = wl.step_inputs_cpu(shape)
    o1, k1, v1, _ = device_step(shape, inp)
    o2, k2, v2, _ = device_step(shape, inp, fused=True)
    assert torch.equal(o1, o2)
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
def test_long_chunk_balanced_pieces(hq, hkv):
    """A 2048-token chunk after 3000 stored tokens (more tile pairs than CTAs:
    the balanced prefill with pieces merged after the grid-wide barrier) with a
    few decodes; sampled rows against the oracle."""
    shape = wl.StepShape(f"long_{hq}x{hkv}", hq, hkv, 128, 16, 1200, q_lens=(1, 2048, 1, 1),
                         ctx_lens=(5000, 3000, 17, 2000), seed=270 + hkv)
    inp = wl.step_inputs_cpu(shape)
    out, _, _, _ = device_step(shape, inp)
    cu = np.concatenate([[0], np.cumsum(shape.q_lens)])
    rows = sorted({0, 1, 7, 8, 500, 1023, 1024, 2046, 2047})
    for r in range(shape.n_reqs):
        rr = rows if shape.q_lens[r] > 1 else None
        ref, rr = sampled_request_oracle(shape, inp, r, rr)
        assert_close(f64(out[cu[r]:cu[r + 1]])[rr], ref, f"{shape.name} request {r}")


@pytest.mark.parametrize("hq,hkv", SHAPES, ids=IDS)
def test_full_size_decode(hq, hkv):
    """256 decodes with contexts uniform in [1024, 16384] over a 20 GB pool (the
    MQA decode workload's shape): sampled requests against the oracle."""
    shape = wl.mqa_decode(n_kv_heads=hkv)
    inp = wl.step_inputs_device(shape, "cuda")
    out, _, _, _ = device_step(shape, inp)
    order = np.argsort(shape.ctx_lens)
    for r in [int(order[0]), int(order[-1]), 0, 100, 255]:
        ref, rows = sampled_request_oracle(shape, inp, r)
        assert_close(f64(out[r:r + 1]), ref, f"{shape.name} request {r}")
    del inp, out
    torch.cuda.empty_cache()
