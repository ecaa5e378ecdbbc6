"""Rolling-window attention on the GPU ([KVB] "Rolling KV Cache", a heading
without a body; reading: a query at position p sees keys p - W + 1 .. p)
through cb_paged_attention_window and cb_kv_append_paged_attention_window,
against the fp64 oracle with the same window.  Every kernel path: the CUDA-core
decode (MHA, GQA 4), the block-tile decode (8, 2 and 1 KV heads), prefill tiles
(round robin and balanced pieces) and the mixed launch.  Blocks wholly before a
request's window hold NaN, so a read of one would show."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import L, assert_close, device_step, f64, oracle_step, sampled_request_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L().lib()


def _poison_outside_windows(shape, inp, window):
    """A copy of the inputs with NaN in every block that no query of the step
    can see: before the window of the request's earliest new token, or not the
    request's at all.  (The oracle reads the clean inputs: its P . V would turn
    a zero weight times NaN into NaN.)"""
    inp = dict(inp)
    keep = torch.zeros(shape.num_blocks, dtype=torch.bool)
    for r, (c, n) in enumerate(zip(shape.ctx_lens, shape.q_lens)):
        lo = max(0, c + 1 - window) if window else 0
        for b in range(lo // shape.block_size, -(-(c + n) // shape.block_size)):
            keep[int(inp["block_tables"][r, b])] = True
    for name in ("k_pool", "v_pool"):
        inp[name] = inp[name].masked_fill(~keep[:, None, None, None], float("nan"))
    return inp


def _window_parity(shape, window, fused=False, scale=None):
    inp = wl.step_inputs_cpu(shape)
    out, _, _, _ = device_step(shape, _poison_outside_windows(shape, inp, window), window=window, fused=fused,
                               scale=scale)
    assert torch.isfinite(out).all()
    return assert_close(f64(out), oracle_step(shape, inp, window=window, scale=scale), f"{shape.name} W={window}")


SHAPES = [(8, 8, 64), (32, 8, 128), (16, 4, 128), (32, 2, 128), (32, 1, 128)]
IDS = ["mha8x64", "gqa32x8", "gqa16x4", "gqa32x2", "mqa32x1"]


@pytest.mark.parametrize("hq,hkv,a", SHAPES, ids=IDS)
@pytest.mark.parametrize("window", [1, 16, 100, 1000])
def test_decode_window(hq, hkv, a, window):
    base = wl.random_step(300 + hkv + window, n_reqs=12, max_ctx=3000, max_q=1, n_q_heads=hq, n_kv_heads=hkv,
                          head_dim=a, p_decode=1.0)
    ctx = list(base.ctx_lens)
    ctx[:6] = [0, 15, window - 1, window, window + 1, 2 * window + 17]
    _window_parity(wl.scaled(base, ctx_lens=ctx, num_blocks=base.num_blocks + 400), window)


@pytest.mark.parametrize("hq,hkv,a", SHAPES, ids=IDS)
@pytest.mark.parametrize("window", [1, 37, 128, 300])
def test_mixed_window(hq, hkv, a, window):
    """Decodes and prefill chunks (several query tiles, stored prefixes) in one
    launch: the chunks' rows see windows that start in different key tiles."""
    shape = wl.StepShape(f"mixed_w_{hq}x{hkv}", hq, hkv, a, 16, 900, q_lens=(1, 300, 1, 129, 2, 77, 1),
                         ctx_lens=(500, 200, 33, 0, 333, 1000, 4000), seed=320 + hkv + window)
    _window_parity(shape, window)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 1)], ids=["gqa32x8", "mqa32x1"])
def test_one_call_window(hq, hkv):
    shape = wl.random_step(340 + hkv, n_reqs=9, max_ctx=2000, max_q=90, n_q_heads=hq, n_kv_heads=hkv, head_dim=128,
                           p_decode=0.5)
    _window_parity(shape, 200, fused=True)


def test_window_at_least_every_context_equals_no_window():
    shape = wl.random_step(350, n_reqs=9, max_ctx=1500, max_q=60, n_q_heads=32, n_kv_heads=8, head_dim=128)
    inp = wl.step_inputs_cpu(shape)
    o0, _, _, _ = device_step(shape, inp)
    o1, _, _, _ = device_step(shape, inp, window=100000)
    o2, _, _, _ = device_step(shape, inp, window=0)
    assert torch.equal(o0, o1) and torch.equal(o0, o2)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 1)], ids=["gqa32x8", "mqa32x1"])
def test_long_chunk_window_balanced_pieces(hq, hkv):
    """A 2048-token chunk after 3000 stored tokens with a 700-key window: more
    tile pairs than CTAs, so the balanced pieces run; each pair starts at the
    key tile its earliest row can see."""
    shape = wl.StepShape(f"long_w_{hq}x{hkv}", hq, hkv, 128, 16, 1200, q_lens=(1, 2048, 1),
                         ctx_lens=(5000, 3000, 17), seed=360 + hkv)
    inp = wl.step_inputs_cpu(shape)
    out, _, _, _ = device_step(shape, _poison_outside_windows(shape, inp, 700), window=700)
    cu = np.concatenate([[0], np.cumsum(shape.q_lens)])
    rows = [0, 1, 7, 8, 500, 1023, 1024, 2046, 2047]
    for r in range(shape.n_reqs):
        rr = rows if shape.q_lens[r] > 1 else None
        ref, rr = sampled_request_oracle(shape, inp, r, rr, window=700)
        assert_close(f64(out[cu[r]:cu[r + 1]])[rr], ref, f"{shape.name} request {r}")


def test_negative_window_is_rejected():
    lib = L()
    shape = wl.tiny()
    inp = wl.step_inputs_cpu(shape)
    with pytest.raises(lib.CBError) as e:
        device_step(shape, inp, window=-1)
    assert e.value.code == lib.CB_EINVAL
