"""GPU parity of cb_kv_append_paged_attention, the whole step of a layer in one
call ([CB] Chunked prefill: the chunk's K/V states are stored, then its queries
attend to the cached prefix and to themselves).

Where the attention launch is cooperative (8 KV heads, head_dim 128, G >= 2)
the append runs inside it, ahead of a grid-wide counter; other shapes run the
append kernel first.  Either way the cache must equal the oracle's append bit
for bit, the outputs must match the fp64 oracle within the attention tolerance,
and, since the attention arithmetic is the same code, equal the two separate
calls' outputs exactly."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import L, assert_close, device_step, f64, oracle_step, sampled_request_oracle
from oracle import paged as op

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L().lib()


def _one_launch(shape):
    return shape.n_kv_heads == 8 and shape.head_dim == 128 and shape.n_q_heads // shape.n_kv_heads >= 2


SHAPES = [
    # decode only, block-tile kernel with the append inside
    wl.scaled(wl.random_step(81, n_reqs=11, max_ctx=3000, max_q=1, n_q_heads=32, n_kv_heads=8, head_dim=128,
                             p_decode=1.0), name="fused_decode_32x8",
              ctx_lens=[0, 15, 16, 2047, 2990, 5, 700, 1, 31, 1200, 64]),
    wl.random_step(82, n_reqs=9, max_ctx=1500, max_q=1, n_q_heads=16, n_kv_heads=8, head_dim=128, p_decode=1.0),
    # mixed: prefill chunks (fresh and after a stored prefix) with decodes
    wl.StepShape("fused_mixed_32x8", 32, 8, 128, 16, 400, q_lens=(1, 300, 1, 129, 1, 1, 40, 200),
                 ctx_lens=(500, 0, 1500, 128, 0, 17, 333, 0), seed=83),
    wl.StepShape("fused_mixed_64x8", 64, 8, 128, 16, 200, q_lens=(1, 77, 1, 1), ctx_lens=(900, 15, 16, 1),
                 seed=84),
    # shapes whose attention launch is not cooperative: two launches
    wl.random_step(85, n_reqs=9, max_ctx=1500, max_q=1, n_q_heads=8, n_kv_heads=8, head_dim=128, p_decode=1.0),
    wl.random_step(86, n_reqs=7, max_ctx=600, max_q=200, n_q_heads=16, n_kv_heads=4, head_dim=64, p_decode=0.5),
    wl.tiny(),
]


def _want_cache(shape, inp, slots):
    want_k = inp["k_pool"].view(torch.int16).numpy().copy()
    want_v = inp["v_pool"].view(torch.int16).numpy().copy()
    op.append_rows(want_k, inp["k_new"].view(torch.int16).numpy(), slots, shape.block_size)
    op.append_rows(want_v, inp["v_new"].view(torch.int16).numpy(), slots, shape.block_size)
    return want_k, want_v


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s.name}_h{s.n_q_heads}_{s.n_kv_heads}_a{s.head_dim}")
def test_fused_step_matches_oracle_cache_and_separate_calls(shape):
    lib = L()
    inp = wl.step_inputs_cpu(shape)
    out, kc, vc, _ = device_step(shape, inp, fused=True)
    assert lib.cb_last_launch_count() == (1 if _one_launch(shape) else 2)
    slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    want_k, want_v = _want_cache(shape, inp, slots)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy(), want_k)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy(), want_v)
    assert_close(f64(out), oracle_step(shape, inp), shape.name)
    out_sep, _, _, _ = device_step(shape, inp)
    assert torch.equal(out.view(torch.int16), out_sep.view(torch.int16))


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2], SHAPES[4]], ids=lambda s: s.name)
def test_fused_negative_slot_skips_and_bad_slot_is_reported(shape):
    """Slot -1 leaves the cache row alone; a slot past the cache is skipped and
    flagged.  Requests whose tokens were all stored still match the oracle."""
    lib = L()
    inp = wl.step_inputs_cpu(shape)
    slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    cu = np.concatenate([[0], np.cumsum(shape.q_lens)])
    skip_r, bad_r = 0, shape.n_reqs - 1            # first token of the first request, last of the last
    slots[cu[skip_r]] = -1
    slots[cu[bad_r + 1] - 1] = shape.num_blocks * shape.block_size + 7
    out, kc, _, status = device_step(shape, inp, fused=True, slots=slots, check=False)
    assert status == lib.CB_EDEVICE
    assert lib.cb_last_error() == 0
    stored = np.where(slots >= shape.num_blocks * shape.block_size, -1, slots)   # the bad slot is not written
    want_k, _ = _want_cache(shape, inp, stored)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy(), want_k)
    ref = oracle_step(shape, inp)
    for r in range(1, shape.n_reqs - 1):
        assert_close(f64(out[cu[r]:cu[r + 1]]), ref[cu[r]:cu[r + 1]], f"{shape.name} request {r}")


def test_fused_empty_step_launches_nothing():
    lib = L()
    shape = wl.StepShape("empty", 32, 8, 128, 16, 8, q_lens=(0, 0), ctx_lens=(5, 0), seed=1)
    inp = wl.step_inputs_cpu(shape)
    device_step(shape, inp, fused=True)
    assert lib.cb_last_launch_count() == 0


def test_fused_zero_length_requests_eight_kv_heads():
    shape = wl.StepShape("fused_zero_q_8kv", 32, 8, 128, 16, 60, q_lens=(0, 3, 0, 1, 40, 0),
                         ctx_lens=(10, 5, 0, 300, 100, 20), seed=87)
    inp = wl.step_inputs_cpu(shape)
    out, _, _, _ = device_step(shape, inp, fused=True)
    assert_close(f64(out), oracle_step(shape, inp), shape.name)


@pytest.mark.parametrize("which", ["gqa_decode48", "mixed"])
def test_full_size_fused_step(which):
    """The full-size GQA 32/8 steps (20 GB pool) through the fused call: sampled
    requests against the oracle, and the newly stored rows read back exactly."""
    shape = wl.mixed()
    if which == "gqa_decode48":
        dec = [i for i, q in enumerate(shape.q_lens) if q == 1]
        shape = wl.scaled(shape, name=which, q_lens=[1] * len(dec), ctx_lens=[shape.ctx_lens[i] for i in dec])
    inp = wl.step_inputs_device(shape, "cuda")
    pool_k = inp["k_pool"]
    lib = L()
    out, kc, _, _ = device_step(shape, inp, fused=True)
    assert kc is pool_k and lib.cb_last_launch_count() == 1
    slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    rows = kc.view(-1, shape.block_size, shape.head_dim)       # [num_blocks * Hkv, bs, A]
    for t in range(0, shape.n_tokens, max(1, shape.n_tokens // 64)):
        b, o = divmod(int(slots[t]), shape.block_size)
        got = rows[b * shape.n_kv_heads:(b + 1) * shape.n_kv_heads, o]
        assert torch.equal(got.view(torch.int16), inp["k_new"][t].view(torch.int16))
    cu = np.concatenate([[0], np.cumsum(shape.q_lens)])
    for r in (0, 11, 47, shape.n_reqs - 1):
        sel = None if shape.q_lens[r] <= 12 else sorted({0, 5, 100, shape.q_lens[r] - 1})
        ref, sel = sampled_request_oracle(shape, inp, r, sel)
        assert_close(f64(out[cu[r]:cu[r + 1]])[sel], ref, f"{shape.name} request {r}")
    del inp, out, kc, rows, pool_k
    torch.cuda.empty_cache()
