"""GPU parity: the C-ABI path (cb_kv_append + cb_paged_attention on GB300)
against the fp64 oracle on the same seeded inputs.

Cache append and block-table indexing: bit-exact.  Attention: max abs error
<= 2e-2 and max abs error / max |reference| <= 1e-2 (bf16 inputs and outputs,
fp32 accumulation)."""
import math

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


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("shape", [wl.tiny(), wl.random_step(3, 12, 90, 40, 8, 2, 128),
                                   wl.random_step(4, 7, 33, 17, 4, 4, 64)], ids=lambda s: s.name)
def test_append_is_bit_exact_including_untouched_slots(shape):
    inp = wl.step_inputs_cpu(shape)
    lib = L()
    slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    assert np.array_equal(slots, op.slot_mapping(inp["block_tables"], shape.q_lens, shape.ctx_lens, shape.block_size))
    kc, vc = inp["k_pool"].cuda(), inp["v_pool"].cuda()
    lib.cb_kv_append(inp["k_new"].cuda(), inp["v_new"].cuda(), torch.from_numpy(slots).cuda(), kc, vc)
    assert lib.cb_last_error() == 0
    want_k = inp["k_pool"].view(torch.int16).numpy().copy()
    want_v = inp["v_pool"].view(torch.int16).numpy().copy()
    op.append_rows(want_k, inp["k_new"].view(torch.int16).numpy(), slots, shape.block_size)
    op.append_rows(want_v, inp["v_new"].view(torch.int16).numpy(), slots, shape.block_size)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy(), want_k)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy(), want_v)


def test_append_negative_slot_skips_and_bad_slot_is_reported():
    shape = wl.tiny()
    inp = wl.step_inputs_cpu(shape)
    lib = L()
    slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    slots[1] = -1
    kc, vc = inp["k_pool"].cuda(), inp["v_pool"].cuda()
    lib.cb_kv_append(inp["k_new"].cuda(), inp["v_new"].cuda(), torch.from_numpy(slots).cuda(), kc, vc)
    assert lib.cb_last_error() == 0
    want = inp["k_pool"].view(torch.int16).numpy().copy()
    op.append_rows(want, inp["k_new"].view(torch.int16).numpy(), slots, shape.block_size)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy(), want)
    slots[0] = shape.num_blocks * shape.block_size + 5          # outside the cache: skipped, flagged
    lib.cb_kv_append(inp["k_new"].cuda(), inp["v_new"].cuda(), torch.from_numpy(slots).cuda(), kc, vc)
    assert lib.cb_last_error() == lib.CB_EDEVICE
    assert lib.cb_last_error() == 0                               # the status is cleared once read


# ------------------------------------------------------------------ attention, small
def _parity(shape, scale=None):
    inp = wl.step_inputs_cpu(shape)
    out, _, _, _ = device_step(shape, inp, scale=scale)
    ref = oracle_step(shape, inp, scale=scale)
    return assert_close(f64(out), ref, shape.name)


def test_tiny_mixed_batch():
    """Two decodes (37 and 100 stored), the second chunk of a 7-token prompt cut at 4,
    a fresh 20-token prefill; MHA 4 heads, head_dim 64."""
    _parity(wl.tiny())


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_decode_only_split_k(group, head_dim):
    base = wl.random_step(10 + group, n_reqs=9, max_ctx=1500, max_q=1, n_q_heads=8, n_kv_heads=8 // group,
                          head_dim=head_dim, p_decode=1.0)
    ctx = list(base.ctx_lens)
    ctx[0], ctx[1], ctx[2] = 0, 15, 2047        # one key; block boundary; many splits with a ragged tail
    _parity(wl.scaled(base, ctx_lens=ctx, num_blocks=base.num_blocks + 200))


@pytest.mark.parametrize("group", [2, 4, 8])
def test_decode_gqa_eight_kv_heads(group):
    """Decode-only steps with 8 KV heads, where one block of every head is one
    128-row tensor-core tile: one key, block boundaries, one and many splits."""
    base = wl.random_step(30 + group, n_reqs=13, max_ctx=3000, max_q=1, n_q_heads=8 * group, n_kv_heads=8,
                          head_dim=128, p_decode=1.0)
    ctx = list(base.ctx_lens)
    ctx[0], ctx[1], ctx[2], ctx[3], ctx[4] = 0, 15, 16, 4095, 8190
    _parity(wl.scaled(base, ctx_lens=ctx, num_blocks=base.num_blocks + 800))


@pytest.mark.parametrize("group", [1, 4])
def test_decode_running_max_rescales(group):
    """A large softmax scale makes later blocks raise the running maximum far
    past the lazy-rescale threshold, so the output accumulator is rescaled."""
    base = wl.random_step(50 + group, n_reqs=6, max_ctx=2500, max_q=1, n_q_heads=8 * group, n_kv_heads=8,
                          head_dim=128, p_decode=1.0)
    _parity(base, scale=0.6)


@pytest.mark.parametrize("shape", [
    wl.random_step(61, n_reqs=9, max_ctx=900, max_q=1, n_q_heads=8, n_kv_heads=8, head_dim=128, p_decode=1.0),
    wl.random_step(62, n_reqs=9, max_ctx=900, max_q=1, n_q_heads=32, n_kv_heads=8, head_dim=128, p_decode=1.0),
    wl.random_step(63, n_reqs=9, max_ctx=900, max_q=1, n_q_heads=8, n_kv_heads=2, head_dim=128, p_decode=1.0),
    wl.random_step(64, n_reqs=7, max_ctx=600, max_q=200, n_q_heads=16, n_kv_heads=8, head_dim=128, p_decode=0.5),
    wl.random_step(65, n_reqs=7, max_ctx=600, max_q=200, n_q_heads=8, n_kv_heads=8, head_dim=64, p_decode=0.5),
], ids=lambda s: f"{s.name}_h{s.n_q_heads}_{s.n_kv_heads}")
def test_unwritten_cache_slots_do_not_leak(shape):
    """Every cache slot a request does not own (past its last key in its last
    block, and every unused block) holds NaN: outputs stay finite and equal."""
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


@pytest.mark.parametrize("group", [1, 4, 8])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_chunked_prefill_tiles(group, head_dim):
    """Prefill chunks spanning several 128-row query tiles and 128-key tiles with
    ragged tails, after stored prefixes of various lengths (0, mid-block, long)."""
    hq = 8
    shape = wl.StepShape(f"prefill_g{group}_a{head_dim}", hq, hq // group, head_dim, 16, 200,
                         q_lens=(300, 129, 2, 77), ctx_lens=(200, 0, 333, 1000), seed=group * 7 + head_dim)
    _parity(shape)


@pytest.mark.parametrize("seed", range(6))
def test_random_mixed_steps(seed):
    group = [1, 2, 4, 8][seed % 4]
    head_dim = [64, 128][seed % 2]
    shape = wl.random_step(100 + seed, n_reqs=11, max_ctx=700, max_q=150, n_q_heads=8, n_kv_heads=8 // group,
                           head_dim=head_dim, p_decode=0.6)
    _parity(shape)


@pytest.mark.parametrize("group", [2, 4, 8])
def test_mixed_steps_eight_kv_heads(group):
    """Mixed prefill + decode steps with 8 KV heads and head_dim 128: the decode
    tokens run the block-tile phase of the mixed kernel."""
    shape = wl.random_step(200 + group, n_reqs=14, max_ctx=2500, max_q=300, n_q_heads=8 * group, n_kv_heads=8,
                           head_dim=128, p_decode=0.7)
    q, c = list(shape.q_lens), list(shape.ctx_lens)
    q[0], c[0] = 1, 0              # a decode with a single key
    q[1], c[1] = 1, 4100           # a decode cut into several splits
    q[2], c[2] = 77, 15            # a prefill chunk after a partial block
    _parity(wl.scaled(shape, q_lens=q, ctx_lens=c, num_blocks=shape.num_blocks + 400))


def test_scale_argument_is_honoured():
    _parity(wl.tiny(), scale=0.05)


def test_chunked_equals_unchunked_on_gpu():
    """[CB] Chunked prefill: a 7-token prompt run as chunks (4 then 3) gives the
    same outputs as one 7-token prefill, through the paged cache."""
    lib = L()
    hq, hk, a, bs = 4, 4, 64, 16
    rng = np.random.default_rng(0)
    q = torch.from_numpy(rng.standard_normal((7, hq, a), dtype=np.float32)).to(torch.bfloat16).cuda()
    k = torch.from_numpy(rng.standard_normal((7, hk, a), dtype=np.float32)).to(torch.bfloat16).cuda()
    v = torch.from_numpy(rng.standard_normal((7, hk, a), dtype=np.float32)).to(torch.bfloat16).cuda()
    table = np.array([[3]], np.int32)

    def run(chunks):
        kc = torch.zeros(8, hk, bs, a, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        outs = []
        start = 0
        for n in chunks:
            slots = lib.cb_build_slot_mapping([n], [start], table, bs)
            lib.cb_kv_append(k[start:start + n], v[start:start + n], torch.from_numpy(slots).cuda(), kc, vc)
            ws = torch.empty(lib.cb_paged_attention_workspace_size(1, n, n, start + n, hq, hk, a, bs),
                             dtype=torch.uint8, device="cuda")
            o = torch.empty(n, hq, a, dtype=torch.bfloat16, device="cuda")
            lib.cb_paged_attention(q[start:start + n].contiguous(), torch.tensor([0, n], dtype=torch.int32).cuda(),
                                   torch.tensor([start], dtype=torch.int32).cuda(), torch.from_numpy(table).cuda(),
                                   kc, vc, o, 1 / math.sqrt(a), ws, max(n, 2), start + n)
            outs.append(o)
            start += n
        assert lib.cb_last_error() == 0
        return torch.cat(outs).float().cpu().numpy()

    full, chunked = run([7]), run([4, 3])
    assert np.abs(full - chunked).max() <= 1e-2


@pytest.mark.parametrize("shape", [
    wl.random_step(7, n_reqs=10, max_ctx=3000, max_q=100, n_q_heads=8, n_kv_heads=2, head_dim=128),
    wl.random_step(8, n_reqs=10, max_ctx=3000, max_q=1, n_q_heads=32, n_kv_heads=8, head_dim=128, p_decode=1.0),
], ids=lambda s: s.name)
def test_outputs_are_deterministic(shape):
    inp = wl.step_inputs_cpu(shape)
    o1 = device_step(shape, inp)[0]
    o2 = device_step(shape, inp)[0]
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


# ------------------------------------------------------------------ edge cases
def test_empty_batch_and_zero_length_requests():
    lib = L()
    shape = wl.StepShape("zero_q", 4, 2, 64, 16, 40, q_lens=(0, 3, 0, 1), ctx_lens=(10, 5, 0, 20), seed=1)
    _parity(shape)
    # an empty step launches nothing and succeeds
    q = torch.empty(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    lib.cb_paged_attention(q, torch.zeros(1, dtype=torch.int32, device="cuda"),
                           torch.zeros(0, dtype=torch.int32, device="cuda"),
                           torch.zeros(0, 1, dtype=torch.int32, device="cuda"),
                           torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device="cuda"),
                           torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device="cuda"), q, 0.125,
                           torch.empty(16, dtype=torch.uint8, device="cuda"), 1, 1)
    assert lib.cb_last_launch_count() == 0


@pytest.mark.parametrize("q_lens,ctx_lens", [((0, 1, 0, 1, 0), (10, 50, 0, 300, 7)),
                                             ((0, 3, 0, 1, 40, 0), (10, 5, 0, 300, 100, 20))],
                         ids=["decode_only", "mixed"])
def test_zero_length_requests_eight_kv_heads(q_lens, ctx_lens):
    """Requests with no new token between decodes and chunks, 8 KV heads: the
    block-tile decode must skip them when it walks the requests' blocks."""
    blocks = sum(-(-(c + q) // 16) for c, q in zip(ctx_lens, q_lens)) + 8
    _parity(wl.StepShape("zero_q_8kv", 32, 8, 128, 16, blocks, q_lens=q_lens, ctx_lens=ctx_lens, seed=3))


def test_bad_block_id_in_mixed_eight_kv_heads_is_reported():
    shape = wl.StepShape("bad_mixed_8kv", 32, 8, 128, 16, 200, q_lens=(1, 1, 60, 1), ctx_lens=(300, 40, 100, 250),
                         seed=4)
    inp = wl.step_inputs_cpu(shape)
    bad = inp["block_tables"].copy()
    bad[1, 1] = shape.num_blocks + 3          # a decode reads it
    lib = L()
    out, _, _, status = device_step(shape, inp, check=False, attn_tables=bad)
    assert status == lib.CB_EDEVICE
    ref = oracle_step(shape, inp)
    cu = np.concatenate([[0], np.cumsum(shape.q_lens)])
    for r in (0, 2, 3):
        assert_close(f64(out[cu[r]:cu[r + 1]]), ref[cu[r]:cu[r + 1]], f"request {r}")


def test_max_requests_mixed_eight_kv_heads():
    """CB_MAX_REQS requests in one mixed launch with 8 KV heads: 2040 decodes
    with short contexts and 8 short prefill chunks."""
    lib = L()
    n = lib.CB_MAX_REQS
    rng = np.random.default_rng(5)
    ctx = [int(c) for c in rng.integers(0, 40, size=n)]
    q = [1] * n
    for r in range(0, n, n // 8):
        q[r] = 20
    shape = wl.StepShape("max_reqs_mixed_8kv", 32, 8, 128, 16, sum(-(-(c + k) // 16) for c, k in zip(ctx, q)) + 4,
                         q_lens=tuple(q), ctx_lens=tuple(ctx), seed=10)
    _parity(shape)


def test_block_and_tile_boundaries():
    """Lengths at exact multiples of the block (16) and tile (128) sizes and one past."""
    shape = wl.StepShape("bounds", 8, 2, 128, 16, 300, q_lens=(1, 1, 128, 129, 16, 1),
                         ctx_lens=(127, 128, 128, 127, 112, 255), seed=5)
    _parity(shape)


def test_bad_block_id_in_gqa_decode_is_reported():
    shape = wl.random_step(71, n_reqs=5, max_ctx=600, max_q=1, n_q_heads=32, n_kv_heads=8, head_dim=128,
                           p_decode=1.0)
    shape = wl.scaled(shape, ctx_lens=[300, 40, 500, 17, 250])
    inp = wl.step_inputs_cpu(shape)
    bad = inp["block_tables"].copy()
    bad[1, 1] = shape.num_blocks + 5
    bad[3, 0] = -1
    lib = L()
    out, _, _, status = device_step(shape, inp, check=False, attn_tables=bad)
    assert status == lib.CB_EDEVICE
    ref = oracle_step(shape, inp)
    for r in (0, 2, 4):
        assert_close(f64(out[r:r + 1]), ref[r:r + 1], f"request {r}")


def test_bad_block_id_is_reported_not_read():
    shape = wl.tiny()
    inp = wl.step_inputs_cpu(shape)
    bad = inp["block_tables"].copy()
    bad[1, 2] = shape.num_blocks + 1000      # decode request 1 reads it
    bad[3, 0] = -7                           # prefill request 3 reads it
    lib = L()
    out, _, _, status = device_step(shape, inp, check=False, attn_tables=bad)
    assert status == lib.CB_EDEVICE
    # the requests that do not touch a bad entry are still right
    ref = oracle_step(shape, inp)
    assert_close(f64(out[0:1]), ref[0:1], "request 0")
    assert_close(f64(out[2:5]), ref[2:5], "request 2")


def test_workspace_too_small_is_rejected():
    shape = wl.tiny()
    inp = wl.step_inputs_cpu(shape)
    with pytest.raises(L().CBError):
        device_step(shape, inp, ws_extra=-64)


@pytest.mark.parametrize("hq,hk,a", [(4, 1, 64), (64, 8, 128)])
def test_max_requests(hq, hk, a):
    """CB_MAX_REQS decode requests with short contexts in one step."""
    lib = L()
    n = lib.CB_MAX_REQS
    rng = np.random.default_rng(3)
    ctx = tuple(int(c) for c in rng.integers(0, 40, size=n))
    shape = wl.StepShape(f"max_reqs_{hq}_{hk}", hq, hk, a, 16, sum(-(-(c + 1) // 16) for c in ctx) + 4,
                         q_lens=(1,) * n, ctx_lens=ctx, seed=9)
    _parity(shape)


# ------------------------------------------------------------------ full-size, sampled
def _full_size(shape, sample, rows_per_req=None):
    inp = wl.step_inputs_device(shape, "cuda")
    out, _, _, _ = device_step(shape, inp)
    cu = np.concatenate([[0], np.cumsum(shape.q_lens)])
    for r in sample:
        rows = None
        if rows_per_req and shape.q_lens[r] > rows_per_req:
            rng = np.random.default_rng(r)
            rows = sorted(set(rng.choice(shape.q_lens[r], rows_per_req - 2, replace=False).tolist())
                          | {0, shape.q_lens[r] - 1})
        ref, rows = sampled_request_oracle(shape, inp, r, rows)
        got = f64(out[cu[r]:cu[r + 1]])[rows]
        assert_close(got, ref, f"{shape.name} request {r}")
    del inp, out
    torch.cuda.empty_cache()


def test_full_size_decode_llama7b_layer():
    """64 decodes, MHA 32 x 128, contexts 512..4096, 20 GB pool: 6 sampled requests."""
    shape = wl.decode()
    order = np.argsort(shape.ctx_lens)
    _full_size(shape, [int(order[0]), int(order[-1]), 0, 17, 40, 63])


def test_full_size_gqa_decode_step():
    """The 48 decodes of the mixed step alone (GQA 32/8, contexts 256..8192)."""
    m = wl.mixed()
    dec = [i for i, q in enumerate(m.q_lens) if q == 1]
    shape = wl.scaled(m, name="gqa_decode48", q_lens=[1] * len(dec), ctx_lens=[m.ctx_lens[i] for i in dec])
    order = np.argsort(shape.ctx_lens)
    _full_size(shape, [int(order[0]), int(order[-1]), 0, 23, 47])


def test_full_size_mixed_gqa_step():
    """48 decodes + two 512-token chunks (after 1024 and 3072 stored), GQA 32/8."""
    shape = wl.mixed()
    _full_size(shape, [0, 11, 47, 48, 49], rows_per_req=12)


def test_full_size_long_context_chunk():
    """Step 15 of a 32768-token prompt in 2048-token chunks (30720 stored) + 16 decodes at 8207."""
    shape = wl.long(15)
    _full_size(shape, [0, 15, 16], rows_per_req=6)


# ------------------------------------------------------------------ balanced prefill pieces
# With more tile pairs than CTAs, the cooperative launch cuts the pairs' key
# tiles into equal ranges per CTA; pieces cut at CTA boundaries are merged by
# log-sum-exp after the grid-wide barrier.  Sizes chosen for 160-240 pairs
# (pairs cut across up to 3 CTAs), small enough for the oracle to check every
# row.
_PRE_REGION = 2 * 160 * 256 * (128 + 2) * 4          # the partials' workspace region (A = 128)


@pytest.mark.parametrize("hq,q_lens,ctx_lens", [
    (16, (2560,), (100,)),                               # G = 2: 128-token pairs, 160 pairs
    (32, (1280,), (100,)),                               # G = 4: 64-token pairs
    (64, (640,), (100,)),                                # G = 8: 32-token pairs
    (32, (1, 700, 1, 600, 1), (3000, 40, 20, 0, 900)),   # with decodes in the same launch
    (16, (3840,), (0,)),                                 # 240 pairs
    (32, (1600,), (1700,)),                              # 200 pairs over longer contexts
    (64, (800,), (1700,)),
    (32, (1, 1000, 1, 700, 1), (3000, 1500, 20, 800, 900)),
], ids=["g2", "g4", "g8", "mixed", "g2_240", "g4_200", "g8_200", "mixed_216"])
def test_balanced_prefill_pieces_match_oracle(hq, q_lens, ctx_lens):
    blocks = sum(-(-(c + q) // 16) for c, q in zip(ctx_lens, q_lens)) + 8
    shape = wl.StepShape(f"balanced_h{hq}", hq, 8, 128, 16, blocks, q_lens=q_lens, ctx_lens=ctx_lens, seed=hq)
    _parity(shape)


def _packed_items_per_cta(q_lens, ctx_lens, n_sms, n_kv_heads=8, tok_per_pair=64):
    """The plan's packing rule restated: items (whole tile pairs of one KV head)
    per CTA when there are fewer items than CTAs: k = 2 if the largest CTA
    load (items longest first, dealt 0..Np-1, then Np-1..0) times
    2.6 us per key tile, with a 30 % margin, fits in the decode bytes at 6 B/ns."""
    lens, dec_blocks = [], 0
    for q, c in zip(q_lens, ctx_lens):
        if q == 1:
            dec_blocks += -(-(c + 1) // 16)
        elif q > 1:
            for pr in range(-(-q // tok_per_pair)):
                lens += [-(-(c + min(q, (pr + 1) * tok_per_pair)) // 128)] * n_kv_heads
    if not 1 < len(lens) <= n_sms:
        return 1
    order = sorted(lens, reverse=True)
    dec_ns = dec_blocks * 2 * n_kv_heads * 16 * 128 * 2 // 6000
    for k in (2,):
        np_ = -(-len(lens) // k)
        load = max(sum(order[r] for q in range(k) for r in [q * np_ + (np_ - 1 - c if q & 1 else c)] if r < len(lens))
                   for c in range(np_))
        if load * 2600 * 13 <= dec_ns * 10:
            return k
    return 1


@pytest.mark.parametrize("q_lens,ctx_lens,k", [
    ((1,) * 16 + (256, 64), tuple(5200 + 37 * i for i in range(16)) + (200, 0), 2),
    ((1,) * 16 + (512,), tuple(8000 + 11 * i for i in range(16)) + (1024,), 2),
    ((1,) * 3 + (512,), (300, 200, 100) + (1024,), 1),
], ids=["short_items", "one_chunk", "too_little_decode"])
def test_prefill_items_packed_onto_fewer_ctas(q_lens, ctx_lens, k):
    """Fewer prefill items than CTAs beside a long decode stream: the plan deals
    whole items to fewer CTAs (longest first, a long one with a short one) so
    that the other CTAs stream the decodes from the start; beside a short
    decode stream they stay one per CTA.  Every row against the oracle."""
    assert _packed_items_per_cta(q_lens, ctx_lens, torch.cuda.get_device_properties(0).multi_processor_count) == k
    blocks = sum(-(-(c + q) // 16) for c, q in zip(ctx_lens, q_lens)) + 8
    shape = wl.StepShape(f"packed_{k}", 32, 8, 128, 16, blocks, q_lens=q_lens, ctx_lens=ctx_lens, seed=40 + k)
    _parity(shape)


def test_prefill_without_room_for_pieces_keeps_pairs_whole():
    """A workspace without the partials' region: the launch keeps tile pairs whole."""
    shape = wl.StepShape("whole_pairs", 32, 8, 128, 16, 240, q_lens=(1600,), ctx_lens=(1700,), seed=5)
    inp = wl.step_inputs_cpu(shape)
    out, _, _, _ = device_step(shape, inp, ws_extra=-_PRE_REGION)
    assert_close(f64(out), oracle_step(shape, inp), shape.name)
