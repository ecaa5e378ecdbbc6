"""Pins of the fp64 attention / paging / size oracle against things other than itself:
values the pages print, closed forms, a library routine (torch SDPA in fp64),
brute force with plain Python loops on tiny inputs, and invariants.

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, a
wrong causal offset, a transposed operand, a swapped GQA mapping, a wrong block
index) fails at least one test here.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as oa
from oracle import paged as op
from oracle import sizes as osz

RNG = np.random.default_rng(1234)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _rand(*shape, rng=RNG):
    return rng.standard_normal(size=shape)


# ----------------------------------------------------------------- softmax / mask
def test_softmax_rows_sum_to_one_and_masked_weights_are_zero():
    nq, nk, a = 9, 23, 16
    Q, K, V = _rand(nq, a), _rand(nk, a), _rand(nk, a)
    mask = RNG.random((nq, nk)) < 0.4
    mask[np.arange(nq), RNG.integers(0, nk, nq)] = True     # every row sees a key
    O, P = oa.masked_softmax_attention(Q, K, V, mask, 0.3)
    assert np.all(P >= 0)
    assert np.all(P[~mask] == 0.0)
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-12, rtol=0)
    assert np.allclose(O, P @ V, atol=1e-13)


def test_empty_row_gives_zero_output_and_never_occurs_in_causal_masks():
    Q, K, V = _rand(2, 4), _rand(3, 4), _rand(3, 4)
    mask = np.array([[True, False, False], [False, False, False]])
    O, P = oa.masked_softmax_attention(Q, K, V, mask, 1.0)
    assert np.all(O[1] == 0) and np.all(P[1] == 0)
    for q in range(1, 6):
        for c in range(0, 7):
            assert oa.chunk_causal_mask(q, c).any(axis=1).all()


def test_identity_mask_means_no_interaction():
    """[CB] §Attention: with every off-diagonal entry False no token sees another,
    so each output row is that token's own value row."""
    n, a = 6, 8
    Q, K, V = _rand(n, a), _rand(n, a), _rand(n, a)
    O, P = oa.masked_softmax_attention(Q, K, V, np.eye(n, dtype=bool), 0.7)
    assert np.array_equal(P, np.eye(n))
    assert np.allclose(O, V, atol=1e-15)


def test_chunk_mask_small_cases_by_hand():
    # q_len 2 after 3 stored tokens: row 0 (position 3) sees keys 0..3, row 1 sees 0..4
    m = oa.chunk_causal_mask(2, 3)
    assert m.tolist() == [[True, True, True, True, False], [True, True, True, True, True]]
    # fresh prefill of 3: lower-triangular
    assert oa.chunk_causal_mask(3, 0).tolist() == [[True, False, False], [True, True, False], [True, True, True]]


# ----------------------------------------------------------------- closed forms
def test_zero_query_gives_mean_of_visible_values():
    n, a = 7, 5
    K, V = _rand(n, a), _rand(n, a)
    Q = np.zeros((n, a))
    mask = oa.chunk_causal_mask(n, 0)
    O, _ = oa.masked_softmax_attention(Q, K, V, mask, 1.0)
    for i in range(n):
        assert np.allclose(O[i], V[: i + 1].mean(axis=0), atol=1e-14)


def test_single_visible_key_returns_its_value():
    Q, K, V = _rand(1, 6), _rand(5, 6), _rand(5, 6)
    mask = np.zeros((1, 5), dtype=bool)
    mask[0, 3] = True
    O, _ = oa.masked_softmax_attention(Q, K, V, mask, 2.0)
    assert np.allclose(O[0], V[3], atol=1e-15)


def test_identical_keys_give_uniform_weights():
    n, a = 8, 4
    k = _rand(a)
    K = np.tile(k, (n, 1))
    Q, V = _rand(3, a), _rand(n, a)
    mask = np.ones((3, n), dtype=bool)
    O, P = oa.masked_softmax_attention(Q, K, V, mask, 1.3)
    assert np.allclose(P, 1.0 / n, atol=1e-15)
    assert np.allclose(O, V.mean(axis=0), atol=1e-14)


def test_two_keys_closed_form_logistic():
    """softmax over two keys is the logistic function of the score difference."""
    Q, K, V = _rand(1, 3), _rand(2, 3), _rand(2, 3)
    s = 0.5
    d = s * (Q[0] @ K[0] - Q[0] @ K[1])
    w0 = 1.0 / (1.0 + math.exp(-d))
    O, _ = oa.masked_softmax_attention(Q, K, V, np.ones((1, 2), bool), s)
    assert np.allclose(O[0], w0 * V[0] + (1 - w0) * V[1], atol=1e-14)


# ----------------------------------------------------------------- brute force
def _brute_force_head(Q, K, V, mask, scale):
    """Plain Python loops and math.exp, no NumPy: a second, independent spelling."""
    nq, nk, a = len(Q), len(K), len(V[0])
    out = []
    for i in range(nq):
        scores = []
        for j in range(nk):
            if mask[i][j]:
                scores.append((j, scale * sum(Q[i][d] * K[j][d] for d in range(a))))
        mx = max(s for _, s in scores)
        w = [(j, math.exp(s - mx)) for j, s in scores]
        z = sum(x for _, x in w)
        out.append([sum(x / z * V[j][d] for j, x in w) for d in range(a)])
    return out


def test_brute_force_tiny_step():
    q_lens, ctx_lens = [1, 3, 2], [4, 0, 5]
    hq, hk, a = 4, 2, 3
    rng = np.random.default_rng(5)
    nq = sum(q_lens)
    q = rng.standard_normal((nq, hq, a))
    ks = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    vs = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    got = oa.attention_step(q, q_lens, ctx_lens, ks, vs, 0.6, hq, hk)
    t0 = 0
    for r, (n, c) in enumerate(zip(q_lens, ctx_lens)):
        mask = [[j <= c + i for j in range(c + n)] for i in range(n)]
        for h in range(hq):
            g = h // (hq // hk)
            want = _brute_force_head(q[t0:t0 + n, h].tolist(), ks[r][:, g].tolist(),
                                     vs[r][:, g].tolist(), mask, 0.6)
            assert np.allclose(got[t0:t0 + n, h], np.array(want), atol=1e-12)
        t0 += n


# ----------------------------------------------------------------- library routine
def test_fresh_prefill_equals_torch_sdpa_causal_fp64():
    n, h, a = 37, 3, 16
    rng = np.random.default_rng(11)
    q, k, v = (rng.standard_normal((n, h, a)) for _ in range(3))
    got = oa.attention_step(q, [n], [0], [k], [v], 1 / math.sqrt(a), h, h)
    t = lambda x: torch.from_numpy(x).permute(1, 0, 2)[None]   # [1, H, n, A]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)[0].permute(1, 0, 2).numpy()
    assert np.allclose(got, ref, atol=1e-12)


def test_gqa_equals_torch_sdpa_enable_gqa_fp64():
    """torch's enable_gqa shares KV head g among query heads g*G .. g*G+G-1."""
    n, hq, hk, a = 21, 8, 2, 16
    rng = np.random.default_rng(12)
    q = rng.standard_normal((n, hq, a))
    k, v = rng.standard_normal((n, hk, a)), rng.standard_normal((n, hk, a))
    got = oa.attention_step(q, [n], [0], [k], [v], 1 / math.sqrt(a), hq, hk)
    t = lambda x: torch.from_numpy(x).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True,
                                         enable_gqa=True)[0].permute(1, 0, 2).numpy()
    assert np.allclose(got, ref, atol=1e-12)


def test_chunk_equals_rows_of_full_sdpa_prefill():
    """A chunk after c stored tokens gives rows c..c+n-1 of the full causal prefill."""
    total, c, hq, hk, a = 40, 29, 4, 1, 8
    rng = np.random.default_rng(13)
    q = rng.standard_normal((total, hq, a))
    k, v = rng.standard_normal((total, hk, a)), rng.standard_normal((total, hk, a))
    got = oa.attention_step(q[c:], [total - c], [c], [k], [v], 0.35, hq, hk)
    t = lambda x: torch.from_numpy(x).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=0.35,
                                         enable_gqa=True)[0].permute(1, 0, 2).numpy()
    assert np.allclose(got, ref[c:], atol=1e-12)


# ----------------------------------------------------------------- chunking / decode
def _prefill_then_chunks(n, m, hq, hk, a, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, hq, a))
    k, v = rng.standard_normal((n, hk, a)), rng.standard_normal((n, hk, a))
    full = oa.attention_step(q, [n], [0], [k], [v], 1 / math.sqrt(a), hq, hk)
    parts = []
    for start, size in zip(range(0, n, m), osz.chunk_sizes(n, m)):
        parts.append(oa.attention_step(q[start:start + size], [size], [start],
                                       [k[: start + size]], [v[: start + size]],
                                       1 / math.sqrt(a), hq, hk))
    return full, np.concatenate(parts, axis=0)


def test_chunked_prefill_worked_example(golden_dir):
    g = _load(golden_dir, "chunking_n7_m4.json")
    assert osz.n_chunks(g["n"], g["m"]) == g["n_chunks"]
    assert osz.chunk_sizes(g["n"], g["m"]) == g["chunk_sizes"]
    full, chunked = _prefill_then_chunks(g["n"], g["m"], 4, 4, 64, seed=0)
    assert np.allclose(full, chunked, atol=1e-12, rtol=0)


@pytest.mark.parametrize("n,m", [(1, 1), (5, 2), (16, 16), (33, 7), (50, 49), (64, 10)])
def test_chunked_equals_unchunked_random(n, m):
    full, chunked = _prefill_then_chunks(n, m, 4, 2, 8, seed=n * 100 + m)
    assert np.allclose(full, chunked, atol=1e-12, rtol=0)


def test_decode_row_equals_last_row_of_full_prefill():
    """[CB] §KV cache: the new token's output with the cache equals what the full
    forward computes for that last token."""
    n, hq, hk, a = 30, 4, 4, 16
    rng = np.random.default_rng(3)
    q = rng.standard_normal((n + 1, hq, a))
    k, v = rng.standard_normal((n + 1, hk, a)), rng.standard_normal((n + 1, hk, a))
    full = oa.attention_step(q, [n + 1], [0], [k], [v], 0.25, hq, hk)
    dec = oa.attention_step(q[n:], [1], [n], [k], [v], 0.25, hq, hk)
    assert np.allclose(dec[0], full[n], atol=1e-12)


def test_attention_rows_match_step():
    n, c, hq, hk, a = 5, 20, 8, 2, 16
    rng = np.random.default_rng(4)
    q = rng.standard_normal((n, hq, a))
    k, v = rng.standard_normal((c + n, hk, a)), rng.standard_normal((c + n, hk, a))
    step = oa.attention_step(q, [n], [c], [k], [v], 0.2, hq, hk)
    rows = oa.attention_rows(q[[0, 3]], k, v, [c, c + 3], 0.2, hq, hk)
    assert np.allclose(rows, step[[0, 3]], atol=1e-13)


# ----------------------------------------------------------------- ragged batching
def test_ragged_block_diagonal_equals_per_request():
    q_lens, ctx_lens = [1, 4, 1, 6], [9, 0, 17, 3]
    hq, hk, a = 4, 2, 8
    rng = np.random.default_rng(8)
    q = rng.standard_normal((sum(q_lens), hq, a))
    ks = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    vs = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    a1 = oa.attention_step(q, q_lens, ctx_lens, ks, vs, 0.3, hq, hk)
    a2 = oa.attention_step_ragged(q, q_lens, ctx_lens, ks, vs, 0.3, hq, hk)
    assert np.allclose(a1, a2, atol=1e-12)
    m = oa.ragged_batch_mask(q_lens, ctx_lens)
    assert m.sum() == sum(n * c + n * (n + 1) // 2 for n, c in zip(q_lens, ctx_lens))


def test_ragged_requests_do_not_interact():
    """Changing one request's keys leaves every other request's output unchanged."""
    q_lens, ctx_lens = [3, 2], [5, 4]
    rng = np.random.default_rng(9)
    q = rng.standard_normal((5, 2, 4))
    ks = [rng.standard_normal((8, 2, 4)), rng.standard_normal((6, 2, 4))]
    vs = [rng.standard_normal((8, 2, 4)), rng.standard_normal((6, 2, 4))]
    a1 = oa.attention_step_ragged(q, q_lens, ctx_lens, ks, vs, 0.5, 2, 2)
    ks2 = [ks[0], ks[1] + 3.0]
    vs2 = [vs[0], -vs[1]]
    a2 = oa.attention_step_ragged(q, q_lens, ctx_lens, ks2, vs2, 0.5, 2, 2)
    assert np.array_equal(a1[:3], a2[:3])
    assert not np.allclose(a1[3:], a2[3:])


# ----------------------------------------------------------------- paging
def test_slot_lookup_hand_worked(golden_dir):
    g = _load(golden_dir, "paged_slots.json")
    got = [op.slot_of(g["table"], p, g["block_size"]) for p in g["positions"]]
    assert got == g["slots"]


def test_gather_equals_numpy_take_reshape():
    """The per-position gather against an independent vectorised spelling:
    pool[table] -> [n_blocks, Hkv, bs, A] -> [n_blocks*bs, Hkv, A]."""
    rng = np.random.default_rng(21)
    nb, hk, bs, a = 30, 3, 4, 5
    pool = rng.standard_normal((nb, hk, bs, a))
    table = rng.permutation(nb)[:7]
    n = 26
    got = op.gather_request(pool, table, n, bs)
    want = np.take(pool, table, axis=0).transpose(0, 2, 1, 3).reshape(-1, hk, a)[:n]
    assert np.array_equal(got, want)


def test_paged_equals_contiguous_under_random_permutations():
    rng = np.random.default_rng(22)
    hq, hk, a, bs = 4, 2, 8, 4
    q_lens, ctx_lens = [1, 5, 1], [13, 6, 2]
    for trial in range(5):
        nb = 40
        perm = rng.permutation(nb)
        tables, off = [], 0
        for c, n in zip(ctx_lens, q_lens):
            cnt = -(-(c + n) // bs)
            tables.append(perm[off:off + cnt])
            off += cnt
        kc = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
        vc = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
        kpool = rng.standard_normal((nb, hk, bs, a))
        vpool = rng.standard_normal((nb, hk, bs, a))
        for r, (c, n) in enumerate(zip(ctx_lens, q_lens)):
            slots = [op.slot_of(tables[r], p, bs) for p in range(c + n)]
            op.append_rows(kpool, kc[r], slots, bs)
            op.append_rows(vpool, vc[r], slots, bs)
        kg = [op.gather_request(kpool, tables[r], c + n, bs) for r, (c, n) in enumerate(zip(ctx_lens, q_lens))]
        vg = [op.gather_request(vpool, tables[r], c + n, bs) for r, (c, n) in enumerate(zip(ctx_lens, q_lens))]
        for r in range(3):
            assert np.array_equal(kg[r], kc[r]) and np.array_equal(vg[r], vc[r])
        q = rng.standard_normal((sum(q_lens), hq, a))
        o1 = oa.attention_step(q, q_lens, ctx_lens, kc, vc, 0.4, hq, hk)
        o2 = oa.attention_step(q, q_lens, ctx_lens, kg, vg, 0.4, hq, hk)
        assert np.array_equal(o1, o2)


def test_slot_mapping_concatenates_requests_in_order():
    bs = 4
    tables = [[3, 1], [0, 2, 5]]
    sm = op.slot_mapping(tables, [2, 3], [5, 9], bs)
    # request 0: positions 5, 6 -> block 1 offsets 1, 2; request 1: positions 9..11 -> block 5 offsets 1..3
    assert sm.tolist() == [5, 6, 21, 22, 23]


def test_append_skips_negative_slots_and_touches_nothing_else():
    pool = np.zeros((4, 2, 4, 3))
    rows = np.arange(3 * 2 * 3, dtype=float).reshape(3, 2, 3) + 1
    op.append_rows(pool, rows, [6, -1, 13], 4)
    assert np.array_equal(pool[1, :, 2], rows[0]) and np.array_equal(pool[3, :, 1], rows[2])
    assert np.count_nonzero(pool) == 2 * 2 * 3


def test_decode_grows_cache_by_one(golden_dir):
    """[KVB] §Batch Decode: after one decode step a 10-token cache holds 11 tokens,
    the first 10 unchanged and the new row last."""
    g = _load(golden_dir, "decode_cache_length.json")
    bs, hk, a = 16, g["num_heads"], g["hidden_dim"] // g["num_heads"]
    rng = np.random.default_rng(2)
    for b in range(g["batch_size"]):
        table = rng.permutation(8)[:2]
        pool = np.zeros((8, hk, bs, a))
        old = rng.standard_normal((g["cached_before"], hk, a))
        op.append_rows(pool, old, op.slot_mapping([table], [g["cached_before"]], [0], bs), bs)
        new = rng.standard_normal((1, hk, a))
        op.append_rows(pool, new, op.slot_mapping([table], [1], [g["cached_before"]], bs), bs)
        got = op.gather_request(pool, table, g["cached_after"], bs)
        assert got.shape[0] == g["cached_after"]
        assert np.array_equal(got[:10], old) and np.array_equal(got[10], new[0])


# ----------------------------------------------------------------- sizes
def test_kv_sizes_printed_on_pages(golden_dir):
    g = _load(golden_dir, "kv_sizes.json")
    l7 = g["llama2_7b"]
    assert osz.kv_values_per_token_per_layer(l7["n_heads"], l7["head_dim"]) == l7["values_per_token_per_layer"]
    assert osz.kv_cache_bytes(1, 1, l7["n_heads"], 1, l7["head_dim"], 2) == l7["bytes_per_token_per_layer"]
    l13 = g["llama_13b"]
    b = osz.kv_cache_bytes(1, l13["n_layers"], l13["n_heads"], l13["seq_len"], l13["head_dim"], 2)
    assert round(b / 1e9, 1) == l13["gb_per_sequence_rounded"]
    q = g["gqa"]
    mha = osz.kv_cache_bytes(1, 32, q["mha_heads"], 100, 128)
    assert osz.kv_cache_bytes(1, 32, q["gqa_kv_heads"], 100, 128) / mha == q["gqa_ratio"]
    assert osz.kv_cache_bytes(1, 32, 1, 100, 128) / mha == q["mqa_ratio"]


def test_kv_formula_scales_linearly_in_batch_and_sequence():
    base = osz.kv_cache_bytes(1, 2, 3, 5, 7, 2)
    assert osz.kv_cache_bytes(4, 2, 3, 5, 7, 2) == 4 * base
    assert osz.kv_cache_bytes(1, 2, 3, 10, 7, 2) == 2 * base
    assert base == 2 * 2 * 3 * 5 * 7 * 2


def test_dynamic_insert_padding_printed_on_page(golden_dir):
    g = _load(golden_dir, "padding_b8_n100.json")
    assert osz.dynamic_insert_padding(g["batch_size"], g["n_prompt"]) == g["pad_tokens"]
    for b in (1, 2, 5):
        for n in (1, 3, 40):
            assert osz.dynamic_insert_padding(b, n) == (n - 1) * (b - 1)


def test_blocks_for_and_ragged_padding_zero():
    assert [osz.blocks_for(n, 16) for n in (0, 1, 16, 17, 32, 33)] == [0, 1, 1, 2, 2, 3]
    # ragged batching concatenates: the token count is the plain sum, no pad rows
    lens = [5, 1, 9]
    assert sum(lens) == sum(row.count("tok") for row in osz.left_padded_batch(lens))


# ----------------------------------------------------------------- rolling window
# [KVB] §Rolling KV Cache has only a heading.  Reading: a query at absolute
# position p sees the keys p - W + 1 .. p (its own included).
def test_window_mask_small_case_by_hand():
    # a 3-token chunk after 2 stored tokens, W = 2: positions 2, 3, 4 see {1, 2}, {2, 3}, {3, 4}
    want = np.array([[0, 1, 1, 0, 0], [0, 0, 1, 1, 0], [0, 0, 0, 1, 1]], dtype=bool)
    assert np.array_equal(oa.chunk_causal_mask(3, 2, window=2), want)


def test_window_at_least_the_context_is_no_window():
    rng = np.random.default_rng(31)
    q_lens, ctx_lens = [1, 5, 3], [9, 0, 4]
    hq, hk, a = 4, 2, 8
    q = rng.standard_normal((sum(q_lens), hq, a))
    ks = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    vs = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    full = oa.attention_step(q, q_lens, ctx_lens, ks, vs, 0.4, hq, hk)
    for w in (10, 11, 1000):
        assert np.array_equal(oa.attention_step(q, q_lens, ctx_lens, ks, vs, 0.4, hq, hk, window=w), full)


def test_window_of_one_returns_each_query_its_own_value():
    rng = np.random.default_rng(32)
    q_lens, ctx_lens = [1, 4], [6, 3]
    q = rng.standard_normal((5, 2, 4))
    ks = [rng.standard_normal((c + n, 2, 4)) for c, n in zip(ctx_lens, q_lens)]
    vs = [rng.standard_normal((c + n, 2, 4)) for c, n in zip(ctx_lens, q_lens)]
    got = oa.attention_step(q, q_lens, ctx_lens, ks, vs, 0.7, 2, 2, window=1)
    assert np.allclose(got[0], vs[0][6], atol=1e-15)
    assert np.allclose(got[1:], vs[1][3:7], atol=1e-15)


def test_window_of_two_is_the_logistic_of_the_last_two_scores():
    rng = np.random.default_rng(33)
    q, k, v = rng.standard_normal((1, 1, 5)), rng.standard_normal((9, 1, 5)), rng.standard_normal((9, 1, 5))
    got = oa.attention_step(q, [1], [8], [k], [v], 0.5, 1, 1, window=2)[0, 0]
    d = 0.5 * (q[0, 0] @ k[8, 0] - q[0, 0] @ k[7, 0])
    w8 = 1.0 / (1.0 + math.exp(-d))
    assert np.allclose(got, w8 * v[8, 0] + (1 - w8) * v[7, 0], atol=1e-14)


def test_window_brute_force_tiny_step():
    q_lens, ctx_lens, w = [1, 4, 2], [7, 0, 5], 3
    hq, hk, a = 4, 1, 3
    rng = np.random.default_rng(34)
    q = rng.standard_normal((sum(q_lens), hq, a))
    ks = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    vs = [rng.standard_normal((c + n, hk, a)) for c, n in zip(ctx_lens, q_lens)]
    got = oa.attention_step(q, q_lens, ctx_lens, ks, vs, 0.6, hq, hk, window=w)
    t0 = 0
    for r, (n, c) in enumerate(zip(q_lens, ctx_lens)):
        mask = [[c + i - w < j <= c + i for j in range(c + n)] for i in range(n)]
        for h in range(hq):
            want = _brute_force_head(q[t0:t0 + n, h].tolist(), ks[r][:, 0].tolist(), vs[r][:, 0].tolist(), mask, 0.6)
            assert np.allclose(got[t0:t0 + n, h], np.array(want), atol=1e-12)
        t0 += n


def test_window_row_equals_sdpa_over_its_last_keys():
    """A query at position p with window W is plain (unmasked) attention over
    keys p - W + 1 .. p: torch's SDPA in fp64 on that slice."""
    rng = np.random.default_rng(35)
    n, c, w, hq, hk, a = 6, 40, 9, 4, 2, 16
    q = rng.standard_normal((n, hq, a))
    k, v = rng.standard_normal((c + n, hk, a)), rng.standard_normal((c + n, hk, a))
    got = oa.attention_step(q, [n], [c], [k], [v], 1 / math.sqrt(a), hq, hk, window=w)
    for i in range(n):
        p = c + i
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(t(q[i:i + 1]), t(k[p - w + 1:p + 1]), t(v[p - w + 1:p + 1]),
                                             enable_gqa=True)[0].permute(1, 0, 2).numpy()
        assert np.allclose(got[i], ref[0], atol=1e-12)


@pytest.mark.parametrize("w", [1, 5, 16, 33])
def test_windowed_chunks_equal_windowed_prefill(w):
    """[CB] §Chunked prefill with the window: chunk after chunk over the stored
    keys equals the unchunked windowed prefill, and a decode row equals the last
    row of a windowed prefill one token longer."""
    rng = np.random.default_rng(36 + w)
    n, hq, hk, a = 50, 2, 1, 8
    q, k, v = rng.standard_normal((n, hq, a)), rng.standard_normal((n, hk, a)), rng.standard_normal((n, hk, a))
    full = oa.attention_step(q, [n], [0], [k], [v], 0.3, hq, hk, window=w)
    for c0, c1 in [(0, 13), (13, 29), (29, 49), (49, 50)]:
        part = oa.attention_step(q[c0:c1], [c1 - c0], [c0], [k[:c1]], [v[:c1]], 0.3, hq, hk, window=w)
        assert np.allclose(part, full[c0:c1], atol=1e-13)
    rows = oa.attention_rows(q[[10, 49]], k, v, [10, 49], 0.3, hq, hk, window=w)
    assert np.allclose(rows, full[[10, 49]], atol=1e-13)
