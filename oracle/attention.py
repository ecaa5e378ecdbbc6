"""fp64 attention oracle (test infrastructure only; see the package docstring).

What one continuous-batching attention step computes, written out plainly:

* [CB] §Attention: Q [nQ, A] and K [nK, A] give scores Q K^T [nQ, nK]; a boolean
  mask of the same shape decides which keys a query may see; a softmax per row
  (per token) follows, and the result multiplies V [nV, A] with nV = nK.
* [KVB] §Batch Decode (batch_decode_step): the scores are divided by the square
  root of head_dim before the softmax.  Here that factor is the ``scale``
  argument (callers pass 1/sqrt(A)).
* [CB] §Chunked prefill: for a chunk, the KV stored by earlier chunks is put in
  front of the chunk's own KV and the mask is shifted accordingly; the result
  equals the unchunked prefill cut in the middle.  Reading: query i of a chunk
  that follows ``n_cached`` stored tokens sits at absolute position n_cached + i
  and sees every key at position <= n_cached + i.
* [CB] §Continuous batching (ragged batching): prompts are concatenated with no
  batch dimension and the mask is block-diagonal, so no token of one request
  sees a token of another.
* [KVN] §MQA/GQA: num_kv_heads = num_query_heads / ratio.  Reading (the page
  does not say which query heads share a KV head): contiguous groups, query
  head h uses KV head h // (Hq / Hkv), as torch's ``enable_gqa`` does.

* [KVB] §Rolling KV Cache (a heading with no body).  Reading: a rolling cache
  keeps each request's W most recent keys, so a query at absolute position p
  sees the keys at positions p - W + 1 .. p (its own included); W = 0 means no
  window.  The cache's memory side (blocks that leave every window are freed)
  belongs to the scheduler oracle.

A row whose mask is all False has an undefined softmax; the oracle returns 0 for
such a row (reading).  The causal step never produces one: every query sees its
own key.
"""
import numpy as np


def masked_softmax_attention(Q, K, V, mask, scale):
    """One attention head, [CB] §Attention.

    Q: [nQ, A], K: [nK, A], V: [nK, A] (float64), mask: bool [nQ, nK]
    (True = key j may influence query i), scale: float multiplying Q K^T.
    Returns (O [nQ, A], P [nQ, nK]) with P the row-softmax weights.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    mask = np.asarray(mask, dtype=bool)
    assert K.shape[0] == V.shape[0], "nK must equal nV"
    assert mask.shape == (Q.shape[0], K.shape[0])
    S = scale * (Q @ K.T)                       # scores [nQ, nK]
    S = np.where(mask, S, -np.inf)              # boolean mask applied pointwise
    P = np.zeros_like(S)
    for i in range(S.shape[0]):                 # softmax per row (per token)
        if not mask[i].any():
            continue                            # empty row -> output 0 (reading)
        row = S[i]
        e = np.exp(row - row.max())             # exp(-inf) = 0 for masked keys
        P[i] = e / e.sum()
    O = P @ V
    return O, P


def chunk_causal_mask(q_len, n_cached, window=0):
    """Mask [q_len, n_cached + q_len] of a chunk after ``n_cached`` stored tokens.

    [CB] §Chunked prefill (stored KV prepended, mask adjusted) on top of the causal
    mask of [CB] §Attention: entry (i, j) is True iff j <= n_cached + i.  A decode
    step is the case q_len = 1 ([CB] §KV cache); a fresh prefill is n_cached = 0.
    With a rolling window W > 0 ([KVB] §Rolling KV Cache, reading above) entry
    (i, j) also needs j > n_cached + i - W.
    """
    mask = np.zeros((q_len, n_cached + q_len), dtype=bool)
    for i in range(q_len):
        lo = max(0, n_cached + i + 1 - window) if window > 0 else 0
        mask[i, lo: n_cached + i + 1] = True
    return mask


def ragged_batch_mask(q_lens, ctx_lens):
    """Block-diagonal mask over a ragged batch, [CB] §Continuous batching.

    Rows are the concatenated new tokens of all requests (sum of q_lens); columns
    are the concatenated keys (each request's stored tokens then its new ones).
    Block r is ``chunk_causal_mask(q_lens[r], ctx_lens[r])``; everything outside
    the diagonal blocks is False.
    """
    nq = int(sum(q_lens))
    nk = int(sum(c + q for c, q in zip(ctx_lens, q_lens)))
    mask = np.zeros((nq, nk), dtype=bool)
    r0 = c0 = 0
    for q, c in zip(q_lens, ctx_lens):
        mask[r0:r0 + q, c0:c0 + c + q] = chunk_causal_mask(q, c)
        r0 += q
        c0 += c + q
    return mask


def kv_head_of(h, n_q_heads, n_kv_heads):
    """KV head used by query head h: contiguous groups ([KVN] §MQA/GQA, reading)."""
    assert n_q_heads % n_kv_heads == 0
    return h // (n_q_heads // n_kv_heads)


def attention_step(q, q_lens, ctx_lens, k_seq, v_seq, scale, n_q_heads, n_kv_heads, window=0):
    """One attention step over a batch, request by request and head by head.

    q:        [nQ, Hq, A]   new query rows, requests concatenated in order.
    q_lens:   new tokens per request; ctx_lens: tokens stored before this step.
    k_seq[r], v_seq[r]: [ctx_lens[r] + q_lens[r], Hkv, A] -- request r's stored
              keys/values followed by the new ones (the contiguous layout of
              [KVB] §连续内存分配).
    window:   rolling-window length W (0: none), see ``chunk_causal_mask``.
    Returns out [nQ, Hq, A] in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    out = np.zeros_like(q)
    t0 = 0
    for r, (ql, cl) in enumerate(zip(q_lens, ctx_lens)):
        K = np.asarray(k_seq[r], dtype=np.float64)
        V = np.asarray(v_seq[r], dtype=np.float64)
        assert K.shape[0] == cl + ql and V.shape[0] == cl + ql
        mask = chunk_causal_mask(ql, cl, window)
        for h in range(n_q_heads):
            g = kv_head_of(h, n_q_heads, n_kv_heads)
            O, _ = masked_softmax_attention(q[t0:t0 + ql, h], K[:, g], V[:, g], mask, scale)
            out[t0:t0 + ql, h] = O
        t0 += ql
    return out


def attention_step_ragged(q, q_lens, ctx_lens, k_seq, v_seq, scale, n_q_heads, n_kv_heads):
    """The same step in the ragged form of [CB] §Continuous batching.

    All requests' keys are concatenated into one K/V of length sum(ctx + q) and one
    explicit block-diagonal boolean mask [nQ, sum(ctx + q)] keeps requests apart.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.concatenate([np.asarray(k, dtype=np.float64) for k in k_seq], axis=0)
    V = np.concatenate([np.asarray(v, dtype=np.float64) for v in v_seq], axis=0)
    mask = ragged_batch_mask(q_lens, ctx_lens)
    out = np.zeros_like(q)
    for h in range(n_q_heads):
        g = kv_head_of(h, n_q_heads, n_kv_heads)
        O, _ = masked_softmax_attention(q[:, h], K[:, g], V[:, g], mask, scale)
        out[:, h] = O
    return out


def attention_rows(q_rows, k, v, positions, scale, n_q_heads, n_kv_heads, window=0):
    """Selected query rows of one request (for sampled checks at large sizes).

    q_rows: [n, Hq, A] query rows at absolute positions ``positions`` (each row i
    sees keys 0..positions[i], or with a rolling window W > 0 the keys
    positions[i] - W + 1 .. positions[i]); k, v: [>= max(positions)+1, Hkv, A].
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(q_rows)
    for i, p in enumerate(positions):
        mask = np.ones((1, p + 1), dtype=bool)
        if window > 0:
            mask[0, : max(0, p + 1 - window)] = False
        for h in range(n_q_heads):
            g = kv_head_of(h, n_q_heads, n_kv_heads)
            O, _ = masked_softmax_attention(q_rows[i:i + 1, h], k[:p + 1, g], v[:p + 1, g], mask, scale)
            out[i, h] = O[0]
    return out
