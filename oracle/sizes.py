"""Size formulas (test infrastructure only; see the package docstring)."""
import math


def kv_cache_bytes(batch, n_layers, n_kv_heads, seq_len, head_dim, bytes_per_value=2):
    """[KVN] §KV Cache内存占用: 2 x batch x layers x heads x seq_len x head_dim x bytes.

    The leading 2 counts K and V ([CB] §KV cache says the same for one token).
    """
    return 2 * batch * n_layers * n_kv_heads * seq_len * head_dim * bytes_per_value


def kv_values_per_token_per_layer(n_kv_heads, head_dim):
    """[CB] §KV cache: 2 x A x H values per token per layer (K and V)."""
    return 2 * n_kv_heads * head_dim


def n_chunks(n, m):
    """[CB] §Chunked prefill: a prompt of n tokens in chunks of m takes ceil(n/m) passes."""
    return -(-n // m)


def chunk_sizes(n, m):
    """The chunk lengths of that split, in order (all m except a shorter last one)."""
    return [min(m, n - s) for s in range(0, n, m)]


def left_padded_batch(lengths):
    """Build the rectangular left-padded batch of [CB] §Continuous batching (batched
    generation): every row padded on the left to the longest length.  Returns the
    rows as lists of 'pad'/'tok' markers, so that padding can be counted by hand.
    """
    width = max(lengths)
    return [["pad"] * (width - n) + ["tok"] * n for n in lengths]


def dynamic_insert_padding(batch_size, n_prompt):
    """Pad tokens when one of B decoding prompts is replaced by a new n-token prompt.

    [CB] §Continuous batching (dynamic scheduling): the new prompt's prefill runs
    next to B-1 prompts that each decode one token, so in the rectangular step the
    B-1 decode rows are padded to width n, and the new prompt needs no padding.
    Counted on the explicit batch built by ``left_padded_batch``.
    """
    rows = left_padded_batch([n_prompt] + [1] * (batch_size - 1))
    return sum(row.count("pad") for row in rows)


def blocks_for(n_tokens, block_size):
    """Physical blocks holding n tokens when a block is taken only once the last one
    is full ([SM] §PagedAttention 批处理)."""
    return math.ceil(n_tokens / block_size)
