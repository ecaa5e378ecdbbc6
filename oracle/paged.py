"""Paged KV layout oracle (test infrastructure only; see the package docstring).

[SM] §PagedAttention 批处理 and [KVB] §思想: each request's KV is cut into
fixed-size logical blocks; a per-request block table maps logical block b to a
physical block of a shared pool; a new physical block is taken only when the
current one is full.

Readings (the pages fix no layout):
* pool layout [num_blocks, Hkv, block_size, A] (head-major blocks);
* the slot of absolute token position p of a request is
  table[p // block_size] * block_size + p % block_size; a negative slot means
  "do not write this row".
"""
import numpy as np


def slot_of(table_row, pos, block_size):
    """Physical slot of token position ``pos`` through one block-table row."""
    return int(table_row[pos // block_size]) * block_size + pos % block_size


def slot_mapping(block_tables, q_lens, ctx_lens, block_size):
    """Slots of every new token of a step, requests concatenated in order.

    Request r's new tokens occupy positions ctx_lens[r] .. ctx_lens[r]+q_lens[r]-1.
    Returns int64 [sum(q_lens)].
    """
    out = []
    for r, (ql, cl) in enumerate(zip(q_lens, ctx_lens)):
        for i in range(ql):
            out.append(slot_of(block_tables[r], cl + i, block_size))
    return np.asarray(out, dtype=np.int64)


def append_rows(cache, rows, slots, block_size):
    """Write ``rows`` [n, Hkv, A] into ``cache`` [num_blocks, Hkv, bs, A] in place.

    Row t goes to physical block slots[t] // bs at in-block offset slots[t] % bs,
    for every KV head.  Rows with a negative slot are skipped.
    """
    for t in range(len(slots)):
        s = int(slots[t])
        if s < 0:
            continue
        cache[s // block_size, :, s % block_size, :] = rows[t]
    return cache


def gather_request(cache, table_row, n_tokens, block_size):
    """A request's first ``n_tokens`` KV rows, read through its block table.

    Returns the contiguous [n_tokens, Hkv, A] view that the contiguous layout of
    [KVB] §连续内存分配 would hold.
    """
    out = np.empty((n_tokens,) + (cache.shape[1], cache.shape[3]), dtype=cache.dtype)
    for p in range(n_tokens):
        s = slot_of(table_row, p, block_size)
        out[p] = cache[s // block_size, :, s % block_size, :]
    return out
