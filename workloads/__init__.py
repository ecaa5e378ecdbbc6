"""Seeded synthetic inputs for the paged-KV continuous-batching attention step.

Shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``; imported by
neither the oracle nor the CUDA library.  It holds only shapes, seeded random
draws and the packing of those draws into buffers -- no attention, masking,
slot-mapping or scheduling arithmetic.

Five workloads, all bf16 with K/V/Q ~ N(0, 1), block_size 16:

tiny      1 layer, 4 q heads = 4 kv heads, head_dim 64; requests (cached, new):
          (37, 1) decode, (100, 1) decode, (4, 3) the second chunk of a 7-token
          prompt cut at 4, (0, 20) fresh prefill; 64-block pool, tables drawn
          from a random permutation of it.
decode    MHA 32 x 128 (a Llama-2-7B attention layer), 64 decode requests with
          cached lengths uniform in [512, 4096]; 20 GB K+V pool, blocks
          randomly scattered.
mixed     GQA 32 q / 8 kv x 128: 48 decodes (cached uniform in [256, 8192]) and
          two 512-token prefill chunks after 1024 and 3072 cached tokens.
          Variant "mixed_budget" keeps to the 560-token step budget: the 48
          decodes and the first chunk only.
long      GQA 32/8 x 128: step k (0..15) of a 32768-token prompt processed in
          2048-token chunks (2048 k cached tokens), co-scheduled with 16 decodes
          at 8192 + k cached tokens.
trace     256 requests for the continuous-batching trace: prompt lengths
          min(8192, round(lognormal(ln 512, 1.0))), output lengths geometric
          with mean 256, Poisson arrivals at 2 per step; 32 layers of GQA 32/8.
"""
from dataclasses import dataclass

import numpy as np

BLOCK_SIZE = 16
GB = 10 ** 9


@dataclass(frozen=True)
class StepShape:
    name: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_lens: tuple
    ctx_lens: tuple
    seed: int = 0

    @property
    def n_reqs(self):
        return len(self.q_lens)

    @property
    def n_tokens(self):
        return int(sum(self.q_lens))

    def kv_block_bytes(self):
        """Bytes of one physical block of K plus V (bf16)."""
        return 2 * self.n_kv_heads * self.block_size * self.head_dim * 2


def pool_blocks(pool_bytes, n_kv_heads, head_dim, block_size=BLOCK_SIZE):
    """How many K+V blocks of bf16 fit in ``pool_bytes``."""
    return int(pool_bytes // (2 * n_kv_heads * block_size * head_dim * 2))


def tiny(seed=0):
    return StepShape("tiny", 4, 4, 64, BLOCK_SIZE, 64,
                     q_lens=(1, 1, 3, 20), ctx_lens=(37, 100, 4, 0), seed=seed)


def decode(seed=0, n_reqs=64, ctx_lo=512, ctx_hi=4096, pool_bytes=20 * GB):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=n_reqs)
    return StepShape("decode", 32, 32, 128, BLOCK_SIZE, pool_blocks(pool_bytes, 32, 128),
                     q_lens=(1,) * n_reqs, ctx_lens=tuple(int(c) for c in ctx), seed=seed)


def mixed(seed=0, budget_variant=False, pool_bytes=20 * GB):
    rng = np.random.default_rng(seed)
    ctx = [int(c) for c in rng.integers(256, 8192 + 1, size=48)]
    q = [1] * 48
    chunks = [(1024, 512)] if budget_variant else [(1024, 512), (3072, 512)]
    for c, n in chunks:
        ctx.append(c)
        q.append(n)
    return StepShape("mixed_budget" if budget_variant else "mixed", 32, 8, 128, BLOCK_SIZE,
                     pool_blocks(pool_bytes, 8, 128), q_lens=tuple(q), ctx_lens=tuple(ctx), seed=seed)


def gqa_decode(seed=0, pool_bytes=20 * GB):
    """The decode requests of ``mixed`` alone: a decode-only step of 48 requests,
    GQA 32/8 x 128, ctx U[256, 8192] (same seed, same lengths)."""
    m = mixed(seed=seed, pool_bytes=pool_bytes)
    ctx = [c for c, q in zip(m.ctx_lens, m.q_lens) if q == 1]
    return StepShape("gqa_decode", m.n_q_heads, m.n_kv_heads, m.head_dim, m.block_size, m.num_blocks,
                     (1,) * len(ctx), tuple(ctx), m.seed)


def mqa_decode(seed=0, n_kv_heads=1, n_reqs=256, ctx_lo=1024, ctx_hi=16384, pool_bytes=20 * GB):
    """Decode-only step of a Llama-2-7B-shaped layer with multi-query attention
    (32 query heads on 1 KV head; n_kv_heads=2: GQA groups of 16): 256 requests,
    stored contexts uniform in [1024, 16384], so the K/V read per step (~1.1 GB
    for one KV head) is still far larger than L2."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=n_reqs)
    name = "mqa_decode" if n_kv_heads == 1 else f"gqa{32 // n_kv_heads}_decode"
    return StepShape(name, 32, n_kv_heads, 128, BLOCK_SIZE, pool_blocks(pool_bytes, n_kv_heads, 128),
                     q_lens=(1,) * n_reqs, ctx_lens=tuple(int(c) for c in ctx), seed=seed)


def long(k=15, seed=0, pool_bytes=20 * GB):
    assert 0 <= k < 16
    q = (1,) * 16 + (2048,)
    ctx = (8192 + k,) * 16 + (2048 * k,)
    return StepShape(f"long_k{k}", 32, 8, 128, BLOCK_SIZE, pool_blocks(pool_bytes, 8, 128),
                     q_lens=q, ctx_lens=ctx, seed=seed)


def scaled(shape, name=None, n_q_heads=None, n_kv_heads=None, head_dim=None,
           q_lens=None, ctx_lens=None, num_blocks=None, seed=None):
    """A copy of ``shape`` with some fields replaced (for small parity cases)."""
    return StepShape(name or shape.name,
                     n_q_heads or shape.n_q_heads, n_kv_heads or shape.n_kv_heads,
                     head_dim or shape.head_dim, shape.block_size,
                     num_blocks or shape.num_blocks,
                     tuple(q_lens) if q_lens is not None else shape.q_lens,
                     tuple(ctx_lens) if ctx_lens is not None else shape.ctx_lens,
                     shape.seed if seed is None else seed)


def random_step(seed, n_reqs, max_ctx, max_q, n_q_heads, n_kv_heads, head_dim,
                p_decode=0.5, extra_blocks=8):
    """A small random ragged step: each request decodes (1 new token) with
    probability p_decode, else takes a chunk of 2..max_q new tokens."""
    rng = np.random.default_rng(seed)
    q, c = [], []
    for _ in range(n_reqs):
        c.append(int(rng.integers(0, max_ctx + 1)))
        q.append(1 if rng.random() < p_decode else int(rng.integers(2, max_q + 1)))
    need = sum(-(-(a + b) // BLOCK_SIZE) for a, b in zip(c, q))
    return StepShape(f"random{seed}", n_q_heads, n_kv_heads, head_dim, BLOCK_SIZE,
                     need + extra_blocks, tuple(q), tuple(c), seed)


def block_tables(shape):
    """Per-request block tables drawn from one seeded permutation of the pool.

    Request r receives the next ceil((ctx + q) / block_size) entries of the
    permutation, so its blocks are scattered over the pool.  Rows are padded with
    -1 to the longest table.  Returns int32 [n_reqs, max_blocks].
    """
    rng = np.random.default_rng(shape.seed + 7919)
    perm = rng.permutation(shape.num_blocks)
    counts = [-(-(c + q) // shape.block_size) for c, q in zip(shape.ctx_lens, shape.q_lens)]
    assert sum(counts) <= shape.num_blocks, "pool too small for this step"
    width = max(max(counts), 1)
    table = np.full((shape.n_reqs, width), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(counts):
        table[r, :n] = perm[off:off + n]
        off += n
    return table


def _bf16_normal_cpu(rng, shape):
    import torch
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def step_inputs_cpu(shape):
    """All inputs of one step as CPU tensors, from NumPy PCG64 (same on every host).

    Returns dict with bf16 tensors q [nQ, Hq, A], k_new/v_new [nQ, Hkv, A],
    k_pool/v_pool [num_blocks, Hkv, bs, A] (every block random, used or not) and
    int32 arrays q_lens, ctx_lens, block_tables.
    """
    rng = np.random.default_rng(shape.seed)
    nq, hq, hk, a = shape.n_tokens, shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    pool = (shape.num_blocks, hk, shape.block_size, a)
    return dict(
        q=_bf16_normal_cpu(rng, (nq, hq, a)),
        k_new=_bf16_normal_cpu(rng, (nq, hk, a)),
        v_new=_bf16_normal_cpu(rng, (nq, hk, a)),
        k_pool=_bf16_normal_cpu(rng, pool),
        v_pool=_bf16_normal_cpu(rng, pool),
        q_lens=np.asarray(shape.q_lens, dtype=np.int32),
        ctx_lens=np.asarray(shape.ctx_lens, dtype=np.int32),
        block_tables=block_tables(shape),
    )


def step_inputs_device(shape, device):
    """The same buffers generated on ``device`` with a seeded torch generator
    (for the full-size workloads, whose pools are tens of GB)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(shape.seed)
    nq, hq, hk, a = shape.n_tokens, shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    pool = (shape.num_blocks, hk, shape.block_size, a)

    def rnd(s):
        return torch.randn(s, generator=g, device=device, dtype=torch.bfloat16)
    return dict(
        q=rnd((nq, hq, a)), k_new=rnd((nq, hk, a)), v_new=rnd((nq, hk, a)),
        k_pool=rnd(pool), v_pool=rnd(pool),
        q_lens=np.asarray(shape.q_lens, dtype=np.int32),
        ctx_lens=np.asarray(shape.ctx_lens, dtype=np.int32),
        block_tables=block_tables(shape),
    )


@dataclass(frozen=True)
class TraceShape:
    name: str
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    token_budget: int
    num_blocks: int
    requests: tuple        # (arrival_step, prompt_len, output_len), arrival order
    seed: int = 0


def trace(seed=0, n_requests=256, pool_bytes=60 * GB, token_budget=2048, n_layers=32,
          rate=2.0, median_prompt=512, sigma=1.0, cap=8192, mean_output=256):
    """The continuous-batching trace: the block pool is shared by all layers, so a
    block id names one block in each layer (pool bytes / (layers x K+V block))."""
    rng = np.random.default_rng(seed)
    gaps = rng.exponential(1.0 / rate, size=n_requests)
    arrivals = np.floor(np.cumsum(gaps)).astype(np.int64)
    prompts = np.minimum(cap, np.maximum(1, np.rint(
        rng.lognormal(np.log(median_prompt), sigma, size=n_requests)))).astype(np.int64)
    outputs = rng.geometric(1.0 / mean_output, size=n_requests).astype(np.int64)
    per_block = n_layers * 2 * 8 * BLOCK_SIZE * 128 * 2
    return TraceShape("trace", n_layers, 32, 8, 128, BLOCK_SIZE, token_budget,
                      int(pool_bytes // per_block),
                      tuple((int(a), int(p), int(o)) for a, p, o in zip(arrivals, prompts, outputs)),
                      seed)


def free_order(num_blocks, seed):
    """Initial free-list order of the block allocator: a seeded permutation."""
    return np.random.default_rng(seed + 104729).permutation(num_blocks).astype(np.int32)


def small_trace(seed, n_requests=24, num_blocks=20, token_budget=48, max_prompt=60,
                mean_output=12, rate=1.5):
    """A small trace whose pool is tight enough to force preemptions."""
    rng = np.random.default_rng(seed)
    arrivals = np.floor(np.cumsum(rng.exponential(1.0 / rate, size=n_requests))).astype(np.int64)
    prompts = rng.integers(1, max_prompt + 1, size=n_requests)
    outputs = rng.geometric(1.0 / mean_output, size=n_requests)
    return TraceShape(f"small_trace{seed}", 1, 4, 4, 64, BLOCK_SIZE, token_budget, num_blocks,
                      tuple((int(a), int(p), int(o)) for a, p, o in zip(arrivals, prompts, outputs)),
                      seed)


def with_prefixes(tr, n_groups, prefix_len, seed=0, share=1.0):
    """The same trace with shared system prompts: each request (with probability
    `share`) joins one of n_groups prefix groups, and its prompt becomes the
    group's prefix_len tokens followed by its own prompt.  Requests become
    (arrival, prompt, output, group, prefix_len), group -1 for none."""
    rng = np.random.default_rng(seed + 7919)
    out = []
    for a, p, o in tr.requests:
        if rng.random() < share:
            out.append((a, p + prefix_len, o, int(rng.integers(n_groups)), prefix_len))
        else:
            out.append((a, p, o, -1, 0))
    return TraceShape(tr.name + f"_prefix{n_groups}x{prefix_len}", tr.n_layers, tr.n_q_heads, tr.n_kv_heads,
                      tr.head_dim, tr.block_size, tr.token_budget, tr.num_blocks, tuple(out), tr.seed)


@dataclass(frozen=True)
class SequenceShape:
    """Consecutive steps that share one KV pool and one set of block tables:
    step k's table rows are rows of ``tables`` (request r of step k uses row
    ``rows[k][r]``)."""
    name: str
    steps: tuple          # StepShape per step
    rows: tuple           # per step, the table row of each request
    tables: np.ndarray    # int32 [n_rows, max_blocks], -1 padded


def long_sequence(seed=0, pool_bytes=20 * GB, n_chunks=16, chunk=2048, n_dec=16, dec_ctx=8192):
    """The long-context workload as a sequence: a 32768-token prompt in 16
    chunks of 2048 (step k: 2048 k stored tokens), each step co-scheduled with
    16 decodes at 8192 + k stored tokens.  One seeded permutation of the pool
    gives the prompt's 2048 blocks and each decode's blocks, so every step's
    table rows are slices of the same tables."""
    num_blocks = pool_blocks(pool_bytes, 8, 128)
    prompt_blocks = chunk * n_chunks // BLOCK_SIZE
    dec_blocks = -(-(dec_ctx + n_chunks) // BLOCK_SIZE)
    assert prompt_blocks + n_dec * dec_blocks <= num_blocks, "pool too small"
    perm = np.random.default_rng(seed + 7919).permutation(num_blocks).astype(np.int32)
    tables = np.full((n_dec + 1, prompt_blocks), -1, np.int32)
    for d in range(n_dec):
        tables[d, :dec_blocks] = perm[prompt_blocks + d * dec_blocks:prompt_blocks + (d + 1) * dec_blocks]
    tables[n_dec] = perm[:prompt_blocks]
    steps = tuple(StepShape(f"long_seq_k{k}", 32, 8, 128, BLOCK_SIZE, num_blocks,
                            q_lens=(1,) * n_dec + (chunk,), ctx_lens=(dec_ctx + k,) * n_dec + (chunk * k,),
                            seed=seed + k) for k in range(n_chunks))
    return SequenceShape("long_seq", steps, tuple(tuple(range(n_dec + 1)) for _ in steps), tables)
