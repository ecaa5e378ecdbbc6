"""CPU oracle of one continuous-batching attention step over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its
Python binding) imports, links or runs anything in this package; only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may use it.  It shares no code, header, table or helper with the CUDA
path.  All floating point is fp64 (NumPy); loops are plain and follow the pages'
definitions in the order the pages give them, so a reader can check them by eye.

Sources cited in this package (pages on KV caching and continuous batching):

[CB]  "Continuous batching from first principles" (Chinese translation,
      news.myit.tw/news/j9529p) -- sections Attention, KV cache, Chunked prefill,
      Continuous batching.  The authority on what attention computes.
[SM]  "AWS SageMaker 推理方案" (clvsit.github.io) -- sections 动态批处理 (dynamic
      batching), 连续批处理 (continuous batching), PagedAttention 批处理.
[KVN] "KV Cache与Continuous Batching" study notes (huajishe.fun) -- sections
      KV Cache内存占用 (memory formula and example table), MQA/GQA,
      Continuous Batching原理 (iteration-level scheduler), 调度策略 (FCFS,
      preemption), Batch大小选择.
[KVB] "kv_cache" blog (klklkl10086.github.io) -- sections 连续内存分配 (the
      contiguous TraditionalKVCache), Batch Decode (batch_decode_step), 思想
      (block table maps logical KV blocks to physical blocks).

Modules:
    attention  -- masked-softmax attention, chunk/causal and ragged block-diagonal
                  masks, the per-request step and the explicit ragged form.
    paged      -- slot mapping from block tables, the append loop, the gather of a
                  request's contiguous K/V from a paged pool.
    sizes      -- KV-cache byte formulas, chunk counts, padding counts.
    scheduler  -- FCFS iteration-level scheduler with a block allocator and
                  recompute preemption (host metadata only).

Every function is pinned by a ``-m "not gpu"`` test against something other than
itself (values the pages print, closed forms, a library routine, brute force on
tiny inputs, invariants).  No function here is "parity unpinned".
"""
