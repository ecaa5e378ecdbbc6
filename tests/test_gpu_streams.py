"""Per-stream device state: each stream's error word is its own.  One step with
a bad block id runs on one stream while a clean step runs on another, both in
flight together; cb_last_error of each stream reports only its own step."""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import L, assert_close, cu_of, f64, oracle_step

pytestmark = pytest.mark.gpu


def _launch(shape, inp, tables, stream):
    lib = L()
    dev = "cuda"
    with torch.cuda.stream(stream):
        kc, vc = inp["k_pool"].to(dev), inp["v_pool"].to(dev)
        slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
        lib.cb_kv_append(inp["k_new"].to(dev), inp["v_new"].to(dev), torch.from_numpy(slots).to(dev), kc, vc,
                         stream=stream)
        max_q = max(shape.q_lens)
        max_kv = max(c + n for c, n in zip(shape.ctx_lens, shape.q_lens))
        ws = torch.empty(lib.cb_paged_attention_workspace_size(shape.n_reqs, shape.n_tokens, max_q, max_kv,
                                                               shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                                                               shape.block_size), dtype=torch.uint8, device=dev)
        out = torch.zeros_like(inp["q"], device=dev)
        lib.cb_paged_attention(inp["q"].to(dev), torch.from_numpy(cu_of(shape.q_lens)).to(dev),
                               torch.tensor(shape.ctx_lens, dtype=torch.int32, device=dev),
                               torch.from_numpy(tables).to(dev), kc, vc, out, 1.0 / math.sqrt(shape.head_dim), ws,
                               max_q, max_kv, stream=stream)
    return out, (kc, vc, ws)


@pytest.mark.parametrize("n_kv_heads", [8, 4], ids=["block_tiles", "cuda_cores"])
def test_error_word_is_per_stream(n_kv_heads):
    lib = L()
    shape = wl.random_step(90 + n_kv_heads, n_reqs=6, max_ctx=700, max_q=40, n_q_heads=32, n_kv_heads=n_kv_heads,
                           head_dim=128)
    inp = wl.step_inputs_cpu(shape)
    bad = inp["block_tables"].copy()
    bad[0, 0] = shape.num_blocks + 7
    s_bad, s_good = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    _, keep_bad = _launch(shape, inp, bad, s_bad)
    out, keep_good = _launch(shape, inp, inp["block_tables"], s_good)
    assert lib.cb_last_error(s_good) == 0           # the other stream's bad id is not reported here
    assert lib.cb_last_error(s_bad) == lib.CB_EDEVICE
    assert lib.cb_last_error(s_bad) == 0            # read and cleared
    assert_close(f64(out), oracle_step(shape, inp), "clean stream")
    torch.cuda.synchronize()
    del keep_bad, keep_good
