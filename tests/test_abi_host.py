"""The C-ABI library without a GPU: it loads, exports every entry point that
include/cbattn.h declares, rejects bad arguments on the host before touching
CUDA, and its pure-host functions (workspace sizing, slot mapping) agree with
the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as wl
from oracle import paged as op

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    from paged_kv_cache_cb_gb300 import _lib as L
    if not os.path.exists(L.LIB_PATH):
        from paged_kv_cache_cb_gb300 import build
        build.build()
    return L


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "cbattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cb_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for must in ("cb_kv_append", "cb_paged_attention", "cb_paged_attention_workspace_size", "cb_last_error",
                 "cb_strerror", "cb_sched_create", "cb_sched_step", "cb_build_slot_mapping"):
        assert must in syms


def test_library_exports_every_declared_symbol():
    L = _lib()
    lib = ctypes.CDLL(L.LIB_PATH)
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing
    bound = {name for name, _, _ in L.SIGNATURES}
    assert set(declared_symbols()) == bound, "binding must cover exactly the header's entry points"


def test_host_side_argument_checks():
    L = _lib().lib()
    V = ctypes.c_void_p
    dummy = V(4096)
    # unsupported head_dim / block_size / group and bad sizes are rejected before any CUDA call
    assert L.cb_kv_append(dummy, dummy, dummy, 4, dummy, dummy, 8, 2, 96, 16, None) == -1
    assert L.cb_kv_append(dummy, dummy, dummy, 4, dummy, dummy, 8, 2, 128, 32, None) == -1
    args = lambda **kw: [kw.get(k, v) for k, v in [
        ("q", dummy), ("cu", dummy), ("ctx", dummy), ("bt", dummy), ("maxb", 4), ("nr", 2), ("nt", 3),
        ("mq", 2), ("mkv", 40), ("kc", dummy), ("vc", dummy), ("nb", 16), ("out", dummy), ("scale", 0.1),
        ("hq", 4), ("hk", 2), ("a", 128), ("bs", 16), ("ws", dummy), ("wsb", 1 << 30), ("s", None)]]
    assert L.cb_paged_attention(*args(hq=6, hk=4)) == -1            # Hq % Hkv != 0
    assert L.cb_paged_attention(*args(hq=64, hk=4)) == -1           # group 16 only with 32 q heads on 2 KV heads
    assert L.cb_paged_attention(*args(hq=16, hk=1)) == -1           # group 16 only with 32 q heads on 2 KV heads
    assert L.cb_paged_attention(*args(hq=32, hk=2, a=64)) == -1     # group 16 and 32: head_dim 128 only
    assert L.cb_paged_attention(*args(hq=64, hk=2)) == -1           # group 32 only with 1 KV head
    assert L.cb_paged_attention(*args(a=96)) == -1
    assert L.cb_paged_attention(*args(bs=8)) == -1
    assert L.cb_paged_attention(*args(nr=5000)) == -1               # more than CB_MAX_REQS
    assert L.cb_paged_attention(*args(scale=0.0)) == -1
    assert L.cb_paged_attention(*args(q=None)) == -1
    assert L.cb_paged_attention(*args(q=V(4100))) == -1             # not 16-byte aligned
    assert L.cb_paged_attention(*args(wsb=16)) == -3                # workspace too small
    assert L.cb_paged_attention(*args(nr=0)) == 0                   # empty batch: nothing to do
    assert L.cb_strerror(-3) == b"workspace too small"
    # the one-call step: the append arguments are checked too
    fargs = lambda **kw: [kw.get("kn", dummy), kw.get("vn", dummy), kw.get("sl", dummy)] + args(**kw)
    assert L.cb_kv_append_paged_attention(*fargs(kn=None)) == -1
    assert L.cb_kv_append_paged_attention(*fargs(vn=V(4104))) == -1   # not 16-byte aligned
    assert L.cb_kv_append_paged_attention(*fargs(a=96)) == -1
    assert L.cb_kv_append_paged_attention(*fargs(wsb=16)) == -3
    assert L.cb_kv_append_paged_attention(*fargs(nr=0)) == 0
    # block copies
    assert L.cb_copy_blocks(dummy, -1, dummy, dummy, 8, 8, 128, 16, None) == -1
    assert L.cb_copy_blocks(dummy, 1, dummy, dummy, 8, 8, 96, 16, None) == -1
    assert L.cb_copy_blocks(dummy, 1, dummy, V(4100), 8, 8, 128, 16, None) == -1
    assert L.cb_copy_blocks(None, 0, None, None, 8, 8, 128, 16, None) == 0   # nothing to copy


def test_workspace_size_query_includes_the_prefill_partials():
    """Block-tile shapes with prefill: the size query leaves room for the balanced
    prefill's partial results (2 x 160 slots of 256 rows x (A + 2) floats); a
    decode-only step or another shape needs none."""
    L = _lib().lib()
    region = 2 * 160 * 256 * (128 + 2) * 4
    with_pre = L.cb_paged_attention_workspace_size(4, 600, 512, 4096, 32, 8, 128, 16)
    dec = L.cb_paged_attention_workspace_size(4, 600, 1, 4096, 32, 8, 128, 16)
    assert with_pre - dec >= region
    mha_pre = L.cb_paged_attention_workspace_size(4, 600, 512, 4096, 32, 32, 128, 16)
    mha_dec = L.cb_paged_attention_workspace_size(4, 600, 1, 4096, 32, 32, 128, 16)
    assert mha_pre == mha_dec


def test_workspace_size_grows_with_requests_and_context():
    L = _lib()
    f = L.cb_paged_attention_workspace_size
    a = f(64, 64, 1, 4097, 32, 32, 128, 16)
    assert a > 0
    assert f(128, 128, 1, 4097, 32, 32, 128, 16) > a
    assert f(64, 64, 1, 8193, 32, 32, 128, 16) > a
    assert f(64, 64, 1, 4097, 32, 32, 96, 16) == 0
    # bound: n_reqs * ceil(ceil(kv/16)/8) splits of (A + 2) floats per q head, plus counters
    splits = 64 * -(-(-(-4097 // 16)) // 8)
    assert a >= splits * 32 * (128 + 2) * 4


@pytest.mark.parametrize("seed", range(4))
def test_host_slot_mapping_matches_oracle(seed):
    L = _lib()
    shape = wl.random_step(seed, n_reqs=9, max_ctx=70, max_q=20, n_q_heads=4, n_kv_heads=2, head_dim=64)
    bt = wl.block_tables(shape)
    got = L.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, bt, shape.block_size)
    want = op.slot_mapping(bt, shape.q_lens, shape.ctx_lens, shape.block_size)
    assert got.dtype == np.int64 and np.array_equal(got, want)


def test_host_slot_mapping_rejects_short_tables():
    L = _lib()
    with pytest.raises(L.CBError):
        L.cb_build_slot_mapping([3], [30], np.array([[1, 2]], np.int32), 16)   # needs 3 blocks
    with pytest.raises(L.CBError):
        L.cb_build_slot_mapping([1], [0], np.array([[-1]], np.int32), 16)


def test_binding_refuses_host_tensors():
    """No CPU fallback: every compute entry point of the binding refuses tensors
    that are not on a CUDA device before anything reaches the library."""
    import torch
    L = _lib()
    bf = torch.bfloat16
    q = torch.zeros(3, 4, 64, dtype=bf)
    kn = torch.zeros(3, 4, 64, dtype=bf)
    sl = torch.zeros(3, dtype=torch.int64)
    cu = torch.tensor([0, 3], dtype=torch.int32)
    ctx = torch.tensor([5], dtype=torch.int32)
    bt = torch.zeros(1, 4, dtype=torch.int32)
    kc = torch.zeros(8, 4, 16, 64, dtype=bf)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        L.cb_kv_append(kn, kn, sl, kc, kc)
    with pytest.raises(ValueError, match="CUDA"):
        L.cb_paged_attention(q, cu, ctx, bt, kc, kc, q.clone(), 0.125, ws, 3, 8)
    with pytest.raises(ValueError, match="CUDA"):
        L.cb_kv_append_paged_attention(kn, kn, sl, q, cu, ctx, bt, kc, kc, q.clone(), 0.125, ws, 3, 8)
    with pytest.raises(ValueError, match="CUDA"):
        L.cb_copy_blocks(torch.zeros(1, 2, dtype=torch.int32), kc, kc)


def test_graph_calls_reject_null_arguments():
    """cb_graph_begin / cb_graph_end check their arguments before any CUDA call."""
    L = _lib()
    lib = L.lib()
    g = lib.cb_graph_create()
    assert g
    try:
        assert lib.cb_graph_begin(g, None) == L.CB_EINVAL      # the legacy default stream cannot be captured
        assert lib.cb_graph_end(g, None) == L.CB_EINVAL
        assert lib.cb_graph_begin(None, 1) == L.CB_EINVAL
        assert lib.cb_graph_end(None, 1) == L.CB_EINVAL
    finally:
        lib.cb_graph_destroy(g)
    lib.cb_graph_destroy(None)                                 # a no-op

