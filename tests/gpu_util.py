"""Shared helpers of the GPU parity tests: run one step through the C-ABI and
build the oracle's view of the same seeded inputs."""
import math
import os

import numpy as np
import torch

import workloads as wl
from oracle import attention as oa
from oracle import paged as op

ATOL = 2e-2          # max abs error, bf16 inputs and output, fp32 accumulation
RTOL_NORM = 1e-2     # max abs error / max |reference|


def L():
    from paged_kv_cache_cb_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from paged_kv_cache_cb_gb300 import build
        build.build()
    return _lib


def cu_of(q_lens):
    return np.concatenate([[0], np.cumsum(np.asarray(q_lens, np.int64))]).astype(np.int32)


def device_step(shape, inp, dev="cuda", scale=None, ws_extra=0, check=True, attn_tables=None, fused=False,
                slots=None, window=None):
    """Append the step's new K/V and run attention; returns (out, k_cache, v_cache, status).
    ``attn_tables`` replaces the block tables that attention reads (the append
    still uses the slots of ``inp["block_tables"]``, or ``slots`` if given).
    ``fused``: one cb_kv_append_paged_attention call instead of the two.
    ``window``: the rolling-window entry points with this window."""
    lib = L()
    scale = scale if scale is not None else 1.0 / math.sqrt(shape.head_dim)
    if slots is None:
        slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    bt = inp["block_tables"] if attn_tables is None else attn_tables
    k_cache = inp["k_pool"].to(dev).clone() if inp["k_pool"].device.type == "cpu" else inp["k_pool"]
    v_cache = inp["v_pool"].to(dev).clone() if inp["v_pool"].device.type == "cpu" else inp["v_pool"]
    q = inp["q"].to(dev)
    k_new, v_new = inp["k_new"].to(dev), inp["v_new"].to(dev)
    d_slots = torch.from_numpy(np.asarray(slots, np.int64)).to(dev)
    if not fused:
        lib.cb_kv_append(k_new, v_new, d_slots, k_cache, v_cache)
    kv = [c + n for c, n in zip(shape.ctx_lens, shape.q_lens)]
    max_q, max_kv = max(max(shape.q_lens), 1), max(max(kv), 1)
    wsb = lib.cb_paged_attention_workspace_size(shape.n_reqs, shape.n_tokens, max_q, max_kv, shape.n_q_heads,
                                                shape.n_kv_heads, shape.head_dim, shape.block_size)
    ws = torch.empty(wsb + ws_extra, dtype=torch.uint8, device=dev)
    out = torch.full_like(q, float("nan"))
    meta = (q, torch.from_numpy(cu_of(shape.q_lens)).to(dev), torch.tensor(shape.ctx_lens, dtype=torch.int32, device=dev),
            torch.from_numpy(bt).to(dev))
    if fused and window is not None:
        lib.cb_kv_append_paged_attention_window(k_new, v_new, d_slots, *meta, k_cache, v_cache, out, scale, ws, max_q,
                                                max_kv, window)
    elif fused:
        lib.cb_kv_append_paged_attention(k_new, v_new, d_slots, *meta, k_cache, v_cache, out, scale, ws, max_q, max_kv)
    elif window is not None:
        lib.cb_paged_attention_window(*meta, k_cache, v_cache, out, scale, ws, max_q, max_kv, window)
    else:
        lib.cb_paged_attention(*meta, k_cache, v_cache, out, scale, ws, max_q, max_kv)
    status = lib.cb_last_error()
    if check:
        assert status == 0, lib.cb_strerror(status)
    return out, k_cache, v_cache, status


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_step(shape, inp, scale=None, window=0):
    """fp64 oracle of the whole step: each request's stored rows read through its
    block table from the initial pool, followed by its new rows."""
    scale = scale if scale is not None else 1.0 / math.sqrt(shape.head_dim)
    kp, vp = f64(inp["k_pool"]), f64(inp["v_pool"])
    kn, vn, q = f64(inp["k_new"]), f64(inp["v_new"]), f64(inp["q"])
    ks, vs = [], []
    t0 = 0
    for r, (c, n) in enumerate(zip(shape.ctx_lens, shape.q_lens)):
        ks.append(np.concatenate([op.gather_request(kp, inp["block_tables"][r], c, shape.block_size), kn[t0:t0 + n]]))
        vs.append(np.concatenate([op.gather_request(vp, inp["block_tables"][r], c, shape.block_size), vn[t0:t0 + n]]))
        t0 += n
    return oa.attention_step(q, shape.q_lens, shape.ctx_lens, ks, vs, scale, shape.n_q_heads, shape.n_kv_heads,
                             window=window)


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref).max() if got.size else 0.0
    den = max(np.abs(ref).max(), 1e-30) if ref.size else 1.0
    assert err <= ATOL, f"{what}: max abs err {err:.3e} > {ATOL}"
    assert err / den <= RTOL_NORM, f"{what}: normwise rel err {err / den:.3e} > {RTOL_NORM}"
    return err


def sampled_request_oracle(shape, inp, r, rows=None, scale=None, window=0):
    """Oracle for (some rows of) request r of a full-size step whose pool lives on
    the GPU: copy just r's physical blocks to the host, then read them through the
    oracle's gather with the table rewritten onto that compact copy."""
    scale = scale if scale is not None else 1.0 / math.sqrt(shape.head_dim)
    c, n = shape.ctx_lens[r], shape.q_lens[r]
    cu = cu_of(shape.q_lens)
    nblk = -(-c // shape.block_size)
    table = inp["block_tables"][r, :max(nblk, 1)]
    idx = torch.from_numpy(table[:nblk].astype(np.int64)).to(inp["k_pool"].device)
    kp = f64(inp["k_pool"].index_select(0, idx)) if nblk else np.zeros((0,) + tuple(inp["k_pool"].shape[1:]))
    vp = f64(inp["v_pool"].index_select(0, idx)) if nblk else np.zeros((0,) + tuple(inp["v_pool"].shape[1:]))
    compact = np.arange(nblk)
    kc = op.gather_request(kp, compact, c, shape.block_size) if nblk else kp.reshape(0, shape.n_kv_heads, shape.head_dim)
    vc = op.gather_request(vp, compact, c, shape.block_size) if nblk else vp.reshape(0, shape.n_kv_heads, shape.head_dim)
    kn = f64(inp["k_new"][cu[r]:cu[r + 1]])
    vn = f64(inp["v_new"][cu[r]:cu[r + 1]])
    k = np.concatenate([kc, kn])
    v = np.concatenate([vc, vn])
    rows = list(range(n)) if rows is None else list(rows)
    q = f64(inp["q"][cu[r]:cu[r + 1]])[rows]
    return oa.attention_rows(q, k, v, [c + i for i in rows], scale, shape.n_q_heads, shape.n_kv_heads,
                             window=window), rows
