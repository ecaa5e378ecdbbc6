"""ctypes binding of libcbattn.so (include/cbattn.h).

Argument marshalling only: every function here checks dtypes/devices/shapes,
turns torch tensors into raw pointers and sizes, calls the C entry point of the
same name and raises ``CBError`` on a non-zero return.  All computation happens
in the library's CUDA kernels (and, for the scheduler, its C++ host code).
There is no fallback: if the library is missing, ``lib()`` raises.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcbattn.so")

CB_OK, CB_EINVAL, CB_ECUDA, CB_EWORKSPACE, CB_EDEVICE, CB_ETIMEOUT, CB_ESTATE = 0, -1, -2, -3, -4, -5, -6
CB_MAX_REQS = 2048

_c_int, _c_size, _c_float, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_intp = ctypes.POINTER(ctypes.c_int)

# (name, restype, argtypes) of every exported entry point, in header order
SIGNATURES = [
    ("cb_kv_append", _c_int, [_vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp]),
    ("cb_copy_blocks", _c_int, [_vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp]),
    ("cb_paged_attention", _c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _c_int,
                                    _vp, _c_float, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp]),
    ("cb_paged_attention_workspace_size", _c_size, [_c_int] * 8),
    ("cb_kv_append_paged_attention", _c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                              _c_int, _vp, _vp, _c_int, _vp, _c_float, _c_int, _c_int, _c_int,
                                              _c_int, _vp, _c_size, _vp]),
    ("cb_paged_attention_window", _c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp,
                                           _c_int, _vp, _c_float, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                           _c_size, _vp]),
    ("cb_kv_append_paged_attention_window", _c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                                     _c_int, _c_int, _vp, _vp, _c_int, _vp, _c_float, _c_int,
                                                     _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp]),
    ("cb_paged_attention_noalloc", _c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp,
                                            _c_int, _vp, _c_float, _c_int, _c_int, _c_int, _c_int, _vp]),
    ("cb_last_error", _c_int, [_vp]),
    ("cb_strerror", ctypes.c_char_p, [_c_int]),
    ("cb_hbm_copy", _c_int, [_vp, _vp, _c_size, _vp]),
    ("cb_last_launch_count", _c_int, []),
    ("cb_graph_create", _vp, []),
    ("cb_graph_destroy", None, [_vp]),
    ("cb_graph_begin", _c_int, [_vp, _vp]),
    ("cb_graph_end", _c_int, [_vp, _vp]),
    ("cb_build_slot_mapping", _c_int, [_i32p, _i32p, _i32p, _c_int, _c_int, _c_int, _i64p]),
    ("cb_sched_create", _vp, [_c_int, _c_int, _c_int, _c_int, _i32p]),
    ("cb_sched_destroy", None, [_vp]),
    ("cb_sched_set_window", _c_int, [_vp, _c_int]),
    ("cb_sched_set_batching", _c_int, [_vp, _c_int, _c_int]),
    ("cb_sched_last_real_tokens", ctypes.c_longlong, [_vp]),
    ("cb_sched_add_request", _c_int, [_vp, _c_int, _c_int, _c_int]),
    ("cb_sched_add_request_prefix", _c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int]),
    ("cb_sched_step", _c_int, [_vp, _i32p, _i32p, _i32p, _i32p, _i32p, _c_int, _i64p, _intp, _intp]),
    ("cb_sched_step_copies", _c_int, [_vp, _i32p, _c_int]),
    ("cb_sched_done", _c_int, [_vp]),
    ("cb_sched_free_blocks", _c_int, [_vp]),
    ("cb_sched_request_info", _c_int, [_vp, _c_int, _intp, _intp, _intp, _intp]),
    ("cb_sched_kv_memory", _c_int, [_vp, _c_int, _i64p]),
]

_LIB = None


class CBError(RuntimeError):
    def __init__(self, fn, code):
        msg = lib().cb_strerror(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


def lib():
    """Load libcbattn.so (built in-tree by paged_kv_cache_cb_gb300.build)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; call paged_kv_cache_cb_gb300.build.build() first")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(fn, rc):
    if rc != CB_OK:
        raise CBError(fn, rc)


_torch = None


def _t():
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _stream(stream):
    """A stream handle: None = torch's current stream; an int is taken as the
    raw cudaStream_t (the cheapest form for tight loops)."""
    if stream is None:
        return _t().cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t, dtype, name, ndim=None):
    """Raw device pointer of a contiguous CUDA tensor of the given dtype and rank."""
    try:
        ok = t.is_cuda and t.dtype is dtype and (ndim is None or t.dim() == ndim) and t.is_contiguous()
    except AttributeError:
        ok = False
    if not ok:
        torch = _t()
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t.data_ptr()


def cb_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None):
    """k_new, v_new: bf16 [n_tokens, Hkv, A]; slot_mapping: int64 [n_tokens];
    k_cache, v_cache: bf16 [num_blocks, Hkv, block_size, A] (written in place)."""
    torch = _t()
    bf = torch.bfloat16
    pk = _dev(k_new, bf, "k_new", 3)
    pv = _dev(v_new, bf, "v_new", 3)
    ps = _dev(slot_mapping, torch.int64, "slot_mapping", 1)
    ck = _dev(k_cache, bf, "k_cache", 4)
    cv = _dev(v_cache, bf, "v_cache", 4)
    n, hk, a = k_new.shape
    if v_new.shape != k_new.shape or slot_mapping.numel() != n or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    nb, hk2, bs, a2 = k_cache.shape
    if (hk2, a2) != (hk, a):
        raise ValueError("cache heads/head_dim differ from k_new")
    _check("cb_kv_append", lib().cb_kv_append(pk, pv, ps, n, ck, cv, nb, hk, a, bs, _stream(stream)))


def cb_copy_blocks(pairs, k_cache, v_cache, stream=None):
    """pairs: int32 CUDA tensor [n, 2] of (src, dst) block ids; caches bf16
    [num_blocks, Hkv, block_size, A]: block dst becomes a copy of block src."""
    torch = _t()
    bf = torch.bfloat16
    pp = _dev(pairs, torch.int32, "pairs", 2)
    ck = _dev(k_cache, bf, "k_cache", 4)
    cv = _dev(v_cache, bf, "v_cache", 4)
    if pairs.shape[1] != 2 or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    nb, hk, bs, a = k_cache.shape
    _check("cb_copy_blocks", lib().cb_copy_blocks(pp, pairs.shape[0], ck, cv, nb, hk, a, bs, _stream(stream)))


def cb_paged_attention_workspace_size(n_reqs, n_tokens, max_q_len, max_kv_len, n_q_heads, n_kv_heads, head_dim,
                                      block_size):
    return int(lib().cb_paged_attention_workspace_size(n_reqs, n_tokens, max_q_len, max_kv_len, n_q_heads,
                                                       n_kv_heads, head_dim, block_size))


def cb_paged_attention(q, cu_q_lens, ctx_lens, block_tables, k_cache, v_cache, out, scale, workspace,
                       max_q_len, max_kv_len, stream=None):
    """q, out: bf16 [n_tokens, Hq, A]; cu_q_lens int32 [n_reqs+1]; ctx_lens int32 [n_reqs];
    block_tables int32 [n_reqs, max_blocks]; caches bf16 [num_blocks, Hkv, bs, A];
    workspace: uint8 CUDA tensor of at least cb_paged_attention_workspace_size bytes."""
    _attention("cb_paged_attention", None, q, cu_q_lens, ctx_lens, block_tables, k_cache, v_cache, out, scale,
               workspace, max_q_len, max_kv_len, stream)


def cb_paged_attention_window(q, cu_q_lens, ctx_lens, block_tables, k_cache, v_cache, out, scale, workspace,
                              max_q_len, max_kv_len, window, stream=None):
    """cb_paged_attention with a rolling window: a query at position p sees the
    keys p - window + 1 .. p (window 0: all)."""
    _attention("cb_paged_attention_window", int(window), q, cu_q_lens, ctx_lens, block_tables, k_cache, v_cache, out,
               scale, workspace, max_q_len, max_kv_len, stream)


def _attention(name, window, q, cu_q_lens, ctx_lens, block_tables, k_cache, v_cache, out, scale, workspace,
               max_q_len, max_kv_len, stream):
    torch = _t()
    bf = torch.bfloat16
    pq = _dev(q, bf, "q", 3)
    po = _dev(out, bf, "out", 3)
    pcu = _dev(cu_q_lens, torch.int32, "cu_q_lens", 1)
    pctx = _dev(ctx_lens, torch.int32, "ctx_lens", 1)
    pbt = _dev(block_tables, torch.int32, "block_tables", 2)
    ck = _dev(k_cache, bf, "k_cache", 4)
    cv = _dev(v_cache, bf, "v_cache", 4)
    pw = _dev(workspace, torch.uint8, "workspace", 1)
    n_tok, hq, a = q.shape
    n_reqs = ctx_lens.numel()
    if out.shape != q.shape or cu_q_lens.numel() != n_reqs + 1 or block_tables.shape[0] != n_reqs:
        raise ValueError("shape mismatch")
    nb, hk, bs, a2 = k_cache.shape
    if v_cache.shape != k_cache.shape or a2 != a:
        raise ValueError("cache shape mismatch")
    w = () if window is None else (window,)
    rc = getattr(lib(), name)(pq, pcu, pctx, pbt, block_tables.shape[1], n_reqs, n_tok, int(max_q_len),
                              int(max_kv_len), ck, cv, nb, po, float(scale), hq, hk, a, bs, *w, pw,
                              workspace.numel(), _stream(stream))
    _check(name, rc)


def cb_kv_append_paged_attention(k_new, v_new, slot_mapping, q, cu_q_lens, ctx_lens, block_tables, k_cache, v_cache,
                                 out, scale, workspace, max_q_len, max_kv_len, stream=None):
    """cb_kv_append of the step's new rows, then cb_paged_attention, as one call
    (one kernel launch where the attention launch is cooperative).  Arguments as
    for those two; k_new, v_new: bf16 [n_tokens, Hkv, A] with n_tokens = q's."""
    _append_attention("cb_kv_append_paged_attention", None, k_new, v_new, slot_mapping, q, cu_q_lens, ctx_lens,
                      block_tables, k_cache, v_cache, out, scale, workspace, max_q_len, max_kv_len, stream)


def cb_kv_append_paged_attention_window(k_new, v_new, slot_mapping, q, cu_q_lens, ctx_lens, block_tables, k_cache,
                                        v_cache, out, scale, workspace, max_q_len, max_kv_len, window, stream=None):
    """cb_kv_append_paged_attention with a rolling window (see
    cb_paged_attention_window)."""
    _append_attention("cb_kv_append_paged_attention_window", int(window), k_new, v_new, slot_mapping, q, cu_q_lens,
                      ctx_lens, block_tables, k_cache, v_cache, out, scale, workspace, max_q_len, max_kv_len, stream)


def _append_attention(name, window, k_new, v_new, slot_mapping, q, cu_q_lens, ctx_lens, block_tables, k_cache,
                      v_cache, out, scale, workspace, max_q_len, max_kv_len, stream):
    torch = _t()
    bf = torch.bfloat16
    pk = _dev(k_new, bf, "k_new", 3)
    pv = _dev(v_new, bf, "v_new", 3)
    ps = _dev(slot_mapping, torch.int64, "slot_mapping", 1)
    pq = _dev(q, bf, "q", 3)
    po = _dev(out, bf, "out", 3)
    pcu = _dev(cu_q_lens, torch.int32, "cu_q_lens", 1)
    pctx = _dev(ctx_lens, torch.int32, "ctx_lens", 1)
    pbt = _dev(block_tables, torch.int32, "block_tables", 2)
    ck = _dev(k_cache, bf, "k_cache", 4)
    cv = _dev(v_cache, bf, "v_cache", 4)
    pw = _dev(workspace, torch.uint8, "workspace", 1)
    n_tok, hq, a = q.shape
    n_reqs = ctx_lens.numel()
    if out.shape != q.shape or cu_q_lens.numel() != n_reqs + 1 or block_tables.shape[0] != n_reqs:
        raise ValueError("shape mismatch")
    nb, hk, bs, a2 = k_cache.shape
    if v_cache.shape != k_cache.shape or a2 != a:
        raise ValueError("cache shape mismatch")
    if k_new.shape != (n_tok, hk, a) or v_new.shape != k_new.shape or slot_mapping.numel() != n_tok:
        raise ValueError("new rows must be [n_tokens, Hkv, A] with one slot per token")
    w = () if window is None else (window,)
    rc = getattr(lib(), name)(pk, pv, ps, pq, pcu, pctx, pbt, block_tables.shape[1], n_reqs, n_tok, int(max_q_len),
                              int(max_kv_len), ck, cv, nb, po, float(scale), hq, hk, a, bs, *w, pw,
                              workspace.numel(), _stream(stream))
    _check(name, rc)


CB_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def cb_paged_attention_noalloc(q, cu_q_lens, ctx_lens, block_tables, k_cache, v_cache, out, scale, max_q_len,
                               max_kv_len, stream=None):
    """cb_paged_attention without a workspace argument: for callers that cannot
    allocate device memory when they run a step.  Its scratch is the library's
    fixed device array (CB_NOALLOC_SCRATCH_BYTES); steps that need more are
    rejected (CBError, CB_EWORKSPACE).  Calls that overlap on the GPU share that
    array and race."""
    torch = _t()
    bf = torch.bfloat16
    pq = _dev(q, bf, "q", 3)
    po = _dev(out, bf, "out", 3)
    pcu = _dev(cu_q_lens, torch.int32, "cu_q_lens", 1)
    pctx = _dev(ctx_lens, torch.int32, "ctx_lens", 1)
    pbt = _dev(block_tables, torch.int32, "block_tables", 2)
    ck = _dev(k_cache, bf, "k_cache", 4)
    cv = _dev(v_cache, bf, "v_cache", 4)
    n_tok, hq, a = q.shape
    n_reqs = ctx_lens.numel()
    if out.shape != q.shape or cu_q_lens.numel() != n_reqs + 1 or block_tables.shape[0] != n_reqs:
        raise ValueError("shape mismatch")
    nb, hk, bs, a2 = k_cache.shape
    if v_cache.shape != k_cache.shape or a2 != a:
        raise ValueError("cache shape mismatch")
    rc = lib().cb_paged_attention_noalloc(pq, pcu, pctx, pbt, block_tables.shape[1], n_reqs, n_tok, int(max_q_len),
                                          int(max_kv_len), ck, cv, nb, po, float(scale), hq, hk, a, bs,
                                          _stream(stream))
    _check("cb_paged_attention_noalloc", rc)


def cb_last_error(stream=None):
    """Synchronise the stream and return (and clear) that stream's error status code."""
    return int(lib().cb_last_error(_stream(stream)))


def cb_strerror(code):
    return lib().cb_strerror(int(code)).decode()


def cb_hbm_copy(dst, src, stream=None):
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() < n or not (src.is_cuda and dst.is_cuda):
        raise ValueError("bad copy buffers")
    _check("cb_hbm_copy", lib().cb_hbm_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), n,
                                            _stream(stream)))


def cb_last_launch_count():
    return int(lib().cb_last_launch_count())


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_i32p)


def cb_build_slot_mapping(q_lens, ctx_lens, block_tables, block_size):
    """Host slot mapping of a step (int64 [sum(q_lens)])."""
    q, pq = _i32(q_lens)
    c, pc = _i32(ctx_lens)
    bt, pbt = _i32(block_tables)
    if bt.ndim != 2 or bt.shape[0] != q.size or c.size != q.size:
        raise ValueError("shape mismatch")
    out = np.empty(int(q.sum()), dtype=np.int64)
    rc = lib().cb_build_slot_mapping(pq, pc, pbt, bt.shape[1], q.size, int(block_size), out.ctypes.data_as(_i64p))
    _check("cb_build_slot_mapping", rc)
    return out


class Graph:
    """cb_graph: record the library calls made on a stream between ``begin`` and
    ``end`` and run them as one CUDA graph (updated in place while the same
    kernels are recorded).  ``stream`` is a raw stream handle or a
    torch.cuda.Stream, never the legacy default stream."""

    def __init__(self):
        self._g = lib().cb_graph_create()
        if not self._g:
            raise CBError("cb_graph_create", CB_ECUDA)

    @staticmethod
    def _handle(stream):
        return stream if isinstance(stream, int) else stream.cuda_stream

    def begin(self, stream):
        _check("cb_graph_begin", lib().cb_graph_begin(self._g, self._handle(stream)))

    def end(self, stream):
        _check("cb_graph_end", lib().cb_graph_end(self._g, self._handle(stream)))

    def close(self):
        if self._g:
            lib().cb_graph_destroy(self._g)
            self._g = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Scheduler:
    """Host FCFS continuous-batching scheduler (cb_sched_* in the library).

    ``step()`` returns a dict with the step's metadata as NumPy arrays
    (req_ids, q_lens, ctx_lens, cu_q_lens, block_tables [B, max_blocks_per_seq],
    slot_mapping) plus ``n_preempted``.
    """

    STATES = ("pending", "waiting", "running", "finished", "rejected")

    def __init__(self, num_blocks, block_size, token_budget, max_batch, free_order, max_blocks_per_seq, window=0,
                 padded_batch=0, max_wait=-1):
        fo, pfo = _i32(free_order)
        self._h = lib().cb_sched_create(num_blocks, block_size, token_budget, max_batch, pfo)
        if not self._h:
            raise CBError("cb_sched_create", CB_EINVAL)
        if window:
            _check("cb_sched_set_window", lib().cb_sched_set_window(self._h, int(window)))
        if padded_batch:
            _check("cb_sched_set_batching", lib().cb_sched_set_batching(self._h, int(padded_batch), int(max_wait)))
        self.max_batch = max_batch
        self.token_budget = token_budget
        self.max_blocks = max_blocks_per_seq
        self._req_ids = np.zeros(max_batch, np.int32)
        self._q = np.zeros(max_batch, np.int32)
        self._c = np.zeros(max_batch, np.int32)
        self._cu = np.zeros(max_batch + 1, np.int32)
        self._bt = np.zeros((max_batch, max_blocks_per_seq), np.int32)
        self._sm = np.zeros(token_budget, np.int64)
        self._pairs = np.zeros((max_batch, 2), np.int32)

    def close(self):
        if self._h:
            lib().cb_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_request(self, arrival_step, prompt_len, output_len, group=-1, prefix_len=0):
        """group >= 0: the first prefix_len prompt tokens are shared by the group."""
        rid = lib().cb_sched_add_request_prefix(self._h, int(arrival_step), int(prompt_len), int(output_len),
                                                int(group), int(prefix_len))
        if rid < 0:
            raise CBError("cb_sched_add_request_prefix", rid)
        return rid

    def step_copies(self):
        """Copy-on-write pairs (src, dst) of the last step, int32 [n, 2]."""
        n = lib().cb_sched_step_copies(self._h, self._pairs.ctypes.data_as(_i32p), self._pairs.shape[0])
        if n < 0:
            raise CBError("cb_sched_step_copies", n)
        return self._pairs[:n].copy()

    def done(self):
        return bool(lib().cb_sched_done(self._h))

    def free_blocks(self):
        return int(lib().cb_sched_free_blocks(self._h))

    def request_info(self, rid):
        vals = [ctypes.c_int() for _ in range(4)]
        _check("cb_sched_request_info", lib().cb_sched_request_info(self._h, rid, *[ctypes.byref(v) for v in vals]))
        produced, stored, preemptions, state = (v.value for v in vals)
        return dict(produced=produced, stored=stored, preemptions=preemptions, state=self.STATES[state])

    def kv_memory(self, max_seq_len):
        """KV memory after the last step: dict(running, stored, paged, contiguous) in
        token slots (cb_sched_kv_memory)."""
        out = np.zeros(4, np.int64)
        _check("cb_sched_kv_memory", lib().cb_sched_kv_memory(self._h, int(max_seq_len), out.ctypes.data_as(_i64p)))
        return dict(running=int(out[0]), stored=int(out[1]), paged=int(out[2]), contiguous=int(out[3]))

    def step(self):
        nr, nt = ctypes.c_int(), ctypes.c_int()
        rc = lib().cb_sched_step(self._h, self._req_ids.ctypes.data_as(_i32p), self._q.ctypes.data_as(_i32p),
                                 self._c.ctypes.data_as(_i32p), self._cu.ctypes.data_as(_i32p),
                                 self._bt.ctypes.data_as(_i32p), self.max_blocks, self._sm.ctypes.data_as(_i64p),
                                 ctypes.byref(nr), ctypes.byref(nt))
        if rc < 0:
            raise CBError("cb_sched_step", rc)
        b, t = nr.value, nt.value
        return dict(req_ids=self._req_ids[:b].copy(), q_lens=self._q[:b].copy(), ctx_lens=self._c[:b].copy(),
                    cu_q_lens=self._cu[:b + 1].copy(), block_tables=self._bt[:b].copy(),
                    slot_mapping=self._sm[:t].copy(), n_preempted=rc,
                    real_tokens=int(lib().cb_sched_last_real_tokens(self._h)))
