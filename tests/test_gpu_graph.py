"""CUDA-graph recording of the library's calls (cb_graph_begin / cb_graph_end).

A recorded step gives the same bits as the direct call (output and both
caches); a new recording of the same kernels updates the graph in place, one
of other kernels instantiates it anew; a kernel error inside a graph reaches
cb_last_error(stream) as it does for a direct call."""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import L, cu_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L().lib()


def _prep(shape, dev="cuda"):
    lib = L()
    inp = wl.step_inputs_cpu(shape)
    slots = lib.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, inp["block_tables"], shape.block_size)
    kv = [c + n for c, n in zip(shape.ctx_lens, shape.q_lens)]
    max_q, max_kv = max(shape.q_lens), max(kv)
    wsb = lib.cb_paged_attention_workspace_size(shape.n_reqs, shape.n_tokens, max_q, max_kv, shape.n_q_heads,
                                                shape.n_kv_heads, shape.head_dim, shape.block_size)
    d = dict(k_new=inp["k_new"].to(dev), v_new=inp["v_new"].to(dev), q=inp["q"].to(dev),
             slots=torch.from_numpy(np.asarray(slots, np.int64)).to(dev),
             cu=torch.from_numpy(cu_of(shape.q_lens)).to(dev),
             ctx=torch.tensor(shape.ctx_lens, dtype=torch.int32, device=dev),
             bt=torch.from_numpy(inp["block_tables"]).to(dev), k0=inp["k_pool"].to(dev), v0=inp["v_pool"].to(dev),
             ws=torch.empty(wsb, dtype=torch.uint8, device=dev), max_q=max_q, max_kv=max_kv,
             scale=1.0 / math.sqrt(shape.head_dim))
    torch.cuda.synchronize()                           # the copies above ran on the default stream
    return d


def _fresh(d):
    return d["k0"].clone(), d["v0"].clone(), torch.full_like(d["q"], float("nan"))


def _step(d, kc, vc, out):
    L().cb_kv_append_paged_attention(d["k_new"], d["v_new"], d["slots"], d["q"], d["cu"], d["ctx"], d["bt"], kc, vc,
                                     out, d["scale"], d["ws"], d["max_q"], d["max_kv"])


def _bits(t):
    return t.view(torch.int16)


# block-tile decode; the same kernel on other lengths (update in place); the
# mixed kernel (new instantiation); MHA on the CUDA-core path (memsets in the
# graph); back to the first
SHAPES = [
    wl.StepShape("g_dec_a", 32, 8, 128, 16, 700, q_lens=(1,) * 6, ctx_lens=(100, 2000, 17, 900, 4000, 33), seed=1),
    wl.StepShape("g_dec_b", 32, 8, 128, 16, 700, q_lens=(1,) * 9, ctx_lens=(5, 3000, 64, 1, 700, 128, 2500, 16, 999),
                 seed=2),
    wl.StepShape("g_mixed", 32, 8, 128, 16, 700, q_lens=(1, 300, 1, 64), ctx_lens=(1500, 100, 40, 0), seed=3),
    wl.StepShape("g_mha", 8, 8, 64, 16, 400, q_lens=(1, 1, 20), ctx_lens=(300, 900, 50), seed=4),
    wl.StepShape("g_dec_a2", 32, 8, 128, 16, 700, q_lens=(1,) * 6, ctx_lens=(100, 2000, 17, 900, 4000, 33), seed=5),
]


def test_recorded_steps_give_the_direct_calls_bits():
    lib = L()
    s = torch.cuda.Stream()
    g = lib.Graph()
    try:
        for shape in SHAPES:
            d = _prep(shape)
            with torch.cuda.stream(s):
                kc, vc, out = _fresh(d)
                _step(d, kc, vc, out)                  # direct (also the shape's first call on the device)
                kc2, vc2, out2 = _fresh(d)
            s.synchronize()
            assert lib.cb_last_error(s) == 0
            g.begin(s)
            with torch.cuda.stream(s):
                _step(d, kc2, vc2, out2)               # recorded, not run
            g.end(s)                                   # updated or instantiated, then launched
            s.synchronize()
            assert lib.cb_last_error(s) == 0, shape.name
            assert not torch.isnan(out2).any(), shape.name
            assert torch.equal(_bits(out2), _bits(out)), shape.name
            assert torch.equal(_bits(kc2), _bits(kc)) and torch.equal(_bits(vc2), _bits(vc)), shape.name
    finally:
        g.close()


def test_repeated_recordings_on_one_graph():
    """Several begin/end pairs on one graph object, the same step each time,
    all launched before one synchronisation: every run is a complete step (the
    launch counters are left at zero between runs)."""
    lib = L()
    s = torch.cuda.Stream()
    g = lib.Graph()
    d = _prep(SHAPES[0])
    try:
        with torch.cuda.stream(s):
            kc, vc, ref = _fresh(d)
            _step(d, kc, vc, ref)
        s.synchronize()
        outs = []
        for _ in range(4):                             # each recording updates the graph while the last runs
            with torch.cuda.stream(s):
                kc2, vc2, out = _fresh(d)
            g.begin(s)
            with torch.cuda.stream(s):
                _step(d, kc2, vc2, out)
            g.end(s)
            outs.append(out)
        s.synchronize()
        assert lib.cb_last_error(s) == 0
        for out in outs:
            assert torch.equal(_bits(out), _bits(ref))
    finally:
        g.close()


def test_kernel_error_inside_a_graph_reaches_last_error():
    lib = L()
    shape = wl.StepShape("g_bad", 32, 8, 128, 16, 200, q_lens=(1, 1, 1), ctx_lens=(300, 40, 250), seed=6)
    d = _prep(shape)
    s = torch.cuda.Stream()
    g = lib.Graph()
    try:
        with torch.cuda.stream(s):
            kc, vc, out = _fresh(d)
            _step(d, kc, vc, out)
        s.synchronize()
        assert lib.cb_last_error(s) == 0
        bad = d["bt"].clone()
        bad[1, 1] = 10_000                             # past the cache: reported, never read
        d["bt"] = bad
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            kc, vc, out = _fresh(d)
        s.synchronize()
        g.begin(s)
        with torch.cuda.stream(s):
            _step(d, kc, vc, out)
        g.end(s)
        assert lib.cb_last_error(s) == lib.CB_EDEVICE
        assert lib.cb_last_error(s) == 0                # read and cleared
    finally:
        g.close()
