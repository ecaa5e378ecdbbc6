#!/usr/bin/env python
"""Benchmark of one continuous-batching attention step over a paged KV cache.

A step = the whole hot path over one batch: the host slot mapping (e2e leg),
the slot-mapped KV append and the paged attention launch (decode split-K,
tensor-core prefill tiles, or both in one launch).  Default workload: 64 decode
requests of a Llama-2-7B attention layer (MHA 32 x 128, contexts uniform in
[512, 4096], block 16, 20 GB pool) -- about 2.4 GB of K/V read per step, far
larger than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead, on bounded samples of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|mixed|mixed_budget|long|tiny]
"""
import os

# the oracle (cpu baseline / reference arm) runs single-threaded, so "cores" is exact
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import workloads as wl  # noqa: E402

METRIC = "mixed-step attention tokens/s; decode KV GB/s as % of measured HBM peak"
UNIT = "tokens/s"
WORKLOADS = {
    "decode": (lambda seed, pool=20: wl.decode(seed=seed, pool_bytes=pool * wl.GB),
               "decode: 64 requests, ctx U[512,4096], MHA 32x128 (Llama-2-7B layer), bf16, block 16, 20 GB pool"),
    "mixed": (lambda seed, pool=20: wl.mixed(seed=seed, pool_bytes=pool * wl.GB),
              "mixed: 48 decodes ctx U[256,8192] + 2x512-token chunks after 1024/3072, GQA 32/8 x128, bf16"),
    "mixed_budget": (lambda seed, pool=20: wl.mixed(seed=seed, budget_variant=True, pool_bytes=pool * wl.GB),
                     "mixed, 560-token budget: 48 decodes + one 512-token chunk after 1024, GQA 32/8 x128"),
    "gqa_decode": (lambda seed, pool=20: wl.gqa_decode(seed=seed, pool_bytes=pool * wl.GB),
                   "gqa_decode: the mixed step's 48 decodes alone, ctx U[256,8192], GQA 32/8 x128, bf16"),
    "long": (lambda seed, pool=20: wl.long(15, seed=seed, pool_bytes=pool * wl.GB),
             "long: 2048-token chunk after 30720 stored (step 15 of a 32768 prompt) + 16 decodes at 8207, GQA 32/8"),
    "tiny": (lambda seed, pool=20: wl.tiny(seed=seed), "tiny: 4 requests (37,1),(100,1),(4,3),(0,20), MHA 4x64"),
}
KERNEL_SOURCES = ["cb_common.cuh", "cb_decode_item.cuh", "cb_decode.cu", "cb_decode_tcb.cuh", "cb_decode_tcb.cu",
                  "cb_mixed.cu", "cb_api.cu"]


# ---------------------------------------------------------------- work accounting
def algorithmic(shape):
    """Algorithmic work of one step: K/V bytes every request must read once
    (valid tokens only), the new-token q/out/append bytes, and the causal-valid
    attention FLOPs (QK^T and PV: 4 * A flops per (query head, key) pair)."""
    a, hq, hk = shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    kv_bytes = dec_kv_bytes = 0
    flops = pre_flops = 0
    for c, n in zip(shape.ctx_lens, shape.q_lens):
        if n == 0:
            continue
        kv_bytes += 2 * (c + n) * hk * a * 2
        pairs = n * c + n * (n + 1) // 2
        flops += 4 * a * hq * pairs
        if n == 1:
            dec_kv_bytes += 2 * (c + 1) * hk * a * 2
        else:
            pre_flops += 4 * a * hq * pairs
    qo_bytes = 2 * shape.n_tokens * hq * a * 2
    append_bytes = 2 * 2 * shape.n_tokens * hk * a * 2        # K and V rows, read + written
    return dict(kv_bytes=kv_bytes, dec_kv_bytes=dec_kv_bytes, attn_bytes=kv_bytes + qo_bytes, flops=flops,
                pre_flops=pre_flops, append_bytes=append_bytes)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def _code_only(text):
    """Source text without comments and with whitespace collapsed: what decides
    the compiled kernels (string literals here hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    """Hash of the kernel sources' code (comments and layout ignored): the traffic
    recorded under profiles/ is reported only for the code it was measured on."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_cb_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary,
    or None when the kernel sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"cb_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- oracle timing
def oracle_on_requests(shape, reqs, fetch):
    """Run the fp64 oracle on whole requests `reqs`; `fetch(r)` returns that
    request's (compact pool k, v, table, q rows, k_new rows, v_new rows) in fp64.
    Returns (seconds, tokens)."""
    from oracle import attention as oa
    from oracle import paged as op
    scale = 1.0 / math.sqrt(shape.head_dim)
    data = [fetch(r) for r in reqs]
    t0 = time.perf_counter()
    toks = 0
    for r, (kp, vp, table, q, kn, vn) in zip(reqs, data):
        c, n = shape.ctx_lens[r], shape.q_lens[r]
        k = np.concatenate([op.gather_request(kp, table, c, shape.block_size), kn])
        v = np.concatenate([op.gather_request(vp, table, c, shape.block_size), vn])
        oa.attention_step(q, [n], [c], [k], [v], scale, shape.n_q_heads, shape.n_kv_heads)
        toks += n
    return time.perf_counter() - t0, toks


def cpu_fetch(shape, seed):
    """Synthetic fp64 inputs of one request generated on the host (for the
    reference arm, which needs no GPU): random blocks in a compact pool,
    scattered by a seeded permutation."""
    def fetch(r):
        rng = np.random.default_rng(seed * 100003 + r)
        c, n = shape.ctx_lens[r], shape.q_lens[r]
        nblk = max(1, -(-c // shape.block_size))
        pool = (nblk, shape.n_kv_heads, shape.block_size, shape.head_dim)
        bf = lambda s: rng.standard_normal(size=s, dtype=np.float32).astype(np.float64)
        kp, vp = bf(pool), bf(pool)
        table = rng.permutation(nblk)
        q = bf((n, shape.n_q_heads, shape.head_dim))
        kn, vn = bf((n, shape.n_kv_heads, shape.head_dim)), bf((n, shape.n_kv_heads, shape.head_dim))
        return kp, vp, table, q, kn, vn
    return fetch


def sample_requests(shape, budget_s, fetch, max_tokens=None):
    """Grow a request sample (decodes first, in order) until ~budget_s of oracle time."""
    order = [r for r in range(shape.n_reqs) if shape.q_lens[r] == 1] + \
            [r for r in range(shape.n_reqs) if shape.q_lens[r] > 1 and shape.q_lens[r] <= 64]
    if not order:
        order = [int(np.argmin([q if q > 0 else 1 << 30 for q in shape.q_lens]))]
    dt, toks = oracle_on_requests(shape, order[:1], fetch)
    per = max(dt, 1e-4)
    n = max(1, min(len(order), int(budget_s / per)))
    if max_tokens:
        n = min(n, max_tokens)
    return order[:n]


def run_reference(args, shape, desc, world, rank):
    if rank != 0:
        return
    fetch = cpu_fetch(shape, shape.seed)
    per_step = max(0.05, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    reqs = sample_requests(shape, per_step, fetch)
    for _ in range(args.warmup):
        oracle_on_requests(shape, reqs[:1], fetch)
    total_t = total_tok = 0.0
    for _ in range(args.steps):
        dt, toks = oracle_on_requests(shape, reqs, fetch)
        total_t += dt
        total_tok += toks
    value = total_tok / total_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "sample": f"{len(reqs)} request(s) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{len(reqs)} of {shape.n_reqs} requests per step, inputs generated on the host"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def run_ours(args, shape, desc, world, rank, local):
    import torch
    from paged_kv_cache_cb_gb300 import _lib as L
    if not os.path.exists(L.LIB_PATH):
        from paged_kv_cache_cb_gb300 import build
        build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    inp = wl.step_inputs_device(shape, dev)
    bt_np = inp["block_tables"]
    kv = [c + n for c, n in zip(shape.ctx_lens, shape.q_lens)]
    max_q, max_kv = max(shape.q_lens), max(kv)
    scale = 1.0 / math.sqrt(shape.head_dim)
    slots_np = L.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, bt_np, shape.block_size)
    cu_np = np.concatenate([[0], np.cumsum(shape.q_lens)]).astype(np.int32)
    ctx_np = np.asarray(shape.ctx_lens, np.int32)
    d_slots = torch.from_numpy(slots_np).to(dev)
    d_cu = torch.from_numpy(cu_np).to(dev)
    d_ctx = torch.from_numpy(ctx_np).to(dev)
    d_bt = torch.from_numpy(bt_np).to(dev)
    wsb = L.cb_paged_attention_workspace_size(shape.n_reqs, shape.n_tokens, max_q, max_kv, shape.n_q_heads,
                                              shape.n_kv_heads, shape.head_dim, shape.block_size)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    out = torch.empty_like(inp["q"])
    kc, vc = inp["k_pool"], inp["v_pool"]
    launches = [0]

    def step(q, k_new, v_new, slots, cu, ctx, bt, o):
        """The step through the public API: append + attention in one call."""
        L.cb_kv_append_paged_attention(k_new, v_new, slots, q, cu, ctx, bt, kc, vc, o, scale, ws, max_q, max_kv,
                                       stream)
        n = L.cb_last_launch_count()
        launches[0] += n
        return n

    args_dev = (inp["q"], inp["k_new"], inp["v_new"], d_slots, d_cu, d_ctx, d_bt, out)
    # one launch: the append runs inside the attention kernel (cooperative
    # launches); else the append kernel runs first and is timed outside the
    # attention's events below
    one_launch = step(*args_dev) == 1
    for _ in range(max(3, args.warmup) - 1):
        step(*args_dev)
    torch.cuda.synchronize()
    status = L.cb_last_error(stream)
    if status != 0:
        raise RuntimeError("warm-up step failed: " + L.cb_strerror(status))

    # HBM copy probe in the same process (context for the measured peak)
    copy_gbs = None
    if rank == 0 and not args.no_copy_probe:
        nb = 4 << 30
        a_ = torch.empty(nb, dtype=torch.uint8, device=dev)
        b_ = torch.empty(nb, dtype=torch.uint8, device=dev)
        for _ in range(3):
            L.cb_hbm_copy(b_, a_, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            L.cb_hbm_copy(b_, a_, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        copy_gbs = 2 * nb * 10 / (e0.elapsed_time(e1) * 1e-3) / 1e9
        del a_, b_
        torch.cuda.empty_cache()

    # ---- device-resident timed region
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    launches[0] = 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if one_launch:
            ev[i][0].record(stream)
            step(*args_dev)
            ev[i][1].record(stream)
        else:
            L.cb_kv_append(inp["k_new"], inp["v_new"], d_slots, kc, vc, stream)
            launches[0] += L.cb_last_launch_count()
            ev[i][0].record(stream)
            L.cb_paged_attention(inp["q"], d_cu, d_ctx, d_bt, kc, vc, out, scale, ws, max_q, max_kv, stream)
            ev[i][1].record(stream)
            launches[0] += L.cb_last_launch_count()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    status = L.cb_last_error(stream)
    if status != 0:
        raise RuntimeError("timed steps failed: " + L.cb_strerror(status))
    elapsed = t_start.elapsed_time(t_end) * 1e-3
    attn_s = sum(a.elapsed_time(b) for a, b in ev) * 1e-3 / args.steps
    elapsed = max_over_ranks(elapsed, world, dev)
    gpu_launches = launches[0]

    # ---- end to end through the C ABI with host buffers
    e2e_steps = max(3, min(args.steps, 200))
    pin = lambda t: t.cpu().pin_memory()
    h_q, h_k, h_v = pin(inp["q"]), pin(inp["k_new"]), pin(inp["v_new"])
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_cu = torch.from_numpy(cu_np).pin_memory()
    h_ctx = torch.from_numpy(ctx_np).pin_memory()
    h_bt = torch.from_numpy(bt_np).pin_memory()
    h_slots = torch.empty(shape.n_tokens, dtype=torch.int64).pin_memory()
    d_q, d_k, d_v = torch.empty_like(inp["q"]), torch.empty_like(inp["k_new"]), torch.empty_like(inp["v_new"])
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_cu, h_ctx, h_bt, h_slots))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        h_slots.numpy()[:] = L.cb_build_slot_mapping(shape.q_lens, shape.ctx_lens, bt_np, shape.block_size)
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_cu.copy_(h_cu, non_blocking=True)
        d_ctx.copy_(h_ctx, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        d_slots.copy_(h_slots, non_blocking=True)
        step(d_q, d_k, d_v, d_slots, d_cu, d_ctx, d_bt, out)
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)

    # ---- cpu baseline: the oracle on a bounded sample of this same step
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cu = cu_np

        def fetch(r):
            c = shape.ctx_lens[r]
            nblk = -(-c // shape.block_size)
            idx = torch.from_numpy(bt_np[r, :nblk].astype(np.int64)).to(dev)
            f = lambda t: t.to("cpu", torch.float64).numpy()
            return (f(kc.index_select(0, idx)), f(vc.index_select(0, idx)), np.arange(nblk),
                    f(inp["q"][cu[r]:cu[r + 1]]), f(inp["k_new"][cu[r]:cu[r + 1]]), f(inp["v_new"][cu[r]:cu[r + 1]]))
        reqs = sample_requests(shape, 12.0, fetch)
        dt, toks = oracle_on_requests(shape, reqs, fetch)
        cpu = {"value": toks / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{len(reqs)} of {shape.n_reqs} requests of the same step ({toks} tokens), fp64 NumPy, "
                         f"{dt:.1f} s"}

    if rank != 0:
        return
    work = algorithmic(shape)
    peaks = load_peaks()
    launch_bytes = work["attn_bytes"] + (work["append_bytes"] if one_launch else 0)
    what = "append + paged attention launch" if one_launch else "paged attention launch"
    t_hbm = launch_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = work["flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved = launch_bytes / attn_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(args.workload),
                "kernel": what + " (split-K decode / mixed)",
                "algorithmic_bytes_per_launch": launch_bytes, "peak_source": peaks["source"] + " hbm_gbs"}
    else:
        achieved = work["flops"] / attn_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": ncu_traffic(args.workload),
                "kernel": what + " (tcgen05 prefill tiles + decode)",
                "algorithmic_flops_per_launch": work["flops"], "peak_source": peaks["source"] + " bf16_tflops"}
    value = shape.n_tokens * args.steps * world / elapsed
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": desc, "n_reqs": shape.n_reqs, "n_tokens": shape.n_tokens,
                   "n_q_heads": shape.n_q_heads, "n_kv_heads": shape.n_kv_heads, "head_dim": shape.head_dim,
                   "block_size": shape.block_size, "num_blocks": shape.num_blocks,
                   "l2": f"inputs larger than L2: {work['kv_bytes'] / 1e9:.2f} GB K/V read per step, no flush",
                   "parallelism": f"replicas x{world} (requests independent, no collective)"},
        "roofline": roof,
        "kv_gbs": work["kv_bytes"] / attn_s / 1e9,
        "kv_frac_of_hbm_peak": work["kv_bytes"] / attn_s / 1e9 / peaks["hbm_gbs"],
        "attention_ms": attn_s * 1e3,
        "append_in_launch": one_launch,
        "prefill_tflops": work["pre_flops"] / attn_s / 1e12 if work["pre_flops"] else None,
        "copy_gbs_same_run": copy_gbs,
        "cpu_baseline": cpu,
        "e2e": {"value": shape.n_tokens * e2e_steps * world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- continuous-batching trace
TRACE_DESC = ("trace: 256 requests, prompts min(8192, lognormal(ln 512, 1)), outputs geometric mean 256, "
              "Poisson 2/step, FCFS budget 2048, 32 layers GQA 32/8 x128 bf16, block 16, 60 GB pool")


def run_trace(args, world, rank, local):
    """Continuous batching end to end: every iteration the host scheduler
    (cb_sched_step) picks the batch and builds its metadata, which is copied
    to the device; then, for each layer, one cb_kv_append_paged_attention
    call appends the new rows and runs the paged attention.  New K/V/Q rows are per-layer seeded random buffers
    (no projections), reused every iteration."""
    import torch
    from paged_kv_cache_cb_gb300 import _lib as L
    if not os.path.exists(L.LIB_PATH):
        from paged_kv_cache_cb_gb300 import build
        build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream            # raw handle: the cheapest form for the per-layer calls
    tr = wl.trace(seed=args.seed + rank, pool_bytes=int(args.trace_pool_gb * wl.GB), n_layers=args.trace_layers)
    if args.trace_prefix_groups > 0:       # shared system prompts: blocks shared, partial last block copied
        tr = wl.with_prefixes(tr, args.trace_prefix_groups, args.trace_prefix_len, seed=args.seed + rank)
    nl, hq, hk, a, bs, budget = tr.n_layers, tr.n_q_heads, tr.n_kv_heads, tr.head_dim, tr.block_size, tr.token_budget
    nb = tr.num_blocks
    bf = torch.bfloat16
    kc = [torch.empty((nb, hk, bs, a), dtype=bf, device=dev) for _ in range(nl)]
    vc = [torch.empty((nb, hk, bs, a), dtype=bf, device=dev) for _ in range(nl)]
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed + 17)
    qn = [torch.randn((budget, hq, a), generator=g, device=dev, dtype=bf) for _ in range(nl)]
    kn = [torch.randn((budget, hk, a), generator=g, device=dev, dtype=bf) for _ in range(nl)]
    vn = [torch.randn((budget, hk, a), generator=g, device=dev, dtype=bf) for _ in range(nl)]
    out = torch.empty((budget, hq, a), dtype=bf, device=dev)
    maxblk = max(-(-(t[1] + t[2] - 1) // bs) for t in tr.requests)
    max_seq = max(t[1] + t[2] - 1 for t in tr.requests)
    def new_scheduler():
        s = L.Scheduler(nb, bs, budget, min(budget, L.CB_MAX_REQS), wl.free_order(nb, tr.seed), maxblk)
        for t in tr.requests:
            s.add_request(*(t[:3] if args.trace_no_share else t))
        return s

    sched = new_scheduler()
    ws = torch.empty(L.cb_paged_attention_workspace_size(min(budget, L.CB_MAX_REQS), budget, budget, max_seq, hq, hk,
                                                         a, bs), dtype=torch.uint8, device=dev)
    d_cu = torch.zeros(budget + 1, dtype=torch.int32, device=dev)
    d_ctx = torch.zeros(budget, dtype=torch.int32, device=dev)
    d_bt = torch.zeros((budget, maxblk), dtype=torch.int32, device=dev)
    d_sl = torch.zeros(budget, dtype=torch.int64, device=dev)
    # double-buffered pinned staging of the metadata
    h = [dict(cu=torch.zeros(budget + 1, dtype=torch.int32).pin_memory(),
              ctx=torch.zeros(budget, dtype=torch.int32).pin_memory(),
              bt=torch.zeros((budget, maxblk), dtype=torch.int32).pin_memory(),
              sl=torch.zeros(budget, dtype=torch.int64).pin_memory(),
              ev=torch.cuda.Event()) for _ in range(2)]
    scale = 1.0 / math.sqrt(a)
    stats = dict(tokens=0, dec=0, pre=0, steps=0, idle=0, launches=0, kv_bytes=0, flops=0, preempted=0, h2d=0, d2h=0,
                 kv_stored=0, kv_paged=0, kv_contig=0)

    d_pairs = torch.zeros((budget, 2), dtype=torch.int32, device=dev)
    for hb in h:
        hb["pairs"] = torch.zeros((budget, 2), dtype=torch.int32).pin_memory()
    # The per-layer step goes straight to the C ABI with pointers taken once, as
    # a native serving loop would call it: every buffer below keeps its address,
    # and a step uses the first t rows / b requests of each.
    step_fn = L.lib().cb_kv_append_paged_attention
    layer_ptrs = [(kn[i].data_ptr(), vn[i].data_ptr(), qn[i].data_ptr(), kc[i].data_ptr(), vc[i].data_ptr())
                  for i in range(nl)]
    fixed = dict(sl=d_sl.data_ptr(), cu=d_cu.data_ptr(), ctx=d_ctx.data_ptr(), bt=d_bt.data_ptr(),
                 out=out.data_ptr(), ws=ws.data_ptr(), wsb=ws.numel())

    def one_step(i, host_io=None):
        m = sched.step()
        pairs = sched.step_copies()             # copy-on-write of shared partial blocks, before the append
        mem = sched.kv_memory(max_seq)          # held after this step: paged blocks vs a max-length reservation
        stats["kv_stored"] += mem["stored"]
        stats["kv_paged"] += mem["paged"]
        stats["kv_contig"] += mem["contiguous"]
        b, t = len(m["req_ids"]), int(m["cu_q_lens"][-1]) if len(m["req_ids"]) else 0
        stats["preempted"] += m["n_preempted"]
        if t == 0:
            stats["idle"] += 1
            return
        hb = h[i & 1]
        hb["ev"].synchronize()                    # this staging buffer's previous copy has finished
        hb["cu"].numpy()[:b + 1] = m["cu_q_lens"]
        hb["ctx"].numpy()[:b] = m["ctx_lens"]
        hb["bt"].numpy()[:b] = m["block_tables"]
        hb["sl"].numpy()[:t] = m["slot_mapping"]
        npairs = len(pairs)
        if npairs:
            hb["pairs"].numpy()[:npairs] = pairs
            d_pairs[:npairs].copy_(hb["pairs"][:npairs], non_blocking=True)
        d_cu[:b + 1].copy_(hb["cu"][:b + 1], non_blocking=True)
        d_ctx[:b].copy_(hb["ctx"][:b], non_blocking=True)
        d_bt[:b].copy_(hb["bt"][:b], non_blocking=True)
        d_sl[:t].copy_(hb["sl"][:t], non_blocking=True)
        hb["ev"].record(stream)
        q_lens, ctx = m["q_lens"], m["ctx_lens"]
        max_q, max_kv = int(q_lens.max()), int((q_lens + ctx).max())
        for layer in range(nl):
            if host_io is not None:                 # end-to-end: this step's rows come from pinned host memory
                qn[layer][:t].copy_(host_io["q"][layer][:t], non_blocking=True)
                kn[layer][:t].copy_(host_io["k"][layer][:t], non_blocking=True)
                vn[layer][:t].copy_(host_io["v"][layer][:t], non_blocking=True)
            if npairs:
                L.cb_copy_blocks(d_pairs[:npairs], kc[layer], vc[layer], sh)
                stats["launches"] += 1
            pk, pv, pq, pkc, pvc = layer_ptrs[layer]
            rc = step_fn(pk, pv, fixed["sl"], pq, fixed["cu"], fixed["ctx"], fixed["bt"], maxblk, b, t, max_q, max_kv,
                         pkc, pvc, nb, fixed["out"], scale, hq, hk, a, bs, fixed["ws"], fixed["wsb"], sh)
            if rc != 0:
                raise RuntimeError("cb_kv_append_paged_attention: " + L.cb_strerror(rc))
            stats["launches"] += L.cb_last_launch_count()
            if host_io is not None:
                host_io["out"][:t].copy_(out[:t], non_blocking=True)
        if host_io is not None:
            stats["h2d"] += nl * t * (hq + 2 * hk) * a * 2 + 4 * (2 * b + 1) + 4 * b * maxblk + 8 * t
            stats["d2h"] += nl * t * hq * a * 2
        stats["tokens"] += t
        stats["steps"] += 1
        dec = int((q_lens == 1).sum())
        stats["dec"] += dec
        stats["pre"] += t - dec
        kvl = (q_lens + ctx).astype(np.int64)
        stats["kv_bytes"] += int(2 * kvl.sum() * hk * a * 2) * nl
        pairs = (q_lens.astype(np.int64) * ctx + q_lens.astype(np.int64) * (q_lens + 1) // 2).sum()
        stats["flops"] += int(4 * a * hq * pairs) * nl
        if host_io is not None:
            stream.synchronize()

    for i in range(args.warmup):
        one_step(i)
    torch.cuda.synchronize()
    if L.cb_last_error(stream) != 0:
        raise RuntimeError("trace warm-up failed")
    for k in list(stats):
        stats[k] = 0
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    def finished_tokens():
        """Requests finished so far and their prompt + output tokens."""
        n = tok = 0
        for rid, t in enumerate(tr.requests):
            if sched.request_info(rid)["state"] == "finished":
                n += 1
                tok += t[1] + t[2]
        return n, tok

    fin0 = finished_tokens()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    i = 0
    while i < args.steps and not sched.done():
        one_step(args.warmup + i)
        i += 1
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    fin1 = finished_tokens()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    status = L.cb_last_error(stream)
    if status != 0:
        raise RuntimeError("trace failed: " + L.cb_strerror(status))
    dev_s = e0.elapsed_time(e1) * 1e-3
    timed = dict(stats)
    elapsed = max_over_ranks(wall, world, dev)
    # end to end: the same iterations again (a fresh scheduler from the trace's
    # start), each layer's new rows copied from pinned host memory and each
    # layer's output returned to the host, the host waiting for every iteration
    host_io = dict(q=[t.cpu().pin_memory() for t in qn], k=[t.cpu().pin_memory() for t in kn],
                   v=[t.cpu().pin_memory() for t in vn], out=torch.empty_like(out, device="cpu").pin_memory())
    sched = new_scheduler()
    for k in list(stats):
        stats[k] = 0
    for j in range(args.warmup):
        one_step(j, host_io)
    for k in list(stats):
        stats[k] = 0
    barrier(world)
    te = time.perf_counter()
    j = 0
    while j < timed["steps"] + timed["idle"] and not sched.done():
        one_step(args.warmup + j, host_io)
        j += 1
    te = max_over_ranks(time.perf_counter() - te, world, dev)
    n_io = max(1, stats["steps"])
    e2e = {"value": stats["tokens"] * world / te if te > 0 else None, "unit": UNIT,
           "h2d_bytes_per_step": int(stats["h2d"] / n_io), "d2h_bytes_per_step": int(stats["d2h"] / n_io),
           "steps": stats["steps"]}
    if rank != 0:
        return
    peaks = load_peaks()
    t_hbm = timed["kv_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = timed["flops"] / (peaks["bf16_tflops_sustained"] * 1e12)
    if t_hbm >= t_tc:
        ach = timed["kv_bytes"] / dev_s / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "traffic": None, "kernel": "whole iteration (32 x append + attention launches), device time",
                "peak_source": peaks["source"] + " hbm_gbs"}
    else:
        ach = timed["flops"] / dev_s / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops_sustained"], "traffic": None,
                "kernel": "whole iteration (32 x append + attention launches), device time",
                "peak_source": peaks["source"] + " bf16_tflops_sustained"}
    line = {
        "metric": METRIC, "value": timed["tokens"] * world / elapsed, "unit": UNIT, "n_gpus": world,
        "steps": timed["steps"], "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / max(1, timed["steps"]),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": TRACE_DESC + (
                       f"; {args.trace_prefix_groups} groups sharing a {args.trace_prefix_len}-token system prompt"
                       + (", computed in full (no sharing)" if args.trace_no_share else
                          ", blocks shared, partial last block copied on write")
                       if args.trace_prefix_groups > 0 else ""),
                   "n_layers": nl, "num_blocks": nb, "token_budget": budget,
                   "decode_tokens": timed["dec"], "prefill_tokens": timed["pre"], "idle_steps": timed["idle"],
                   "preemptions": timed["preempted"],
                   "l2": "inputs larger than L2: each iteration reads every running request's K/V in 32 layers",
                   "parallelism": f"replicas x{world} (independent traces, no collective)"},
        "roofline": roof, "device_s": dev_s, "wall_s": wall,
        "finished_in_timed_region": {"requests": fin1[0] - fin0[0], "prompt_plus_output_tokens": fin1[1] - fin0[1],
                                     "requests_per_s": (fin1[0] - fin0[0]) / elapsed},
        "kv_memory": {"paged_waste": 1 - timed["kv_stored"] / max(1, timed["kv_paged"]),
                      "contiguous_waste": 1 - timed["kv_stored"] / max(1, timed["kv_contig"]),
                      "contiguous_max_seq_len": max_seq,
                      "definition": "slots held but not stored, summed over steps: paged blocks taken only when "
                                    "full vs a cache reserving max_seq_len slots per running request"},
        "cpu_baseline": None, "e2e": e2e, "gpu_launches": timed["launches"], "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS) + ["trace"])
    ap.add_argument("--trace-pool-gb", type=float, default=60.0, help="trace: K+V pool of all layers")
    ap.add_argument("--trace-layers", type=int, default=32, help="trace: attention layers per iteration")
    ap.add_argument("--trace-prefix-groups", type=int, default=0,
                    help="trace: requests join this many groups sharing a system prompt (0: none)")
    ap.add_argument("--trace-prefix-len", type=int, default=1000, help="trace: shared system prompt tokens")
    ap.add_argument("--trace-no-share", action="store_true",
                    help="trace with prefix groups: compute every prompt in full (no block sharing)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-copy-probe", action="store_true", help="skip the in-process HBM copy probe")
    ap.add_argument("--pool-gb", type=float, default=20.0,
                    help="K+V block pool size (blocks stay randomly scattered over it)")
    args = ap.parse_args(argv)
    world, rank, local = dist_env()
    if args.workload == "trace":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "trace workload: the reference arm times single steps"}))
            return
        run_trace(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    make, desc = WORKLOADS[args.workload]
    if args.pool_gb != 20.0:
        desc = desc.replace("20 GB pool", f"{args.pool_gb:g} GB pool") + f" (pool {args.pool_gb:g} GB)"
    if args.impl == "reference":
        run_reference(args, make(args.seed, args.pool_gb), desc, world, rank)
        return
    # weak scaling: each rank runs its own batch of the same workload (its own seed)
    run_ours(args, make(args.seed + rank, args.pool_gb), desc, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
