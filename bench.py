#!/usr/bin/env python
"""Benchmark of the continuous-batching attention step over a paged KV cache.

A step = the whole hot path over one batch: the host slot mapping (e2e leg),
the slot-mapped KV append and the paged attention (decode split-K, tensor-core
prefill tiles, or both in one launch), through the library's one-call
append + attention.  Default workload: the mixed continuous-batching step --
48 decodes (contexts uniform in [256, 8192]) and two 512-token prefill chunks
after 1024 and 3072 stored tokens, GQA 32/8 x 128, block 16, 20 GB pool --
reported as tokens/s; the same run also measures the 64-request Llama-2-7B
decode step (MHA 32 x 128) and reports its K/V read rate as a fraction of the
HBM peak (``decode``).  Both read far more K/V than L2 holds, so no flush is
needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead, on bounded samples of the same workload, on all host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--workload mixed|decode|mixed_budget|gqa_decode|mqa_decode|gqa16_decode|long|long_seq|tiny|trace]
"""
import os

# every oracle process runs single-threaded BLAS; parallelism is by processes
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
    "mixed": (lambda seed, pool: wl.mixed(seed=seed, pool_bytes=pool),
              "mixed: 48 decodes ctx U[256,8192] + 2x512-token chunks after 1024/3072, GQA 32/8 x128, bf16, "
              "block 16, 20 GB pool"),
    "decode": (lambda seed, pool: wl.decode(seed=seed, pool_bytes=pool),
               "decode: 64 requests, ctx U[512,4096], MHA 32x128 (Llama-2-7B layer), bf16, block 16, 20 GB pool"),
    "mixed_budget": (lambda seed, pool: wl.mixed(seed=seed, budget_variant=True, pool_bytes=pool),
                     "mixed, 560-token budget: 48 decodes + one 512-token chunk after 1024, GQA 32/8 x128"),
    "gqa_decode": (lambda seed, pool: wl.gqa_decode(seed=seed, pool_bytes=pool),
                   "gqa_decode: the mixed step's 48 decodes alone, ctx U[256,8192], GQA 32/8 x128, bf16"),
    "long": (lambda seed, pool: wl.long(15, seed=seed, pool_bytes=pool),
             "long: 2048-token chunk after 30720 stored (step 15 of a 32768 prompt) + 16 decodes at 8207, GQA 32/8"),
    "long_seq": (lambda seed, pool: wl.long_sequence(seed=seed, pool_bytes=pool),
                 "long_seq: a 32768-token prompt in 16 chained 2048-token chunks, each appended and attended over "
                 "the growing paged cache, each co-scheduled with 16 decodes at 8192 + k, GQA 32/8 x128, bf16"),
    "mqa_decode": (lambda seed, pool: wl.mqa_decode(seed=seed, pool_bytes=pool),
                   "mqa_decode: 256 requests, ctx U[1024,16384], MQA 32 q heads on 1 KV head x128, bf16, block 16, "
                   "20 GB pool"),
    "gqa16_decode": (lambda seed, pool: wl.mqa_decode(seed=seed, n_kv_heads=2, pool_bytes=pool),
                     "gqa16_decode: 256 requests, ctx U[1024,16384], GQA 32 q heads on 2 KV heads x128, bf16, "
                     "block 16, 20 GB pool"),
    "tiny": (lambda seed, pool: wl.tiny(seed=seed), "tiny: 4 requests (37,1),(100,1),(4,3),(0,20), MHA 4x64"),
}
KERNEL_SOURCES = ["cb_common.cuh", "cb_decode_item.cuh", "cb_decode.cu", "cb_decode_tcb.cuh", "cb_decode_tcb.cu",
                  "cb_mixed.cu", "cb_api.cu"]


def make_job(workload, seed, pool_gb):
    """A workload as a job: its steps (one, or a sequence sharing one pool and
    one set of block tables) and its description."""
    make, desc = WORKLOADS[workload]
    if pool_gb != 20.0:
        desc = desc.replace("20 GB pool", f"{pool_gb:g} GB pool") + f" (pool {pool_gb:g} GB)"
    x = make(seed, int(pool_gb * wl.GB))
    if isinstance(x, wl.SequenceShape):
        return {"steps": list(x.steps), "seq": x, "desc": desc}
    return {"steps": [x], "seq": None, "desc": desc}


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
# The oracle (fp64 NumPy, as it stands) timed on the host's cores: worker
# processes started with "spawn" (safe after CUDA is initialised in this one),
# each with single-threaded BLAS, each running its share of a bounded sample of
# the workload's query rows.  Rows are sampled uniformly within every step:
# the same fraction of its decode requests and of each prefill request's rows,
# so the sample's mix of short and long rows is the step's.
def sample_tasks(steps, frac, seed):
    """[(step index, request, rows)]: a fraction `frac` of each step's decode
    requests (at least one) and of each prefill request's rows (at least one)."""
    rng = np.random.default_rng(seed)
    tasks = []
    for k, sh in enumerate(steps):
        dec = [r for r in range(sh.n_reqs) if sh.q_lens[r] == 1]
        if dec:
            nd = min(len(dec), max(1, int(round(frac * len(dec)))))
            tasks += [(k, int(r), [0]) for r in sorted(rng.choice(dec, nd, replace=False))]
        for r in range(sh.n_reqs):
            n = sh.q_lens[r]
            if n > 1:
                m = min(n, max(1, int(round(frac * n))))
                tasks.append((k, r, sorted(int(i) for i in rng.choice(n, m, replace=False))))
    return tasks


def task_cost(steps, t):
    """Keys the oracle reads for a task (its cost, up to a constant)."""
    sh = steps[t[0]]
    c = sh.ctx_lens[t[1]]
    return sum(c + i + 1 for i in t[2]) * sh.n_q_heads * sh.head_dim


def _host_inputs(sh, r, rows):
    """Inputs of request r's sampled rows generated on the host (fp64): a
    compact pool of its stored blocks in a seeded order, the table that reads
    it, its new K/V rows up to the last sampled row and those rows' queries."""
    rng = np.random.default_rng(sh.seed * 100003 + r)
    c, hk, hq, a, bs = sh.ctx_lens[r], sh.n_kv_heads, sh.n_q_heads, sh.head_dim, sh.block_size
    nblk = max(1, -(-c // bs))
    f = lambda shape: rng.standard_normal(size=shape, dtype=np.float32).astype(np.float64)
    kp, vp = f((nblk, hk, bs, a)), f((nblk, hk, bs, a))
    table = rng.permutation(nblk)
    n = max(rows) + 1
    return kp, vp, table, f((n, hk, a)), f((n, hk, a)), f((len(rows), hq, a))


def oracle_rows(sh, r, rows, data):
    """The oracle on request r's sampled rows: its stored keys gathered through
    its block table ([SM] PagedAttention), its new keys after them, then the
    masked softmax attention of each row ([CB] Attention)."""
    from oracle import attention as oa
    from oracle import paged as op
    kp, vp, table, kn, vn, q = data
    c = sh.ctx_lens[r]
    k = np.concatenate([op.gather_request(kp, table, c, sh.block_size), kn])
    v = np.concatenate([op.gather_request(vp, table, c, sh.block_size), vn])
    return oa.attention_rows(q, k, v, [c + i for i in rows], 1.0 / math.sqrt(sh.head_dim), sh.n_q_heads,
                             sh.n_kv_heads)


def _oracle_worker(steps, rounds, barrier, queue, wid):
    """One worker: for each round, build its tasks' inputs, meet the other
    workers at the barrier, then time the oracle on them."""
    res = []
    for tasks in rounds:
        data = [_host_inputs(steps[k], r, rows) for k, r, rows in tasks]
        barrier.wait(timeout=900)
        t0 = time.perf_counter()
        n = 0
        for (k, r, rows), d in zip(tasks, data):
            oracle_rows(steps[k], r, rows, d)
            n += len(rows)
        res.append((time.perf_counter() - t0, n))
    queue.put((wid, res))


def time_oracle(steps, rounds_tasks, n_procs):
    """Runs every round's tasks split over n_procs spawned workers (balanced by
    cost); returns per round (wall seconds = slowest worker, rows)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    shares = [[[] for _ in rounds_tasks] for _ in range(n_procs)]
    for ri, tasks in enumerate(rounds_tasks):
        load = [0] * n_procs
        for t in sorted(tasks, key=lambda t: -task_cost(steps, t)):
            w = int(np.argmin(load))
            shares[w][ri].append(t)
            load[w] += task_cost(steps, t)
    barrier = ctx.Barrier(n_procs)
    queue = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(steps, shares[w], barrier, queue, w)) for w in range(n_procs)]
    for p in procs:
        p.start()
    got = dict(queue.get(timeout=3600) for _ in procs)
    for p in procs:
        p.join()
    return [(max(got[w][ri][0] for w in range(n_procs)), sum(got[w][ri][1] for w in range(n_procs)))
            for ri in range(len(rounds_tasks))]


def oracle_frac(steps, seconds, seed):
    """Fraction of the job's rows that the oracle, on one core, runs in about
    `seconds` (from a short pilot timed here)."""
    pilot = sample_tasks(steps, 1e-9, seed)[:3]
    data = [_host_inputs(steps[k], r, rows) for k, r, rows in pilot]
    t0 = time.perf_counter()
    for (k, r, rows), d in zip(pilot, data):
        oracle_rows(steps[k], r, rows, d)
    per_unit = (time.perf_counter() - t0) / max(1, sum(task_cost(steps, t) for t in pilot))
    full = sum(task_cost(steps, t) for t in sample_tasks(steps, 1.0, seed))
    return min(1.0, max(1e-6, seconds / (per_unit * full)))


def cpu_baseline(steps, seed, tokens_per_row=1.0, par_seconds=3.0, single_seconds=8.0):
    """The oracle's rate on all host cores and on one, on bounded samples of the
    job (tokens per second: sampled rows / time, divided by tokens_per_row, the
    layers a token passes through in the workload)."""
    n_procs = os.cpu_count() or 1
    frac = oracle_frac(steps, par_seconds * n_procs, seed)       # par_seconds of work for each process
    par = sample_tasks(steps, frac, seed + 1)
    single = sample_tasks(steps, oracle_frac(steps, single_seconds, seed), seed + 2)
    (dt_p, rows_p), = time_oracle(steps, [par], n_procs)
    (dt_1, rows_1), = time_oracle(steps, [single], 1)
    return {"value": rows_p / dt_p / tokens_per_row, "unit": UNIT, "cores": n_procs, "kind": "oracle",
            "single_thread": {"value": rows_1 / dt_1 / tokens_per_row, "cores": 1,
                              "sample": f"{rows_1} rows in {dt_1:.1f} s"},
            "sample": f"{rows_p} query rows ({frac:.4f} of the job's rows, sampled uniformly per request), "
                      f"inputs generated on the host, fp64 NumPy, {n_procs} processes x 1 BLAS thread, "
                      f"{dt_p:.1f} s wall"
                      + (f"; rate per token = per row / {tokens_per_row:g} layers" if tokens_per_row != 1 else "")}


def run_reference(args, job, desc, world, rank, tokens_per_row=1.0):
    """The reference arm: the oracle as it stands on the host's cores, each step
    a bounded sample of the job's rows."""
    if rank != 0:
        return
    steps = job["steps"]
    n_procs = os.cpu_count() or 1
    per_step = max(0.05, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    frac = oracle_frac(steps, per_step * n_procs, args.seed)
    rounds = [sample_tasks(steps, frac, args.seed + 10 + i) for i in range(args.warmup + args.steps)]
    res = time_oracle(steps, rounds, n_procs)[args.warmup:]
    total_t = sum(dt for dt, _ in res)
    rows = sum(n for _, n in res)
    value = rows / total_t / tokens_per_row
    sample = (f"{rows // max(1, args.steps)} query rows per step ({frac:.4f} of the job's rows, sampled uniformly "
              f"per request), inputs generated on the host, fp64 NumPy, {n_procs} processes x 1 BLAS thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_procs, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def _tables(job, k):
    """Block tables of step k of the job."""
    if job["seq"] is not None:
        return np.ascontiguousarray(job["seq"].tables[list(job["seq"].rows[k])])
    return wl.block_tables(job["steps"][k])


def measure(args, job, dev, stream, world, e2e=True, probe_copy=False):
    """Times the job's steps through the public API (append + attention, one call
    per step of the job; K timed iterations of the whole job after W warm-up
    iterations) with inputs resident in HBM, then end to end with host buffers.
    Returns a dict of timings and counts."""
    import torch
    from paged_kv_cache_cb_gb300 import _lib as L
    steps = job["steps"]
    first = steps[0]
    g = torch.Generator(device=dev)
    g.manual_seed(first.seed)
    pool = (first.num_blocks, first.n_kv_heads, first.block_size, first.head_dim)
    kc = torch.randn(pool, generator=g, device=dev, dtype=torch.bfloat16)
    vc = torch.randn(pool, generator=g, device=dev, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(first.head_dim)
    per = []
    for k, sh in enumerate(steps):
        gk = torch.Generator(device=dev)
        gk.manual_seed(sh.seed * 7 + 1 + k)
        rnd = lambda s: torch.randn(s, generator=gk, device=dev, dtype=torch.bfloat16)
        bt = _tables(job, k)
        kv = [c + n for c, n in zip(sh.ctx_lens, sh.q_lens)]
        slots = L.cb_build_slot_mapping(sh.q_lens, sh.ctx_lens, bt, sh.block_size)
        cu = np.concatenate([[0], np.cumsum(sh.q_lens)]).astype(np.int32)
        ctx = np.asarray(sh.ctx_lens, np.int32)
        d = dict(q=rnd((sh.n_tokens, sh.n_q_heads, sh.head_dim)), k_new=rnd((sh.n_tokens, sh.n_kv_heads, sh.head_dim)),
                 v_new=rnd((sh.n_tokens, sh.n_kv_heads, sh.head_dim)), slots=torch.from_numpy(slots).to(dev),
                 cu=torch.from_numpy(cu).to(dev), ctx=torch.from_numpy(ctx).to(dev), bt=torch.from_numpy(bt).to(dev),
                 max_q=max(sh.q_lens), max_kv=max(kv), bt_np=bt, cu_np=cu, ctx_np=ctx, shape=sh)
        d["out"] = torch.empty_like(d["q"])
        d["ws"] = torch.empty(L.cb_paged_attention_workspace_size(sh.n_reqs, sh.n_tokens, d["max_q"], d["max_kv"],
                                                                  sh.n_q_heads, sh.n_kv_heads, sh.head_dim,
                                                                  sh.block_size), dtype=torch.uint8, device=dev)
        per.append(d)
    launches = [0]

    def call(d, q, k_new, v_new, slots, cu, ctx, bt):
        L.cb_kv_append_paged_attention(k_new, v_new, slots, q, cu, ctx, bt, kc, vc, d["out"], scale, d["ws"],
                                       d["max_q"], d["max_kv"], stream)
        n = L.cb_last_launch_count()
        launches[0] += n
        return n

    dev_args = lambda d: (d["q"], d["k_new"], d["v_new"], d["slots"], d["cu"], d["ctx"], d["bt"])
    one_launch = all(call(d, *dev_args(d)) == 1 for d in per)
    for _ in range(max(3, args.warmup) - 1):
        for d in per:
            call(d, *dev_args(d))
    torch.cuda.synchronize()
    status = L.cb_last_error(stream)
    if status != 0:
        raise RuntimeError("warm-up step failed: " + L.cb_strerror(status))

    copy_gbs = None
    if probe_copy:                      # HBM copy probe in the same process (context for the measured peak)
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

    # ---- device-resident timed region: K iterations of the whole job
    launches[0] = 0
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in per]
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        for j, d in enumerate(per):
            if one_launch:
                ev[i][j][0].record(stream)
                call(d, *dev_args(d))
                ev[i][j][1].record(stream)
            else:                       # the append kernel runs outside the attention launch's events
                L.cb_kv_append(d["k_new"], d["v_new"], d["slots"], kc, vc, stream)
                launches[0] += L.cb_last_launch_count()
                ev[i][j][0].record(stream)
                L.cb_paged_attention(d["q"], d["cu"], d["ctx"], d["bt"], kc, vc, d["out"], scale, d["ws"],
                                     d["max_q"], d["max_kv"], stream)
                ev[i][j][1].record(stream)
                launches[0] += L.cb_last_launch_count()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    status = L.cb_last_error(stream)
    if status != 0:
        raise RuntimeError("timed steps failed: " + L.cb_strerror(status))
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) * 1e-3, world, dev)
    launch_s = [sum(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(args.steps)) * 1e-3 / args.steps
                for j in range(len(per))]
    res = dict(elapsed=elapsed, launch_s=launch_s, attn_s=sum(launch_s), one_launch=one_launch,
               gpu_launches=launches[0], copy_gbs=copy_gbs)
    if e2e:
        res["e2e"] = _measure_e2e(args, per, call, stream, world, dev)
    del kc, vc, per
    torch.cuda.empty_cache()
    return res


def _measure_e2e(args, per, call, stream, world, dev):
    """The job end to end through the C ABI: every step's inputs copied from
    pinned host memory and its output read back, the host waiting for each."""
    import torch
    from paged_kv_cache_cb_gb300 import _lib as L
    e2e_steps = max(3, min(args.steps, max(3, 200 // len(per))))
    pin = lambda t: t.cpu().pin_memory()
    host = []
    for d in per:
        h = dict(q=pin(d["q"]), k=pin(d["k_new"]), v=pin(d["v_new"]), cu=torch.from_numpy(d["cu_np"]).pin_memory(),
                 ctx=torch.from_numpy(d["ctx_np"]).pin_memory(), bt=torch.from_numpy(d["bt_np"]).pin_memory(),
                 slots=torch.empty(d["shape"].n_tokens, dtype=torch.int64).pin_memory(),
                 out=torch.empty(d["out"].shape, dtype=d["out"].dtype).pin_memory())
        h["dq"], h["dk"], h["dv"] = torch.empty_like(d["q"]), torch.empty_like(d["k_new"]), torch.empty_like(d["v_new"])
        host.append(h)
    h2d = sum(t.numel() * t.element_size() for h in host for t in (h["q"], h["k"], h["v"], h["cu"], h["ctx"], h["bt"],
                                                                  h["slots"]))
    d2h = sum(h["out"].numel() * h["out"].element_size() for h in host)

    def e2e_job():
        for d, h in zip(per, host):
            sh = d["shape"]
            h["slots"].numpy()[:] = L.cb_build_slot_mapping(sh.q_lens, sh.ctx_lens, d["bt_np"], sh.block_size)
            h["dq"].copy_(h["q"], non_blocking=True)
            h["dk"].copy_(h["k"], non_blocking=True)
            h["dv"].copy_(h["v"], non_blocking=True)
            d["cu"].copy_(h["cu"], non_blocking=True)
            d["ctx"].copy_(h["ctx"], non_blocking=True)
            d["bt"].copy_(h["bt"], non_blocking=True)
            d["slots"].copy_(h["slots"], non_blocking=True)
            call(d, h["dq"], h["dk"], h["dv"], d["slots"], d["cu"], d["ctx"], d["bt"])
            h["out"].copy_(d["out"], non_blocking=True)
            stream.synchronize()

    for _ in range(2):
        e2e_job()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_job()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    tokens = sum(d["shape"].n_tokens for d in per)
    return {"value": tokens * e2e_steps * world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": e2e_steps}


def job_work(job):
    """Algorithmic work of one iteration of the job (all its steps)."""
    tot = {}
    for sh in job["steps"]:
        for key, v in algorithmic(sh).items():
            tot[key] = tot.get(key, 0) + v
    return tot


def roofline_of(job, res, workload):
    """The dominant bound of the job's launches: achieved = algorithmic bytes (or
    FLOPs) per iteration / the launches' summed CUDA-event time."""
    work = job_work(job)
    peaks = load_peaks()
    launch_bytes = work["attn_bytes"] + (work["append_bytes"] if res["one_launch"] else 0)
    what = "append + paged attention launch" if res["one_launch"] else "paged attention launch"
    n = len(job["steps"])
    per = f" ({n} launches per iteration, {n} steps of the job)" if n > 1 else ""
    t = res["attn_s"]
    if launch_bytes / (peaks["hbm_gbs"] * 1e9) >= work["flops"] / (peaks["bf16_tflops"] * 1e12):
        a = launch_bytes / t / 1e9
        return {"bound": "hbm", "achieved": a, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": a / peaks["hbm_gbs"],
                "traffic": ncu_traffic(workload), "kernel": what + " (split-K decode / mixed)" + per,
                "algorithmic_bytes_per_launch": launch_bytes / n, "peak_source": peaks["source"] + " hbm_gbs"}
    a = work["flops"] / t / 1e12
    return {"bound": "tensor", "achieved": a, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": a / peaks["bf16_tflops"], "traffic": ncu_traffic(workload),
            "kernel": what + " (tcgen05 prefill tiles + decode)" + per,
            "algorithmic_flops_per_launch": work["flops"] / n, "peak_source": peaks["source"] + " bf16_tflops"}


def decode_summary(args, dev, stream, world):
    """The decode workload (64 decodes, MHA 32 x 128, 20 GB pool) measured in the
    same run: its K/V read rate and fraction of the HBM peak."""
    job = make_job("decode", args.seed, 20.0)
    res = measure(args, job, dev, stream, world, e2e=False)
    work = job_work(job)
    roof = roofline_of(job, res, "decode")
    sh = job["steps"][0]
    return {"workload": job["desc"], "ms_per_step": 1e3 * res["elapsed"] / args.steps,
            "tokens_per_s": sh.n_tokens * args.steps * world / res["elapsed"],
            "attention_ms": res["attn_s"] * 1e3, "kv_gbs": work["kv_bytes"] / res["attn_s"] / 1e9,
            "frac": work["kv_bytes"] / res["attn_s"] / 1e9 / load_peaks()["hbm_gbs"],
            "traffic": roof["traffic"], "roofline": roof, "gpu_launches": res["gpu_launches"],
            "l2": f"inputs larger than L2: {work['kv_bytes'] / 1e9:.2f} GB K/V read per step, no flush"}


def run_ours(args, job, world, rank, local):
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
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    res = measure(args, job, dev, stream, world, e2e=True, probe_copy=rank == 0 and not args.no_copy_probe)
    dec = decode_summary(args, dev, stream, world) if args.workload == "mixed" and not args.no_decode else None
    clocks = sampler.stop() if sampler else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(job["steps"], args.seed)
    if rank != 0:
        return
    work = job_work(job)
    steps = job["steps"]
    tokens = sum(sh.n_tokens for sh in steps)
    first = steps[0]
    line = {
        "metric": METRIC, "value": tokens * args.steps * world / res["elapsed"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * res["elapsed"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": job["desc"], "steps_per_iteration": len(steps),
                   "n_reqs": [sh.n_reqs for sh in steps] if len(steps) > 1 else first.n_reqs,
                   "n_tokens": tokens, "n_q_heads": first.n_q_heads, "n_kv_heads": first.n_kv_heads,
                   "head_dim": first.head_dim, "block_size": first.block_size, "num_blocks": first.num_blocks,
                   "l2": f"inputs larger than L2: {work['kv_bytes'] / 1e9:.2f} GB K/V read per iteration, no flush",
                   "parallelism": f"replicas x{world} (requests independent, no collective)"},
        "roofline": roofline_of(job, res, args.workload),
        "kv_gbs": work["kv_bytes"] / res["attn_s"] / 1e9,
        "kv_frac_of_hbm_peak": work["kv_bytes"] / res["attn_s"] / 1e9 / load_peaks()["hbm_gbs"],
        "attention_ms": res["attn_s"] * 1e3,
        "launch_ms": [round(1e3 * t, 4) for t in res["launch_s"]] if len(steps) > 1 else None,
        "append_in_launch": res["one_launch"],
        "prefill_tflops": work["pre_flops"] / res["attn_s"] / 1e12 if work["pre_flops"] else None,
        "copy_gbs_same_run": res["copy_gbs"],
        "decode": dec,
        "cpu_baseline": cpu,
        "e2e": res["e2e"],
        "gpu_launches": res["gpu_launches"],
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- continuous-batching trace
def trace_oracle_steps(tr, max_steps, seed, n_pick=24):
    """A bounded sample of the trace's iterations for the oracle: the FCFS
    scheduler oracle runs the trace (host only) for up to max_steps iterations,
    and n_pick of the iterations that run tokens are drawn uniformly; each is one
    layer's step (every layer of an iteration has the same shape)."""
    from oracle.scheduler import FCFSScheduler
    s = FCFSScheduler(tr.requests, tr.token_budget, tr.block_size, tr.num_blocks, wl.free_order(tr.num_blocks, tr.seed))
    shapes = []
    n = 0
    while not s.done() and n < max_steps:
        m = s.step()
        n += 1
        if len(m.q_lens):
            shapes.append(wl.StepShape(f"trace_it{m.step}", tr.n_q_heads, tr.n_kv_heads, tr.head_dim, tr.block_size,
                                       tr.num_blocks, tuple(int(x) for x in m.q_lens),
                                       tuple(int(x) for x in m.ctx_lens), seed=seed * 100003 + m.step))
    pick = sorted(np.random.default_rng(seed).choice(len(shapes), min(n_pick, len(shapes)), replace=False))
    return [shapes[i] for i in pick]


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
    # a stream of its own: the legacy default stream cannot be recorded into a graph
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    sh = stream.cuda_stream            # raw handle: the cheapest form for the per-layer calls
    tr = wl.trace(seed=args.seed + rank, pool_bytes=int(args.trace_pool_gb * wl.GB), n_layers=args.trace_layers)
    if args.trace_prefix_groups > 0:       # shared system prompts: blocks shared, partial last block copied
        tr = wl.with_prefixes(tr, args.trace_prefix_groups, args.trace_prefix_len, seed=args.seed + rank)
    nl, hq, hk, a, bs = tr.n_layers, tr.n_q_heads, tr.n_kv_heads, tr.head_dim, tr.block_size
    nb = tr.num_blocks
    # padded batching (static / dynamic): a step holds up to batch_size x the
    # longest prompt tokens, and one buffer of new rows serves every layer
    padded = args.trace_batching != "continuous"
    pB = args.trace_batch_size
    max_prompt = max(t[1] for t in tr.requests)
    max_out = max(t[2] for t in tr.requests)
    budget = pB * max_prompt if padded else tr.token_budget          # tokens per step the buffers hold
    max_reqs = pB if padded else min(budget, L.CB_MAX_REQS)
    nbuf = 1 if padded else nl
    bf = torch.bfloat16
    kc = [torch.empty((nb, hk, bs, a), dtype=bf, device=dev) for _ in range(nl)]
    vc = [torch.empty((nb, hk, bs, a), dtype=bf, device=dev) for _ in range(nl)]
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed + 17)
    qn = [torch.randn((budget, hq, a), generator=g, device=dev, dtype=bf) for _ in range(nbuf)]
    kn = [torch.randn((budget, hk, a), generator=g, device=dev, dtype=bf) for _ in range(nbuf)]
    vn = [torch.randn((budget, hk, a), generator=g, device=dev, dtype=bf) for _ in range(nbuf)]
    out = torch.empty((budget, hq, a), dtype=bf, device=dev)
    if padded:
        max_seq = max_prompt + max_out - 1
        maxblk = -(-max_seq // bs)
    else:
        maxblk = max(-(-(t[1] + t[2] - 1) // bs) for t in tr.requests)
        max_seq = max(t[1] + t[2] - 1 for t in tr.requests)
    window = args.trace_window

    def new_scheduler():
        s = L.Scheduler(nb, bs, budget, max_reqs, wl.free_order(nb, tr.seed), maxblk, window=window,
                        padded_batch=pB if padded else 0,
                        max_wait=args.trace_max_wait if args.trace_batching == "dynamic" else -1)
        for t in tr.requests:
            s.add_request(*(t[:3] if args.trace_no_share or padded else t))
        return s

    sched = new_scheduler()
    ws = torch.empty(L.cb_paged_attention_workspace_size(max_reqs, budget, budget, max_seq, hq, hk, a, bs),
                     dtype=torch.uint8, device=dev)
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
                 kv_stored=0, kv_paged=0, kv_contig=0, real=0)

    d_pairs = torch.zeros((budget, 2), dtype=torch.int32, device=dev)
    for hb in h:
        hb["pairs"] = torch.zeros((budget, 2), dtype=torch.int32).pin_memory()
    # The per-layer step goes straight to the C ABI with pointers taken once, as
    # a native serving loop would call it: every buffer below keeps its address,
    # and a step uses the first t rows / b requests of each.
    if window:
        wfn = L.lib().cb_kv_append_paged_attention_window

        def step_fn(*x):       # the window goes after block_size
            return wfn(*x[:21], window, *x[21:])
    else:
        step_fn = L.lib().cb_kv_append_paged_attention
    layer_ptrs = [(kn[i % nbuf].data_ptr(), vn[i % nbuf].data_ptr(), qn[i % nbuf].data_ptr(), kc[i].data_ptr(),
                   vc[i].data_ptr()) for i in range(nl)]
    fixed = dict(sl=d_sl.data_ptr(), cu=d_cu.data_ptr(), ctx=d_ctx.data_ptr(), bt=d_bt.data_ptr(),
                 out=out.data_ptr(), ws=ws.data_ptr(), wsb=ws.numel())

    # Each iteration's layer calls recorded as one CUDA graph and launched at once
    # (kernels of a graph start ~0.8 us after their predecessor instead of ~2.8
    # us); one graph per kind of iteration, updated in place while its kernels
    # stay the same.  A kind's first iteration runs directly: the library sets up
    # a kernel's per-device state on its first call, outside any recording.
    graphs, seen = {}, set()
    use_graphs = not args.trace_eager

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
        kind = (max_q > 1, npairs > 0)
        graph = None
        if use_graphs and host_io is None and kind in seen:
            graph = graphs.setdefault(kind, L.Graph())
            graph.begin(sh)
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
        if graph is not None:
            graph.end(sh)
        seen.add(kind)
        if host_io is not None:
            stats["h2d"] += nl * t * (hq + 2 * hk) * a * 2 + 4 * (2 * b + 1) + 4 * b * maxblk + 8 * t
            stats["d2h"] += nl * t * hq * a * 2
        stats["tokens"] += t
        stats["real"] += m["real_tokens"]
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
    e2e = None
    if not padded:
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
    cpu = None
    if world == 1 and not args.no_cpu_baseline and not padded and not window:
        cpu = cpu_baseline(trace_oracle_steps(tr, args.steps, args.seed), args.seed, tokens_per_row=nl)
        cpu["sample"] = "24 iterations of the trace drawn uniformly (one layer each); " + cpu["sample"]
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
        "config": {"workload": TRACE_DESC + {"continuous": "", "static": f"; static batching with padding, batches of {pB}",
                                              "dynamic": f"; dynamic batching with padding, batches of {pB}, "
                                                         f"max wait {args.trace_max_wait} steps"}[args.trace_batching]
                   + (f"; rolling window {window}" if window else "") + (
                       f"; {args.trace_prefix_groups} groups sharing a {args.trace_prefix_len}-token system prompt"
                       + (", computed in full (no sharing)" if args.trace_no_share else
                          ", blocks shared, partial last block copied on write")
                       if args.trace_prefix_groups > 0 else ""),
                   "n_layers": nl, "num_blocks": nb, "token_budget": budget,
                   "launch": ("per layer, directly" if args.trace_eager else
                              "each iteration's layer calls recorded as one CUDA graph (cb_graph_begin / "
                              "cb_graph_end, updated in place per kind of iteration); the end-to-end run directly"),
                   "decode_tokens": timed["dec"], "prefill_tokens": timed["pre"], "idle_steps": timed["idle"],
                   "preemptions": timed["preempted"],
                   "l2": "inputs larger than L2: each iteration reads every running request's K/V in 32 layers",
                   "parallelism": f"replicas x{world} (independent traces, no collective)"},
        "roofline": roof, "device_s": dev_s, "wall_s": wall,
        "useful": {"tokens": timed["real"], "pad_tokens": timed["tokens"] - timed["real"],
                   "tokens_per_s": timed["real"] * world / elapsed,
                   "definition": "prompt tokens and decoded positions of the requests, without pads; under "
                                 "continuous batching every processed token (recomputed prefills included)"},
        "finished_in_timed_region": {"requests": fin1[0] - fin0[0], "prompt_plus_output_tokens": fin1[1] - fin0[1],
                                     "requests_per_s": (fin1[0] - fin0[0]) / elapsed},
        "kv_memory": {"paged_waste": 1 - timed["kv_stored"] / max(1, timed["kv_paged"]),
                      "contiguous_waste": 1 - timed["kv_stored"] / max(1, timed["kv_contig"]),
                      "contiguous_max_seq_len": max_seq,
                      "definition": "slots held but not stored, summed over steps: paged blocks taken only when "
                                    "full vs a cache reserving max_seq_len slots per running request"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": timed["launches"], "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed", choices=sorted(WORKLOADS) + ["trace"])
    ap.add_argument("--trace-pool-gb", type=float, default=60.0, help="trace: K+V pool of all layers")
    ap.add_argument("--trace-layers", type=int, default=32, help="trace: attention layers per iteration")
    ap.add_argument("--trace-prefix-groups", type=int, default=0,
                    help="trace: requests join this many groups sharing a system prompt (0: none)")
    ap.add_argument("--trace-prefix-len", type=int, default=1000, help="trace: shared system prompt tokens")
    ap.add_argument("--trace-batching", default="continuous", choices=["continuous", "static", "dynamic"],
                    help="trace: continuous batching, or padded static / dynamic batching on the same kernels")
    ap.add_argument("--trace-batch-size", type=int, default=32, help="trace, padded batching: requests per batch")
    ap.add_argument("--trace-max-wait", type=int, default=8, help="trace, dynamic batching: steps a request waits")
    ap.add_argument("--trace-window", type=int, default=0,
                    help="trace: rolling window (keys per query; 0: none); blocks outside every window are freed")
    ap.add_argument("--trace-eager", action="store_true",
                    help="trace: launch every layer's call directly instead of recording each iteration's calls as "
                         "one CUDA graph (cb_graph_begin / cb_graph_end)")
    ap.add_argument("--trace-no-share", action="store_true",
                    help="trace with prefix groups: compute every prompt in full (no block sharing)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-copy-probe", action="store_true", help="skip the in-process HBM copy probe")
    ap.add_argument("--no-decode", action="store_true",
                    help="mixed workload: skip the decode step measured in the same run")
    ap.add_argument("--pool-gb", type=float, default=20.0,
                    help="K+V block pool size (blocks stay randomly scattered over it)")
    args = ap.parse_args(argv)
    world, rank, local = dist_env()
    if args.workload == "trace":
        if args.impl == "reference":
            if rank == 0:
                tr = wl.trace(seed=args.seed, pool_bytes=int(args.trace_pool_gb * wl.GB), n_layers=args.trace_layers)
                if args.trace_prefix_groups > 0:
                    tr = wl.with_prefixes(tr, args.trace_prefix_groups, args.trace_prefix_len, seed=args.seed)
                    if args.trace_no_share:
                        tr = wl.TraceShape(tr.name, tr.n_layers, tr.n_q_heads, tr.n_kv_heads, tr.head_dim,
                                           tr.block_size, tr.token_budget, tr.num_blocks,
                                           tuple(t[:3] for t in tr.requests), tr.seed)
                steps = trace_oracle_steps(tr, args.steps, args.seed)
                run_reference(args, {"steps": steps, "seq": None}, TRACE_DESC + "; 24 iterations drawn uniformly, "
                              "one layer each, rate per token through all layers", world, rank,
                              tokens_per_row=tr.n_layers)
            return
        run_trace(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.impl == "reference":
        job = make_job(args.workload, args.seed, args.pool_gb)
        run_reference(args, job, job["desc"], world, rank)
        return
    # weak scaling: each rank runs its own batch of the same workload (its own seed)
    job = make_job(args.workload, args.seed + rank, args.pool_gb)
    run_ours(args, job, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
