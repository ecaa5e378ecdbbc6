"""The roofline's algorithmic work (bench.py): worked by hand on the tiny step.

Decode/prefill K/V bytes count each request's valid keys once, 2 (K, V) x keys x
Hkv x A x 2 bytes; attention FLOPs count the causal-valid (query, key) pairs,
4 A flops per pair and query head (QK^T and PV); the append reads and writes
each new row's K and V."""
import bench
import workloads as wl


def test_algorithmic_work_of_the_tiny_step():
    s = wl.tiny()                       # (ctx, q): (37, 1), (100, 1), (4, 3), (0, 20); Hq = Hkv = 4, A = 64
    w = bench.algorithmic(s)
    keys = (37 + 1) + (100 + 1) + (4 + 3) + (0 + 20)          # 166
    assert w["kv_bytes"] == 2 * keys * 4 * 64 * 2
    assert w["dec_kv_bytes"] == 2 * ((37 + 1) + (100 + 1)) * 4 * 64 * 2
    # causal-valid pairs: a decode sees ctx + 1 keys; query i of a chunk sees ctx + i + 1
    pairs = 38 + 101 + (5 + 6 + 7) + sum(range(1, 21))
    assert w["flops"] == 4 * 64 * 4 * pairs
    assert w["pre_flops"] == 4 * 64 * 4 * ((5 + 6 + 7) + sum(range(1, 21)))
    assert w["append_bytes"] == 2 * 2 * 25 * 4 * 64 * 2
    assert w["attn_bytes"] == w["kv_bytes"] + 2 * 25 * 4 * 64 * 2   # plus q read and out written


def test_code_only_hash_ignores_comments_and_layout():
    a = "int x = 1; // one\n/* block\n comment */ float y;"
    b = "int x = 1;   /* other */\n\n float y; // two"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(a.replace("x = 1", "x = 2"))
