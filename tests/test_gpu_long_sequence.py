"""Long-context chunked prefill as [CB] §Chunked prefill describes it: one
32768-token prompt processed in 16 chunks of 2048 tokens, each chunk's K/V
appended through the block table and attended together with everything the
earlier chunks stored, co-scheduled in every step with 16 decodes whose stored
contexts grow from 8192 by one token per step.  Each step is one
cb_kv_append_paged_attention call on the cache that the previous steps wrote;
the prompt's blocks start out filled with NaN, so a read of a position that no
append has written yet would show.  Checked against the oracle at every step:
six rows of the chunk (the first, the last and four inside) and all 16
decodes, over the keys the oracle assembles from the generated inputs."""
import math

import numpy as np
import pytest
import torch

from gpu_util import L, assert_close, cu_of, f64
from oracle import attention as oa
from oracle import paged as op

pytestmark = pytest.mark.gpu

HQ, HKV, A, BS = 32, 8, 128, 16
CHUNK, N_CHUNKS, N_DEC, DEC_CTX = 2048, 16, 16, 8192


def test_long_prompt_in_sixteen_chained_chunks():
    lib = L()
    dev = "cuda"
    prompt_blocks = CHUNK * N_CHUNKS // BS
    dec_blocks = -(-(DEC_CTX + N_CHUNKS) // BS)
    num_blocks = prompt_blocks + N_DEC * dec_blocks + 1000
    rng = np.random.default_rng(11)
    perm = rng.permutation(num_blocks).astype(np.int32)
    prompt_table = perm[:prompt_blocks]
    dec_tables = perm[prompt_blocks:prompt_blocks + N_DEC * dec_blocks].reshape(N_DEC, dec_blocks)
    tables = np.full((N_DEC + 1, prompt_blocks), -1, np.int32)
    tables[:N_DEC, :dec_blocks] = dec_tables
    tables[N_DEC] = prompt_table
    d_tables = torch.from_numpy(tables).to(dev)

    g = torch.Generator(device=dev)
    g.manual_seed(11)
    kc = torch.randn((num_blocks, HKV, BS, A), generator=g, device=dev, dtype=torch.bfloat16)
    vc = torch.randn((num_blocks, HKV, BS, A), generator=g, device=dev, dtype=torch.bfloat16)
    pidx = torch.from_numpy(prompt_table.astype(np.int64)).to(dev)
    kc[pidx] = float("nan")
    vc[pidx] = float("nan")

    # the oracle's contiguous keys: the decodes' first 8192 stored positions (read
    # from the initial pool through their tables), then every appended row
    dec_k = np.zeros((N_DEC, DEC_CTX + N_CHUNKS, HKV, A))
    dec_v = np.zeros_like(dec_k)
    compact = np.arange(DEC_CTX // BS)
    for d in range(N_DEC):
        idx = torch.from_numpy(dec_tables[d, :DEC_CTX // BS].astype(np.int64)).to(dev)
        dec_k[d, :DEC_CTX] = op.gather_request(f64(kc.index_select(0, idx)), compact, DEC_CTX, BS)
        dec_v[d, :DEC_CTX] = op.gather_request(f64(vc.index_select(0, idx)), compact, DEC_CTX, BS)
    prompt_k = np.zeros((CHUNK * N_CHUNKS, HKV, A))
    prompt_v = np.zeros_like(prompt_k)

    scale = 1.0 / math.sqrt(A)
    q_lens = [1] * N_DEC + [CHUNK]
    d_cu = torch.from_numpy(cu_of(q_lens)).to(dev)
    n_tok = N_DEC + CHUNK
    gi = torch.Generator(device=dev)
    for k in range(N_CHUNKS):
        ctx = [DEC_CTX + k] * N_DEC + [CHUNK * k]
        gi.manual_seed(1000 + k)
        q = torch.randn((n_tok, HQ, A), generator=gi, device=dev, dtype=torch.bfloat16)
        k_new = torch.randn((n_tok, HKV, A), generator=gi, device=dev, dtype=torch.bfloat16)
        v_new = torch.randn((n_tok, HKV, A), generator=gi, device=dev, dtype=torch.bfloat16)
        slots = lib.cb_build_slot_mapping(q_lens, ctx, tables, BS)
        max_q, max_kv = CHUNK, max(DEC_CTX + k + 1, CHUNK * (k + 1))
        ws = torch.empty(lib.cb_paged_attention_workspace_size(N_DEC + 1, n_tok, max_q, max_kv, HQ, HKV, A, BS),
                         dtype=torch.uint8, device=dev)
        out = torch.full_like(q, float("nan"))
        lib.cb_kv_append_paged_attention(k_new, v_new, torch.from_numpy(slots).to(dev), q, d_cu,
                                         torch.tensor(ctx, dtype=torch.int32, device=dev), d_tables, kc, vc, out,
                                         scale, ws, max_q, max_kv)
        assert lib.cb_last_error() == 0, f"chunk {k}"
        qh, kn, vn, got = f64(q), f64(k_new), f64(v_new), f64(out)
        prompt_k[CHUNK * k:CHUNK * (k + 1)] = kn[N_DEC:]
        prompt_v[CHUNK * k:CHUNK * (k + 1)] = vn[N_DEC:]
        dec_k[:, DEC_CTX + k] = kn[:N_DEC]
        dec_v[:, DEC_CTX + k] = vn[:N_DEC]
        rows = sorted({0, CHUNK - 1} | set(np.random.default_rng(k).choice(np.arange(1, CHUNK - 1), 4,
                                                                            replace=False).tolist()))
        hi = CHUNK * (k + 1)
        ref = oa.attention_rows(qh[N_DEC:][rows], prompt_k[:hi], prompt_v[:hi], [CHUNK * k + i for i in rows],
                                scale, HQ, HKV)
        assert_close(got[N_DEC:][rows], ref, f"chunk {k} rows {rows}")
        for d in range(N_DEC):
            ref = oa.attention_rows(qh[d:d + 1], dec_k[d, :DEC_CTX + k + 1], dec_v[d, :DEC_CTX + k + 1],
                                    [DEC_CTX + k], scale, HQ, HKV)
            assert_close(got[d:d + 1], ref, f"chunk step {k} decode {d}")
        del ws, out
    del kc, vc
    torch.cuda.empty_cache()
