"""attn_decode_paged_noalloc: paged decode for callers that cannot allocate.

Some users of this library cannot call cudaMalloc (code hosted by another
runtime that owns all device memory, programs with a fixed memory budget,
loops that must not risk cudaMalloc/cudaFree synchronising the device).  For
them the library keeps its split-K scratch in a fixed buffer compiled into it.

These tests call that entry point through the C ABI several times in a row.
It runs the same kernels with the same split plan as attn_decode_paged, so
each result must equal attn_decode_paged's bit for bit on the same inputs,
and match the FP64 oracle within the tolerance of the other parity tests.
The second call keeps the first call's shape (sequences, heads, table width)
but has much shorter contexts, so every row finds finite partials from the
first call in splits past its own: they must be ignored.  The third call has
another shape.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import oracle
import workloads as W
from gpu_util import assert_close, device_error_clean, host

pytestmark = pytest.mark.gpu


def _problem(lens, seed, max_blocks=128):
    cfg = W.DecodeConfig("noalloc", len(lens), 16, 8, max_blocks_per_seq=max_blocks)
    inp = W.decode_inputs(cfg, seed=seed, seq_lens=np.asarray(lens, np.int32))
    dev = [torch.from_numpy(x).cuda() for x in (inp.q, inp.k_cache, inp.v_cache,
                                                 inp.block_tables, inp.seq_lens)]
    return inp, dev


def _existing(t):
    out = torch.full_like(t[0], float("nan"))
    ag.attn_decode_paged(t[0], t[1], t[2], out, t[3], t[4])
    torch.cuda.synchronize()
    return host(out)


def _noalloc(t):
    out = torch.full_like(t[0], float("nan"))
    ag.attn_decode_paged_noalloc(t[0], t[1], t[2], out, t[3], t[4])
    torch.cuda.synchronize()
    return host(out)


def test_noalloc_matches_existing_entry_point_and_oracle_on_three_calls():
    long_lens = [2048, 1, 700, 17, 0, 1333, 16, 2000] * 8
    short_lens = [1 + (7 * i) % 40 for i in range(len(long_lens))]     # 1..40 tokens
    calls = [("first call", _problem(long_lens, seed=21)),
             ("second call, same shape, short contexts", _problem(short_lens, seed=23)),
             ("third call, another shape", _problem([5, 900, 128, 2048, 64, 1500], seed=22))]
    for name, (inp, t) in calls:
        got = _noalloc(t)
        assert np.array_equal(got.view(np.uint16), _existing(t).view(np.uint16)), \
            f"{name}: noalloc differs from attn_decode_paged"
        ref = oracle.decode_paged(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.seq_lens)
        assert_close(got, ref, f"noalloc vs oracle, {name}")
    assert device_error_clean()


def test_noalloc_refuses_problem_larger_than_its_scratch():
    # 1024 sequences x 16 heads x 16 splits (of 64 pages) of partials need ~135 MB > 32 MiB
    N, H_q, H_kv, mb = 1024, 16, 8, 1024
    need = ag.attn_decode_paged_workspace_bytes(N, H_q, H_kv, 128, mb, 16, 0)
    assert need > ag.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(N, H_q, 128, dtype=torch.float16, device="cuda")
    kc = torch.zeros(1, H_kv, 16, 128, dtype=torch.float16, device="cuda")
    bt = torch.zeros(N, mb, dtype=torch.int32, device="cuda")
    sl = torch.ones(N, dtype=torch.int32, device="cuda")
    with pytest.raises(ag.AttnError) as e:
        ag.attn_decode_paged_noalloc(q, kc, kc, torch.empty_like(q), bt, sl)
    assert e.value.status == ag.ATTN_ERR_WORKSPACE
