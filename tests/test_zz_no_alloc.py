"""attn_decode_paged_noalloc: paged decode for callers that cannot allocate.

Some users of this library cannot call cudaMalloc (code hosted by another
runtime that owns all device memory, programs with a fixed memory budget,
loops that must not risk cudaMalloc/cudaFree synchronising the device).  For
them the library keeps its split-K scratch in a fixed buffer compiled into it.
These tests call that entry point through the C ABI twice in a row, on two
different problems, and check each result against attn_decode_paged on the
same inputs within the tolerance the other parity tests use; the second call
also shows that what the first call left in the shared buffer does no harm.
This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import workloads as W
from gpu_util import assert_close, device_error_clean, host

pytestmark = pytest.mark.gpu


def _problem(lens, seed, max_blocks=128):
    cfg = W.DecodeConfig("noalloc", len(lens), 16, 8, max_blocks_per_seq=max_blocks)
    inp = W.decode_inputs(cfg, seed=seed, seq_lens=np.asarray(lens, np.int32))
    return [torch.from_numpy(x).cuda() for x in (inp.q, inp.k_cache, inp.v_cache,
                                                  inp.block_tables, inp.seq_lens)]


def _existing(t):
    out = torch.empty_like(t[0])
    ag.attn_decode_paged(t[0], t[1], t[2], out, t[3], t[4])
    torch.cuda.synchronize()
    return host(out).astype(np.float64)


def _noalloc(t):
    out = torch.full_like(t[0], float("nan"))
    ag.attn_decode_paged_noalloc(t[0], t[1], t[2], out, t[3], t[4])
    torch.cuda.synchronize()
    return host(out)


def test_noalloc_matches_existing_entry_point_on_two_calls():
    first = _problem([2048, 1, 700, 17, 0, 1333, 16, 2000] * 8, seed=21)
    second = _problem([5, 900, 128, 2048, 64, 1500], seed=22)
    for name, t in (("first call", first), ("second call", second)):
        got = _noalloc(t)
        assert_close(got, _existing(t), f"noalloc vs attn_decode_paged, {name}")
    assert device_error_clean()


def test_noalloc_refuses_problem_larger_than_its_scratch():
    # 1024 sequences x 16 heads x 8 splits of partials need ~68 MB > 32 MiB
    N, H_q, H_kv, mb = 1024, 16, 8, 128
    need = ag.attn_decode_paged_workspace_bytes(N, H_q, H_kv, 128, mb, 16, 0)
    assert need > ag.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(N, H_q, 128, dtype=torch.float16, device="cuda")
    kc = torch.zeros(1, H_kv, 16, 128, dtype=torch.float16, device="cuda")
    bt = torch.zeros(N, mb, dtype=torch.int32, device="cuda")
    sl = torch.ones(N, dtype=torch.int32, device="cuda")
    with pytest.raises(ag.AttnError) as e:
        ag.attn_decode_paged_noalloc(q, kc, kc, torch.empty_like(q), bt, sl)
    assert e.value.status == ag.ATTN_ERR_WORKSPACE
