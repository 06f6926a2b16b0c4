"""GPU parity of attn_prefill_paged (packed query chunks against a paged
cache with cached prefixes) against the FP64 oracle.

Covers ragged batches with and without prefixes, causal and full, even
(head-paired) and odd (row-paired) GQA groups, chunks longer than one and two
128-row tiles, NaN in unused cache slots, permuted pages, the special cases
that reduce to the contiguous prefill and to paged decode, and the
device-side length checks."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import oracle
import workloads as W
from gpu_util import assert_close, dev, device_error_clean, host
from test_oracle_pins import _paged_problem
from test_parity_prefill import stratified_rows

pytestmark = pytest.mark.gpu


def run(Q, kc, vc, cu, skv, table, causal=True, max_q=None):
    O = torch.full(Q.shape, float("nan"), dtype=torch.float16, device="cuda")
    mq = max_q if max_q is not None else int(np.diff(cu).max())
    ag.attn_prefill_paged(dev(Q), dev(kc), dev(vc), O, dev(cu), dev(skv), dev(table), mq, causal)
    torch.cuda.synchronize()
    return host(O)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("heads", [(16, 8), (32, 8), (6, 2), (3, 3)])
def test_ragged_chunks_with_prefixes(causal, heads):
    H_q, H_kv = heads
    rng = np.random.default_rng(60 + H_q)
    lens_kv = [1, 130, 600, 300, 1000, 257]
    lens_q = [1, 130, 129, 17, 400, 1]
    _, _, kc, vc, table, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q, H_q, H_kv, 128)
    out = run(Q, kc, vc, cu, skv, table, causal)
    ref = oracle.prefill_paged(Q, kc, vc, cu, skv, table, causal=causal)
    assert_close(out, ref, f"paged prefill heads={heads} causal={causal}")
    assert device_error_clean()


def test_no_prefix_equals_contiguous_prefill():
    B, S, H_q, H_kv = 3, 333, 8, 2
    Qc, Kc, Vc = W.prefill_inputs(W.PrefillConfig("t", B, S, H_q, H_kv), seed=61)
    Oc = torch.empty(Qc.shape, dtype=torch.float16, device="cuda")
    ag.attn_prefill(dev(Qc), dev(Kc), dev(Vc), Oc, causal=True)
    npg = (S + 15) // 16
    table = np.arange(B * npg, dtype=np.int32).reshape(B, npg)
    kc = np.zeros((B * npg, H_kv, 16, 128), np.float16)
    vc = np.zeros_like(kc)
    for b in range(B):
        for p in range(npg):
            t0, t1 = 16 * p, min(S, 16 * p + 16)
            kc[table[b, p], :, :t1 - t0] = Kc[b, t0:t1].transpose(1, 0, 2)
            vc[table[b, p], :, :t1 - t0] = Vc[b, t0:t1].transpose(1, 0, 2)
    cu = np.arange(0, (B + 1) * S, S, dtype=np.int32)
    out = run(Qc.reshape(B * S, H_q, 128), kc, vc, cu, np.full(B, S, np.int32), table)
    assert_close(out.reshape(B, S, H_q, 128), host(Oc).astype(np.float64), "paged vs contiguous")


def test_single_query_chunks_equal_decode():
    cfg = W.DecodeConfig("t", 32, 16, 8, max_blocks_per_seq=64)
    inp = W.decode_inputs(cfg, seed=62, seq_lens=W.uniform_int(62, 3, 32, 1, 1024))
    cu = np.arange(33, dtype=np.int32)
    out = run(inp.q, inp.k_cache, inp.v_cache, cu, inp.seq_lens, inp.block_tables)
    dec = torch.empty(inp.q.shape, dtype=torch.float16, device="cuda")
    ag.attn_decode_paged(dev(inp.q), dev(inp.k_cache), dev(inp.v_cache), dec, dev(inp.block_tables),
                         dev(inp.seq_lens))
    torch.cuda.synchronize()
    ref = oracle.decode_paged(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.seq_lens)
    assert_close(out, ref, "paged prefill L_q=1 vs oracle decode")
    assert_close(out, host(dec).astype(np.float64), "paged prefill L_q=1 vs GPU decode")


def test_chunked_prefill_workload_sampled():
    # 4 sequences with 2-4k cached tokens each and a 512-1024-token new chunk, H 32/8
    rng = np.random.default_rng(63)
    lens_q = [512, 1024, 777, 600]
    lens_kv = [q + p for q, p in zip(lens_q, [3000, 2048, 3333, 4000])]
    _, _, kc, vc, table, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q, 32, 8, 128)
    out = run(Q, kc, vc, cu, skv, table)
    ref = oracle.prefill_paged(Q, kc, vc, cu, skv, table)
    assert_close(out, ref, "chunked prefill")


@pytest.mark.parametrize("causal", [True, False])
def test_chunked_prefill_bench_workload_stratified(causal):
    # the benchmark's launch: 4 x (6144 cached + 2048 new), H 32/8, one random row
    # per (sequence, 128-row block, head) plus all rows of the first and last
    # chunk blocks for three heads: every CTA of the launch is checked
    cfg = W.CHUNKED_PREFILL
    Q, kc, vc, cu, skv, table = W.chunked_prefill_inputs(cfg, seed=0)
    out = run(Q, kc, vc, cu, skv, table, causal=causal, max_q=cfg.chunk)
    assert np.isfinite(out.astype(np.float32)).all(), "rows left unwritten"
    n_mb = cfg.chunk // 128
    rows = stratified_rows(cfg.num_seqs, cfg.chunk, cfg.H_q, seed=2, diag_blocks=(0, n_mb - 1),
                           diag_heads=(0, 17, cfg.H_q - 1))
    ref = oracle.prefill_paged_rows(Q, kc, vc, cu, skv, table, rows, causal=causal)
    got = out[cu[rows[:, 0]] + rows[:, 1], rows[:, 2]]
    assert_close(got, ref, f"{cfg.name} causal={causal}: {len(rows)} stratified rows")
    assert device_error_clean()


def test_device_length_checks():
    rng = np.random.default_rng(64)
    _, _, kc, vc, table, Q, cu, skv = _paged_problem(rng, [50, 300], [10, 200], 4, 2, 128)
    bad = skv.copy()
    bad[1] = 150                                 # chunk of 200 longer than its 150-key context
    out = run(Q, kc, vc, cu, bad, table)
    assert ag.attn_get_device_error(reset=True) & 64
    ref = oracle.prefill_paged(Q[:10], kc, vc, cu[:2], skv[:1], table[:1])
    assert_close(out[:10], ref, "good sequence next to a bad one")
    assert np.isnan(out[10:].astype(np.float32)).all()   # the bad sequence is skipped
    # max_seqlen_q = 100 sizes the launch for one 128-row tile: the 200-row chunk
    # overruns it and is flagged, its first 128 rows are still right
    out = run(Q, kc, vc, cu, skv, table, max_q=100)
    assert ag.attn_get_device_error(reset=True) & 64
    ref = oracle.prefill_paged(Q, kc, vc, cu, skv, table)
    assert_close(out[:10 + 128], ref[:10 + 128], "rows within max_seqlen_q")


def test_chunk_offsets_outside_packed_rows_are_skipped():
    rng = np.random.default_rng(66)
    _, _, kc, vc, table, Q, cu, skv = _paged_problem(rng, [300, 400], [200, 150], 4, 2, 128)
    bad = cu.copy()
    bad[2] = cu[2] + 40                          # the second chunk would run past packed Q / O
    out = run(Q, kc, vc, bad, skv, table, max_q=200)
    assert ag.attn_get_device_error(reset=True) & 64
    ref = oracle.prefill_paged(Q[:200], kc, vc, cu[:2], skv[:1], table[:1])
    assert_close(out[:200], ref, "good sequence next to one outside packed Q")
    assert np.isnan(out[200:].astype(np.float32)).all()
    bad = cu.copy()
    bad[1] = -8                                  # negative offset: both chunks are skipped
    out = run(Q, kc, vc, bad, skv, table, max_q=200)
    assert ag.attn_get_device_error(reset=True) & 64
    assert np.isnan(out.astype(np.float32)).all()


@pytest.mark.parametrize("heads", [(32, 2), (5, 1), (64, 64)])
def test_wide_groups_and_many_heads(heads):
    H_q, H_kv = heads
    rng = np.random.default_rng(65 + H_q)
    lens_q, prefix = [150, 1, 300], [200, 63, 0]
    _, _, kc, vc, table, Q, cu, skv = _paged_problem(rng, [q + p for q, p in zip(lens_q, prefix)],
                                                     lens_q, H_q, H_kv, 128)
    out = run(Q, kc, vc, cu, skv, table)
    assert_close(out, oracle.prefill_paged(Q, kc, vc, cu, skv, table), f"paged prefill heads={heads}")
    assert device_error_clean()


def test_one_long_chunk_without_prefix():
    # a single 8192-token chunk with an empty cache prefix (the whole prompt at once)
    rng = np.random.default_rng(67)
    _, _, kc, vc, table, Q, cu, skv = _paged_problem(rng, [8192], [8192], 16, 8, 128, nan_unused=False)
    out = run(Q, kc, vc, cu, skv, table)
    assert np.isfinite(out.astype(np.float32)).all(), "rows left unwritten"
    rows = stratified_rows(1, 8192, 16, seed=5, diag_blocks=(0, 63), diag_heads=(0, 15))
    ref = oracle.prefill_paged_rows(Q, kc, vc, cu, skv, table, rows)
    assert_close(out[cu[rows[:, 0]] + rows[:, 1], rows[:, 2]], ref, "one 8192-token chunk")
    assert device_error_clean()
