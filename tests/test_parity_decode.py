"""GPU parity of the paged decode path (split-K + combine, through the C ABI)
against the FP64 oracle.

Covers the pages' own decode shapes (identity block table, equal lengths),
both decode workloads at full size (256 sequences with lengths uniform on
[128, 2048]; 8 sequences of 32768 tokens) in the configuration the benchmark
times, ragged lengths including 0, 1 and page boundaries, NaN-poisoned unused
cache slots and table entries, block relocation (bitwise invariant), every
split size, decode == last prefill row, group sizes 1..16, the standalone
combine kernel on oracle partials, and the device-side input checks."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import golden_cases
import oracle
import workloads as W
from gpu_util import assert_close, dev, device_error_clean, host

pytestmark = pytest.mark.gpu


def to_dev(inp: W.DecodeInputs):
    return (dev(inp.q), dev(inp.k_cache), dev(inp.v_cache), dev(inp.block_tables), dev(inp.seq_lens))


def run_decode(inp: W.DecodeInputs, pages_per_split=None, tensors=None):
    q, kc, vc, bt, sl = tensors or to_dev(inp)
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    if pages_per_split is None:
        ag.attn_decode_paged(q, kc, vc, out, bt, sl)
    else:
        nbytes = ag.attn_decode_paged_workspace_bytes(q.shape[0], q.shape[1], kc.shape[1], 128,
                                                      bt.shape[1], 16, pages_per_split)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        ag.attn_decode_paged_ws(q, kc, vc, out, bt, sl, ws, pages_per_split)
    torch.cuda.synchronize()
    return host(out)


def oracle_decode(inp: W.DecodeInputs):
    return oracle.decode_paged(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.seq_lens)


def make(num_seqs, H_q, H_kv, lens, max_blocks=None, seed=0):
    lens = np.asarray(lens, np.int32)
    mb = max_blocks or max(1, int(np.ceil(lens.max() / 16)) if len(lens) else 1)
    cfg = W.DecodeConfig("t", num_seqs, H_q, H_kv, max_blocks_per_seq=mb)
    return W.decode_inputs(cfg, seed=seed, seq_lens=lens)


def poison(inp: W.DecodeInputs):
    """NaN in every cache slot past a sequence's length and in unused blocks;
    -1 is already in unused table entries."""
    kc, vc = inp.k_cache.copy(), inp.v_cache.copy()
    used = np.zeros(kc.shape[0], bool)
    for n, L in enumerate(inp.seq_lens):
        pages = (int(L) + 15) // 16
        for p in range(pages):
            b = inp.block_tables[n, p]
            used[b] = True
            valid = min(16, int(L) - 16 * p)
            kc[b, :, valid:, :] = np.nan
            vc[b, :, valid:, :] = np.nan
    kc[~used] = np.nan
    vc[~used] = np.nan
    return W.DecodeInputs(inp.q, kc, vc, inp.block_tables, inp.seq_lens)


@pytest.mark.parametrize("case", golden_cases.load()[1])
def test_page_decode_cases_identity_table(case):
    N, L, H_q, H_kv, D = case
    npg = (L + 15) // 16
    table = np.arange(N * npg, dtype=np.int32).reshape(N, npg)
    q = W.normal_fp16(L, 0, (N, H_q, D))
    kc = W.normal_fp16(L, 1, (N * npg, H_kv, 16, D))
    vc = W.normal_fp16(L, 2, (N * npg, H_kv, 16, D))
    inp = W.DecodeInputs(q, kc, vc, table, np.full(N, L, np.int32))
    assert_close(run_decode(inp), oracle_decode(inp), f"page decode {case}")
    assert device_error_clean()


@pytest.mark.parametrize("cfg", [W.DECODE_MIX, W.DECODE_LONG, W.DECODE_GQA8], ids=lambda c: c.name)
def test_decode_workloads_full(cfg):
    inp = W.decode_inputs(cfg, seed=0)
    assert_close(run_decode(inp), oracle_decode(inp), cfg.name)
    assert device_error_clean()


def test_ragged_lengths_poisoned_slots():
    lens = [0, 1, 2, 15, 16, 17, 31, 32, 33, 100, 255, 256, 257, 1000, 2047, 2048]
    inp = poison(make(len(lens), 16, 8, lens, max_blocks=128, seed=3))
    out = run_decode(inp)
    ref = oracle_decode(inp)
    assert np.all(out[0] == 0)                 # empty context -> zeros
    assert_close(out, ref, "ragged+poison")
    assert device_error_clean()


@pytest.mark.parametrize("pps", [1, 2, 3, 7, 16, 64, 128])
def test_every_split_size_matches(pps):
    lens = [1, 16, 17, 333, 2048, 1500, 64, 900]
    inp = make(len(lens), 16, 8, lens, max_blocks=128, seed=4)
    assert_close(run_decode(inp, pages_per_split=pps), oracle_decode(inp), f"pages_per_split={pps}")


def test_block_relocation_is_bitwise_invariant():
    lens = [50, 700, 1, 2048, 129]
    inp = make(len(lens), 16, 8, lens, max_blocks=128, seed=5)
    a = run_decode(inp)
    nb = inp.num_blocks
    p = np.random.default_rng(6).permutation(nb).astype(np.int32)
    kc2, vc2 = np.empty_like(inp.k_cache), np.empty_like(inp.v_cache)
    kc2[p], vc2[p] = inp.k_cache, inp.v_cache
    bt2 = np.where(inp.block_tables >= 0, p[np.maximum(inp.block_tables, 0)], -1).astype(np.int32)
    b = run_decode(W.DecodeInputs(inp.q, kc2, vc2, bt2, inp.seq_lens))
    assert np.array_equal(a, b)


# groups of 1 to 16 heads fill one tile of 16 head rows; 20 and 32 take two tiles
# (the second one partly empty for 20)
@pytest.mark.parametrize("heads", [(8, 8), (16, 8), (12, 4), (32, 8), (16, 2), (10, 2), (16, 1),
                                   (40, 2), (64, 2)])
def test_group_sizes(heads):
    H_q, H_kv = heads
    lens = [5, 77, 300, 1024]
    inp = make(len(lens), H_q, H_kv, lens, max_blocks=64, seed=H_q + H_kv)
    assert_close(run_decode(inp), oracle_decode(inp), f"heads={heads}")


def test_decode_equals_last_prefill_row():
    B, S, H_q, H_kv = 3, 517, 16, 8
    Q, K, V = W.prefill_inputs(W.PrefillConfig("t", B, S, H_q, H_kv), seed=8)
    O = torch.empty(Q.shape, dtype=torch.float16, device="cuda")
    ag.attn_prefill(dev(Q), dev(K), dev(V), O, causal=True)
    npg = (S + 15) // 16
    perm = W.permutation(8, 4, B * npg)
    table = perm.reshape(B, npg).astype(np.int32)
    kc = np.zeros((B * npg, H_kv, 16, 128), np.float16)
    vc = np.zeros_like(kc)
    for b in range(B):
        for p in range(npg):
            t0, t1 = 16 * p, min(S, 16 * p + 16)
            kc[table[b, p], :, :t1 - t0] = K[b, t0:t1].transpose(1, 0, 2)
            vc[table[b, p], :, :t1 - t0] = V[b, t0:t1].transpose(1, 0, 2)
    inp = W.DecodeInputs(Q[:, S - 1].copy(), kc, vc, table, np.full(B, S, np.int32))
    dec = run_decode(inp)
    pre = host(O)[:, S - 1]
    ref = oracle.prefill_rows(Q, K, V, [(b, S - 1, h) for b in range(B) for h in range(H_q)])
    assert_close(dec, ref.reshape(B, H_q, 128), "decode vs oracle")
    assert_close(dec, pre.astype(np.float64), "decode vs GPU prefill", max_abs=4e-3, mean_abs=5e-4)


@pytest.mark.parametrize("cuts", [[0, 700], [0, 1, 2, 350, 700], [0, 0, 100, 100, 700, 700], [0, 16, 32, 48, 64, 700]])
def test_combine_kernel_on_oracle_partials(cuts):
    H_q, H_kv, L = 8, 2, 700
    rng = np.random.default_rng(len(cuts))
    q = W.normal_fp16(11, 0, (H_q, 128))
    Kseq, Vseq = W.normal_fp16(11, 1, (L, H_kv, 128)), W.normal_fp16(11, 2, (L, H_kv, 128))
    O_part, lse_part = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        n = b - a
        kc = Kseq[a:b][:, :, None, :].copy() if n else np.zeros((1, H_kv, 1, 128), np.float16)
        vc = Vseq[a:b][:, :, None, :].copy() if n else np.zeros((1, H_kv, 1, 128), np.float16)
        o, l = oracle.decode_paged(q[None], kc, vc, np.arange(max(n, 1), dtype=np.int32)[None],
                                   np.array([n], np.int32), with_lse=True)
        O_part.append(o[0])
        lse_part.append(l[0])
    O_part = np.stack(O_part, 1)
    lse_part = np.stack(lse_part, 1)
    ref = oracle.lse_combine(O_part, lse_part)
    out = torch.empty(H_q, 128, dtype=torch.float16, device="cuda")
    ag.attn_lse_combine(dev(O_part.astype(np.float32)), dev(lse_part.astype(np.float32)), out)
    torch.cuda.synchronize()
    assert_close(host(out), ref, f"combine cuts={cuts}")
    del rng


def test_combine_all_empty_rows_give_zero():
    O_part = torch.ones(3, 4, 128, device="cuda")
    lse = torch.full((3, 4), float("-inf"), device="cuda")
    out = torch.full((3, 128), 7.0, dtype=torch.float16, device="cuda")
    ag.attn_lse_combine(O_part, lse, out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_device_checks_flag_bad_inputs():
    lens = [40, 40]
    inp = make(2, 16, 8, lens, max_blocks=4, seed=12)
    assert device_error_clean()
    bt = inp.block_tables.copy()
    bt[1, 1] = -7                                   # a hole inside sequence 1's pages
    run_decode(W.DecodeInputs(inp.q, inp.k_cache, inp.v_cache, bt, inp.seq_lens))
    assert ag.attn_get_device_error(reset=True) == 2
    sl = np.array([40, 40 + 4 * 16], np.int32)      # longer than the table holds
    run_decode(W.DecodeInputs(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, sl))
    assert ag.attn_get_device_error(reset=True) & 4
    assert device_error_clean()


def test_empty_batch_noop_and_library_workspace_release():
    q = torch.zeros(0, 16, 128, dtype=torch.float16, device="cuda")
    kc = torch.zeros(1, 8, 16, 128, dtype=torch.float16, device="cuda")
    bt = torch.zeros(0, 4, dtype=torch.int32, device="cuda")
    sl = torch.zeros(0, dtype=torch.int32, device="cuda")
    ag.attn_decode_paged(q, kc, kc, q.clone(), bt, sl)
    ag.attn_release_workspace()


@pytest.mark.parametrize("pps", [None, 4])
def test_split_of_negative_block_ids_contributes_nothing(pps):
    # sequence 0: pages 4..7 (one whole split at 4 pages per split) hold -1;
    # sequence 1: every page holds -1; sequence 2 is clean.  The skipped pages
    # drop out of the softmax, so the result is the oracle's over the pages
    # that remain (listed contiguously in a compacted table).
    lens = [315, 100, 500]
    inp = make(len(lens), 16, 8, lens, max_blocks=32, seed=13)
    bt = inp.block_tables.copy()
    bt[0, 4:8] = -1
    bt[1, :7] = -1
    out = run_decode(W.DecodeInputs(inp.q, inp.k_cache, inp.v_cache, bt, inp.seq_lens),
                     pages_per_split=pps)
    assert ag.attn_get_device_error(reset=True) == 2
    keep0 = [p for p in range(20) if not 4 <= p < 8]
    ct = np.full_like(bt, -1)
    ct[0, :len(keep0)] = inp.block_tables[0, keep0]
    ct[2] = inp.block_tables[2]
    cl = np.array([315 - 64, 0, 500], np.int32)
    ref = oracle.decode_paged(inp.q, inp.k_cache, inp.v_cache, ct, cl)
    assert np.all(out[1] == 0)
    assert_close(out, ref, f"negative-id split, pages_per_split={pps}")


def test_many_sequences_short_contexts():
    # 4096 sequences of 0..64 tokens: a grid of 8192 CTAs, most splits past the context
    lens = W.uniform_int(79, 3, 4096, 0, 64)
    inp = make(len(lens), 16, 8, lens, max_blocks=8, seed=79)
    out = run_decode(inp)
    assert np.all(out[np.asarray(lens) == 0] == 0)
    assert_close(out, oracle_decode(inp), "4096 short sequences")
    assert device_error_clean()
