"""GPU parity of attn_prefill (called through the C ABI) against the FP64 oracle.

Covers the pages' own test shapes, the small and Qwen3-shaped workloads in
full, the long workload (B=2, S=8192, H 32/8, causal and full) on sampled rows
with the launch configuration the benchmark times, ragged sequence lengths
around the 128-row tiles, group sizes 1..8 (even groups pair heads in a CTA,
odd ones pair row tiles), and the closed-form invariants."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import golden_cases
import oracle
import workloads as W
from gpu_util import assert_close, dev, device_error_clean, host

pytestmark = pytest.mark.gpu


def run_prefill(Q, K, V, causal=True):
    O = torch.empty(Q.shape, dtype=torch.float16, device="cuda")
    ag.attn_prefill(dev(Q), dev(K), dev(V), O, causal=causal)
    torch.cuda.synchronize()
    return host(O)


def rand_inputs(B, S, H_q, H_kv, seed):
    cfg = W.PrefillConfig("t", B, S, H_q, H_kv)
    return W.prefill_inputs(cfg, seed=seed)


@pytest.mark.parametrize("case", golden_cases.load()[0])
def test_page_prefill_cases(case):
    B, S, H_q, H_kv, D = case
    Q, K, V = rand_inputs(B, S, H_q, H_kv, seed=S)
    assert_close(run_prefill(Q, K, V), oracle.prefill(Q, K, V), f"page case {case}")
    assert device_error_clean()


def test_small_workload_seed0():
    cfg = W.PREFILL_SMALL
    Q, K, V = W.prefill_inputs(cfg, seed=0)
    assert_close(run_prefill(Q, K, V), oracle.prefill(Q, K, V), cfg.name)


@pytest.mark.parametrize("S", [1, 2, 17, 127, 128, 129, 255, 256, 300, 383, 513])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("heads", [(4, 2), (3, 3), (6, 2), (8, 1)])
def test_ragged_lengths_and_groups(S, causal, heads):
    H_q, H_kv = heads
    Q, K, V = rand_inputs(2, S, H_q, H_kv, seed=S * 7 + H_q)
    assert_close(run_prefill(Q, K, V, causal), oracle.prefill(Q, K, V, causal=causal),
                 f"S={S} causal={causal} heads={heads}")


def test_qwen_shape_full_compare():
    cfg = W.PREFILL_QWEN
    Q, K, V = W.prefill_inputs(cfg, seed=0)
    assert_close(run_prefill(Q, K, V), oracle.prefill(Q, K, V), cfg.name)
    assert device_error_clean()


def stratified_rows(B, S, H_q, seed, diag_blocks, diag_heads):
    """Rows (b, i, h) that reach every CTA of a full-size launch on both of its
    Q tiles: one random row in every (b, 128-row block, q head), plus every
    row of the listed 128-row blocks (diagonal tiles under the causal mask)
    for the listed heads of each batch entry."""
    rng = np.random.default_rng(seed)
    n_mb = (S + 127) // 128
    b, mb, h = np.meshgrid(np.arange(B), np.arange(n_mb), np.arange(H_q), indexing="ij")
    b, mb, h = b.ravel(), mb.ravel(), h.ravel()
    width = np.minimum(128, S - mb * 128)
    i = mb * 128 + (rng.random(b.size) * width).astype(np.int64)
    rows = [np.stack([b, i, h], 1)]
    for bb in range(B):
        for blk in diag_blocks:
            r = np.arange(blk * 128, min(S, blk * 128 + 128))
            for hh in diag_heads:
                rows.append(np.stack([np.full_like(r, bb), r, np.full_like(r, hh)], 1))
    return np.unique(np.concatenate(rows).astype(np.int32), axis=0)


@pytest.mark.parametrize("cfg", [W.PREFILL_LONG, W.PREFILL_LONG_FULL], ids=lambda c: c.name)
def test_long_workload_stratified_rows(cfg):
    # the launch the benchmark times (B 2, S 8192, H 32/8), every CTA checked
    Q, K, V = W.prefill_inputs(cfg, seed=0)
    O = torch.full(Q.shape, float("nan"), dtype=torch.float16, device="cuda")
    ag.attn_prefill(dev(Q), dev(K), dev(V), O, causal=cfg.causal)
    torch.cuda.synchronize()
    O = host(O)
    n_mb = cfg.S // 128
    rows = stratified_rows(cfg.B, cfg.S, cfg.H_q, seed=1, diag_blocks=(0, n_mb // 2, n_mb - 1),
                           diag_heads=(0, 13, cfg.H_q - 1))
    assert len(rows) >= cfg.B * n_mb * cfg.H_q
    ref = oracle.prefill_rows(Q, K, V, rows, causal=cfg.causal)
    got = O[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, ref, f"{cfg.name}: {len(rows)} stratified rows")
    assert np.isfinite(O.astype(np.float32)).all(), "rows left unwritten"
    assert device_error_clean()


def test_invariants_identical_v_row0_and_determinism():
    B, S, H_q, H_kv = 2, 300, 8, 2
    Q, K, V = rand_inputs(B, S, H_q, H_kv, seed=5)
    # identical V rows: the output is that row (to FP16 rounding of a weighted mean of equal values)
    Vc = np.broadcast_to(V[:, :1], V.shape).copy()
    O = run_prefill(Q, K, Vc)
    g = (np.arange(H_q) * H_kv) // H_q
    expect = np.broadcast_to(Vc[:, :1][:, :, g, :], O.shape).astype(np.float64)
    assert_close(O, expect, "identical V rows")
    # causal row 0 attends to V[0] alone (weight 1 up to the rounding of exp2 near 0)
    O = run_prefill(Q, K, V)
    assert_close(O[:, 0], V[:, 0][:, g].astype(np.float64), "causal row 0", max_abs=1e-3, mean_abs=1e-5)
    # identical K rows: causal row i is the mean of V[0..i]
    Kc = np.broadcast_to(K[:, :1], K.shape).copy()
    O = run_prefill(Q, Kc, V)
    Vd = V.astype(np.float64)
    means = np.cumsum(Vd, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    assert_close(O, means[:, :, g, :], "identical K rows")
    # run-to-run determinism
    a = run_prefill(Q, K, V)
    b = run_prefill(Q, K, V)
    assert np.array_equal(a, b)


def test_mha_equals_per_head():
    B, S, H = 1, 200, 3
    Q, K, V = rand_inputs(B, S, H, H, seed=9)
    O = run_prefill(Q, K, V)
    for h in range(H):
        Oh = run_prefill(Q[:, :, h:h + 1].copy(), K[:, :, h:h + 1].copy(), V[:, :, h:h + 1].copy())
        assert np.array_equal(O[:, :, h:h + 1], Oh)


def test_empty_problem_is_noop():
    Q = torch.zeros(1, 0, 4, 128, dtype=torch.float16, device="cuda")
    K = torch.zeros(1, 0, 2, 128, dtype=torch.float16, device="cuda")
    ag.attn_prefill(Q, K, K, Q.clone())
    torch.cuda.synchronize()


def test_unsupported_head_dim_raises():
    Q = torch.zeros(1, 8, 2, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(ag.AttnError) as e:
        ag.attn_prefill(Q, Q[:, :, :1].contiguous(), Q[:, :, :1].contiguous(), Q.clone())
    assert e.value.status == ag.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("heads", [(32, 2), (15, 3), (48, 4), (64, 64)])
def test_wide_groups_and_many_heads(causal, heads):
    # group 16 and 12 (head pairs), group 5 (odd: row pairs), and 64-head MHA
    H_q, H_kv = heads
    S = 333
    Q, K, V = rand_inputs(1, S, H_q, H_kv, seed=H_q * 31 + H_kv)
    assert_close(run_prefill(Q, K, V, causal), oracle.prefill(Q, K, V, causal=causal),
                 f"S={S} causal={causal} heads={heads}")
    assert device_error_clean()


def test_long_single_sequence_stratified():
    # the largest sequence here: S 32768, one batch entry, H 8/1 (group 8: head pairs)
    B, S, H_q, H_kv = 1, 32768, 8, 1
    Q, K, V = rand_inputs(B, S, H_q, H_kv, seed=77)
    O = torch.full(Q.shape, float("nan"), dtype=torch.float16, device="cuda")
    ag.attn_prefill(dev(Q), dev(K), dev(V), O, causal=True)
    torch.cuda.synchronize()
    O = host(O)
    assert np.isfinite(O.astype(np.float32)).all(), "rows left unwritten"
    rows = stratified_rows(B, S, H_q, seed=4, diag_blocks=(0, S // 128 - 1), diag_heads=(0, H_q - 1))
    ref = oracle.prefill_rows(Q, K, V, rows, causal=True)
    assert_close(O[rows[:, 0], rows[:, 1], rows[:, 2]], ref, f"S={S}: {len(rows)} stratified rows")
    assert device_error_clean()


@pytest.mark.parametrize("causal", [True, False])
def test_many_tiny_batches(causal):
    # 64 batch entries of 16 tokens: one ragged tile per CTA, 512 CTAs
    Q, K, V = rand_inputs(64, 16, 16, 8, seed=78)
    assert_close(run_prefill(Q, K, V, causal), oracle.prefill(Q, K, V, causal=causal), f"B=64 S=16 causal={causal}")
    assert device_error_clean()
