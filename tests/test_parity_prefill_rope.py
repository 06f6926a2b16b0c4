"""GPU parity of attn_prefill_paged_qk_norm_rope -- the chunked prefill with the
query side of the attention-input prologue (per-head QK-norm, then NeoX RoPE at
each query's position) folded into the kernel's Q load -- against the FP64
oracle chain in the pages' layer order: QK-norm -> RoPE (queries and keys in
FP64, rounded to the FP16 the kernels hold) -> KV append -> paged prefill.

The keys go through the keys-only form of attn_qk_norm_rope_append (Q = NULL).
Covers even (head-paired) and odd (row-paired) GQA groups, causal and full,
with and without the norm weight, ragged chunks after cached prefixes, the
benchmark's chunked workload at full size on stratified rows, that Q is only
read, agreement with the unfused two-call path, and positions outside the
cos/sin table (flagged, left unrotated)."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import oracle
import workloads as W
from gpu_util import assert_close, dev, device_error_clean, host
from test_oracle_pins import _paged_problem
from test_parity_prefill import stratified_rows
from test_parity_prologue import BASE, EPS, rand_weights, table

pytestmark = pytest.mark.gpu


def _layer(seed, lens_q, prefix, H_q, H_kv):
    """Cached prefixes already in the cache (rotated keys, as a previous step
    left them), the chunk's raw q, k, v, norm weights, positions and slots."""
    rng = np.random.default_rng(seed)
    lens_kv = [q + p for q, p in zip(lens_q, prefix)]
    _, _, kc, vc, tb, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q, H_q, H_kv, 128, nan_unused=False)
    T = int(cu[-1])
    Knew = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    Vnew = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    qw, kw = rand_weights(rng), rand_weights(rng)
    pos = np.concatenate([np.arange(p, p + q) for p, q in zip(prefix, lens_q)]).astype(np.int32)
    slots = np.concatenate([tb[b, pos[cu[b]:cu[b + 1]] // 16].astype(np.int64) * 16 + pos[cu[b]:cu[b + 1]] % 16
                            for b in range(len(lens_q))])
    return dict(Q=Q, kc=kc, vc=vc, tb=tb, cu=cu, skv=skv, Knew=Knew, Vnew=Vnew, qw=qw, kw=kw, pos=pos,
                slots=slots, max_q=max(lens_q), H_q=H_q)


def run_fused(L, causal=True, norm=True, max_pos=4096):
    dQ, dkc, dvc = dev(L["Q"]), dev(L["kc"]), dev(L["vc"])
    tab = table(max_pos)
    ag.attn_qk_norm_rope_append(None, dev(L["Knew"]), dev(L["Vnew"]), None,
                                dev(L["kw"]) if norm else None, tab, dev(L["pos"]), dev(L["slots"]),
                                dkc, dvc, eps=EPS, H_q=L["H_q"])
    O = torch.full_like(dQ, float("nan"))
    ag.attn_prefill_paged_qk_norm_rope(dQ, dkc, dvc, O, dev(L["cu"]), dev(L["skv"]), dev(L["tb"]),
                                       dev(L["qw"]) if norm else None, tab, L["max_q"], eps=EPS,
                                       causal=causal)
    torch.cuda.synchronize()
    return host(O), host(dQ)


def oracle_chain(L, causal=True, norm=True):
    qw = L["qw"] if norm else None
    kw = L["kw"] if norm else None
    q_r = oracle.qk_norm_rope(L["Q"], qw, L["pos"], BASE, EPS).astype(np.float16)
    k_r = oracle.qk_norm_rope(L["Knew"], kw, L["pos"], BASE, EPS).astype(np.float16)
    kc2, vc2, bad = oracle.kv_append(k_r, L["Vnew"], L["kc"], L["vc"], L["slots"])
    assert bad == 0
    return oracle.prefill_paged(q_r, kc2, vc2, L["cu"], L["skv"], L["tb"], causal=causal)


@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("heads", [(16, 4), (32, 8), (6, 2), (5, 5)])
def test_fused_query_prologue_matches_oracle_chain(heads, causal, norm):
    H_q, H_kv = heads
    L = _layer(90 + H_q, [100, 257, 1, 130], [300, 0, 77, 1000], H_q, H_kv)
    out, q_after = run_fused(L, causal, norm)
    assert np.array_equal(q_after.view(np.uint16), L["Q"].view(np.uint16)), "Q was modified"
    assert_close(out, oracle_chain(L, causal, norm), f"fused prologue heads={heads} causal={causal} norm={norm}")
    assert device_error_clean()


def test_fused_equals_unfused_two_call_path():
    # the same layer step through attn_qk_norm_rope_append (queries rotated in
    # place) and attn_prefill_paged: only the FP32 order of the sum of squares
    # differs, so the outputs agree far inside the oracle tolerance
    L = _layer(95, [512, 333, 64], [1024, 2000, 5], 32, 8)
    fused, _ = run_fused(L)
    dQ, dkc, dvc = dev(L["Q"]), dev(L["kc"]), dev(L["vc"])
    tab = table(4096)
    ag.attn_qk_norm_rope_append(dQ, dev(L["Knew"]), dev(L["Vnew"]), dev(L["qw"]), dev(L["kw"]), tab,
                                dev(L["pos"]), dev(L["slots"]), dkc, dvc, eps=EPS)
    O = torch.empty_like(dQ)
    ag.attn_prefill_paged(dQ, dkc, dvc, O, dev(L["cu"]), dev(L["skv"]), dev(L["tb"]), L["max_q"])
    torch.cuda.synchronize()
    d = np.abs(fused.astype(np.float64) - host(O).astype(np.float64))
    assert d.max() <= 2e-3 and d.mean() <= 5e-5, f"fused vs unfused: max {d.max():.2e} mean {d.mean():.2e}"


@pytest.mark.parametrize("causal", [True, False])
def test_bench_workload_stratified(causal):
    # the benchmark's chunked workload (4 x (6144 cached + 2048 new), H 32/8) with
    # raw queries: every CTA of the launch checked on stratified rows
    cfg = W.CHUNKED_PREFILL
    Q, kc, vc, cu, skv, tb = W.chunked_prefill_inputs(cfg, seed=0)
    qw = (1.0 + 0.25 * W.normal_fp16(0, 13, (128,)).astype(np.float32)).astype(np.float16)
    O = torch.full(Q.shape, float("nan"), dtype=torch.float16, device="cuda")
    ag.attn_prefill_paged_qk_norm_rope(dev(Q), dev(kc), dev(vc), O, dev(cu), dev(skv), dev(tb), dev(qw),
                                       table(cfg.prefix + cfg.chunk), cfg.chunk, eps=EPS, causal=causal)
    torch.cuda.synchronize()
    O = host(O)
    assert np.isfinite(O.astype(np.float32)).all(), "rows left unwritten"
    pos = np.tile(np.arange(cfg.prefix, cfg.prefix + cfg.chunk, dtype=np.int32), cfg.num_seqs)
    q_r = oracle.qk_norm_rope(Q, qw, pos, BASE, EPS).astype(np.float16)
    rows = stratified_rows(cfg.num_seqs, cfg.chunk, cfg.H_q, seed=3, diag_blocks=(0, cfg.chunk // 128 - 1),
                           diag_heads=(0, cfg.H_q - 1))
    ref = oracle.prefill_paged_rows(q_r, kc, vc, cu, skv, tb, rows, causal=causal)
    assert_close(O[cu[rows[:, 0]] + rows[:, 1], rows[:, 2]], ref, f"{cfg.name} fused prologue causal={causal}")
    assert device_error_clean()


def test_positions_outside_the_table_are_flagged_and_left_unrotated():
    # context 300 + 100: positions 300..399, but the table has 350 positions
    L = _layer(96, [100], [300], 8, 2)
    out, _ = run_fused(L, max_pos=350)
    assert ag.attn_get_device_error(reset=True) & 128
    good = L["pos"] < 350
    ref = oracle_chain(L)
    assert_close(out[good], ref[good], "rows inside the table")
    # Rows past the table attend with their raw query.  The append skipped the
    # tokens past the table too (flagged), so their cache slots keep what they held.
    k_r = oracle.qk_norm_rope(L["Knew"], L["kw"], L["pos"], BASE, EPS).astype(np.float16)
    kc2, vc2, _ = oracle.kv_append(k_r[good], L["Vnew"][good], L["kc"], L["vc"], L["slots"][good])
    raw = oracle.prefill_paged(L["Q"], kc2, vc2, L["cu"], L["skv"], L["tb"])
    assert_close(out[~good], raw[~good], "rows past the table, unrotated")
