"""GPU parity of the attention-input prologue (QK-norm, NeoX RoPE, KV append)
against the FP64 oracle.

Tolerance: the outputs are single FP16 roundings of FP32 arithmetic, so each
element must lie within half an FP16 ulp of the exact value plus the FP32
error: |gpu - ref| <= 2^-11 |ref| + 2e-6 * (largest |ref| of its row) + 2^-25.
Besides the bound, at least 99 % of the elements must equal the oracle's value
rounded to FP16 (the rest sit next to a rounding tie)."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import oracle
import workloads as W
from gpu_util import assert_close, dev, device_error_clean, host, rope_table_entries
from test_oracle_pins import _paged_problem

pytestmark = pytest.mark.gpu

BASE = 1.0e6
EPS = 1e-6


def table(max_pos, base=BASE):
    cs = torch.empty((max_pos, 128), dtype=torch.float32, device="cuda")
    ag.attn_rope_cos_sin_table(cs, base)
    return cs


def assert_rounded(gpu, ref, what):
    gpu = gpu.astype(np.float64)
    assert np.isfinite(gpu).all(), f"{what}: non-finite"
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    bound = 2.0 ** -11 * np.abs(ref) + 2e-6 * scale + 2.0 ** -25
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside the rounding bound, worst " \
        f"{float((np.abs(gpu - ref) - bound).max()):.3e}"
    exact = np.mean(gpu == ref.astype(np.float16).astype(np.float64))
    assert exact >= 0.99, f"{what}: only {exact:.4f} of elements equal the rounded oracle value"


def rand_weights(rng, D=128):
    return rng.uniform(0.5, 1.5, D).astype(np.float16)


def test_table_matches_fp64_cos_sin():
    max_pos = 70000
    c, s = (host(x).astype(np.float64) for x in rope_table_entries(table(max_pos)))
    p = np.arange(max_pos, dtype=np.float64)[:, None]
    a = p * BASE ** (-2.0 * np.arange(64) / 128)
    # one rounding of the exact value to FP32 (relative 2^-24, |cos|,|sin| <= 1)
    assert np.abs(c - np.cos(a)).max() <= 2.0 ** -24
    assert np.abs(s - np.sin(a)).max() <= 2.0 ** -24


@pytest.mark.parametrize("heads", [(32, 8), (16, 8), (3, 1), (5, 7)])
def test_in_place_matches_oracle(heads):
    H_q, H_kv = heads
    rng = np.random.default_rng(80 + H_q)
    T = 777                                          # a ragged tail for the row grid
    Q = (rng.standard_normal((T, H_q, 128)) * 2).astype(np.float16)
    K = (rng.standard_normal((T, H_kv, 128)) * 0.3).astype(np.float16)
    qw, kw = rand_weights(rng), rand_weights(rng)
    pos = rng.integers(0, 60000, T).astype(np.int32)
    dQ, dK = dev(Q), dev(K)
    ag.attn_qk_norm_rope(dQ, dK, dev(qw), dev(kw), table(60000), dev(pos), eps=EPS)
    torch.cuda.synchronize()
    assert_rounded(host(dQ), oracle.qk_norm_rope(Q, qw, pos, BASE, EPS), f"Q {heads}")
    assert_rounded(host(dK), oracle.qk_norm_rope(K, kw, pos, BASE, EPS), f"K {heads}")
    assert device_error_clean()


def test_rope_only_and_mixed_weights():
    rng = np.random.default_rng(81)
    T, H_q, H_kv = 300, 8, 2
    Q = rng.standard_normal((T, H_q, 128)).astype(np.float16)
    K = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    kw = rand_weights(rng)
    pos = rng.integers(0, 5000, T).astype(np.int32)
    dQ, dK = dev(Q), dev(K)
    ag.attn_qk_norm_rope(dQ, dK, None, dev(kw), table(5000), dev(pos))
    torch.cuda.synchronize()
    assert_rounded(host(dQ), oracle.qk_norm_rope(Q, None, pos, BASE), "RoPE only")
    assert_rounded(host(dK), oracle.qk_norm_rope(K, kw, pos, BASE, EPS), "norm + RoPE")


def test_position_zero_and_small_and_large_rows():
    rng = np.random.default_rng(82)
    T, H = 64, 4
    Q = rng.standard_normal((T, H, 128)).astype(np.float16)
    Q[:16] *= np.float16(1e-3)                       # rows where eps matters
    Q[16:32] *= np.float16(200.0)                    # large rows: sum of squares in FP32
    Q[40] = 0                                        # an all-zero row stays zero
    K = rng.standard_normal((T, 1, 128)).astype(np.float16)
    w = rand_weights(rng)
    pos = np.zeros(T, np.int32)
    pos[32:] = rng.integers(0, 100, T - 32)
    dQ = dev(Q)
    ag.attn_qk_norm_rope(dQ, dev(K), dev(w), dev(w), table(128), dev(pos), eps=EPS)
    torch.cuda.synchronize()
    out = host(dQ)
    assert_rounded(out, oracle.qk_norm_rope(Q, w, pos, BASE, EPS), "edge rows")
    assert np.all(out[40] == 0)


def test_bad_positions_skip_the_token():
    rng = np.random.default_rng(83)
    T, H_q, H_kv, max_pos = 40, 4, 2, 1000
    Q = rng.standard_normal((T, H_q, 128)).astype(np.float16)
    K = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    pos = rng.integers(0, max_pos, T).astype(np.int32)
    pos[[3, 17]] = [max_pos, -1]
    dQ, dK = dev(Q), dev(K)
    ag.attn_qk_norm_rope(dQ, dK, None, None, table(max_pos), dev(pos))
    torch.cuda.synchronize()
    assert ag.attn_get_device_error(reset=True) == 128
    out_q, out_k = host(dQ), host(dK)
    ok = np.setdiff1d(np.arange(T), [3, 17])
    assert np.array_equal(out_q[[3, 17]].view(np.uint16), Q[[3, 17]].view(np.uint16))
    assert np.array_equal(out_k[[3, 17]].view(np.uint16), K[[3, 17]].view(np.uint16))
    assert_rounded(out_q[ok], oracle.qk_norm_rope(Q[ok], None, pos[ok], BASE), "good tokens")


def _append_case(rng, T, H_q, H_kv, nb, max_pos):
    Q = rng.standard_normal((T, H_q, 128)).astype(np.float16)
    K = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    V = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    qw, kw = rand_weights(rng), rand_weights(rng)
    pos = rng.integers(0, max_pos, T).astype(np.int32)
    slots = rng.choice(nb * 16, T, replace=False).astype(np.int64)
    return Q, K, V, qw, kw, pos, slots


def test_append_writes_rotated_k_and_raw_v_to_slots():
    rng = np.random.default_rng(84)
    T, H_q, H_kv, nb, max_pos = 333, 16, 8, 40, 4096
    Q, K, V, qw, kw, pos, slots = _append_case(rng, T, H_q, H_kv, nb, max_pos)
    slots[[5, 6]] = -1                               # padding tokens: cache untouched
    slots[9] = nb * 16 + 1                           # out of range: flagged, skipped
    kc = np.full((nb, H_kv, 16, 128), np.nan, np.float16)
    vc = kc.copy()
    dQ, dK, dV, dkc, dvc = dev(Q), dev(K), dev(V), dev(kc), dev(vc)
    ag.attn_qk_norm_rope_append(dQ, dK, dV, dev(qw), dev(kw), table(max_pos), dev(pos), dev(slots),
                                dkc, dvc, eps=EPS)
    torch.cuda.synchronize()
    assert ag.attn_get_device_error(reset=True) == 32
    assert_rounded(host(dQ), oracle.qk_norm_rope(Q, qw, pos, BASE, EPS), "Q in place")
    assert np.array_equal(host(dK).view(np.uint16), K.view(np.uint16))   # K itself is only read
    ok = (slots >= 0) & (slots < nb * 16)
    gk, gv = host(dkc), host(dvc)
    kref = oracle.qk_norm_rope(K[ok], kw, pos[ok], BASE, EPS)
    s = slots[ok]
    assert_rounded(gk[s // 16, :, s % 16, :], kref, "K in the cache")
    assert np.array_equal(gv[s // 16, :, s % 16, :].view(np.uint16), V[ok].view(np.uint16))
    # every other slot keeps its NaN
    mask = np.ones((nb * 16,), bool)
    mask[s] = False
    rest = np.nonzero(mask)[0]
    assert np.isnan(gk[rest // 16, :, rest % 16, :].astype(np.float32)).all()
    assert np.isnan(gv[rest // 16, :, rest % 16, :].astype(np.float32)).all()


def test_prologue_then_chunked_prefill_matches_oracle_chain():
    """A layer's attention step in the pages' order: QK-norm -> RoPE -> KV append
    -> attention, for chunks after cached prefixes (the prefix keys are already
    in the cache; only the chunk's own keys pass through the prologue)."""
    rng = np.random.default_rng(85)
    H_q, H_kv = 16, 4
    lens_q, prefix = [100, 257, 1], [300, 0, 77]
    lens_kv = [q + p for q, p in zip(lens_q, prefix)]
    _, _, kc, vc, table_b, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q, H_q, H_kv, 128,
                                                       nan_unused=False)
    T = int(cu[-1])
    Knew = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    Vnew = rng.standard_normal((T, H_kv, 128)).astype(np.float16)
    qw, kw = rand_weights(rng), rand_weights(rng)
    pos = np.concatenate([np.arange(p, p + q) for p, q in zip(prefix, lens_q)]).astype(np.int32)
    slots = np.concatenate([
        table_b[b, (pos[cu[b]:cu[b + 1]] // 16)].astype(np.int64) * 16 + pos[cu[b]:cu[b + 1]] % 16
        for b in range(len(lens_q))])
    dQ, dkc, dvc = dev(Q), dev(kc), dev(vc)
    ag.attn_qk_norm_rope_append(dQ, dev(Knew), dev(Vnew), dev(qw), dev(kw), table(2048), dev(pos),
                                dev(slots), dkc, dvc, eps=EPS)
    O = torch.empty_like(dQ)
    ag.attn_prefill_paged(dQ, dkc, dvc, O, dev(cu), dev(skv), dev(table_b), max(lens_q))
    torch.cuda.synchronize()
    # the oracle chain: prologue in FP64, rounded to the FP16 the cache holds
    q_r = oracle.qk_norm_rope(Q, qw, pos, BASE, EPS).astype(np.float16)
    k_r = oracle.qk_norm_rope(Knew, kw, pos, BASE, EPS).astype(np.float16)
    kc2, vc2, bad = oracle.kv_append(k_r, Vnew, kc, vc, slots)
    assert bad == 0
    ref = oracle.prefill_paged(q_r, kc2, vc2, cu, skv, table_b)
    assert_close(host(O), ref, "prologue + chunked prefill")
    assert device_error_clean()


def test_prologue_then_decode_step():
    cfg = W.DecodeConfig("t", 24, 16, 8, max_blocks_per_seq=40)
    inp = W.decode_inputs(cfg, seed=86, seq_lens=W.uniform_int(86, 3, 24, 1, 600))
    rng = np.random.default_rng(86)
    N = cfg.num_seqs
    Ls = inp.seq_lens.astype(np.int64)
    pos = (Ls - 1).astype(np.int32)                  # the new token is the last of each sequence
    slots = inp.block_tables[np.arange(N), (Ls - 1) // 16].astype(np.int64) * 16 + (Ls - 1) % 16
    kn = rng.standard_normal((N, 8, 128)).astype(np.float16)
    vn = rng.standard_normal((N, 8, 128)).astype(np.float16)
    qw, kw = rand_weights(rng), rand_weights(rng)
    dq, dkc, dvc = dev(inp.q), dev(inp.k_cache), dev(inp.v_cache)
    ag.attn_qk_norm_rope_append(dq, dev(kn), dev(vn), dev(qw), dev(kw), table(1024), dev(pos),
                                dev(slots), dkc, dvc, eps=EPS)
    out = torch.empty_like(dq)
    ag.attn_decode_paged(dq, dkc, dvc, out, dev(inp.block_tables), dev(inp.seq_lens))
    torch.cuda.synchronize()
    q_r = oracle.qk_norm_rope(inp.q, qw, pos, BASE, EPS).astype(np.float16)
    k_r = oracle.qk_norm_rope(kn, kw, pos, BASE, EPS).astype(np.float16)
    kc2, vc2, _ = oracle.kv_append(k_r, vn, inp.k_cache, inp.v_cache, slots)
    ref = oracle.decode_paged(q_r, kc2, vc2, inp.block_tables, inp.seq_lens)
    assert_close(host(out), ref, "prologue + decode")


def test_bench_workload_sampled():
    """The benchmark's prologue (2 x 8192 tokens, H 32/8) in the launch the
    bench times; sampled tokens (and the first and last of each sequence)
    checked against the oracle."""
    cfg = W.PROLOGUE
    Q, K, V, qw, kw, pos, slots, nb = W.prologue_inputs(cfg, seed=0)
    kc = torch.zeros((nb, cfg.H_kv, 16, 128), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    dQ = dev(Q)
    ag.attn_qk_norm_rope_append(dQ, dev(K), dev(V), dev(qw), dev(kw), table(cfg.seq_len, cfg.base),
                                dev(pos), dev(slots), kc, vc, eps=EPS)
    torch.cuda.synchronize()
    assert device_error_clean()
    pick = np.sort(np.random.default_rng(87).choice(cfg.tokens, 512, replace=False))
    pick = np.union1d(pick, [0, cfg.seq_len - 1, cfg.seq_len, cfg.tokens - 1])
    out_q = host(dQ)[pick]
    assert_rounded(out_q, oracle.qk_norm_rope(Q[pick], qw, pos[pick], cfg.base, EPS), "Q sample")
    s = slots[pick]
    gk = host(kc)[s // 16, :, s % 16, :]
    gv = host(vc)[s // 16, :, s % 16, :]
    assert_rounded(gk, oracle.qk_norm_rope(K[pick], kw, pos[pick], cfg.base, EPS), "K sample")
    assert np.array_equal(gv.view(np.uint16), V[pick].view(np.uint16))


def test_append_at_the_row_limit():
    # H_q + 2 * H_kv = 192 rows per token: the most one token may stage
    rng = np.random.default_rng(88)
    T, H_q, H_kv, nb, max_pos = 37, 96, 48, 4, 500
    Q, K, V, qw, kw, pos, slots = _append_case(rng, T, H_q, H_kv, nb, max_pos)
    kc = torch.zeros((nb, H_kv, 16, 128), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    dQ = dev(Q)
    ag.attn_qk_norm_rope_append(dQ, dev(K), dev(V), dev(qw), dev(kw), table(max_pos), dev(pos),
                                dev(slots), kc, vc, eps=EPS)
    torch.cuda.synchronize()
    assert device_error_clean()
    assert_rounded(host(dQ), oracle.qk_norm_rope(Q, qw, pos, BASE, EPS), "Q at the row limit")
    gk, gv = host(kc), host(vc)
    assert_rounded(gk[slots // 16, :, slots % 16, :], oracle.qk_norm_rope(K, kw, pos, BASE, EPS), "K")
    assert np.array_equal(gv[slots // 16, :, slots % 16, :].view(np.uint16), V.view(np.uint16))
