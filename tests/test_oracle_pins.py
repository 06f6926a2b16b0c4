"""Pins for the FP64 oracle against things other than itself (CPU only).

Each check is chosen so that a plausible slip in the oracle (a wrong GQA head
map, a dropped 1/sqrt(D), an off-by-one causal bound, a transposed operand, a
wrong page index) fails at least one of them:

* a library special case: torch float64 ``scaled_dot_product_attention`` with
  ``enable_gqa`` (its K/V heads are repeat-interleaved, i.e. q head h uses kv
  head h // (H_q/H_kv) = floor(h*H_kv/H_q));
* closed forms: identical V rows, identical K rows (mean of the allowed V
  rows), causal row 0, zero keys (lse = ln n), a one-hot query against a
  large-margin key;
* invariants: paged == contiguous, decode == last prefill row, block-table
  permutation, splitting the keys and merging by lse.

Sources of the definitions: "Tutorial: Adding a New Kernel to RL.cu"
(add-cuda-kernel page), include/kernels/attention.cuh and
tests/test_attention.cu (reference attention, scale 1/sqrt(D), causal j <= i,
GQA map, paged layout); the Kimi-K2.6 KernelBench trace for the online-softmax
identity that the lse merge relies on.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W


def _rand16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def _sdpa(Q, K, V, causal):
    # [B,S,H,D] -> [B,H,S,D], float64 on CPU
    q = torch.from_numpy(Q.astype(np.float64)).permute(0, 2, 1, 3)
    k = torch.from_numpy(K.astype(np.float64)).permute(0, 2, 1, 3)
    v = torch.from_numpy(V.astype(np.float64)).permute(0, 2, 1, 3)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=causal, enable_gqa=True)
    return o.permute(0, 2, 1, 3).numpy()


def test_half_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


SHAPES = [  # (B, S, H_q, H_kv, D)
    (1, 16, 2, 1, 128),   # first prefill case of the page's test file
    (2, 7, 4, 2, 4),
    (1, 9, 6, 3, 8),
    (1, 5, 4, 4, 16),     # H_kv == H_q (MHA)
    (2, 11, 8, 2, 32),    # 4:1 groups
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_matches_torch_sdpa_float64(shape, causal):
    B, S, H_q, H_kv, D = shape
    rng = np.random.default_rng(1234 + S)
    Q, K, V = _rand16(rng, (B, S, H_q, D)), _rand16(rng, (B, S, H_kv, D)), _rand16(rng, (B, S, H_kv, D))
    O = oracle.prefill(Q, K, V, causal=causal)
    ref = _sdpa(Q, K, V, causal)
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


def test_prefill_gqa_map_distinguishes_groups():
    # each kv head's V is a constant vector equal to its index: O row = g(h)
    B, S, H_q, H_kv, D = 1, 6, 8, 2, 4
    rng = np.random.default_rng(7)
    Q, K = _rand16(rng, (B, S, H_q, D)), _rand16(rng, (B, S, H_kv, D))
    V = np.zeros((B, S, H_kv, D), np.float16)
    for g in range(H_kv):
        V[:, :, g, :] = g + 1
    O = oracle.prefill(Q, K, V, causal=True)
    for h in range(H_q):
        np.testing.assert_allclose(O[:, :, h, :], (h * H_kv) // H_q + 1, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_identical_v_rows_give_that_row(causal):
    B, S, H_q, H_kv, D = 2, 13, 4, 2, 16
    rng = np.random.default_rng(3)
    Q, K = _rand16(rng, (B, S, H_q, D), 2.0), _rand16(rng, (B, S, H_kv, D), 2.0)
    row = _rand16(rng, (B, 1, H_kv, D))
    V = np.broadcast_to(row, (B, S, H_kv, D)).copy()
    O = oracle.prefill(Q, K, V, causal=causal)
    g = (np.arange(H_q) * H_kv) // H_q
    expect = np.broadcast_to(row[:, :, g, :].astype(np.float64), O.shape)
    np.testing.assert_allclose(O, expect, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_identical_k_rows_give_mean_of_allowed_v(causal):
    B, S, H_q, H_kv, D = 1, 12, 4, 2, 8
    rng = np.random.default_rng(4)
    Q = _rand16(rng, (B, S, H_q, D))
    krow = _rand16(rng, (B, 1, H_kv, D))
    K = np.broadcast_to(krow, (B, S, H_kv, D)).copy()
    V = _rand16(rng, (B, S, H_kv, D))
    O, lse = oracle.prefill(Q, K, V, causal=causal, with_lse=True)
    Vd = V.astype(np.float64)
    for h in range(H_q):
        g = h * H_kv // H_q
        for i in range(S):
            n = i + 1 if causal else S
            np.testing.assert_allclose(O[0, i, h], Vd[0, :n, g].mean(axis=0), atol=1e-14)
            s = float(np.dot(Q[0, i, h].astype(np.float64), krow[0, 0, g].astype(np.float64))) / math.sqrt(D)
            assert abs(lse[0, i, h] - (s + math.log(n))) < 1e-12


def test_causal_row0_is_v0_and_zero_keys_lse():
    B, S, H_q, H_kv, D = 2, 9, 4, 1, 128
    rng = np.random.default_rng(5)
    Q, K, V = _rand16(rng, (B, S, H_q, D), 3.0), _rand16(rng, (B, S, H_kv, D), 3.0), _rand16(rng, (B, S, H_kv, D))
    O = oracle.prefill(Q, K, V, causal=True)
    for h in range(H_q):
        assert np.array_equal(O[:, 0, h], V[:, 0, 0].astype(np.float64))
    Kz = np.zeros_like(K)
    _, lse = oracle.prefill(Q, Kz, V, causal=True, with_lse=True)
    np.testing.assert_allclose(lse[0, :, 0], np.log(np.arange(1, S + 1)), atol=1e-14)
    _, lse = oracle.prefill(Q, Kz, V, causal=False, with_lse=True)
    np.testing.assert_allclose(lse, math.log(S), atol=1e-14)


def test_one_hot_query_selects_large_margin_key():
    # q = c*e_0, key j* has k[0] = 1 and the others 0: weight of j* is
    # 1 / (1 + (n-1) e^{-c/sqrt(D)}); with c/sqrt(D) = 64 it is 1 to 1e-27.
    B, S, H_q, H_kv, D = 1, 8, 2, 1, 4
    Q = np.zeros((B, S, H_q, D), np.float16)
    Q[..., 0] = 128.0
    K = np.zeros((B, S, H_kv, D), np.float16)
    K[0, 3, 0, 0] = 1.0
    rng = np.random.default_rng(6)
    V = _rand16(rng, (B, S, H_kv, D))
    O = oracle.prefill(Q, K, V, causal=False)
    np.testing.assert_allclose(O[0, :, 0], np.broadcast_to(V[0, 3, 0].astype(np.float64), (S, D)), atol=1e-20)
    # causal rows before the key cannot see it: uniform mean over their prefix
    O = oracle.prefill(Q, K, V, causal=True)
    np.testing.assert_allclose(O[0, 2, 1], V[0, :3, 0].astype(np.float64).mean(0), atol=1e-15)


def test_mha_heads_independent():
    B, S, H, D = 1, 10, 3, 16
    rng = np.random.default_rng(8)
    Q, K, V = _rand16(rng, (B, S, H, D)), _rand16(rng, (B, S, H, D)), _rand16(rng, (B, S, H, D))
    O = oracle.prefill(Q, K, V)
    for h in range(H):
        Oh = oracle.prefill(Q[:, :, h:h + 1].copy(), K[:, :, h:h + 1].copy(), V[:, :, h:h + 1].copy())
        assert np.array_equal(O[:, :, h:h + 1], Oh)


def test_prefill_rows_equal_full():
    B, S, H_q, H_kv, D = 2, 20, 4, 2, 32
    rng = np.random.default_rng(9)
    Q, K, V = _rand16(rng, (B, S, H_q, D)), _rand16(rng, (B, S, H_kv, D)), _rand16(rng, (B, S, H_kv, D))
    for causal in (True, False):
        O, lse = oracle.prefill(Q, K, V, causal=causal, with_lse=True)
        rows = [(1, 19, 3), (0, 0, 0), (1, 7, 2), (0, 13, 1)]
        Or, lr = oracle.prefill_rows(Q, K, V, rows, causal=causal, with_lse=True)
        for r, (b, i, h) in enumerate(rows):
            assert np.array_equal(Or[r], O[b, i, h]) and lr[r] == lse[b, i, h]


def test_thread_count_does_not_change_results():
    # every output row is one independent loop: one thread or many, same bits
    B, S, H_q, H_kv, D = 1, 24, 4, 2, 16
    rng = np.random.default_rng(17)
    Q, K, V = _rand16(rng, (B, S, H_q, D)), _rand16(rng, (B, S, H_kv, D)), _rand16(rng, (B, S, H_kv, D))
    O, lse = oracle.prefill(Q, K, V, with_lse=True)
    before = oracle.num_threads()
    with oracle.threads(1):
        assert oracle.num_threads() == 1
        O1, lse1 = oracle.prefill(Q, K, V, with_lse=True)
    assert oracle.num_threads() == before
    assert np.array_equal(O, O1) and np.array_equal(lse, lse1)


# ------------------------------------------------------------------ decode

def _page(K, bs, perm):
    """Contiguous per-sequence K [N, L, H_kv, D] -> paged cache via perm of pages."""
    N, L, H_kv, D = K.shape
    npg = (L + bs - 1) // bs
    cache = np.full((N * npg, H_kv, bs, D), np.nan, np.float16)
    table = np.full((N, npg + 2), -1, np.int32)
    for n in range(N):
        for p in range(npg):
            phys = int(perm[n * npg + p])
            table[n, p] = phys
            t0, t1 = p * bs, min(L, (p + 1) * bs)
            cache[phys, :, : t1 - t0, :] = K[n, t0:t1].transpose(1, 0, 2)
    return cache, table


@pytest.mark.parametrize("bs", [16, 5])
def test_decode_paged_equals_last_prefill_row(bs):
    B, S, H_q, H_kv, D = 3, 37, 4, 2, 16
    rng = np.random.default_rng(10)
    Q, K, V = _rand16(rng, (B, S, H_q, D)), _rand16(rng, (B, S, H_kv, D)), _rand16(rng, (B, S, H_kv, D))
    O = oracle.prefill(Q, K, V, causal=True)
    perm = rng.permutation(B * ((S + bs - 1) // bs)).astype(np.int32)
    kc, table = _page(K, bs, perm)
    vc, _ = _page(V, bs, perm)
    out = oracle.decode_paged(Q[:, S - 1].copy(), kc, vc, table, np.full(B, S, np.int32))
    np.testing.assert_allclose(out, O[:, S - 1], rtol=0, atol=1e-14)
    # unused (NaN-poisoned) slots of the last page were never read
    assert np.isfinite(out).all()


def test_decode_matches_sdpa_on_gathered_keys_ragged():
    N, H_q, H_kv, D, bs = 4, 8, 2, 32, 16
    rng = np.random.default_rng(11)
    lens = np.array([1, 16, 17, 50], np.int32)
    tables, nb = W.decode_layout(lens, bs, 5, seed=3)
    kc, vc = _rand16(rng, (nb, H_kv, bs, D)), _rand16(rng, (nb, H_kv, bs, D))
    q = _rand16(rng, (N, H_q, D))
    out = oracle.decode_paged(q, kc, vc, tables, lens)
    for n in range(N):
        L = int(lens[n])
        t = np.arange(L)
        kk = kc[tables[n, t // bs], :, t % bs, :]  # [L, H_kv, D]
        vv = vc[tables[n, t // bs], :, t % bs, :]
        ref = _sdpa(q[n][None, None], kk[None], vv[None], causal=False)[0, 0]
        np.testing.assert_allclose(out[n], ref, atol=1e-12)


def test_decode_empty_sequence_gives_zero_and_neg_inf_lse():
    N, H_q, H_kv, D, bs = 2, 2, 1, 8, 16
    rng = np.random.default_rng(12)
    lens = np.array([0, 3], np.int32)
    tables = np.array([[-1], [0]], np.int32)
    kc, vc = _rand16(rng, (1, H_kv, bs, D)), _rand16(rng, (1, H_kv, bs, D))
    out, lse = oracle.decode_paged(_rand16(rng, (N, H_q, D)), kc, vc, tables, lens, with_lse=True)
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(lse[1]))


def test_decode_block_permutation_invariant_and_rows():
    cfg = W.DecodeConfig("t", 5, 4, 2, D=16, block_size=4, len_lo=1, len_hi=30, max_blocks_per_seq=8)
    inp = W.decode_inputs(cfg, seed=2)
    out = oracle.decode_paged(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.seq_lens)
    # move every physical block to a new place and rewrite the tables to match
    nb = inp.num_blocks
    p = np.random.default_rng(13).permutation(nb).astype(np.int32)
    kc2 = np.empty_like(inp.k_cache)
    vc2 = np.empty_like(inp.v_cache)
    kc2[p] = inp.k_cache
    vc2[p] = inp.v_cache
    bt2 = np.where(inp.block_tables >= 0, p[np.maximum(inp.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle.decode_paged(inp.q, kc2, vc2, bt2, inp.seq_lens)
    assert np.array_equal(out, out2)
    rows = [(4, 3), (0, 0), (2, 1)]
    orow = oracle.decode_paged_rows(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.seq_lens, rows)
    for r, (n, h) in enumerate(rows):
        assert np.array_equal(orow[r], out[n, h])


# ----------------------------------------------------------------- combine

def _segment_partials(q, Kseq, Vseq, cuts):
    """Oracle decode over each key segment [cuts[i], cuts[i+1]) of one sequence,
    each laid out as its own single-sequence paged problem (block size 1)."""
    H_q, D = q.shape
    H_kv = Kseq.shape[1]
    O_part, lse_part = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        L = b - a
        kc = Kseq[a:b][:, :, None, :].copy() if L else np.zeros((1, H_kv, 1, D), np.float16)
        vc = Vseq[a:b][:, :, None, :].copy() if L else np.zeros((1, H_kv, 1, D), np.float16)
        table = np.arange(max(L, 1), dtype=np.int32)[None]
        o, l = oracle.decode_paged(q[None], kc, vc, table, np.array([L], np.int32), with_lse=True)
        O_part.append(o[0])
        lse_part.append(l[0])
    return np.stack(O_part, 1), np.stack(lse_part, 1)  # [H_q, n_split, D], [H_q, n_split]


@pytest.mark.parametrize("cuts", [[0, 40], [0, 17, 40], [0, 1, 2, 33, 40], [0, 0, 13, 13, 40, 40]])
def test_lse_merge_of_segments_equals_whole(cuts):
    H_q, H_kv, D, L = 4, 2, 16, 40
    rng = np.random.default_rng(14)
    q = _rand16(rng, (H_q, D), 2.0)
    Kseq, Vseq = _rand16(rng, (L, H_kv, D), 2.0), _rand16(rng, (L, H_kv, D))
    O_part, lse_part = _segment_partials(q, Kseq, Vseq, cuts)
    out, lse = oracle.lse_combine(O_part, lse_part, with_lse=True)
    full, lfull = oracle.decode_paged(q[None], Kseq[:, :, None, :].copy(), Vseq[:, :, None, :].copy(),
                                      np.arange(L, dtype=np.int32)[None], np.array([L], np.int32),
                                      with_lse=True)
    np.testing.assert_allclose(out, full[0], atol=1e-13)
    np.testing.assert_allclose(lse, lfull[0], atol=1e-12)


def test_lse_merge_all_empty():
    out, lse = oracle.lse_combine(np.ones((2, 3, 4)), np.full((2, 3), -np.inf), with_lse=True)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_lse_merge_two_known_partials():
    # two singleton segments with scores a, b: weights e^a/(e^a+e^b), e^b/(e^a+e^b)
    a, b = 0.3, -1.1
    O_part = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    out, lse = oracle.lse_combine(O_part, np.array([[a, b]]), with_lse=True)
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(out[0], [wa, 1 - wa], atol=1e-15)
    assert abs(lse[0] - math.log(math.exp(a) + math.exp(b))) < 1e-15


def test_kv_append_matches_fancy_indexing_scatter():
    rng = np.random.default_rng(40)
    nb, H_kv, bs, D, T = 7, 3, 16, 8, 9
    kc, vc = _rand16(rng, (nb, H_kv, bs, D)), _rand16(rng, (nb, H_kv, bs, D))
    kn, vn = _rand16(rng, (T, H_kv, D)), _rand16(rng, (T, H_kv, D))
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[2] = -1                       # padding token: skipped
    slots[5] = nb * bs + 3              # out of range: skipped and counted
    k2, v2, bad = oracle.kv_append(kn, vn, kc, vc, slots)
    assert bad == 1
    ek, ev = kc.copy(), vc.copy()
    ok = (slots >= 0) & (slots < nb * bs)
    ek[slots[ok] // bs, :, slots[ok] % bs, :] = kn[ok]
    ev[slots[ok] // bs, :, slots[ok] % bs, :] = vn[ok]
    assert np.array_equal(k2.view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(v2.view(np.uint16), ev.view(np.uint16))


# ---------------------------------------------------------- paged prefill

def _paged_problem(rng, lens_kv, lens_q, H_q, H_kv, D, bs=16, nan_unused=True):
    """Contiguous K/V per sequence, the same keys in a permuted paged cache
    (unused slots NaN), and packed queries for the last lens_q positions."""
    B = len(lens_kv)
    K = [_rand16(rng, (L, H_kv, D)) for L in lens_kv]
    V = [_rand16(rng, (L, H_kv, D)) for L in lens_kv]
    pages = [(L + bs - 1) // bs for L in lens_kv]
    nb = sum(pages)
    perm = rng.permutation(nb).astype(np.int32)
    mb = max(pages) + 1
    kc = np.full((nb, H_kv, bs, D), np.nan if nan_unused else 0.0, np.float16)
    vc = kc.copy()
    table = np.full((B, mb), -1, np.int32)
    off = 0
    for b in range(B):
        for p in range(pages[b]):
            phys = perm[off + p]
            table[b, p] = phys
            t0, t1 = p * bs, min(lens_kv[b], (p + 1) * bs)
            kc[phys, :, :t1 - t0] = K[b][t0:t1].transpose(1, 0, 2)
            vc[phys, :, :t1 - t0] = V[b][t0:t1].transpose(1, 0, 2)
        off += pages[b]
    Qs = [_rand16(rng, (Lq, H_q, D)) for Lq in lens_q]
    cu = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    return K, V, kc, vc, table, np.concatenate(Qs), cu, np.array(lens_kv, np.int32)


def test_prefill_paged_equals_last_rows_of_full_causal_prefill():
    rng = np.random.default_rng(50)
    lens_kv, lens_q, H_q, H_kv, D = [40, 17, 70], [9, 17, 1], 4, 2, 16
    K, V, kc, vc, table, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q, H_q, H_kv, D)
    out = oracle.prefill_paged(Q, kc, vc, cu, skv, table, causal=True)
    assert np.isfinite(out).all()           # NaN in unused slots never read
    for b, (Lkv, Lq) in enumerate(zip(lens_kv, lens_q)):
        # a full causal prefill of the whole sequence, whose last Lq query rows are the chunk
        Qfull = _rand16(rng, (1, Lkv, H_q, D))
        Qfull[0, Lkv - Lq:] = Q[cu[b]:cu[b + 1]]
        ref = _sdpa(Qfull, K[b][None], V[b][None], causal=True)[0, Lkv - Lq:]
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ref, atol=1e-12)


def test_prefill_paged_noncausal_and_decode_special_case():
    rng = np.random.default_rng(51)
    lens_kv, lens_q, H_q, H_kv, D = [33, 5], [1, 1], 8, 2, 32
    K, V, kc, vc, table, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q, H_q, H_kv, D)
    # one new query per sequence: paged prefill == paged decode (causal or not)
    for causal in (True, False):
        out = oracle.prefill_paged(Q, kc, vc, cu, skv, table, causal=causal)
        dec = oracle.decode_paged(Q, kc, vc, table, skv)
        np.testing.assert_allclose(out, dec, atol=1e-14)
    # non-causal chunk: every query sees all L_kv keys
    lens_q2 = [6, 3]
    K, V, kc, vc, table, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q2, H_q, H_kv, D)
    out = oracle.prefill_paged(Q, kc, vc, cu, skv, table, causal=False)
    for b in range(2):
        ref = _sdpa(Q[cu[b]:cu[b + 1]][None], K[b][None], V[b][None], causal=False)[0]
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ref, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_paged_rows_match_sdpa(causal):
    # selected rows (b, i, h) against torch float64 SDPA over each sequence's own keys
    rng = np.random.default_rng(52)
    lens_kv, lens_q, H_q, H_kv, D = [40, 23, 70], [9, 23, 5], 6, 2, 16
    K, V, kc, vc, table, Q, cu, skv = _paged_problem(rng, lens_kv, lens_q, H_q, H_kv, D)
    rows = np.array([(b, i, h) for b in range(3) for i in range(lens_q[b]) for h in range(H_q)
                     if (b * 7 + i * 3 + h) % 4 == 0], np.int32)
    got = oracle.prefill_paged_rows(Q, kc, vc, cu, skv, table, rows, causal=causal)
    for r, (b, i, h) in enumerate(rows):
        Lkv, Lq = lens_kv[b], lens_q[b]
        if causal:
            Qfull = np.zeros((1, Lkv, H_q, D), np.float16)
            Qfull[0, Lkv - Lq:] = Q[cu[b]:cu[b + 1]]
            ref = _sdpa(Qfull, K[b][None], V[b][None], causal=True)[0, Lkv - Lq + i, h]
        else:
            ref = _sdpa(Q[cu[b] + i][None, None], K[b][None], V[b][None], causal=False)[0, 0, h]
        np.testing.assert_allclose(got[r], ref, atol=1e-12)


# ------------------------------------------------ QK-norm + RoPE prologue

ROPE_BASE = 1.0e6


def _complex_turn(y, positions, freqs):
    """Rotate each split-half pair (y_i, y_{i+D/2}) as the complex number
    y_i + 1j*y_{i+D/2} multiplied by exp(1j*pos*freq_i)."""
    h = y.shape[-1] // 2
    z = (y[..., :h] + 1j * y[..., h:]) * np.exp(1j * np.multiply.outer(positions, freqs))[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1)


def _recovered_freqs(D, base):
    # a unit vector in pair i (element i = 1, element i+D/2 = 0) at position 1
    # turns by freq_i; read the angle back with atan2 (freq <= 1 < pi)
    h = D // 2
    x = np.zeros((h, 1, D), np.float16)
    x[np.arange(h), 0, np.arange(h)] = 1.0
    out = oracle.qk_norm_rope(x, None, np.ones(h, np.int32), base)
    i = np.arange(h)
    return np.arctan2(out[i, 0, i + h], out[i, 0, i])


@pytest.mark.parametrize("D", [128, 16])
def test_rope_frequencies_are_geometric_from_one(D):
    f = _recovered_freqs(D, ROPE_BASE)
    assert abs(f[0] - 1.0) < 1e-15                               # pair 0 turns one radian per position
    np.testing.assert_allclose(f[1:] / f[:-1], ROPE_BASE ** (-2.0 / D), rtol=1e-12)
    # extrapolating one pair past the end reaches 1/base
    assert abs(f[-1] * ROPE_BASE ** (-2.0 / D) * ROPE_BASE - 1.0) < 1e-9


def test_rope_equals_complex_rotation():
    rng = np.random.default_rng(70)
    T, H, D = 11, 3, 128
    x = _rand16(rng, (T, H, D))
    pos = rng.integers(0, 40000, T).astype(np.int32)
    pos[0] = 0
    out = oracle.qk_norm_rope(x, None, pos, ROPE_BASE)
    freqs = _recovered_freqs(D, ROPE_BASE)
    ref = _complex_turn(x.astype(np.float64), pos.astype(np.float64), freqs)
    np.testing.assert_allclose(out, ref, atol=1e-9)
    np.testing.assert_array_equal(out[0], x[0].astype(np.float64))     # position 0 is the identity
    # every pair keeps its length
    h = D // 2
    np.testing.assert_allclose(out[..., :h] ** 2 + out[..., h:] ** 2,
                               x[..., :h].astype(np.float64) ** 2 + x[..., h:].astype(np.float64) ** 2,
                               rtol=1e-12, atol=1e-14)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(71)
    D = 128
    q, k = _rand16(rng, (1, 1, D)), _rand16(rng, (1, 1, D))

    def score(m, n):
        a = oracle.qk_norm_rope(q, None, np.array([m], np.int32), ROPE_BASE)
        b = oracle.qk_norm_rope(k, None, np.array([n], np.int32), ROPE_BASE)
        return float((a * b).sum())
    s = score(37, 5)
    for c in (1, 100, 9000):
        assert abs(score(37 + c, 5 + c) - s) < 1e-9 * (1 + abs(s))
    assert abs(score(5, 37) - s) > 1e-3                               # the sign of m - n matters


@pytest.mark.parametrize("scale", [1.0, 30.0, 1e-4])
def test_qk_norm_equals_torch_rms_norm_at_position_zero(scale):
    rng = np.random.default_rng(72)
    T, H, D = 7, 4, 128
    x = _rand16(rng, (T, H, D), scale)
    w = (1.0 + 0.5 * rng.standard_normal(D)).astype(np.float16)
    out = oracle.qk_norm_rope(x, w, np.zeros(T, np.int32), ROPE_BASE, eps=1e-6)
    ref = F.rms_norm(torch.from_numpy(x.astype(np.float64)), (D,),
                     torch.from_numpy(w.astype(np.float64)), eps=1e-6).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_qk_norm_then_rope_order_and_weights():
    # RMSNorm first, RoPE second: with non-uniform weights the two do not commute
    rng = np.random.default_rng(73)
    T, H, D = 9, 2, 128
    x = _rand16(rng, (T, H, D))
    w = rng.uniform(0.2, 3.0, D).astype(np.float16)
    pos = rng.integers(1, 30000, T).astype(np.int32)
    out = oracle.qk_norm_rope(x, w, pos, ROPE_BASE)
    normed = F.rms_norm(torch.from_numpy(x.astype(np.float64)), (D,),
                        torch.from_numpy(w.astype(np.float64)), eps=1e-6).numpy()
    ref = _complex_turn(normed, pos.astype(np.float64), _recovered_freqs(D, ROPE_BASE))
    np.testing.assert_allclose(out, ref, atol=1e-9)
    wrong_order = _complex_turn(x.astype(np.float64), pos.astype(np.float64),
                                _recovered_freqs(D, ROPE_BASE))
    wrong_order = F.rms_norm(torch.from_numpy(wrong_order), (D,),
                             torch.from_numpy(w.astype(np.float64)), eps=1e-6).numpy()
    assert np.abs(out - wrong_order).max() > 0.1
