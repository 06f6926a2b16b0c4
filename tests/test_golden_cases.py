"""The pages' own test shapes, run through the oracle (CPU only).

Prefill cases are compared with torch float64 SDPA; decode cases are laid out
both with the identity block table the page uses and with a random
permutation, and must equal the last causal prefill row of the same keys."""
import numpy as np
import pytest

import golden_cases
import oracle
from test_oracle_pins import _page, _rand16, _sdpa

PREFILL, DECODE = golden_cases.load()


def test_fixture_has_the_pages_cases():
    assert len(PREFILL) == 5 and len(DECODE) == 4
    assert all(c[-1] == 128 for c in PREFILL + DECODE)


@pytest.mark.parametrize("case", PREFILL)
def test_page_prefill_case(case):
    B, S, H_q, H_kv, D = case
    rng = np.random.default_rng(S)
    Q, K, V = _rand16(rng, (B, S, H_q, D)), _rand16(rng, (B, S, H_kv, D)), _rand16(rng, (B, S, H_kv, D))
    np.testing.assert_allclose(oracle.prefill(Q, K, V), _sdpa(Q, K, V, True), atol=1e-12)


@pytest.mark.parametrize("case", DECODE)
@pytest.mark.parametrize("identity", [True, False])
def test_page_decode_case(case, identity):
    N, L, H_q, H_kv, D = case
    bs = 16
    rng = np.random.default_rng(L + N)
    Q, K, V = _rand16(rng, (N, L, H_q, D)), _rand16(rng, (N, L, H_kv, D)), _rand16(rng, (N, L, H_kv, D))
    npg = N * ((L + bs - 1) // bs)
    perm = np.arange(npg, dtype=np.int32) if identity else rng.permutation(npg).astype(np.int32)
    kc, table = _page(K, bs, perm)
    vc, _ = _page(V, bs, perm)
    out = oracle.decode_paged(Q[:, L - 1].copy(), kc, vc, table, np.full(N, L, np.int32))
    np.testing.assert_allclose(out, oracle.prefill(Q, K, V)[:, L - 1], atol=1e-13)
