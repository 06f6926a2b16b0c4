"""GPU parity of the KV append (reshape-and-cache) and of one decode step with
its append, against the oracle.  Cache contents must match bit for bit."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import oracle
import workloads as W
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def test_kv_append_bitwise_with_skips_and_flags():
    rng = np.random.default_rng(41)
    nb, H_kv, T = 40, 8, 300
    kc, vc = W.normal_fp16(41, 1, (nb, H_kv, 16, 128)), W.normal_fp16(41, 2, (nb, H_kv, 16, 128))
    kn, vn = W.normal_fp16(41, 5, (T, H_kv, 128)), W.normal_fp16(41, 6, (T, H_kv, 128))
    slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[::7] = -1
    dk, dv = dev(kc), dev(vc)
    ag.attn_kv_append(dev(kn), dev(vn), dk, dv, dev(slots))
    ek, ev, bad = oracle.kv_append(kn, vn, kc, vc, slots)
    assert bad == 0
    assert np.array_equal(host(dk).view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(host(dv).view(np.uint16), ev.view(np.uint16))
    assert ag.attn_get_device_error(reset=True) == 0
    # an out-of-range slot is skipped and flagged; the others still land
    slots2 = np.array([5, nb * 16 + 1, 7], np.int64)
    kn2, vn2 = kn[:3].copy(), vn[:3].copy()
    ag.attn_kv_append(dev(kn2), dev(vn2), dk, dv, dev(slots2))
    e2k, _, bad2 = oracle.kv_append(kn2, vn2, ek, ev, slots2)
    assert bad2 == 1 and ag.attn_get_device_error(reset=True) == 32
    assert np.array_equal(host(dk).view(np.uint16), e2k.view(np.uint16))


@pytest.mark.parametrize("cfg", [W.DECODE_MIX], ids=lambda c: c.name)
def test_decode_step_with_append(cfg):
    inp = W.decode_inputs(cfg, seed=42)
    N, H_kv = cfg.num_seqs, cfg.H_kv
    # the new token of sequence n is its last position, seq_lens[n] - 1
    L = inp.seq_lens.astype(np.int64)
    slots = inp.block_tables[np.arange(N), (L - 1) // 16].astype(np.int64) * 16 + (L - 1) % 16
    kn, vn = W.normal_fp16(42, 7, (N, H_kv, 128)), W.normal_fp16(42, 8, (N, H_kv, 128))
    q, kc, vc, bt, sl = (dev(x) for x in (inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.seq_lens))
    out = torch.empty_like(q)
    ag.attn_decode_paged_append(q, dev(kn), dev(vn), kc, vc, out, dev(slots), bt, sl)
    torch.cuda.synchronize()
    ek, ev, _ = oracle.kv_append(kn, vn, inp.k_cache, inp.v_cache, slots)
    assert np.array_equal(host(kc).view(np.uint16), ek.view(np.uint16))
    ref = oracle.decode_paged(inp.q, ek, ev, inp.block_tables, inp.seq_lens)
    assert_close(host(out), ref, "decode + append")
    assert ag.attn_get_device_error(reset=True) == 0
