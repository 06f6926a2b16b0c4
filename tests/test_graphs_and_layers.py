"""CUDA-graph capture and multi-layer KV pools (GPU).

* attn_decode_paged_ws allocates nothing and its launch shapes depend only on
  the sizes (max_blocks_per_seq, not the device-side seq_lens), so it can be
  captured once and replayed after the inputs change in place.
* attn_prefill builds its TMA descriptors on the host when called; captured,
  it replays on the same buffers.
* A multi-layer pool [layers, num_blocks, H_kv, 16, D] is served by passing
  each layer's base pointer (layer * num_blocks * H_kv * 16 * D elements in):
  the "GRPO-CUDA Project Memory" page's "Known bugs fixed" records the bug of
  always passing layer 0's base."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import oracle
import workloads as W
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def test_decode_ws_graph_capture_and_replay():
    cfg = W.DecodeConfig("graph", 16, 16, 8, max_blocks_per_seq=32)
    a = W.decode_inputs(cfg, seed=31, seq_lens=W.uniform_int(31, 3, 16, 1, 512))
    q, kc, vc, bt, sl = (dev(x) for x in (a.q, a.k_cache, a.v_cache, a.block_tables, a.seq_lens))
    out = torch.empty_like(q)
    ws = torch.empty(ag.attn_decode_paged_workspace_bytes(16, 16, 8, 128, 32, 16), dtype=torch.uint8,
                     device="cuda")
    ag.attn_decode_paged_ws(q, kc, vc, out, bt, sl, ws)   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ag.attn_decode_paged_ws(q, kc, vc, out, bt, sl, ws)
    for step in range(3):
        # new query and shorter contexts, written in place into the captured buffers
        q_new = W.normal_fp16(100 + step, 0, a.q.shape)
        lens = np.maximum(a.seq_lens - 7 * step, 0).astype(np.int32)
        q.copy_(torch.from_numpy(q_new))
        sl.copy_(torch.from_numpy(lens))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.decode_paged(q_new, a.k_cache, a.v_cache, a.block_tables, lens)
        assert_close(host(out), ref, f"graph replay {step}")


def test_prefill_graph_capture_and_replay():
    cfg = W.PrefillConfig("g", 1, 300, 4, 2)
    Q, K, V = W.prefill_inputs(cfg, seed=32)
    dQ, dK, dV = dev(Q), dev(K), dev(V)
    O = torch.empty_like(dQ)
    ag.attn_prefill(dQ, dK, dV, O)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ag.attn_prefill(dQ, dK, dV, O)
    Q2, K2, V2 = W.prefill_inputs(cfg, seed=33)
    dQ.copy_(torch.from_numpy(Q2)); dK.copy_(torch.from_numpy(K2)); dV.copy_(torch.from_numpy(V2))
    g.replay()
    torch.cuda.synchronize()
    assert_close(host(O), oracle.prefill(Q2, K2, V2), "prefill graph replay")


def test_multi_layer_pool_per_layer_base():
    layers, N, H_q, H_kv = 3, 6, 16, 8
    lens = np.array([1, 17, 100, 256, 33, 200], np.int32)
    tables, nb = W.decode_layout(lens, 16, 16, seed=34)
    kpool = W.normal_fp16(34, 1, (layers, nb, H_kv, 16, 128))
    vpool = W.normal_fp16(34, 2, (layers, nb, H_kv, 16, 128))
    q = W.normal_fp16(34, 0, (layers, N, H_q, 128))
    dk, dv, dq = dev(kpool), dev(vpool), dev(q)
    bt, sl = dev(tables), dev(lens)
    for l in range(layers):
        out = torch.empty(N, H_q, 128, dtype=torch.float16, device="cuda")
        ag.attn_decode_paged(dq[l], dk[l], dv[l], out, bt, sl)   # dk[l]: the layer's base pointer
        torch.cuda.synchronize()
        ref = oracle.decode_paged(q[l], kpool[l], vpool[l], tables, lens)
        assert_close(host(out), ref, f"layer {l}")
        if l > 0:   # reading layer 0 instead would give a different answer
            wrong = oracle.decode_paged(q[l], kpool[0], vpool[0], tables, lens)
            assert np.abs(host(out).astype(np.float64) - wrong).max() > 0.1
