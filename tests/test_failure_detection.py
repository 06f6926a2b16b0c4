"""Failure detection on the GPU without a fault: the prefill kernel is run
with one key tile withheld (attn_debug_prefill_stall), so its bounded
mbarrier waits expire.  The kernel must exit by itself, release its tensor
memory, and report ATTN_ERR_TIMEOUT through the device error word; the
context must stay usable and the next normal call must be correct."""
import numpy as np
import pytest
import torch

import attention_gqa_causal_gb300 as ag
import oracle
import workloads as W
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("stall_tile", [0, 1])
def test_withheld_tile_times_out_and_context_survives(stall_tile):
    # two CTAs; tile 0 (sent before the set-up barrier) stalls both, tile 1 the
    # one with two key tiles
    B, S, H_q, H_kv = 1, 256, 2, 1
    Q, K, V = W.prefill_inputs(W.PrefillConfig("t", B, S, H_q, H_kv), seed=3)
    dQ, dK, dV = dev(Q), dev(K), dev(V)
    O = torch.zeros(Q.shape, dtype=torch.float16, device="cuda")
    assert ag.attn_get_device_error(reset=True) == 0
    ag.attn_debug_prefill_stall(dQ, dK, dV, O, stall_tile=stall_tile)
    torch.cuda.synchronize()                 # returns: the waits are bounded
    code = ag.attn_get_device_error(reset=True)
    assert code & 1, f"expected the timeout bit, got {code}"
    # the context is still usable and a normal call is correct afterwards
    O2 = torch.empty_like(O)
    ag.attn_prefill(dQ, dK, dV, O2, causal=True)
    torch.cuda.synchronize()
    assert_close(host(O2), oracle.prefill(Q, K, V), "after timeout")
    assert ag.attn_get_device_error(reset=True) == 0


def test_stall_hook_rejects_negative_tile():
    Q = torch.zeros(1, 8, 2, 128, dtype=torch.float16, device="cuda")
    K = torch.zeros(1, 8, 1, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(ag.AttnError) as e:
        ag.attn_debug_prefill_stall(Q, K, K, Q.clone(), stall_tile=-1)
    assert e.value.status == ag.ATTN_ERR_INVALID_ARG
