"""Helpers for the GPU parity tests: device transfer and the error check.

Tolerances (the target's stated bar, FP16 output against the unrounded FP64
oracle): max |gpu - oracle| <= 4e-3 and mean |gpu - oracle| <= 5e-4 over all
compared elements."""
import numpy as np
import torch

MAX_ABS = 4e-3
MEAN_ABS = 5e-4


def dev(a: np.ndarray) -> torch.Tensor:
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def errors(gpu: np.ndarray, ref: np.ndarray):
    d = np.abs(gpu.astype(np.float64) - ref)
    return float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0


def assert_close(gpu, ref, what="", max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    if isinstance(gpu, torch.Tensor):
        gpu = host(gpu)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu.astype(np.float64)).all(), f"{what}: non-finite output"
    mx, mn = errors(gpu, ref)
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max_abs={mx:.3e} mean_abs={mn:.3e}"
    return mx, mn


def device_error_clean():
    import attention_gqa_causal_gb300 as ag
    return ag.attn_get_device_error(reset=True) == 0


def rope_table_entries(cos_sin):
    """(cos, sin), each [max_pos, 64] in pair order, from a table filled by
    attn_rope_cos_sin_table: entry (p, i, m) = p*32 + i*8 + m of its float4
    view holds {cos j, cos j+1, sin j, sin j+1} for pair j = 8m + 2i (the
    entry order include/attn.h documents)."""
    t = cos_sin.reshape(-1, 4, 8, 4)                 # [p, i, m, 4]
    j_even = t[..., [0, 2]].permute(0, 2, 1, 3)      # [p, m, i, (cos, sin)] of pair 8m+2i
    j_odd = t[..., [1, 3]].permute(0, 2, 1, 3)       # pair 8m+2i+1
    pairs = torch.stack([j_even, j_odd], dim=3).reshape(t.shape[0], 64, 2)
    return pairs[..., 0], pairs[..., 1]
