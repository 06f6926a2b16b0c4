"""ctypes binding of libattn_gb300 (the C ABI declared in include/attn.h).

Argument marshalling only: tensors are checked for device, dtype and layout,
turned into raw pointers, and passed with the current CUDA stream.  Every
computation runs in the library's CUDA kernels.  There is no fallback: if the
library cannot be built or loaded, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build as _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_CUDA = -3
ATTN_ERR_TIMEOUT = -4
ATTN_ERR_BAD_INPUT = -5
ATTN_ERR_WORKSPACE = -6

EXPORTED = [
    "attn_prefill", "attn_decode_paged", "attn_decode_paged_workspace_bytes",
    "attn_decode_paged_ws", "attn_lse_combine", "attn_release_workspace",
    "attn_get_device_error", "attn_last_cuda_error", "attn_status_string", "attn_version",
    "attn_decode_paged_noalloc", "attn_debug_prefill_stall", "attn_kv_append",
    "attn_decode_paged_append", "attn_prefill_paged", "attn_rope_cos_sin_table",
    "attn_qk_norm_rope", "attn_qk_norm_rope_append", "attn_prefill_paged_qk_norm_rope",
]

# Size of the scratch buffer compiled into the library for attn_decode_paged_noalloc.
NOALLOC_SCRATCH_BYTES = 32 << 20

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)} ({status})"
        if status == ATTN_ERR_CUDA and _lib is not None:
            msg += f", cudaError {_lib.attn_last_cuda_error()}"
        super().__init__(msg)


def load():
    """Build (if stale) and load libattn_gb300.so; returns the ctypes handle."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.attn_prefill.argtypes = [p, p, p, p, i, i, i, i, i, i, p]
            lib.attn_decode_paged.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p]
            lib.attn_decode_paged_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
            lib.attn_decode_paged_workspace_bytes.restype = sz
            lib.attn_decode_paged_ws.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, p, sz, p]
            lib.attn_lse_combine.argtypes = [p, p, p, i, i, i, p]
            lib.attn_release_workspace.argtypes = []
            lib.attn_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), i]
            lib.attn_last_cuda_error.argtypes = []
            lib.attn_status_string.argtypes = [i]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_version.argtypes = []
            lib.attn_decode_paged_noalloc.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p]
            lib.attn_debug_prefill_stall.argtypes = [p, p, p, p, i, i, i, i, i, i, i, p]
            ll = ctypes.c_longlong
            lib.attn_kv_append.argtypes = [p, p, p, p, p, i, i, i, i, ll, p]
            lib.attn_decode_paged_append.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i,
                                                     ll, p]
            lib.attn_prefill_paged.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, ll, i, p]
            f, d = ctypes.c_float, ctypes.c_double
            lib.attn_rope_cos_sin_table.argtypes = [p, i, i, d, p]
            lib.attn_qk_norm_rope.argtypes = [p, p, p, p, p, i, p, i, i, i, i, f, p]
            lib.attn_qk_norm_rope_append.argtypes = [p, p, p, p, p, p, i, p, p, p, p, i, i, i, i, i,
                                                     ll, f, p]
            lib.attn_prefill_paged_qk_norm_rope.argtypes = [p, p, p, p, p, p, p, p, p, i, f, i, i, i,
                                                            i, i, i, i, i, ll, i, p]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def _stream(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def attn_prefill(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor,
                 causal: bool = True, stream=None) -> None:
    """O <- attention(Q, K, V) for [B,S,H,128] FP16 tensors (GQA, causal or full)."""
    if Q.dim() != 4 or K.dim() != 4 or V.shape != K.shape or O.shape != Q.shape:
        raise ValueError("expected Q,O [B,S,H_q,D] and K,V [B,S,H_kv,D]")
    B, S, H_q, D = Q.shape
    if K.shape[0] != B or K.shape[1] != S or K.shape[3] != D:
        raise ValueError("K/V batch, sequence and head_dim must match Q")
    args = [_dev(Q, "Q", torch.float16), _dev(K, "K", torch.float16),
            _dev(V, "V", torch.float16), _dev(O, "O", torch.float16)]
    st = _stream(stream, Q.device)
    _check(load().attn_prefill(*args, B, S, H_q, K.shape[2], D, int(bool(causal)),
                               ctypes.c_void_p(st)), "attn_prefill")


def _paged_prefill_args(Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv, block_tables):
    if Q.dim() != 3 or O.shape != Q.shape or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected Q,O [total_q,H_q,D] and caches [num_blocks,H_kv,block_size,D]")
    B = seq_lens_kv.shape[0]
    if cu_seqlens_q.shape != (B + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("expected cu_seqlens_q [B+1], seq_lens_kv [B], block_tables [B, max_blocks]")
    return [_dev(Q, "Q", torch.float16), _dev(k_cache, "k_cache", torch.float16),
            _dev(v_cache, "v_cache", torch.float16), _dev(O, "O", torch.float16),
            _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32), _dev(seq_lens_kv, "seq_lens_kv", torch.int32),
            _dev(block_tables, "block_tables", torch.int32)]


def attn_prefill_paged(Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv, block_tables,
                       max_seqlen_q: int, causal: bool = True, stream=None) -> None:
    """Prefill of packed query chunks (Q, O [total_q, H_q, D]; cu_seqlens_q [B+1])
    against a paged cache holding seq_lens_kv[b] keys per sequence (its last
    L_q keys are the chunk's own): query i sits at position L_kv - L_q + i."""
    ptrs = _paged_prefill_args(Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv, block_tables)
    total_q, H_q, D = Q.shape
    st = _stream(stream, Q.device)
    _check(load().attn_prefill_paged(*ptrs, seq_lens_kv.shape[0], int(max_seqlen_q), total_q, H_q,
                                     k_cache.shape[1], D, block_tables.shape[1], k_cache.shape[2],
                                     k_cache.shape[0], int(bool(causal)), ctypes.c_void_p(st)),
           "attn_prefill_paged")


def attn_prefill_paged_qk_norm_rope(Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv,
                                    block_tables, q_weight, cos_sin, max_seqlen_q: int,
                                    eps: float = 1e-6, causal: bool = True, stream=None) -> None:
    """attn_prefill_paged on raw query projections: each query row is first
    normalised (q_weight [D], None = no norm) and rotated at its position with
    the cos/sin table [max_pos, D] inside the kernel; Q is only read."""
    ptrs = _paged_prefill_args(Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv, block_tables)
    total_q, H_q, D = Q.shape
    if cos_sin.dim() != 2 or cos_sin.shape[1] != D:
        raise ValueError("expected cos_sin [max_pos, D] float32")
    if q_weight is not None and q_weight.shape != (D,):
        raise ValueError("expected q_weight [D]")
    w = None if q_weight is None else _dev(q_weight, "q_weight", torch.float16)
    cs = _dev(cos_sin, "cos_sin", torch.float32)
    st = _stream(stream, Q.device)
    _check(load().attn_prefill_paged_qk_norm_rope(
        *ptrs, w, cs, cos_sin.shape[0], float(eps), seq_lens_kv.shape[0], int(max_seqlen_q), total_q,
        H_q, k_cache.shape[1], D, block_tables.shape[1], k_cache.shape[2], k_cache.shape[0],
        int(bool(causal)), ctypes.c_void_p(st)), "attn_prefill_paged_qk_norm_rope")


def attn_debug_prefill_stall(Q, K, V, O, stall_tile: int, causal: bool = True, stream=None) -> None:
    """Failure-detection test hook: attn_prefill with key tile ``stall_tile``
    withheld, so the kernel's bounded waits run out (about a second) and it
    reports ATTN_ERR_TIMEOUT through attn_get_device_error."""
    B, S, H_q, D = Q.shape
    args = [_dev(Q, "Q", torch.float16), _dev(K, "K", torch.float16),
            _dev(V, "V", torch.float16), _dev(O, "O", torch.float16)]
    st = _stream(stream, Q.device)
    _check(load().attn_debug_prefill_stall(*args, B, S, H_q, K.shape[2], D, int(bool(causal)),
                                           int(stall_tile), ctypes.c_void_p(st)),
           "attn_debug_prefill_stall")


def _decode_args(q, k_cache, v_cache, out, block_tables, seq_lens):
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("expected q,out [N,H_q,D] and caches [num_blocks,H_kv,block_size,D]")
    N, H_q, D = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != N or seq_lens.shape != (N,):
        raise ValueError("expected block_tables [N,max_blocks_per_seq] and seq_lens [N]")
    ptrs = [_dev(q, "q", torch.float16), _dev(k_cache, "k_cache", torch.float16),
            _dev(v_cache, "v_cache", torch.float16), _dev(out, "out", torch.float16),
            _dev(block_tables, "block_tables", torch.int32), _dev(seq_lens, "seq_lens", torch.int32)]
    sizes = [N, H_q, k_cache.shape[1], D, block_tables.shape[1], k_cache.shape[2]]
    return ptrs, sizes


def attn_decode_paged(q, k_cache, v_cache, out, block_tables, seq_lens, stream=None) -> None:
    """out <- single-token attention of q over the paged cache (library-owned scratch)."""
    ptrs, sizes = _decode_args(q, k_cache, v_cache, out, block_tables, seq_lens)
    st = _stream(stream, q.device)
    _check(load().attn_decode_paged(*ptrs, *sizes, ctypes.c_void_p(st)), "attn_decode_paged")


def attn_kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """Write new K/V rows [T, H_kv, D] into their paged slots (int64 slot_mapping, -1 skips)."""
    if k_new.dim() != 3 or v_new.shape != k_new.shape or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected k_new/v_new [T,H_kv,D] and caches [num_blocks,H_kv,block_size,D]")
    T, H_kv, D = k_new.shape
    if slot_mapping.shape != (T,):
        raise ValueError("expected slot_mapping [T]")
    ptrs = [_dev(k_new, "k_new", torch.float16), _dev(v_new, "v_new", torch.float16),
            _dev(k_cache, "k_cache", torch.float16), _dev(v_cache, "v_cache", torch.float16),
            _dev(slot_mapping, "slot_mapping", torch.int64)]
    st = _stream(stream, k_new.device)
    _check(load().attn_kv_append(*ptrs, T, H_kv, D, k_cache.shape[2], k_cache.shape[0],
                                 ctypes.c_void_p(st)), "attn_kv_append")


def attn_decode_paged_append(q, k_new, v_new, k_cache, v_cache, out, slot_mapping, block_tables,
                             seq_lens, stream=None) -> None:
    """One decode step: append each sequence's new K/V row, then paged decode."""
    ptrs, sizes = _decode_args(q, k_cache, v_cache, out, block_tables, seq_lens)
    N = q.shape[0]
    if k_new.shape != (N, k_cache.shape[1], q.shape[2]) or v_new.shape != k_new.shape or slot_mapping.shape != (N,):
        raise ValueError("expected k_new/v_new [N,H_kv,D] and slot_mapping [N]")
    extra = [_dev(k_new, "k_new", torch.float16), _dev(v_new, "v_new", torch.float16),
             _dev(slot_mapping, "slot_mapping", torch.int64)]
    st = _stream(stream, q.device)
    # C order: q, k_new, v_new, k_cache, v_cache, out, slot_mapping, block_tables, seq_lens
    _check(load().attn_decode_paged_append(ptrs[0], extra[0], extra[1], ptrs[1], ptrs[2], ptrs[3],
                                           extra[2], ptrs[4], ptrs[5], *sizes, k_cache.shape[0],
                                           ctypes.c_void_p(st)), "attn_decode_paged_append")


def attn_rope_cos_sin_table(cos_sin: torch.Tensor, base: float, stream=None) -> None:
    """Fill cos_sin [max_pos, 128] FP32 with the rotary table: the (cos, sin) of
    p * base^(-2j/128) for every position p and pair j, computed in FP64 on the
    device and rounded once, in the entry order include/attn.h documents."""
    if cos_sin.dim() != 2 or cos_sin.shape[1] != 128:
        raise ValueError("expected cos_sin [max_pos, 128] float32")
    ptr = _dev(cos_sin, "cos_sin", torch.float32)
    st = _stream(stream, cos_sin.device)
    _check(load().attn_rope_cos_sin_table(ptr, cos_sin.shape[0], 128, float(base), ctypes.c_void_p(st)),
           "attn_rope_cos_sin_table")


def _prologue_args(Q, K, q_weight, k_weight, cos_sin, positions):
    """Q may be None (keys-only form of the append)."""
    if K.dim() != 3 or (Q is not None and (Q.dim() != 3 or K.shape[0] != Q.shape[0] or K.shape[2] != Q.shape[2])):
        raise ValueError("expected Q [T,H_q,D] and K [T,H_kv,D]")
    D = K.shape[2]
    if cos_sin.dim() != 2 or cos_sin.shape[1] != D:
        raise ValueError("expected cos_sin [max_pos, D] float32")
    if positions.shape != (K.shape[0],):
        raise ValueError("expected positions [T] int32")
    w = []
    for name, t in (("q_weight", q_weight), ("k_weight", k_weight)):
        if t is None:
            w.append(None)
        else:
            if t.shape != (D,):
                raise ValueError(f"expected {name} [D]")
            w.append(_dev(t, name, torch.float16))
    return w, _dev(cos_sin, "cos_sin", torch.float32), _dev(positions, "positions", torch.int32)


def attn_qk_norm_rope(Q, K, q_weight, k_weight, cos_sin, positions, eps: float = 1e-6,
                      stream=None) -> None:
    """In place: per-head RMSNorm (weight None = none) then NeoX RoPE of
    Q [T,H_q,128] and K [T,H_kv,128] at positions [T]."""
    if Q is None:
        raise ValueError("attn_qk_norm_rope rewrites Q in place: Q is required")
    w, cs, pos = _prologue_args(Q, K, q_weight, k_weight, cos_sin, positions)
    T, H_q, D = Q.shape
    st = _stream(stream, Q.device)
    _check(load().attn_qk_norm_rope(_dev(Q, "Q", torch.float16), _dev(K, "K", torch.float16),
                                    w[0], w[1], cs, cos_sin.shape[0], pos, T, H_q, K.shape[1], D,
                                    float(eps), ctypes.c_void_p(st)), "attn_qk_norm_rope")


def attn_qk_norm_rope_append(Q, K, V, q_weight, k_weight, cos_sin, positions, slot_mapping,
                             k_cache, v_cache, eps: float = 1e-6, stream=None, H_q: int = 0) -> None:
    """Q normalised and rotated in place; K normalised and rotated, and V as is,
    written to their paged slots (int64 slot_mapping, -1 skipped).  Q=None
    processes keys and values only (the queries' part then runs inside
    attn_prefill_paged_qk_norm_rope); H_q is the query head count for the
    checks in that case (it defaults to the KV head count)."""
    w, cs, pos = _prologue_args(Q, K, q_weight, k_weight, cos_sin, positions)
    T, H_kv, D = K.shape
    hq = Q.shape[1] if Q is not None else (H_q or H_kv)
    if V.shape != K.shape or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected V like K and caches [num_blocks,H_kv,block_size,D]")
    if slot_mapping.shape != (T,):
        raise ValueError("expected slot_mapping [T]")
    st = _stream(stream, K.device)
    q = None if Q is None else _dev(Q, "Q", torch.float16)
    _check(load().attn_qk_norm_rope_append(
        q, _dev(K, "K", torch.float16), _dev(V, "V", torch.float16),
        w[0], w[1], cs, cos_sin.shape[0], pos, _dev(slot_mapping, "slot_mapping", torch.int64),
        _dev(k_cache, "k_cache", torch.float16), _dev(v_cache, "v_cache", torch.float16), T, hq,
        H_kv, D, k_cache.shape[2], k_cache.shape[0], float(eps), ctypes.c_void_p(st)),
        "attn_qk_norm_rope_append")


def attn_decode_paged_workspace_bytes(num_seqs: int, H_q: int, H_kv: int, D: int,
                                      max_blocks_per_seq: int, block_size: int,
                                      pages_per_split: int = 0) -> int:
    return int(load().attn_decode_paged_workspace_bytes(num_seqs, H_q, H_kv, D,
                                                        max_blocks_per_seq, block_size,
                                                        pages_per_split))


def attn_decode_paged_ws(q, k_cache, v_cache, out, block_tables, seq_lens,
                         workspace: torch.Tensor, pages_per_split: int = 0, stream=None) -> None:
    """attn_decode_paged with a caller-owned scratch tensor (any dtype, contiguous, on device)."""
    ptrs, sizes = _decode_args(q, k_cache, v_cache, out, block_tables, seq_lens)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    st = _stream(stream, q.device)
    _check(load().attn_decode_paged_ws(*ptrs, *sizes, int(pages_per_split),
                                       ctypes.c_void_p(workspace.data_ptr()), nbytes,
                                       ctypes.c_void_p(st)), "attn_decode_paged_ws")


def attn_decode_paged_noalloc(q, k_cache, v_cache, out, block_tables, seq_lens,
                              stream=None) -> None:
    """attn_decode_paged for callers that cannot allocate device memory.

    Meant for code that has no CUDA allocator of its own to call (for example
    when another runtime owns all device memory), that runs under a fixed
    memory budget, or that must not risk the device-wide synchronisation of
    cudaMalloc/cudaFree.  The split-K scratch is a fixed NOALLOC_SCRATCH_BYTES
    buffer inside the library, so nothing is allocated; a problem that needs
    more scratch raises AttnError(ATTN_ERR_WORKSPACE).  The first call on a
    device looks the buffer up (make it before any stream capture), and calls
    that overlap on the GPU share the buffer and race: serialise them.
    """
    ptrs, sizes = _decode_args(q, k_cache, v_cache, out, block_tables, seq_lens)
    st = _stream(stream, q.device)
    _check(load().attn_decode_paged_noalloc(*ptrs, *sizes, ctypes.c_void_p(st)),
           "attn_decode_paged_noalloc")


def attn_lse_combine(O_part: torch.Tensor, lse: torch.Tensor, out: torch.Tensor,
                     stream=None) -> None:
    """out[r] <- merge of O_part[r, i] weighted by exp(lse[r, i]) (FP32 in, FP16 out)."""
    if O_part.dim() != 3 or lse.shape != O_part.shape[:2] or out.shape != (O_part.shape[0], O_part.shape[2]):
        raise ValueError("expected O_part [R,n_split,D], lse [R,n_split], out [R,D]")
    R, n_split, D = O_part.shape
    ptrs = [_dev(O_part, "O_part", torch.float32), _dev(lse, "lse", torch.float32),
            _dev(out, "out", torch.float16)]
    st = _stream(stream, O_part.device)
    _check(load().attn_lse_combine(*ptrs, R, n_split, D, ctypes.c_void_p(st)), "attn_lse_combine")


def attn_release_workspace() -> None:
    _check(load().attn_release_workspace(), "attn_release_workspace")


def attn_get_device_error(reset: bool = True) -> int:
    """Raw device error bits of the current device (synchronises); 0 when clean."""
    code = ctypes.c_int(0)
    st = load().attn_get_device_error(ctypes.byref(code), int(bool(reset)))
    if st not in (ATTN_OK, ATTN_ERR_TIMEOUT, ATTN_ERR_BAD_INPUT):
        raise AttnError(st, "attn_get_device_error")
    return code.value


def attn_version() -> int:
    return int(load().attn_version())
