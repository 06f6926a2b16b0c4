"""FP64 CPU oracle for grouped-query attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and it
never calls the CUDA library: the two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain loops in double precision,
one function per definition; see the header of that file for the formulas and
the passages of the pages they follow).  This module only compiles it with the
host C compiler, loads it with ctypes and converts numpy arrays to pointers.

Inputs are FP16 arrays (numpy ``float16``); they are passed as their raw bits
and decoded exactly to double inside the oracle.  Outputs are unrounded
float64 arrays.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so with gcc -O2 -fopenmp."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    p = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    lib.oracle_set_num_threads.argtypes = [i]
    lib.oracle_set_num_threads.restype = None
    lib.oracle_prefill.argtypes = [p, p, p, i, i, i, i, i, i, p, p]
    lib.oracle_prefill.restype = None
    lib.oracle_prefill_rows.argtypes = [p, p, p, i, i, i, i, i, i, p, i, p, p]
    lib.oracle_prefill_rows.restype = None
    lib.oracle_decode_paged.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, p]
    lib.oracle_decode_paged.restype = None
    lib.oracle_decode_paged_rows.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, i, p, p]
    lib.oracle_decode_paged_rows.restype = None
    lib.oracle_lse_combine.argtypes = [p, p, i, i, i, p, p]
    lib.oracle_lse_combine.restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _half(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float16:
        raise TypeError(f"oracle inputs are FP16 arrays, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.int32:
        raise TypeError(f"expected int32, got {a.dtype}")
    return a


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


@contextlib.contextmanager
def threads(n: int):
    """Run the oracle's calls inside the block on ``n`` OpenMP threads."""
    lib = _load()
    saved = int(lib.oracle_num_threads())
    lib.oracle_set_num_threads(int(n))
    try:
        yield
    finally:
        lib.oracle_set_num_threads(saved)


def half_to_double(bits: int) -> float:
    """Exact IEEE binary16 decode of one 16-bit pattern."""
    return float(_load().oracle_half_to_double(ctypes.c_uint16(bits)))


def prefill(Q, K, V, causal: bool = True, with_lse: bool = False):
    """O = softmax(Q K^T / sqrt(D) [+ causal mask]) V per (b, h), GQA map g = h*H_kv//H_q.

    Q: [B,S,H_q,D] fp16; K,V: [B,S,H_kv,D] fp16.  Returns O [B,S,H_q,D] float64
    (and lse [B,S,H_q] if ``with_lse``).
    """
    Q, K, V = _half(Q), _half(K), _half(V)
    B, S, H_q, D = Q.shape
    H_kv = K.shape[2]
    assert K.shape == (B, S, H_kv, D) and V.shape == K.shape
    O = np.empty((B, S, H_q, D), np.float64)
    lse = np.empty((B, S, H_q), np.float64)
    _load().oracle_prefill(_ptr(Q), _ptr(K), _ptr(V), B, S, H_q, H_kv, D, int(bool(causal)),
                           _ptr(O), _ptr(lse))
    return (O, lse) if with_lse else O


def prefill_rows(Q, K, V, rows, causal: bool = True, with_lse: bool = False):
    """Oracle rows (b, i, h) of a prefill only: returns [n_rows, D] float64."""
    Q, K, V = _half(Q), _half(K), _half(V)
    B, S, H_q, D = Q.shape
    H_kv = K.shape[2]
    rows = _i32(np.asarray(rows, np.int32).reshape(-1, 3))
    out = np.empty((rows.shape[0], D), np.float64)
    lse = np.empty((rows.shape[0],), np.float64)
    _load().oracle_prefill_rows(_ptr(Q), _ptr(K), _ptr(V), B, S, H_q, H_kv, D,
                                int(bool(causal)), _ptr(rows), rows.shape[0], _ptr(out),
                                _ptr(lse))
    return (out, lse) if with_lse else out


def decode_paged(q, k_cache, v_cache, block_tables, seq_lens, with_lse: bool = False):
    """Single-token decode over a paged cache.

    q: [N,H_q,D] fp16; caches: [num_blocks,H_kv,block_size,D] fp16;
    block_tables: [N,max_blocks_per_seq] int32; seq_lens: [N] int32.
    Returns out [N,H_q,D] float64 (and lse [N,H_q]).
    """
    q, kc, vc = _half(q), _half(k_cache), _half(v_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    N, H_q, D = q.shape
    H_kv, bs = kc.shape[1], kc.shape[2]
    out = np.empty((N, H_q, D), np.float64)
    lse = np.empty((N, H_q), np.float64)
    _load().oracle_decode_paged(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl), N, H_q, H_kv,
                                D, bt.shape[1], bs, _ptr(out), _ptr(lse))
    return (out, lse) if with_lse else out


def decode_paged_rows(q, k_cache, v_cache, block_tables, seq_lens, rows, with_lse=False):
    """Oracle rows (n, h) of a paged decode only: returns [n_rows, D] float64."""
    q, kc, vc = _half(q), _half(k_cache), _half(v_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    N, H_q, D = q.shape
    H_kv, bs = kc.shape[1], kc.shape[2]
    rows = _i32(np.asarray(rows, np.int32).reshape(-1, 2))
    out = np.empty((rows.shape[0], D), np.float64)
    lse = np.empty((rows.shape[0],), np.float64)
    _load().oracle_decode_paged_rows(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl), N, H_q,
                                     H_kv, D, bt.shape[1], bs, _ptr(rows), rows.shape[0],
                                     _ptr(out), _ptr(lse))
    return (out, lse) if with_lse else out


def lse_combine(O_part, lse_part, with_lse: bool = False):
    """Merge partials over disjoint key segments.

    O_part: [R, n_split, D] float64 (each normalised over its segment);
    lse_part: [R, n_split] float64 (-inf for an empty segment).
    """
    O_part = np.ascontiguousarray(O_part, np.float64)
    lse_part = np.ascontiguousarray(lse_part, np.float64)
    R, n_split, D = O_part.shape
    out = np.empty((R, D), np.float64)
    lse = np.empty((R,), np.float64)
    _load().oracle_lse_combine(_ptr(O_part), _ptr(lse_part), R, n_split, D, _ptr(out),
                               _ptr(lse))
    return (out, lse) if with_lse else out


@contextlib.contextmanager
def variant(lib_path: str):
    """Route every call of this module through another build of attn_oracle.c
    for the duration of the block.  Used by the planted-mistake tests, which
    compile a deliberately altered copy of the oracle and check that the pins
    reject it."""
    global _lib
    saved = _load()
    _lib = _bind(ctypes.CDLL(lib_path))
    try:
        yield
    finally:
        _lib = saved


def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping):
    """Return copies of the caches with the new rows written to their slots
    (int64 slot_mapping, -1 skipped) and the count of out-of-range slots."""
    k_new, v_new = _half(k_new), _half(v_new)
    kc, vc = _half(k_cache).copy(), _half(v_cache).copy()
    sm = np.ascontiguousarray(slot_mapping, np.int64)
    T, H_kv, D = k_new.shape
    lib = _load()
    lib.oracle_kv_append.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 + [ctypes.c_long]
    lib.oracle_kv_append.restype = ctypes.c_int
    bad = lib.oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc), _ptr(sm), T, H_kv, D,
                               kc.shape[2], kc.shape[0])
    return kc, vc, int(bad)


def prefill_paged(Q, k_cache, v_cache, cu_seqlens_q, seq_lens_kv, block_tables, causal=True,
                  with_lse=False):
    """New query chunks (packed Q [total_q, H_q, D], cu_seqlens_q [B+1]) against
    a paged cache holding L_kv = seq_lens_kv[b] keys per sequence, the last
    L_q of them the chunk's own; query i sits at position L_kv - L_q + i."""
    Q, kc, vc = _half(Q), _half(k_cache), _half(v_cache)
    cu, sl, bt = _i32(cu_seqlens_q), _i32(seq_lens_kv), _i32(block_tables)
    total_q, H_q, D = Q.shape
    B = sl.shape[0]
    assert cu.shape == (B + 1,) and cu[-1] == total_q
    H_kv, bs = kc.shape[1], kc.shape[2]
    O = np.empty((total_q, H_q, D), np.float64)
    lse = np.empty((total_q, H_q), np.float64)
    lib = _load()
    p, i = ctypes.c_void_p, ctypes.c_int
    lib.oracle_prefill_paged.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, p, p]
    lib.oracle_prefill_paged.restype = None
    lib.oracle_prefill_paged(_ptr(Q), _ptr(kc), _ptr(vc), _ptr(cu), _ptr(sl), _ptr(bt), B, H_q,
                             H_kv, D, bt.shape[1], bs, int(bool(causal)), _ptr(O), _ptr(lse))
    return (O, lse) if with_lse else O


def prefill_paged_rows(Q, k_cache, v_cache, cu_seqlens_q, seq_lens_kv, block_tables, rows,
                       causal=True, with_lse=False):
    """Oracle rows (b, i, h) of prefill_paged only (query i of sequence b's
    chunk, head h): returns [n_rows, D] float64."""
    Q, kc, vc = _half(Q), _half(k_cache), _half(v_cache)
    cu, sl, bt = _i32(cu_seqlens_q), _i32(seq_lens_kv), _i32(block_tables)
    total_q, H_q, D = Q.shape
    B = sl.shape[0]
    assert cu.shape == (B + 1,) and cu[-1] == total_q
    rows = _i32(np.asarray(rows, np.int32).reshape(-1, 3))
    lq = np.diff(cu)
    assert np.all((rows[:, 0] >= 0) & (rows[:, 0] < B)), "sequence index out of range"
    assert np.all((rows[:, 1] >= 0) & (rows[:, 1] < lq[rows[:, 0]])), "query index out of range"
    assert np.all((rows[:, 2] >= 0) & (rows[:, 2] < H_q)), "head index out of range"
    H_kv, bs = kc.shape[1], kc.shape[2]
    out = np.empty((rows.shape[0], D), np.float64)
    lse = np.empty((rows.shape[0],), np.float64)
    lib = _load()
    p, i = ctypes.c_void_p, ctypes.c_int
    lib.oracle_prefill_paged_rows.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, p, i, p, p]
    lib.oracle_prefill_paged_rows.restype = None
    lib.oracle_prefill_paged_rows(_ptr(Q), _ptr(kc), _ptr(vc), _ptr(cu), _ptr(sl), _ptr(bt), B,
                                  H_q, H_kv, D, bt.shape[1], bs, int(bool(causal)), _ptr(rows),
                                  rows.shape[0], _ptr(out), _ptr(lse))
    return (out, lse) if with_lse else out


def qk_norm_rope(x, weight, positions, base, eps=1e-6):
    """Per-head RMSNorm (skipped when ``weight`` is None) then NeoX rotary
    embedding of x [T, H, D] at ``positions`` [T]; float64 result."""
    x = _half(x)
    T, H, D = x.shape
    assert D % 2 == 0 and D <= 1024
    w = None if weight is None else _half(weight)
    assert w is None or w.shape == (D,)
    pos = _i32(positions)
    assert pos.shape == (T,)
    out = np.empty((T, H, D), np.float64)
    lib = _load()
    p, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.oracle_qk_norm_rope.argtypes = [p, p, p, i, i, i, d, d, p]
    lib.oracle_qk_norm_rope.restype = None
    lib.oracle_qk_norm_rope(_ptr(x), None if w is None else _ptr(w), _ptr(pos), T, H, D,
                            float(base), float(eps), _ptr(out))
    return out
