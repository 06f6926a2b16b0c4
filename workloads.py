"""Seeded synthetic inputs for the attention workloads.

This module holds random-number generation and input structure only (shapes,
paged block tables, sequence-length mixes): none of the attention arithmetic.
Both the FP64 oracle and the CUDA library consume what it produces; neither
imports the other.

Generator definition (the contract for "N(0,1) from seed s"):

* splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; the finaliser constants of Vigna's public
  splitmix64): the i-th output (i >= 0) of stream ``sid`` under seed ``s`` is
  ``mix(base + (i+1)*GAMMA)`` with ``base = mix(s*GAMMA + sid)``, arithmetic
  mod 2^64.  Being counter based, any element can be generated independently,
  so generation is chunked over threads.
* uniform in (0,1]: ``((x >> 11) + 1) * 2^-53``; uniform in [0,1): ``(x >> 11) * 2^-53``.
* standard normal: Box-Muller on consecutive pairs (u1 in (0,1], u2 in [0,1)):
  ``r = sqrt(-2 ln u1)``, element 2k = ``r cos(2 pi u2)``, element 2k+1 = ``r sin(2 pi u2)``.
* FP16: round-to-nearest-even from the double (numpy's float64 -> float16 cast).

Streams: prefill Q=0, K=1, V=2.  Decode q=0, k_cache=1, v_cache=2,
seq_lens=3, block permutation=4.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, sid: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = np.array([seed], np.uint64) * GAMMA + np.uint64(sid)
    return _mix(a)[0]


def _raw(base: np.uint64, start: int, n: int) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GAMMA)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def uint64_stream(seed: int, sid: int, n: int) -> np.ndarray:
    """First n raw 64-bit outputs of stream ``sid``."""
    base = _base(seed, sid)
    return _raw(base, 0, n)


def _normal_chunk(base, out, start, n):
    # n even, start even: pairs stay aligned with the Box-Muller pairing
    x = _raw(base, start, n)
    u1 = ((x[0::2] >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53
    u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    z = np.empty(n, np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    out[start:start + n] = z.astype(np.float16)


def normal_fp16(seed: int, sid: int, shape) -> np.ndarray:
    """FP16 array of i.i.d. N(0,1) draws from stream ``sid`` (row-major fill)."""
    total = int(np.prod(shape))
    padded = total + (total & 1)
    out = np.empty(padded, np.float16)
    base = _base(seed, sid)
    starts = list(range(0, padded, _CHUNK))
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(lambda s: _normal_chunk(base, out, s, min(_CHUNK, padded - s)), starts))
    return out[:total].reshape(shape)


def uniform_int(seed: int, sid: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform on [lo, hi] (inclusive): lo + floor(u * (hi-lo+1)), u in [0,1)."""
    x = uint64_stream(seed, sid, n)
    u = (x >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


def permutation(seed: int, sid: int, n: int) -> np.ndarray:
    """Seeded random permutation of 0..n-1: stable argsort of n raw 64-bit keys."""
    return np.argsort(uint64_stream(seed, sid, n), kind="stable").astype(np.int32)


# ----------------------------------------------------------------- workloads

@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    S: int
    H_q: int
    H_kv: int
    D: int = 128
    causal: bool = True

    def flops(self) -> float:
        """Algorithmic FLOPs: 2*B*H_q*S^2*D causal, 4*B*H_q*S^2*D full."""
        f = 2.0 * self.B * self.H_q * self.S * self.S * self.D
        return f if self.causal else 2.0 * f

    def io_bytes(self) -> int:
        return 2 * self.D * self.B * self.S * (2 * self.H_q + 2 * self.H_kv)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    num_seqs: int
    H_q: int
    H_kv: int
    D: int = 128
    block_size: int = 16
    len_lo: int = 128
    len_hi: int = 2048
    max_blocks_per_seq: int = 128


PREFILL_SMALL = PrefillConfig("prefill_b1_s64_h4_kv2", 1, 64, 4, 2)
PREFILL_QWEN = PrefillConfig("prefill_b4_s1024_h16_kv8", 4, 1024, 16, 8)
PREFILL_LONG = PrefillConfig("prefill_b2_s8192_h32_kv8_causal", 2, 8192, 32, 8)
PREFILL_LONG_FULL = PrefillConfig("prefill_b2_s8192_h32_kv8_full", 2, 8192, 32, 8,
                                  causal=False)
DECODE_MIX = DecodeConfig("decode_n256_len128to2048_h16_kv8", 256, 16, 8)
DECODE_LONG = DecodeConfig("decode_n8_len32768_h16_kv8", 8, 16, 8, len_lo=32768,
                           len_hi=32768, max_blocks_per_seq=2048)
# the same length mix with eight query heads per kv head (a GQA-8 model's decode)
DECODE_GQA8 = DecodeConfig("decode_n256_len128to2048_h64_kv8", 256, 64, 8)


def prefill_inputs(cfg: PrefillConfig, seed: int = 0):
    """Q [B,S,H_q,D], K,V [B,S,H_kv,D]: FP16 N(0,1), streams 0/1/2."""
    Q = normal_fp16(seed, 0, (cfg.B, cfg.S, cfg.H_q, cfg.D))
    K = normal_fp16(seed, 1, (cfg.B, cfg.S, cfg.H_kv, cfg.D))
    V = normal_fp16(seed, 2, (cfg.B, cfg.S, cfg.H_kv, cfg.D))
    return Q, K, V


@dataclass
class DecodeInputs:
    q: np.ndarray            # [N, H_q, D] fp16
    k_cache: np.ndarray      # [num_blocks, H_kv, bs, D] fp16
    v_cache: np.ndarray      # [num_blocks, H_kv, bs, D] fp16
    block_tables: np.ndarray  # [N, max_blocks_per_seq] int32, unused entries -1
    seq_lens: np.ndarray     # [N] int32

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    def kv_bytes(self) -> int:
        """Bytes of K and V the decode must read: valid tokens only."""
        H_kv, D = self.k_cache.shape[1], self.k_cache.shape[3]
        return int(self.seq_lens.astype(np.int64).sum()) * H_kv * D * 2 * 2


def decode_layout(seq_lens: np.ndarray, block_size: int, max_blocks_per_seq: int,
                  seed: int = 0):
    """Block tables for ``seq_lens``: seq n's logical pages take consecutive
    entries of a seeded permutation of 0..num_blocks-1 (stream 4), with
    num_blocks = sum ceil(L/bs).  Unused table entries are -1."""
    pages = (seq_lens.astype(np.int64) + block_size - 1) // block_size
    if np.any(pages > max_blocks_per_seq):
        raise ValueError("a sequence needs more pages than max_blocks_per_seq")
    num_blocks = int(pages.sum())
    perm = permutation(seed, 4, num_blocks)
    tables = np.full((len(seq_lens), max_blocks_per_seq), -1, np.int32)
    off = 0
    for n, p in enumerate(pages):
        tables[n, :p] = perm[off:off + p]
        off += p
    return tables, num_blocks


def decode_inputs(cfg: DecodeConfig, seed: int = 0, seq_lens=None) -> DecodeInputs:
    """Paged decode inputs.  seq_lens uniform on [len_lo, len_hi] (stream 3)
    unless given; q, k_cache, v_cache N(0,1) FP16 (streams 0/1/2)."""
    if seq_lens is None:
        seq_lens = uniform_int(seed, 3, cfg.num_seqs, cfg.len_lo, cfg.len_hi)
    seq_lens = np.asarray(seq_lens, np.int32)
    tables, num_blocks = decode_layout(seq_lens, cfg.block_size, cfg.max_blocks_per_seq, seed)
    q = normal_fp16(seed, 0, (cfg.num_seqs, cfg.H_q, cfg.D))
    shape = (max(num_blocks, 1), cfg.H_kv, cfg.block_size, cfg.D)
    k = normal_fp16(seed, 1, shape)
    v = normal_fp16(seed, 2, shape)
    return DecodeInputs(q, k, v, tables, seq_lens)


@dataclass(frozen=True)
class ChunkedPrefillConfig:
    """New query chunks after a cached prefix, K/V in the paged cache."""
    name: str
    num_seqs: int
    prefix: int
    chunk: int
    H_q: int
    H_kv: int
    D: int = 128
    causal: bool = True

    def flops(self) -> float:
        """4*D*H_q per (query, visible key) pair: query i of a chunk sees
        prefix + i + 1 keys (causal) or prefix + chunk keys."""
        Lq, off = self.chunk, self.prefix
        pairs = Lq * off + Lq * (Lq + 1) / 2 if self.causal else Lq * (off + Lq)
        return 4.0 * self.D * self.H_q * self.num_seqs * pairs


CHUNKED_PREFILL = ChunkedPrefillConfig("prefill_paged_n4_prefix6144_chunk2048_h32_kv8", 4, 6144,
                                       2048, 32, 8)


def chunked_prefill_inputs(cfg: ChunkedPrefillConfig, seed: int = 0):
    """Packed Q [total_q, H_q, D] (stream 0), paged K/V caches (streams 1/2)
    laid out by decode_layout, cu_seqlens_q and seq_lens_kv."""
    lens_kv = np.full(cfg.num_seqs, cfg.prefix + cfg.chunk, np.int32)
    tables, nb = decode_layout(lens_kv, 16, (cfg.prefix + cfg.chunk + 15) // 16, seed)
    kc = normal_fp16(seed, 1, (nb, cfg.H_kv, 16, cfg.D))
    vc = normal_fp16(seed, 2, (nb, cfg.H_kv, 16, cfg.D))
    Q = normal_fp16(seed, 0, (cfg.num_seqs * cfg.chunk, cfg.H_q, cfg.D))
    cu = np.arange(0, (cfg.num_seqs + 1) * cfg.chunk, cfg.chunk, dtype=np.int32)
    return Q, kc, vc, cu, lens_kv, tables


@dataclass(frozen=True)
class PrologueConfig:
    """The attention-input prologue (QK-norm, RoPE, KV append) over the new
    tokens of num_seqs sequences of seq_len tokens, at positions 0..seq_len-1."""
    name: str
    num_seqs: int
    seq_len: int
    H_q: int
    H_kv: int
    D: int = 128
    base: float = 1.0e6     # RoPE base; the pages print none (Qwen3 models use 1e6)

    @property
    def tokens(self) -> int:
        return self.num_seqs * self.seq_len

    def bytes(self) -> float:
        """HBM bytes the op must move: each token's q, k and v rows read once
        and written once (q in place, k and v to their cache slots), plus its
        64 (cos, sin) FP32 pairs, its int32 position and its int64 slot."""
        row = self.D * 2
        per_token = 2 * row * (self.H_q + 2 * self.H_kv) + (self.D // 2) * 8 + 4 + 8
        return float(per_token * self.tokens)


PROLOGUE = PrologueConfig("qk_norm_rope_append_b2_s8192_h32_kv8", 2, 8192, 32, 8)


def prologue_inputs(cfg: PrologueConfig, seed: int = 0):
    """Q [T, H_q, D] and K, V [T, H_kv, D] (streams 10-12), RMSNorm weights
    1 + N(0, 1)/4 (streams 13/14), positions 0..seq_len-1 per sequence, and
    each token's cache slot from a seeded permutation of ceil(T/16)*16 slots
    (stream 15).  Returns (Q, K, V, q_weight, k_weight, positions, slots,
    num_blocks)."""
    T = cfg.tokens
    Q = normal_fp16(seed, 10, (T, cfg.H_q, cfg.D))
    K = normal_fp16(seed, 11, (T, cfg.H_kv, cfg.D))
    V = normal_fp16(seed, 12, (T, cfg.H_kv, cfg.D))
    qw = (1.0 + 0.25 * normal_fp16(seed, 13, (cfg.D,)).astype(np.float32)).astype(np.float16)
    kw = (1.0 + 0.25 * normal_fp16(seed, 14, (cfg.D,)).astype(np.float32)).astype(np.float16)
    positions = np.tile(np.arange(cfg.seq_len, dtype=np.int32), cfg.num_seqs)
    num_blocks = (T + 15) // 16
    slots = permutation(seed, 15, num_blocks * 16)[:T].astype(np.int64)
    return Q, K, V, qw, kw, positions, slots, num_blocks


def chunked_layer_inputs(cfg: ChunkedPrefillConfig, seed: int = 0):
    """One layer's attention step on the chunked workload, before its prologue:
    the chunked-prefill inputs (Q as raw query projections; the caches hold the
    cached prefixes), the chunk's own raw K and V rows [total_q, H_kv, D]
    (streams 11/12), RMSNorm weights 1 + N(0,1)/4 (streams 13/14), each new
    token's position (prefix .. prefix + chunk - 1) and its cache slot (the slot
    of that position in its sequence's pages).  Returns a dict."""
    Q, kc, vc, cu, lens_kv, tables = chunked_prefill_inputs(cfg, seed)
    T = Q.shape[0]
    K = normal_fp16(seed, 11, (T, cfg.H_kv, cfg.D))
    V = normal_fp16(seed, 12, (T, cfg.H_kv, cfg.D))
    qw = (1.0 + 0.25 * normal_fp16(seed, 13, (cfg.D,)).astype(np.float32)).astype(np.float16)
    kw = (1.0 + 0.25 * normal_fp16(seed, 14, (cfg.D,)).astype(np.float32)).astype(np.float16)
    pos = np.tile(np.arange(cfg.prefix, cfg.prefix + cfg.chunk, dtype=np.int32), cfg.num_seqs)
    seq = np.repeat(np.arange(cfg.num_seqs), cfg.chunk)
    slots = tables[seq, pos // 16].astype(np.int64) * 16 + pos % 16
    return dict(Q=Q, k_cache=kc, v_cache=vc, cu_seqlens_q=cu, seq_lens_kv=lens_kv,
                block_tables=tables, K=K, V=V, q_weight=qw, k_weight=kw, positions=pos,
                slot_mapping=slots, max_pos=cfg.prefix + cfg.chunk)
