"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/attn.h declares, and rejects bad arguments
before launching anything.  Pointers here are fake addresses: every call below
returns from argument validation without touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

import attention_gqa_causal_gb300 as ag

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

P = ctypes.c_void_p
A16 = 0x10000          # a 16-byte aligned fake device address
A16B = 0x20000000
MIS = 0x10008          # 8-byte aligned only


def declared():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_all_bound_symbols():
    names = set(declared())
    assert names == set(ag.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = ag.load()
    for name in declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (attn_\w+)", out))
    assert set(declared()) <= exported


def test_version_and_status_strings():
    assert ag.attn_version() == 100
    assert ag.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5, -6):
        assert ag.status_string(code) not in ("ok", "unknown status")
    assert ag.status_string(-99) == "unknown status"


def prefill(Q=A16, K=A16 + 0x100000, V=A16 + 0x200000, O=A16B, B=1, S=64, Hq=4, Hkv=2, D=128, causal=1):
    return ag.load().attn_prefill(P(Q), P(K), P(V), P(O), B, S, Hq, Hkv, D, causal, P(0))


def test_prefill_validation():
    assert prefill(D=64) == ag.ATTN_ERR_UNSUPPORTED
    assert prefill(D=256) == ag.ATTN_ERR_UNSUPPORTED
    assert prefill(Hq=6, Hkv=4) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(Hq=0) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(Hkv=0) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(B=-1) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(S=-5) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(Q=0) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(O=0) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(K=MIS) == ag.ATTN_ERR_INVALID_ARG
    assert prefill(O=A16 + 64) == ag.ATTN_ERR_INVALID_ARG      # O overlaps Q
    assert prefill(O=A16 + 0x100000 + 16) == ag.ATTN_ERR_INVALID_ARG  # O overlaps K
    # empty problems are valid no-ops (nothing launched, no device needed)
    assert prefill(B=0) == ag.ATTN_OK
    assert prefill(S=0) == ag.ATTN_OK
    assert prefill(B=0, Q=0, K=0, V=0, O=0) == ag.ATTN_OK


def decode(q=A16, kc=A16 + 0x100000, vc=A16 + 0x200000, out=A16B, bt=A16 + 0x300000, sl=A16 + 0x400000,
           N=4, Hq=16, Hkv=8, D=128, mb=128, bs=16):
    return ag.load().attn_decode_paged(P(q), P(kc), P(vc), P(out), P(bt), P(sl), N, Hq, Hkv, D, mb, bs, P(0))


def test_decode_validation():
    assert decode(bs=32) == ag.ATTN_ERR_UNSUPPORTED
    assert decode(bs=8) == ag.ATTN_ERR_UNSUPPORTED
    assert decode(D=64) == ag.ATTN_ERR_UNSUPPORTED
    assert decode(Hq=12, Hkv=8) == ag.ATTN_ERR_INVALID_ARG
    assert decode(N=-1) == ag.ATTN_ERR_INVALID_ARG
    assert decode(mb=0) == ag.ATTN_ERR_INVALID_ARG
    assert decode(bt=0) == ag.ATTN_ERR_INVALID_ARG
    assert decode(sl=A16 + 2) == ag.ATTN_ERR_INVALID_ARG
    assert decode(kc=MIS) == ag.ATTN_ERR_INVALID_ARG
    assert decode(out=A16 + 32) == ag.ATTN_ERR_INVALID_ARG      # out overlaps q
    assert decode(N=0) == ag.ATTN_OK
    assert decode(N=0, q=0, kc=0, vc=0, out=0, bt=0, sl=0) == ag.ATTN_OK


def test_workspace_sizes_and_checks():
    ws = ag.attn_decode_paged_workspace_bytes
    # default split of 64 pages: 128 pages -> 2 splits; [N*H_q*2*128] f32 + [N*H_q*2] f32, 256-aligned
    n = ws(256, 16, 8, 128, 128, 16, 0)
    assert n == 256 * 16 * 2 * 128 * 4 + ((256 * 16 * 2 * 4 + 255) // 256) * 256
    # a small grid gets smaller splits: 4 seqs x 8 kv heads x ceil(128/pps) CTAs < 1824 down to pps = 4
    assert ws(4, 16, 8, 128, 128, 16, 0) == ws(4, 16, 8, 128, 128, 16, 4)
    assert ws(256, 16, 8, 128, 128, 16, 1) == 256 * 16 * 128 * 128 * 4 + 256 * 16 * 128 * 4
    assert ws(8, 16, 8, 128, 2048, 16, 16) == 8 * 16 * 128 * 128 * 4 + ((8 * 16 * 128 * 4 + 255) // 256) * 256
    assert ws(4, 16, 8, 64, 128, 16, 0) == 0
    assert ws(4, 16, 8, 128, 128, 32, 0) == 0
    lib = ag.load()
    need = ws(4, 16, 8, 128, 128, 16, 0)
    args = [P(A16), P(A16 + 0x100000), P(A16 + 0x200000), P(A16B), P(A16 + 0x300000), P(A16 + 0x400000),
            4, 16, 8, 128, 128, 16, 0]
    assert lib.attn_decode_paged_ws(*args, P(0x40000000), need - 1, P(0)) == ag.ATTN_ERR_WORKSPACE
    assert lib.attn_decode_paged_ws(*args, P(0), need, P(0)) == ag.ATTN_ERR_WORKSPACE
    assert lib.attn_decode_paged_ws(*args, P(0x40000010), need, P(0)) == ag.ATTN_ERR_WORKSPACE


def test_combine_validation():
    lib = ag.load()
    assert lib.attn_lse_combine(P(A16), P(A16B), P(A16 + 0x300000), 4, 3, 64, P(0)) == ag.ATTN_ERR_UNSUPPORTED
    assert lib.attn_lse_combine(P(A16), P(A16B), P(A16 + 0x300000), -1, 3, 128, P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_lse_combine(P(A16), P(A16B), P(A16 + 0x300000), 4, 0, 128, P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_lse_combine(P(0), P(A16B), P(A16 + 0x300000), 4, 3, 128, P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_lse_combine(P(0), P(0), P(0), 0, 3, 128, P(0)) == ag.ATTN_OK


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 4, 2, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        ag.attn_prefill(x, x[:, :, :1], x[:, :, :1], x.clone())


def test_kv_append_validation():
    lib = ag.load()
    LL = ctypes.c_longlong

    def app(kn=A16, vn=A16 + 0x10000, kc=A16B, vc=A16B + 0x1000000, sm=A16 + 0x20000, T=4, Hkv=8, D=128,
            bs=16, nb=16):
        return lib.attn_kv_append(P(kn), P(vn), P(kc), P(vc), P(sm), T, Hkv, D, bs, LL(nb), P(0))

    assert app(D=64) == ag.ATTN_ERR_UNSUPPORTED
    assert app(bs=8) == ag.ATTN_ERR_UNSUPPORTED
    assert app(T=-1) == ag.ATTN_ERR_INVALID_ARG
    assert app(sm=A16 + 0x20004) == ag.ATTN_ERR_INVALID_ARG      # slot_mapping must be 8-byte aligned
    assert app(kn=0) == ag.ATTN_ERR_INVALID_ARG
    assert app(kc=A16) == ag.ATTN_ERR_INVALID_ARG                # cache overlaps the new rows
    assert app(T=0) == ag.ATTN_OK


def test_prefill_paged_validation():
    lib = ag.load()
    LL = ctypes.c_longlong

    def pp(Q=A16, kc=A16B, vc=A16B + 0x1000000, O=A16 + 0x100000, cu=A16 + 0x200000, sl=A16 + 0x200100,
           bt=A16 + 0x200200, B=2, mq=64, tq=100, Hq=4, Hkv=2, D=128, mb=8, bs=16, nb=16, causal=1):
        return lib.attn_prefill_paged(P(Q), P(kc), P(vc), P(O), P(cu), P(sl), P(bt), B, mq, tq, Hq, Hkv, D,
                                      mb, bs, LL(nb), causal, P(0))

    assert pp(D=64) == ag.ATTN_ERR_UNSUPPORTED
    assert pp(bs=32) == ag.ATTN_ERR_UNSUPPORTED
    assert pp(Hq=6, Hkv=4) == ag.ATTN_ERR_INVALID_ARG
    assert pp(B=-1) == ag.ATTN_ERR_INVALID_ARG
    assert pp(mb=0) == ag.ATTN_ERR_INVALID_ARG
    assert pp(nb=0) == ag.ATTN_ERR_INVALID_ARG
    assert pp(cu=0) == ag.ATTN_ERR_INVALID_ARG
    assert pp(O=A16 + 64) == ag.ATTN_ERR_INVALID_ARG          # O overlaps Q
    assert pp(O=A16B + 128) == ag.ATTN_ERR_INVALID_ARG        # O overlaps the K cache
    assert pp(B=0) == ag.ATTN_OK and pp(tq=0) == ag.ATTN_OK and pp(mq=0) == ag.ATTN_OK


def test_rope_table_validation():
    lib = ag.load()
    D = ctypes.c_double
    assert lib.attn_rope_cos_sin_table(P(A16), 100, 64, D(1e4), P(0)) == ag.ATTN_ERR_UNSUPPORTED
    assert lib.attn_rope_cos_sin_table(P(A16), -1, 128, D(1e4), P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_rope_cos_sin_table(P(A16), 100, 128, D(0.0), P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_rope_cos_sin_table(P(A16), 100, 128, D(float("inf")), P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_rope_cos_sin_table(P(MIS), 100, 128, D(1e4), P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_rope_cos_sin_table(P(0), 100, 128, D(1e4), P(0)) == ag.ATTN_ERR_INVALID_ARG
    assert lib.attn_rope_cos_sin_table(P(A16), 0, 128, D(1e4), P(0)) == ag.ATTN_OK


def test_qk_norm_rope_validation():
    lib = ag.load()
    F = ctypes.c_float
    # Q 4 tokens x 8 heads x 256 B = 8 KB at A16; K 4 KB at A16 + 0x4000
    base = dict(Q=A16, K=A16 + 0x4000, qw=A16 + 0x8000, kw=A16 + 0x8100, cs=A16 + 0x10000,
                mp=64, pos=A16 + 0x20000, T=4, Hq=8, Hkv=4, D=128, eps=1e-6)

    def qr(**kw):
        a = dict(base, **kw)
        return lib.attn_qk_norm_rope(P(a["Q"]), P(a["K"]), P(a["qw"]), P(a["kw"]), P(a["cs"]), a["mp"],
                                     P(a["pos"]), a["T"], a["Hq"], a["Hkv"], a["D"], F(a["eps"]), P(0))

    assert qr(D=64) == ag.ATTN_ERR_UNSUPPORTED
    assert qr(T=-1) == ag.ATTN_ERR_INVALID_ARG
    assert qr(Hkv=0) == ag.ATTN_ERR_INVALID_ARG
    assert qr(mp=0) == ag.ATTN_ERR_INVALID_ARG
    assert qr(eps=-1.0) == ag.ATTN_ERR_INVALID_ARG
    assert qr(eps=float("nan")) == ag.ATTN_ERR_INVALID_ARG
    assert qr(pos=0) == ag.ATTN_ERR_INVALID_ARG
    assert qr(cs=MIS) == ag.ATTN_ERR_INVALID_ARG                  # table must be 16-byte aligned
    assert qr(qw=A16 + 0x8008) == ag.ATTN_ERR_INVALID_ARG         # weight must be 16-byte aligned
    assert qr(K=A16 + 0x1000) == ag.ATTN_ERR_INVALID_ARG          # K overlaps Q
    assert qr(qw=A16 + 0x100) == ag.ATTN_ERR_INVALID_ARG          # a weight inside Q
    assert qr(cs=A16 + 0x1000) == ag.ATTN_ERR_INVALID_ARG         # the table inside Q
    assert qr(Q=A16B, Hq=190, Hkv=3) == ag.ATTN_ERR_UNSUPPORTED   # more than 192 rows per token
    assert qr(T=0) == ag.ATTN_OK
    assert qr(T=0, qw=0, kw=0) == ag.ATTN_OK                      # null weights are allowed


def test_qk_norm_rope_append_validation():
    lib = ag.load()
    F, LL = ctypes.c_float, ctypes.c_longlong
    base = dict(Q=A16, K=A16 + 0x4000, V=A16 + 0x6000, qw=A16 + 0x8000, kw=A16 + 0x8100,
                cs=A16 + 0x10000, mp=64, pos=A16 + 0x20000, sm=A16 + 0x20100, kc=A16B,
                vc=A16B + 0x1000000, T=4, Hq=8, Hkv=4, D=128, bs=16, nb=16, eps=1e-6)

    def qa(**kw):
        a = dict(base, **kw)
        return lib.attn_qk_norm_rope_append(
            P(a["Q"]), P(a["K"]), P(a["V"]), P(a["qw"]), P(a["kw"]), P(a["cs"]), a["mp"], P(a["pos"]),
            P(a["sm"]), P(a["kc"]), P(a["vc"]), a["T"], a["Hq"], a["Hkv"], a["D"], a["bs"], LL(a["nb"]),
            F(a["eps"]), P(0))

    assert qa(D=64) == ag.ATTN_ERR_UNSUPPORTED
    assert qa(bs=32) == ag.ATTN_ERR_UNSUPPORTED
    assert qa(nb=-1) == ag.ATTN_ERR_INVALID_ARG
    assert qa(V=0) == ag.ATTN_ERR_INVALID_ARG
    assert qa(sm=A16 + 0x20104) == ag.ATTN_ERR_INVALID_ARG         # slot_mapping must be 8-byte aligned
    assert qa(V=A16 + 0x1000) == ag.ATTN_ERR_INVALID_ARG          # V overlaps Q
    assert qa(kc=A16) == ag.ATTN_ERR_INVALID_ARG                  # cache overlaps Q
    assert qa(vc=A16B + 0x100) == ag.ATTN_ERR_INVALID_ARG         # the two caches overlap
    assert qa(vc=A16 + 0x10000) == ag.ATTN_ERR_INVALID_ARG        # cache over the cos/sin table
    assert qa(Q=A16B + 0x4000000, Hq=180, Hkv=7) == ag.ATTN_ERR_UNSUPPORTED   # 194 rows per token
    assert qa(T=0) == ag.ATTN_OK


def test_qk_norm_rope_append_keys_only_validation():
    # Q = NULL: keys and values only; the row limit then counts 2 * H_kv alone
    lib = ag.load()
    F, LL = ctypes.c_float, ctypes.c_longlong

    def qa(Q=0, K=A16 + 0x4000, V=A16 + 0x6000, T=4, Hq=8, Hkv=4, nb=16, eps=1e-6):
        return lib.attn_qk_norm_rope_append(
            P(Q), P(K), P(V), P(A16 + 0x8000), P(A16 + 0x8100), P(A16 + 0x10000), 64, P(A16 + 0x20000),
            P(A16 + 0x20100), P(A16B), P(A16B + 0x1000000), T, Hq, Hkv, 128, 16, LL(nb), F(eps), P(0))

    assert qa(K=0) == ag.ATTN_ERR_INVALID_ARG
    assert qa(Hq=0) == ag.ATTN_ERR_INVALID_ARG
    assert qa(Hq=97, Hkv=97, K=A16B + 0x4000000, V=A16B + 0x5000000) == ag.ATTN_ERR_UNSUPPORTED  # 194 rows
    assert qa(T=0) == ag.ATTN_OK


def test_prefill_paged_qk_norm_rope_validation():
    lib = ag.load()
    F, LL = ctypes.c_float, ctypes.c_longlong

    def pr(Q=A16, kc=A16B, vc=A16B + 0x1000000, O=A16 + 0x100000, cu=A16 + 0x200000,
           sl=A16 + 0x200100, bt=A16 + 0x200200, qw=A16 + 0x300000, cs=A16 + 0x400000, mp=4096,
           eps=1e-6, B=2, mq=64, tq=100, Hq=4, Hkv=2, D=128, mb=8, bs=16, nb=16, causal=1):
        return lib.attn_prefill_paged_qk_norm_rope(
            P(Q), P(kc), P(vc), P(O), P(cu), P(sl), P(bt), P(qw), P(cs), mp, F(eps), B, mq, tq, Hq, Hkv,
            D, mb, bs, LL(nb), causal, P(0))

    assert pr(D=64) == ag.ATTN_ERR_UNSUPPORTED
    assert pr(bs=32) == ag.ATTN_ERR_UNSUPPORTED
    assert pr(mp=0) == ag.ATTN_ERR_INVALID_ARG
    assert pr(eps=-1.0) == ag.ATTN_ERR_INVALID_ARG
    assert pr(eps=float("inf")) == ag.ATTN_ERR_INVALID_ARG
    assert pr(cs=0) == ag.ATTN_ERR_INVALID_ARG
    assert pr(cs=MIS) == ag.ATTN_ERR_INVALID_ARG                  # table must be 16-byte aligned
    assert pr(qw=A16 + 0x300008) == ag.ATTN_ERR_INVALID_ARG       # weight must be 16-byte aligned
    assert pr(O=A16 + 0x400000 - 0x1000) == ag.ATTN_ERR_INVALID_ARG   # O over the table
    assert pr(O=A16 + 64) == ag.ATTN_ERR_INVALID_ARG              # O overlaps Q
    assert pr(Hq=6, Hkv=4) == ag.ATTN_ERR_INVALID_ARG
    assert pr(B=0) == ag.ATTN_OK and pr(tq=0) == ag.ATTN_OK
    assert pr(B=0, qw=0) == ag.ATTN_OK                            # no norm weight is allowed
