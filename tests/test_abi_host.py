"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* libkvc.so loads and exports every function include/kvc.h declares;
* the ctypes signatures in the binding cover exactly those functions;
* argument errors are rejected on the host with KVC_ERR_INVALID /
  KVC_ERR_UNSUPPORTED before any CUDA call (so they work without a GPU);
* the status strings are stable.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")
LIB = os.path.join(ROOT, "kv_cache_compression_attention_b300", "libkvc.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kvc_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from kv_cache_compression_attention_b300 import build
        build.build()
    from kv_cache_compression_attention_b300 import binding
    return binding.load(LIB)


def test_header_declares_the_path():
    names = declared_functions()
    for required in ("kvc_score_attn", "kvc_score_linear", "kvc_select", "kvc_compact",
                     "kvc_decode_attn", "kvc_fidelity"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_match_header():
    from kv_cache_compression_attention_b300 import binding
    assert sorted(binding.SIGNATURES) == declared_functions()


def test_status_strings(lib):
    assert lib.kvc_status_string(0) == b"ok"
    assert lib.kvc_status_string(-1) == b"invalid argument"
    assert lib.kvc_status_string(-5) == b"device wait timed out"
    assert lib.kvc_status_string(12345) == b"unknown status"
    assert lib.kvc_version() >= 100


P = ctypes.c_void_p(16)   # a non-null, 16-byte aligned dummy pointer (never dereferenced)


def test_score_attn_rejects_bad_arguments(lib):
    f = lib.kvc_score_attn
    ok = dict(q=P, k=P, dt=1, U=1, Hq=8, Hkv=4, T=64, W=8, d=128, scale=0.1, hs=None, causal=1,
              scores=P, ws=None, wsb=0, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["dt"], a["U"], a["Hq"], a["Hkv"], a["T"], a["W"], a["d"],
                 a["scale"], a["hs"], a["causal"], a["scores"], a["ws"], a["wsb"], a["s"])

    assert call(q=None) == -1
    assert call(scores=None) == -1
    assert call(dt=7) == -1
    assert call(Hq=6) == -1              # Hq % Hkv
    assert call(W=65) == -1              # W > T
    assert call(T=0) == -1
    assert call(scale=float("nan")) == -1
    assert call(scale=0.0) == -1
    assert call(scale=-0.1) == -1
    assert call(d=96) == -2


def test_score_attn_agg_rejects_bad_arguments(lib):
    f = lib.kvc_score_attn_agg

    def call(agg, **kw):
        a = dict(q=P, k=P, dt=1, U=1, Hq=8, Hkv=4, T=64, W=8, d=128, scale=0.1, scores=P)
        a.update(kw)
        return f(a["q"], a["k"], a["dt"], a["U"], a["Hq"], a["Hkv"], a["T"], a["W"], a["d"],
                 a["scale"], None, 1, agg, a["scores"], None, 0, None)

    assert call(2) == -1                 # aggregation outside the enum
    assert call(-1) == -1
    assert call(1, q=None) == -1
    assert call(1, W=65) == -1
    assert call(1, d=96) == -2


def test_select_rejects_bad_arguments(lib):
    f = lib.kvc_select

    def call(scores=P, U=1, Hkv=2, T=16, mode=0, ratio=0.5, tau=0.0, hb=None, ns=1, nr=1,
             kept=P, counts=P, offs=P):
        return f(scores, U, Hkv, T, mode, ratio, tau, hb, ns, nr, kept, counts, offs, None, 0, None)

    assert call(scores=None) == -1
    assert call(mode=3) == -1
    assert call(ratio=1.5) == -1
    assert call(ratio=float("nan")) == -1
    assert call(ns=-1) == -1
    assert call(mode=2, hb=None) == -1
    assert call(T=(1 << 24) + 1, mode=1) == -2    # pool larger than supported
    assert call(Hkv=1025, T=1 << 14) == -2         # more than 2^24 keys pooled across heads
    assert call(Hkv=600, T=16) == -2               # more than 512 heads in one pool


def test_select_compact_rejects_bad_arguments(lib):
    f = lib.kvc_select_compact

    def call(scores=P, U=1, Hkv=2, T=16, mode=0, ratio=0.5, tau=0.0, hb=None, ns=1, nr=1,
             k=P, v=P, dtype=1, d=128, slack=0, kc=P, vc=P, cap=64, kept=P, counts=P, offs=P,
             start=P, length=P):
        return f(scores, U, Hkv, T, mode, ratio, tau, hb, ns, nr, k, v, dtype, d, slack, kc, vc,
                 cap, kept, counts, offs, start, length, None, 0, None)

    assert call(scores=None) == -1            # the select's rules
    assert call(mode=3) == -1
    assert call(ratio=1.5) == -1
    assert call(T=(1 << 24) + 1, mode=1) == -2
    assert call(k=None) == -1                 # the compaction's rules
    assert call(length=None) == -1
    assert call(dtype=7) == -1
    assert call(slack=-1) == -1
    assert call(d=100) == -2                  # 200-byte rows
    assert call(d=4096) == -2                 # 8 KB rows
    # the hand-off record: one pool only, up to 8 heads per pool
    # (16 CTA ranges x (threshold, tie cut, a count per head and 512-token sub-range))
    assert lib.kvc_select_compact_workspace(1, 8, 32768, 0) == 16 * (2 + 8 * 64) * 4
    assert lib.kvc_select_compact_workspace(1, 1, 4096, 1) == 16 * (2 + 64) * 4
    assert lib.kvc_select_compact_workspace(2, 8, 32768, 0) == 0
    assert lib.kvc_select_compact_workspace(1, 9, 32768, 0) == 0
    assert lib.kvc_select_compact_workspace(1, 4, 131072, 1) == 0     # four per-head pools


def test_compact_and_decode_reject_bad_arguments(lib):
    c = lib.kvc_compact
    assert c(None, P, 1, 1, 1, 8, 128, P, P, P, 0, P, P, 8, P, P, None) == -1
    assert c(P, P, 1, 1, 1, 8, 128, P, P, P, -1, P, P, 8, P, P, None) == -1
    assert c(P, P, 1, 1, 1, 8, 100, P, P, P, 0, P, P, 8, P, P, None) == -2   # 200-byte rows
    dec = lib.kvc_decode_attn
    args = [P, P, P, P, P, None, None, 1, 1, 8, 2, 128, 64, 0.1, P, P, P, 1 << 20, None]
    bad = list(args); bad[0] = None
    assert dec(*bad) == -1
    bad = list(args); bad[5] = P              # k_new without v_new
    assert dec(*bad) == -1
    bad = list(args); bad[9] = 3              # Hq % Hkv
    assert dec(*bad) == -1
    bad = list(args); bad[11] = 80            # d
    assert dec(*bad) == -2
    bad = list(args); bad[17] = 0             # workspace too small
    assert dec(*bad) == -3


def test_workspace_queries_are_pure_host(lib):
    assert lib.kvc_select_workspace(1, 8, 32768, 0) == 0
    n = lib.kvc_decode_workspace(64, 32, 8, 128, 10086, 1)
    chunks = (10086 + 1023) // 1024
    assert n == 64 * 8 * chunks * 4 * (128 + 2) * 4
    # tensor-core scoring path: per-CTA row partials (2 buffers x 1024 CTAs x G*W rows,
    # each (max, sum) as two tagged 64-bit words), independent of U and T; the SIMT
    # path keeps one lse per window row
    tc = 2 * 1024 * 256 * 16
    assert lib.kvc_score_attn_workspace(1, 32, 8, 32768, 64, 128, 1) == tc
    assert lib.kvc_score_attn_workspace(128, 32, 8, 16384, 64, 128, 1) == tc
    assert lib.kvc_score_attn_workspace(1, 8, 4, 1024, 32, 64, 0) == 8 * 32 * 4


def test_quantize_and_q8_decode_reject_bad_arguments(lib):
    qz = lib.kvc_quantize_rows
    assert qz(None, 1, 4, 128, P, P, None) == -1
    assert qz(P, 7, 4, 128, P, P, None) == -1                 # unknown dtype
    assert qz(P, 1, -1, 128, P, P, None) == -1                # negative row count
    assert qz(P, 1, 4, 96, P, P, None) == -2                  # d outside {64, 128}
    assert qz(P, 0, 4, 128, P, P, None) == -2                 # f32 rows
    dq = lib.kvc_decode_attn_q8
    args = [P, P, P, P, P, P, P, None, None, 1, 1, 8, 2, 128, 64, 0.1, P, P, P, 1 << 20, None]
    bad = list(args); bad[1] = None                           # no K codes
    assert dq(*bad) == -1
    bad = list(args); bad[7] = P                              # k_new without v_new
    assert dq(*bad) == -1
    bad = list(args); bad[12] = 3                             # Hq % Hkv
    assert dq(*bad) == -1
    bad = list(args); bad[13] = 64                            # d
    assert dq(*bad) == -2
    bad = list(args); bad[11] = 32; bad[12] = 2               # 16 query heads per kv head
    assert dq(*bad) == -2
    bad = list(args); bad[2] = ctypes.c_void_p(24)            # unaligned scale/offset pairs
    assert dq(*bad) == -2
    bad = list(args); bad[19] = 0                             # workspace too small
    assert dq(*bad) == -3


def test_prune_and_gather_reject_bad_arguments(lib):
    def arr(t, *v):
        return (t * len(v))(*v)
    pools = arr(ctypes.c_void_p, 16, 32)
    rb = arr(ctypes.c_int, 256, 256)
    pr = lib.kvc_decode_prune
    ok = [pools, rb, 2, P, P, P, P, 8, 16, 4, 0.5, 1000, None]
    for k, v, want in [(0, None, -1), (2, 0, -1), (2, 5, -1), (3, None, -1), (8, 0, -1),
                       (9, -1, -1), (10, float("nan"), -1), (11, -1, -1), (7, -1, -1)]:
        bad = list(ok); bad[k] = v
        assert pr(*bad) == want, (k, v)
    bad = list(ok); bad[0] = arr(ctypes.c_void_p, 16, None)
    assert pr(*bad) == -1                                     # a null pool
    bad = list(ok); bad[1] = arr(ctypes.c_int, 256, 24)
    assert pr(*bad) == -2                                     # rows not whole 16-byte vectors
    bad = list(ok); bad[0] = arr(ctypes.c_void_p, 16, 40)
    assert pr(*bad) == -2                                     # unaligned pool
    ga = lib.kvc_gather_scores
    assert ga(None, 1, 8, 64, P, P, P, P, 100, None) == -1
    assert ga(P, -1, 8, 64, P, P, P, P, 100, None) == -1
    assert ga(P, 1, 8, 64, P, P, P, P, -1, None) == -1
    assert ga(P, 9000, 8, 64, P, P, P, P, 100, None) == -2    # more heads than grid rows


def test_vector_entry_points_reject_bad_arguments(lib):
    r = lib.kvc_vector_residual
    ok = [P, P, P, 1, 1, 8, 64, 128, P, P, 4, 16, P, None]
    assert r(*ok[:0], None, *ok[1:]) == -1                      # no K
    for k, v, want in [(3, 7, -1), (5, 0, -1), (10, -1, -1), (7, 64, -2), (3, 0, -2)]:
        bad = list(ok); bad[k] = v
        assert r(*bad) == want, (k, v)
    bad = list(ok); bad[2] = ctypes.c_void_p(24)
    assert r(*bad) == -2                                        # unaligned W
    sv = lib.kvc_vector_select
    oks = [P, 1, 8, 32768, P, 3932, P, P, P, None]
    for k, v, want in [(0, None, -1), (4, None, -1), (8, None, -1), (1, 0, -1), (3, -5, -1),
                       (5, -1, -1), (5, 8 * 32768 + 1, -1), (3, 1 << 22, -2)]:
        bad = list(oks); bad[k] = v
        assert sv(*bad) == want, (k, v)
    c = lib.kvc_vector_compact
    okc = [P, P, 1, 1, 8, 64, 128, P, P, P, P, P, P, 0, P, 100, P, 100, P, P, P, P, None]
    bad = list(okc); bad[9] = None
    assert c(*bad) == -1                                        # no approximated positions
    bad = list(okc); bad[13] = -1
    assert c(*bad) == -1                                        # negative slack
    bad = list(okc); bad[6] = 64
    assert c(*bad) == -2                                        # d
    d = lib.kvc_decode_attn_vector
    okd = [P, P, P, P, P, P, P, P, None, None, 1, 1, 8, 2, 128, 64, 0.1, P, P, P, 1 << 20, None]
    bad = list(okd); bad[7] = None
    assert d(*bad) == -1                                        # no predictor
    bad = list(okd); bad[8] = P
    assert d(*bad) == -1                                        # k_new without v_new
    bad = list(okd); bad[14] = 64
    assert d(*bad) == -2
    bad = list(okd); bad[20] = 0
    assert d(*bad) == -3                                        # workspace too small
    # one more split-K chunk than the plain decode: approximated and exact rows
    # are chunked apart
    assert lib.kvc_decode_vector_workspace(64, 32, 8, 128, 10086) == \
        64 * 8 * (10 + 1) * 4 * 130 * 4


def test_score_mlp_rejects_bad_arguments(lib):
    f = lib.kvc_score_mlp
    ws = ctypes.c_void_p(256)
    ok = [P, P, P, P, P, 1, 1, 128, 3584, 448, 4, P, ws, 1 << 40, None]
    bad = list(ok); bad[0] = None
    assert f(*bad) == -1
    bad = list(ok); bad[10] = 9
    assert f(*bad) == -2                                        # more than 8 kv heads
    bad = list(ok); bad[9] = 452
    assert f(*bad) == -2                                        # Dm not a multiple of 8
    bad = list(ok); bad[9] = 2048
    assert f(*bad) == -2                                        # Dm beyond 1024
    bad = list(ok); bad[12] = P
    assert f(*bad) == -2                                        # workspace not 256-byte aligned
    bad = list(ok); bad[13] = 1000
    assert f(*bad) == -3
    assert lib.kvc_score_mlp_workspace(3584, 448) == 448 * 3584 * 2        # w1 transposed
    assert lib.kvc_score_mlp_workspace(512, 16) == 32 * 512 * 2            # rows padded to 32
    assert lib.kvc_score_mlp_workspace(4096, 1000) == 1024 * 4096 * 2      # two passes of 512
    assert lib.kvc_score_mlp_workspace(0, 448) == 0


def test_score_kvzip_plus_rejects_bad_arguments(lib):
    f = lib.kvc_score_kvzip_plus
    ws = ctypes.c_void_p(256)
    ok = [P, P, P, P, P, 1, 1, 32, 8, 4096, 64, 128, 0.09, None, 1, P, ws, 1 << 40, None]
    for k, v, want in [(4, None, -1), (9, 3, -1), (10, 5000, -1), (12, 0.0, -1), (11, 64, -2),
                       (5, 0, -2), (17, 100, -3)]:
        bad = list(ok); bad[k] = v
        assert f(*bad) == want, (k, v)
    bad = list(ok); bad[16] = P
    assert f(*bad) == -2                                        # workspace not 256-byte aligned
    # value norms, then the tensor-core scorer's row partials (G*W = 256, W = 64)
    assert lib.kvc_score_kvzip_plus_workspace(1, 32, 8, 32768, 64) == \
        32 * 32768 * 4 + 2 * 1024 * 256 * 16
    # G*W = 256 with W = 32: quarters span two heads, the SIMT pass (one lse per row)
    assert lib.kvc_score_kvzip_plus_workspace(1, 32, 4, 1024, 32) == 32 * 1024 * 4 + 32 * 32 * 4


def test_prune_ring_rejects_bad_arguments(lib):
    def arr(t, *v):
        return (t * len(v))(*v)
    pools = arr(ctypes.c_void_p, 16, 32)
    rb = arr(ctypes.c_int, 256, 256)
    pr = lib.kvc_decode_prune_ring
    ok = [pools, rb, 2, P, P, P, P, 1000, P, 8, 16, 4, 0.5, 1000, None]
    for k, v, want in [(0, None, -1), (2, 0, -1), (2, 5, -1), (3, None, -1), (6, None, -1),
                       (7, -1, -1), (8, None, -1), (10, 0, -1), (11, -1, -1),
                       (12, float("nan"), -1), (13, -1, -1), (9, -1, -1)]:
        bad = list(ok); bad[k] = v
        assert pr(*bad) == want, (k, v)
    bad = list(ok); bad[1] = arr(ctypes.c_int, 256, 24)
    assert pr(*bad) == -2                                     # rows not whole 16-byte vectors
    bad = list(ok); bad[0] = arr(ctypes.c_void_p, 16, 40)
    assert pr(*bad) == -2                                     # unaligned pool
    ri = lib.kvc_prune_ring_init
    assert ri(None, 8, 16, 100, P, None) == -1
    assert ri(P, 8, 16, 100, None, None) == -1
    assert ri(P, -1, 16, 100, P, None) == -1
    assert ri(P, 8, 0, 100, P, None) == -1
    assert ri(P, 8, 16, -1, P, None) == -1
