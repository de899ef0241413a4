"""kvc_decode_attn_noalloc: the decode step for callers that cannot allocate.

A plug-in inside a host engine that owns every device allocation, or a
caller whose device-memory budget is fixed at start-up, cannot hand
kvc_decode_attn a workspace.  kvc_decode_attn_noalloc takes its split-K
scratch from a fixed array in the library's own device memory instead.  The
GPU test first leaves non-zero records of a larger call in that array, then
calls both entry points through the C ABI on identical copies of one
compressed cache, two decode steps in a row (each appending a token): both
run the same kernels on the same split, so outputs, lse, lengths and the
appended rows must agree bit for bit; the outputs are also checked against
the CPU oracle's decode within the tolerance of the other decode tests.  The
host test checks the refusals that happen before any CUDA call.

This file is collected last on purpose: the shared scratch array keeps the
previous call's contents, and the test must pass after every other test as
well as alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.kvc_testutil import TOL, lse_err, np64, row_rel_err


def test_noalloc_refuses_on_the_host():
    from kv_cache_compression_attention_b300 import binding
    try:
        lib = binding.lib()
    except ImportError:
        pytest.skip("libkvc.so not built")
    limit = lib.kvc_decode_noalloc_scratch_bytes()
    assert limit == 16 << 20
    P = ctypes.c_void_p(16)
    f = lib.kvc_decode_attn_noalloc
    # 64 x 8 kv heads, G = 4, d = 128: 15360 rows fit, 15361 rows do not
    ok_need = lib.kvc_decode_workspace(64, 32, 8, 128, 15360, 1)
    assert ok_need <= limit < lib.kvc_decode_workspace(64, 32, 8, 128, 15361, 1)
    assert f(P, P, P, P, P, None, None, 1, 64, 32, 8, 128, 15361, 0.1, P, P, None) == -3
    assert f(None, P, P, P, P, None, None, 1, 64, 32, 8, 128, 64, 0.1, P, P, None) == -1
    assert f(P, P, P, P, P, None, None, 1, 0, 32, 8, 128, 64, 0.1, P, P, None) == -1


def _pool(lens, slack, d, dtype, seed):
    lens = np.asarray(lens)
    start = np.concatenate([[0], np.cumsum(lens + slack)[:-1]]).astype(np.int64)
    rows = int((lens + slack).sum())
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn((rows, d), generator=g).to(dtype)
    vc = torch.randn((rows, d), generator=g).to(dtype)
    return kc, vc, torch.from_numpy(start), torch.from_numpy(lens.astype(np.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_entry_point_two_calls(dtype):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kv_cache_compression_attention_b300 import binding as B
    from oracle import kvc_oracle as O
    B.lib()
    U, Hkv, G, d, slack = 2, 3, 4, 128, 2
    g = torch.Generator().manual_seed(22)
    # a larger call first, with other lengths, so that the shared array holds
    # non-zero records at the offsets the checked calls use
    dl = [3000, 7, 1500, 2999, 640, 1]
    dk, dv, ds, dn = [t.cuda() for t in _pool(dl, 1, d, dtype, 23)]
    dq = torch.randn((U, Hkv * G, d), generator=g).to(dtype).cuda()
    dout = torch.empty_like(dq)
    B.kvc_decode_attn_noalloc(dq, dk, dv, ds, dn, dout, None, max_len=max(dl) + 1,
                              scale=d ** -0.5)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    del dk, dv, ds, dn, dq, dout

    lens = [0, 1, 511, 512, 513, 2000]
    kc, vc, start, length = _pool(lens, slack, d, dtype, 21)
    # two identical copies: one for each entry point
    a = [t.cuda() for t in (kc, vc, start, length)]
    b = [t.clone().cuda() for t in (kc, vc, start, length)]
    # the oracle's own copy of the cache state (float64 arrays)
    o_kc, o_vc = np64(kc), np64(vc)
    o_start, o_len = start.numpy(), length.numpy()
    max_len = max(lens) + slack
    for step in range(2):
        q = torch.randn((U, Hkv * G, d), generator=g).to(dtype).cuda()
        kn = torch.randn((U, Hkv, d), generator=g).to(dtype).cuda()
        vn = torch.randn((U, Hkv, d), generator=g).to(dtype).cuda()
        out_a = torch.full_like(q, float("nan"))
        out_b = torch.full_like(q, float("nan"))
        lse_a = torch.full((U, Hkv * G), float("nan"), device="cuda")
        lse_b = torch.full_like(lse_a, float("nan"))
        B.kvc_decode_attn(q, a[0], a[1], a[2], a[3], out_a, lse_a, k_new=kn, v_new=vn,
                          max_len=max_len, scale=d ** -0.5)
        B.kvc_decode_attn_noalloc(q, b[0], b[1], b[2], b[3], out_b, lse_b, k_new=kn,
                                  v_new=vn, max_len=max_len, scale=d ** -0.5)
        torch.cuda.synchronize()
        assert B.kvc_device_status() == 0
        # same kernels, same split: identical bits
        np.testing.assert_array_equal(out_b.cpu().float().numpy(), out_a.cpu().float().numpy())
        np.testing.assert_array_equal(lse_b.cpu().numpy(), lse_a.cpu().numpy())
        np.testing.assert_array_equal(b[3].cpu().numpy(), a[3].cpu().numpy())
        np.testing.assert_array_equal(b[0].cpu().float().numpy(), a[0].cpu().float().numpy())
        np.testing.assert_array_equal(b[1].cpu().float().numpy(), a[1].cpu().float().numpy())
        # and the oracle's decode of the same step
        r_out, r_lse, o_kc, o_vc, o_len = O.decode_attn(np64(q), o_kc, o_vc, o_start, o_len,
                                                        np64(kn), np64(vn), d ** -0.5)
        assert row_rel_err(np64(out_b).reshape(-1, d), r_out.reshape(-1, d)) <= TOL[dtype]
        assert lse_err(np64(lse_b), r_lse) <= TOL[dtype]
    np.testing.assert_array_equal(b[3].cpu().numpy(), np.asarray(lens) + 2)
