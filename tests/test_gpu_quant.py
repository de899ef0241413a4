"""GPU group quantisation of the compacted cache ([KVTC] §2B: groups of 32
sharing a scale and an offset) and decode over the quantised pool, through
the C ABI and against the CPU oracle: the codes and (scale, offset) pairs
bit for bit, the decode outputs within the bf16 tolerance of the oracle's
decode over the dequantised pool, the appended rows quantised bit for bit.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_attention_b300 import inputs
from oracle import kvc_oracle as O
from tests.kvc_testutil import lse_err, np64, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kv_cache_compression_attention_b300 import binding
    binding.lib()
    return binding


def gpu_quantize(B, x):
    rows, d = x.shape
    codes = torch.empty((rows, d), dtype=torch.uint8, device="cuda")
    params = torch.empty((rows, d // 32, 2), dtype=torch.float16, device="cuda")
    B.kvc_quantize_rows(x, codes, params)
    torch.cuda.synchronize()
    return codes, params


def test_quantize_rows_bit_exact(B):
    g = torch.Generator().manual_seed(31)
    x = torch.randn((777, 128), generator=g) * torch.tensor([1.0, 8.0, 0.02, 3.0]).repeat(32)
    x[5, :32] = 0.75                              # a constant group
    x[6, 32:64] = torch.arange(32.0) * 8          # an integer ramp
    x = x.to(torch.bfloat16)
    codes, params = gpu_quantize(B, x.cuda())
    rc, rp = O.quantize_rows(x.float().numpy())
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(params.cpu().numpy().view(np.uint16), rp.view(np.uint16))
    x64 = torch.randn((100, 64), generator=g).to(torch.bfloat16)
    c64, p64 = gpu_quantize(B, x64.cuda())
    rc64, rp64 = O.quantize_rows(x64.float().numpy())
    np.testing.assert_array_equal(c64.cpu().numpy(), rc64)
    np.testing.assert_array_equal(p64.cpu().numpy().view(np.uint16), rp64.view(np.uint16))


def pool(lens, slack, d, seed):
    lens = np.asarray(lens)
    start = np.concatenate([[0], np.cumsum(lens + slack)[:-1]]).astype(np.int64)
    rows = int((lens + slack).sum())
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn((rows, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((rows, d), generator=g).to(torch.bfloat16)
    return kc, vc, start, lens.astype(np.int32)


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("append", [True, False])
def test_decode_q8_small(B, G, append):
    U, Hkv, d = 2, 3, 128
    lens = [0, 1, 511, 512, 513, 2000]
    kc, vc, start, lens = pool(lens, 1, d, 32)
    g = torch.Generator().manual_seed(33)
    q = torch.randn((U, Hkv * G, d), generator=g).to(torch.bfloat16)
    kn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16) if append else None
    vn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16) if append else None
    kq, kp = gpu_quantize(B, kc.cuda())
    vq, vp = gpu_quantize(B, vc.cuda())
    st, ln = torch.from_numpy(start).cuda(), torch.from_numpy(lens).cuda()
    out = torch.full((U, Hkv * G, d), float("nan"), device="cuda").to(torch.bfloat16)
    lse = torch.full((U, Hkv * G), float("nan"), device="cuda")
    B.kvc_decode_attn_q8(q.cuda(), kq, kp, vq, vp, st, ln, out, lse,
                         k_new=None if kn is None else kn.cuda(),
                         v_new=None if vn is None else vn.cuda(), max_len=int(lens.max()) + 1)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    rkq, rkp = O.quantize_rows(kc.float().numpy())
    rvq, rvp = O.quantize_rows(vc.float().numpy())
    kd, vd = O.dequantize_rows(rkq, rkp), O.dequantize_rows(rvq, rvp)
    ro, rl, _, _, rlen = O.decode_attn(np64(q), kd, vd, start, lens,
                                       None if kn is None else np64(kn),
                                       None if vn is None else np64(vn), d ** -0.5)
    assert row_rel_err(np64(out).reshape(-1, d), ro.reshape(-1, d)) <= 2e-2
    assert lse_err(np64(lse), rl) <= 2e-2
    np.testing.assert_array_equal(ln.cpu().numpy(), rlen)
    if append:
        # the appended rows, quantised like every other row
        rows = [int(start[i] + lens[i]) for i in range(U * Hkv)]
        akq, akp = O.quantize_rows(kn.float().numpy().reshape(-1, d))
        avq, avp = O.quantize_rows(vn.float().numpy().reshape(-1, d))
        np.testing.assert_array_equal(kq.cpu().numpy()[rows], akq)
        np.testing.assert_array_equal(vq.cpu().numpy()[rows], avq)
        np.testing.assert_array_equal(kp.cpu().numpy()[rows].view(np.uint16), akp.view(np.uint16))
        np.testing.assert_array_equal(vp.cpu().numpy()[rows].view(np.uint16), avp.view(np.uint16))


@pytest.mark.parametrize("G", [1, 3, 8])
def test_decode_q8_chunk_edges(B, G):
    """Lengths around the quantised kernel's 2048-row chunks and 64-row
    stages, with appends, against the oracle's decode over the dequantised pool."""
    U, Hkv, d = 1, 6, 128
    kc, vc, start, lens = pool([63, 1025, 2047, 2048, 2049, 4097], 2, d, 4)
    g = torch.Generator().manual_seed(34 + G)
    q = torch.randn((U, Hkv * G, d), generator=g).to(torch.bfloat16)
    kn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16)
    vn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16)
    kq, kp = gpu_quantize(B, kc.cuda())
    vq, vp = gpu_quantize(B, vc.cuda())
    st, ln = torch.from_numpy(start).cuda(), torch.from_numpy(lens).cuda()
    out = torch.full((U, Hkv * G, d), float("nan"), device="cuda").to(torch.bfloat16)
    lse = torch.full((U, Hkv * G), float("nan"), device="cuda")
    B.kvc_decode_attn_q8(q.cuda(), kq, kp, vq, vp, st, ln, out, lse, k_new=kn.cuda(),
                         v_new=vn.cuda(), max_len=int(lens.max()) + 1)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    rkq, rkp = O.quantize_rows(kc.float().numpy())
    rvq, rvp = O.quantize_rows(vc.float().numpy())
    kd, vd = O.dequantize_rows(rkq, rkp), O.dequantize_rows(rvq, rvp)
    # the new token is attended exactly (it is appended quantised afterwards)
    ro, rl, _, _, rlen = O.decode_attn(np64(q), kd, vd, start, lens, np64(kn), np64(vn),
                                       d ** -0.5)
    assert row_rel_err(np64(out).reshape(-1, d), ro.reshape(-1, d)) <= 2e-2
    assert lse_err(np64(lse), rl) <= 2e-2
    np.testing.assert_array_equal(ln.cpu().numpy(), rlen)


def test_decode_q8_batch64_sampled(B):
    """The batch-64 compressed caches: quantised once, four decode steps
    (appends quantised), sampled sequences against the oracle at steps 0 and 3."""
    w = inputs.WORKLOADS["c5_decode"]
    lens = inputs.head_budgets(w, "cpu")
    kc, vc, start, length = inputs.compressed_pool(w, lens, "cuda")
    kq, kp = gpu_quantize(B, kc)
    vq, vp = gpu_quantize(B, vc)
    max_len = int(lens.max()) + 8
    ws = torch.empty(B.kvc_decode_workspace(w.U, w.Hq, w.Hkv, w.d, max_len), dtype=torch.uint8,
                     device="cuda")
    sample_u = [3, 60]
    heads = [u * w.Hkv + g for u in sample_u for g in range(w.Hkv)]
    st_np, ln0 = start.cpu().numpy(), length.cpu().numpy()
    # the sampled heads' rows (dequantised by the oracle), re-based into a small pool
    rkq, rkp = O.quantize_rows(kc.float().cpu().numpy())
    rvq, rvp = O.quantize_rows(vc.float().cpu().numpy())
    np.testing.assert_array_equal(kq.cpu().numpy(), rkq)
    pk, pv, pstart, base = [], [], [], 0
    for i in heads:
        rows = slice(int(st_np[i]), int(st_np[i]) + int(ln0[i]) + w.slack)
        pk.append(O.dequantize_rows(rkq[rows], rkp[rows]))
        pv.append(O.dequantize_rows(rvq[rows], rvp[rows]))
        pstart.append(base)
        base += int(ln0[i]) + w.slack
    okc, ovc = np.concatenate(pk), np.concatenate(pv)
    ostart = np.array(pstart, dtype=np.int64)
    olen = ln0[heads].astype(np.int32)
    for step in range(4):
        q, kn, vn = inputs.decode_step_inputs(w, step, "cuda")
        out = torch.empty_like(q)
        lse = torch.empty((w.U, w.Hq), device="cuda")
        B.kvc_decode_attn_q8(q, kq, kp, vq, vp, start, length, out, lse, k_new=kn, v_new=vn,
                             max_len=max_len, scale=w.scale, workspace=ws)
        qs, kns, vns = np64(q[sample_u]), np64(kn[sample_u]), np64(vn[sample_u])
        # the oracle appends the dequantised quantisation of the new rows
        kqd = O.dequantize_rows(*O.quantize_rows(kn[sample_u].float().cpu().numpy().reshape(-1, w.d)))
        vqd = O.dequantize_rows(*O.quantize_rows(vn[sample_u].float().cpu().numpy().reshape(-1, w.d)))
        ro, rl, _, _, _ = O.decode_attn(qs, okc, ovc, ostart, olen, kns, vns, w.scale)
        for x, i in enumerate(range(len(heads))):
            okc[ostart[i] + olen[i]] = kqd[x]
            ovc[ostart[i] + olen[i]] = vqd[x]
        olen = olen + 1
        if step in (0, 3):
            got = np64(out[sample_u]).reshape(-1, w.d)
            assert row_rel_err(got, ro.reshape(-1, w.d)) <= 2e-2, step
            assert lse_err(np64(lse[sample_u]), rl) <= 2e-2, step
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    np.testing.assert_array_equal(length.cpu().numpy(), ln0 + 4)
