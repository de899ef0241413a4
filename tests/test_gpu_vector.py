"""GPU VECTOR three-way routing through the C ABI against the CPU oracle:
reconstruction-error keys within fp32 tolerance (NaN pattern exact), the
lowest-error choice and the K-for-all / V-for-exact compaction bit-exact on
the same keys, decode over the routed cache (values of approximated rows
rebuilt as W k) within the bf16 tolerance; the full 32k Llama-shaped layer
with p_c = 0.9, p_a = 0.05, and the batch-64 decode over VECTOR caches.
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


def bits(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


def key_close(got, ref):
    """NaN pattern exact; values within 1e-3 relative (fp32 accumulation of the
    d x d product against float64)."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    if ok.any():
        err = np.abs(got[ok] - ref[ok]) / (np.abs(ref[ok]) + 1e-3)
        assert err.max() <= 1e-3, err.max()


def small_case(seed, U=2, Hkv=3, T=300, d=128, keep=0.4, n_sink=4, n_recent=16):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn((U, Hkv, T, d), generator=g).to(torch.bfloat16)
    W = (torch.randn((Hkv, d, d), generator=g) / d ** 0.5).to(torch.bfloat16)
    sigma = torch.rand((U, Hkv, T, 1), generator=g)
    v = (torch.einsum("ugty,gxy->ugtx", k.float(), W.float()) +
         sigma * torch.randn((U, Hkv, T, d), generator=g)).to(torch.bfloat16).contiguous()
    scores = torch.randn((U, Hkv, T), generator=g)
    kept, counts, offsets = O.select(scores.numpy(), "global", keep_ratio=keep, n_sink=n_sink,
                                     n_recent=n_recent)
    return k, v, W, kept, counts, offsets


def run_gpu_routing(B, k, v, W, kept, counts, offsets, A, n_sink, n_recent, slack):
    """residual -> top-A of the keys over the pool positions -> VECTOR
    compaction, all on the GPU; the choice is also made by the plain global
    select over all positions, which must agree bit for bit."""
    U, Hkv, T, d = k.shape
    n = U * Hkv
    kept_t, counts_t = torch.as_tensor(kept).cuda(), torch.as_tensor(counts).cuda()
    offs_t = torch.as_tensor(offsets).cuda()
    key = torch.full((U, Hkv, T), 7.0, device="cuda")
    B.kvc_vector_residual(k, v, W, kept_t, counts_t, key, n_sink, n_recent)
    apos = torch.empty((n, T), dtype=torch.int32, device="cuda")
    acnt = torch.empty(n, dtype=torch.int32, device="cuda")
    aoff = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    B.kvc_vector_select(key, counts_t, A, apos, acnt, aoff)
    apos2, acnt2, aoff2 = torch.empty_like(apos), torch.empty_like(acnt), torch.empty_like(aoff)
    B.kvc_select(key, "global", apos2, acnt2, aoff2, keep_ratio=(A + 0.5) / (Hkv * T))
    torch.cuda.synchronize()
    assert torch.equal(acnt, acnt2) and torch.equal(aoff, aoff2)
    for i in range(n):
        c = int(acnt[i])
        assert torch.equal(apos[i, :c], apos2[i, :c]), i
    rows_k = int(np.sum(counts)) + n * slack
    rows_v = int(np.sum(counts)) - U * A + n * slack
    kc = torch.zeros((rows_k, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((rows_v, d), dtype=torch.bfloat16, device="cuda")
    ks = torch.empty(n, dtype=torch.int64, device="cuda")
    kl = torch.empty(n, dtype=torch.int32, device="cuda")
    vs = torch.empty(n, dtype=torch.int64, device="cuda")
    na = torch.empty(n, dtype=torch.int32, device="cuda")
    B.kvc_vector_compact(k, v, kept_t, counts_t, offs_t, apos, acnt, aoff, kc, vc, ks, kl, vs,
                         na, slack=slack)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    return key, apos, acnt, kc, vc, ks, kl, vs, na


def test_vector_routing_small(B):
    n_sink, n_recent, slack = 4, 16, 3
    k, v, W, kept, counts, offsets = small_case(81, n_sink=n_sink, n_recent=n_recent)
    U, Hkv, T, d = k.shape
    A = 100
    key, apos, acnt, kc, vc, ks, kl, vs, na = run_gpu_routing(
        B, k.cuda(), v.cuda(), W.cuda(), kept, counts, offsets, A, n_sink, n_recent, slack)
    ref_key = O.vector_residual(k.float().numpy(), v.float().numpy(), W.float().numpy(), kept,
                                counts, n_sink, n_recent)
    key_close(key.cpu().numpy(), ref_key)
    # the choice, on the GPU's keys, is the oracle's choice bit for bit
    gk = key.cpu().numpy()
    rpos, rcnt = O.vector_approx(gk, A)
    np.testing.assert_array_equal(acnt.cpu().numpy(), rcnt)
    for i in range(U * Hkv):
        np.testing.assert_array_equal(apos.cpu().numpy()[i, :rcnt[i]], rpos[i, :rcnt[i]])
    rkc, rvc, rks, rkl, rvs, rna = O.vector_compact(k.float().numpy(), v.float().numpy(), kept,
                                                    counts, rpos, rcnt, slack=slack)
    np.testing.assert_array_equal(ks.cpu().numpy(), rks)
    np.testing.assert_array_equal(kl.cpu().numpy(), rkl)
    np.testing.assert_array_equal(vs.cpu().numpy(), rvs)
    np.testing.assert_array_equal(na.cpu().numpy(), rna)
    gkc, gvc = kc.float().cpu().numpy(), vc.float().cpu().numpy()
    for i in range(U * Hkv):
        r = slice(int(rks[i]), int(rks[i] + rkl[i]))
        np.testing.assert_array_equal(gkc[r], rkc[r])
        r = slice(int(rvs[i]), int(rvs[i] + rkl[i] - rna[i]))
        np.testing.assert_array_equal(gvc[r], rvc[r])


def vselect(B, key, counts, A):
    U, Hkv, T = key.shape
    n = U * Hkv
    apos = torch.full((n, T), -7, dtype=torch.int32, device="cuda")
    acnt = torch.empty(n, dtype=torch.int32, device="cuda")
    aoff = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    B.kvc_vector_select(key.cuda(), torch.as_tensor(counts, dtype=torch.int32).cuda(), A, apos,
                        acnt, aoff)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    return apos.cpu().numpy(), acnt.cpu().numpy(), aoff.cpu().numpy()


@pytest.mark.parametrize("U,Hkv,T", [(1, 8, 32768), (3, 8, 1000), (2, 5, 997), (4, 1, 4096)])
def test_vector_select_pool_positions(B, U, Hkv, T):
    """The choice over pool positions j < counts[i] against the oracle's
    choice on keys that hold NaN from counts[i] on (as the residual writes
    them), with ties, +-0, +-inf and NaN inside the pools; heads with empty
    and full pools; budgets up to every number-valued key."""
    g = torch.Generator().manual_seed(U * 1000 + Hkv * 10 + T)
    n = U * Hkv
    counts = torch.randint(0, max(2, T // 5), (n,), generator=g).to(torch.int32)
    counts[0] = 0
    counts[-1] = T
    key = -torch.rand((U, Hkv, T), generator=g).square()
    key = torch.where(torch.rand((U, Hkv, T), generator=g) < 0.3, key.round(decimals=2), key)
    flat = key.view(n, T)
    flat[-1, :4] = torch.tensor([0.0, -0.0, float("inf"), -float("inf")])
    flat[-1, 4:9] = float("nan")
    pos = torch.arange(T)
    flat[pos[None, :] >= counts[:, None].long()] = float("nan")
    kn = key.numpy()
    valid = np.array([int((~np.isnan(kn[u])).sum()) for u in range(U)])
    for A in sorted({0, 1, int(valid.min()) // 3, int(valid.min())}):
        apos, acnt, aoff = vselect(B, key, counts.numpy(), A)
        rpos, rcnt = O.vector_approx(kn, A)
        np.testing.assert_array_equal(acnt, rcnt)
        np.testing.assert_array_equal(aoff, np.concatenate([[0], np.cumsum(rcnt)]))
        for i in range(n):
            np.testing.assert_array_equal(apos[i, :rcnt[i]], rpos[i, :rcnt[i]])


def test_vector_select_budget_beyond_the_pool(B):
    """A budget above the candidates keeps every pool position, NaN or not,
    and nothing past a head's count."""
    U, Hkv, T = 2, 4, 640
    g = torch.Generator().manual_seed(5)
    counts = np.array([0, 7, 640, 300, 1, 64, 0, 129], dtype=np.int32)
    key = torch.randn((U, Hkv, T), generator=g)
    key.view(-1)[::7] = float("nan")
    for A in (int(counts[:4].sum()), int(counts[:4].sum()) + 5, Hkv * T):
        apos, acnt, _ = vselect(B, key, counts, A)
        np.testing.assert_array_equal(acnt, counts)
        for i in range(U * Hkv):
            np.testing.assert_array_equal(apos[i, :counts[i]], np.arange(counts[i]))


def test_vector_residual_edges(B):
    """Every position protected or empty: all keys NaN; a head with an empty pool."""
    k, v, W, kept, counts, offsets = small_case(82, T=40, keep=0.2, n_sink=4, n_recent=16)
    counts = counts.copy()
    counts[1] = 0
    kept_t = torch.as_tensor(kept).cuda()
    key = torch.zeros((2, 3, 40), device="cuda")
    B.kvc_vector_residual(k.cuda(), v.cuda(), W.cuda(), kept_t, torch.as_tensor(counts).cuda(),
                          key, 20, 20)
    torch.cuda.synchronize()
    assert torch.isnan(key).all()
    B.kvc_vector_residual(k.cuda(), v.cuda(), W.cuda(), kept_t, torch.as_tensor(counts).cuda(),
                          key, 4, 16)
    ref = O.vector_residual(k.float().numpy(), v.float().numpy(), W.float().numpy(), kept, counts,
                            4, 16)
    key_close(key.cpu().numpy(), ref)


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("append", [True, False])
def test_decode_vector_small(B, G, append):
    n_sink, n_recent, slack = 4, 16, 2
    # a long pool so that heads span several chunks of both kinds (1024 exact,
    # 2048 approximated rows)
    k, v, W, kept, counts, offsets = small_case(83 + G, U=2, Hkv=2, T=2600, keep=0.9,
                                                n_sink=n_sink, n_recent=n_recent)
    U, Hkv, T, d = k.shape
    key = O.vector_residual(k.float().numpy(), v.float().numpy(), W.float().numpy(), kept, counts,
                            n_sink, n_recent)
    rpos, rcnt = O.vector_approx(key, 1500)
    rpos[0, :] = -1
    rcnt[0] = 0                                   # a head without approximated rows
    kc, vc, ks, kl, vs, na = O.vector_compact(k.float().numpy(), v.float().numpy(), kept, counts,
                                              rpos, rcnt, slack=slack)
    g = torch.Generator().manual_seed(90 + G)
    q = torch.randn((U, Hkv * G, d), generator=g).to(torch.bfloat16)
    kn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16) if append else None
    vn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16) if append else None
    kc_t = torch.from_numpy(kc).to(torch.bfloat16).cuda()
    vc_t = torch.from_numpy(vc).to(torch.bfloat16).cuda()
    kl_t = torch.from_numpy(kl).cuda()
    out = torch.full((U, Hkv * G, d), float("nan"), device="cuda").to(torch.bfloat16)
    lse = torch.full((U, Hkv * G), float("nan"), device="cuda")
    B.kvc_decode_attn_vector(q.cuda(), kc_t, vc_t, torch.from_numpy(ks).cuda(), kl_t,
                             torch.from_numpy(vs).cuda(), torch.from_numpy(na).cuda(), W.cuda(),
                             out, lse, k_new=None if kn is None else kn.cuda(),
                             v_new=None if vn is None else vn.cuda(), max_len=int(kl.max()) + 1)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    ro, rl, rkc, rvc, rkl = O.decode_attn_vector(
        np64(q), kc, vc, ks, kl, vs, na, W.float().numpy(),
        None if kn is None else np64(kn), None if vn is None else np64(vn), d ** -0.5)
    assert row_rel_err(np64(out).reshape(-1, d), ro.reshape(-1, d)) <= 2e-2
    assert lse_err(np64(lse), rl) <= 2e-2
    np.testing.assert_array_equal(kl_t.cpu().numpy(), rkl)
    if append:
        np.testing.assert_array_equal(kc_t.float().cpu().numpy(), rkc)
        np.testing.assert_array_equal(vc_t.float().cpu().numpy(), rvc)


def test_vector_layer_llama32k(B):
    """The 32k Llama-3-8B-shaped layer with p_c = 0.9, p_a = 0.05: attention-mass
    scores -> pool of 0.15 (global top-k) -> residual -> 0.10 approximated ->
    compaction; keys sampled against the oracle, the choice and the layout
    exact on the GPU's keys, the memory accounting exact."""
    w = inputs.WORKLOADS["c2_llama32k"]
    p_c, p_a = 0.9, 0.05
    q_win = inputs.window_queries(w, "cuda")
    k, _ = inputs.keys_values(w, q_win, "cuda")
    W = inputs.vector_predictor(w, "cuda")
    v = inputs.vector_values(w, k, W, "cuda")
    n = w.U * w.Hkv
    scores = torch.empty((w.U, w.Hkv, w.T), device="cuda")
    B.kvc_score_attn(q_win, k, scores, scale=w.scale)
    ratio, Bpool, A = O.vector_budgets(p_c, p_a, w.Hkv, w.T, w.n_sink, w.n_recent)
    kept = torch.empty((n, w.T), dtype=torch.int32, device="cuda")
    counts = torch.empty(n, dtype=torch.int32, device="cuda")
    offs = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    B.kvc_select(scores, "global", kept, counts, offs, keep_ratio=ratio, n_sink=w.n_sink,
                 n_recent=w.n_recent)
    torch.cuda.synchronize()
    assert int(counts.sum()) == Bpool
    key, apos, acnt, kc, vc, ks, kl, vs, na = run_gpu_routing(
        B, k, v, W, kept.cpu().numpy(), counts.cpu().numpy(), offs.cpu().numpy(), A, w.n_sink,
        w.n_recent, 0)
    assert int(acnt.sum()) == A
    # memory accounting: K rows for the pool + V rows for the exact tokens
    assert int(kl.sum()) + int((kl - na).sum()) == 2 * Bpool - A
    assert abs((2 * Bpool - A) - 2 * (1 - p_c) * w.Hkv * w.T) <= 2
    # keys of the first 256 pool positions of every head against the oracle
    kept_np, counts_np = kept.cpu().numpy(), counts.cpu().numpy()
    sub = np.full((n, w.T), -1, dtype=np.int32)
    sub[:, :256] = kept_np[:, :256]
    sub_counts = np.minimum(counts_np, 256)
    ref = O.vector_residual(k.float().cpu().numpy(), v.float().cpu().numpy(),
                            W.float().cpu().numpy(), sub, sub_counts, w.n_sink, w.n_recent)
    key_close(key.cpu().numpy()[:, :, :256], ref[:, :, :256])
    # the choice, on the GPU's keys, bit for bit
    gk = key.cpu().numpy()
    rpos, rcnt = O.vector_approx(gk, A)
    np.testing.assert_array_equal(acnt.cpu().numpy(), rcnt)
    ap = apos.cpu().numpy()
    for i in range(n):
        np.testing.assert_array_equal(ap[i, :rcnt[i]], rpos[i, :rcnt[i]])
    # the layout of two heads, rows against the source tokens
    kcn, vcn = bits(kc), bits(vc)
    kb, vb = bits(k), bits(v)
    for i in (0, n - 1):
        g = i % w.Hkv
        pool = kept_np[i, :counts_np[i]]
        approx = set(rpos[i, :rcnt[i]].tolist())
        order = [pool[j] for j in rpos[i, :rcnt[i]]] + [pool[j] for j in range(counts_np[i])
                                                        if j not in approx]
        s0 = int(ks[i])
        np.testing.assert_array_equal(kcn[s0: s0 + len(order)], kb[0, g, order])
        exact = [pool[j] for j in range(counts_np[i]) if j not in approx]
        v0 = int(vs[i])
        np.testing.assert_array_equal(vcn[v0: v0 + len(exact)], vb[0, g, exact])


def test_decode_vector_batch64_sampled(B):
    """Batch 64 of VECTOR caches (pool lengths ~ U(0.1, 0.3) x 32768 per head,
    two thirds of every pool approximated): four decode steps with appends,
    two sequences against the oracle at steps 0 and 3."""
    w = inputs.WORKLOADS["c5_decode"]
    lens = inputs.head_budgets(w, "cpu")
    nap = (lens.to(torch.int64) * 2 // 3).to(torch.int32)
    kc, vc, ks, kl, vs, na = inputs.vector_pool(w, lens, nap, "cuda")
    W = inputs.vector_predictor(w, "cuda")
    max_len = int(lens.max()) + 8
    ws = torch.empty(B.kvc_decode_vector_workspace(w.U, w.Hq, w.Hkv, w.d, max_len),
                     dtype=torch.uint8, device="cuda")
    sample_u = [5, 62]
    heads = [u * w.Hkv + g for u in sample_u for g in range(w.Hkv)]
    ks_np, kl0, vs_np, na_np = ks.cpu().numpy(), kl.cpu().numpy(), vs.cpu().numpy(), na.cpu().numpy()
    pk, pv, pks, pvs, kb, vb = [], [], [], [], 0, 0
    for i in heads:
        pk.append(kc[ks_np[i]: ks_np[i] + kl0[i] + w.slack].float().cpu().numpy())
        pv.append(vc[vs_np[i]: vs_np[i] + kl0[i] - na_np[i] + w.slack].float().cpu().numpy())
        pks.append(kb)
        pvs.append(vb)
        kb += kl0[i] + w.slack
        vb += kl0[i] - na_np[i] + w.slack
    okc, ovc = np.concatenate(pk), np.concatenate(pv)
    oks, ovs = np.array(pks, np.int64), np.array(pvs, np.int64)
    okl, ona = kl0[heads].astype(np.int32), na_np[heads].astype(np.int32)
    Wn = W.float().cpu().numpy()
    for step in range(4):
        q, kn, vn = inputs.decode_step_inputs(w, step, "cuda")
        out = torch.empty_like(q)
        lse = torch.empty((w.U, w.Hq), device="cuda")
        B.kvc_decode_attn_vector(q, kc, vc, ks, kl, vs, na, W, out, lse, k_new=kn, v_new=vn,
                                 max_len=max_len, scale=w.scale, workspace=ws)
        ro, rl, okc, ovc, okl = O.decode_attn_vector(np64(q[sample_u]), okc, ovc, oks, okl, ovs,
                                                     ona, Wn, np64(kn[sample_u]),
                                                     np64(vn[sample_u]), w.scale)
        if step in (0, 3):
            got = np64(out[sample_u]).reshape(-1, w.d)
            assert row_rel_err(got, ro.reshape(-1, w.d)) <= 2e-2, step
            assert lse_err(np64(lse[sample_u]), rl) <= 2e-2, step
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    np.testing.assert_array_equal(kl.cpu().numpy(), kl0 + 4)


def test_decode_vector_many_chunks(B):
    """A head with more split-K chunks than the merge stages in shared memory
    (72 000 approximated + 72 000 exact rows: 36 + 71 chunks)."""
    d, G, na, ne = 128, 2, 72000, 72000
    g = torch.Generator().manual_seed(95)
    kc = torch.randn((na + ne + 1, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((ne + 1, d), generator=g).to(torch.bfloat16)
    W = (torch.randn((1, d, d), generator=g) / d ** 0.5).to(torch.bfloat16)
    q = torch.randn((1, G, d), generator=g).to(torch.bfloat16)
    kn = torch.randn((1, 1, d), generator=g).to(torch.bfloat16)
    vn = torch.randn((1, 1, d), generator=g).to(torch.bfloat16)
    ks, vs = np.zeros(1, np.int64), np.zeros(1, np.int64)
    kl, nap = np.array([na + ne], np.int32), np.array([na], np.int32)
    kc_t, vc_t, kl_t = kc.cuda(), vc.cuda(), torch.from_numpy(kl).cuda()
    out = torch.empty((1, G, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, G), device="cuda")
    B.kvc_decode_attn_vector(q.cuda(), kc_t, vc_t, torch.from_numpy(ks).cuda(), kl_t,
                             torch.from_numpy(vs).cuda(), torch.from_numpy(nap).cuda(), W.cuda(),
                             out, lse, k_new=kn.cuda(), v_new=vn.cuda(), max_len=na + ne + 1)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    ro, rl, _, _, rkl = O.decode_attn_vector(np64(q), kc.float().numpy(), vc.float().numpy(), ks,
                                             kl, vs, nap, W.float().numpy(), np64(kn), np64(vn),
                                             d ** -0.5)
    assert row_rel_err(np64(out).reshape(-1, d), ro.reshape(-1, d)) <= 2e-2
    assert lse_err(np64(lse), rl) <= 2e-2
    np.testing.assert_array_equal(kl_t.cpu().numpy(), rkl)
