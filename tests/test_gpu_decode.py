"""GPU varlen decode attention (+ append), the fidelity probe, the whole
score -> select -> compact -> decode chain, and the bounded-wait self-test,
all through the C ABI and against the CPU oracle.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_attention_b300 import inputs
from oracle import kvc_oracle as O
from tests.kvc_testutil import TOL, lse_err, mass_rel_err, np64, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kv_cache_compression_attention_b300 import binding
    binding.lib()
    return binding


def run_decode(B, q, kc, vc, start, length, kn, vn, max_len, scale):
    U, Hq, d = q.shape
    out = torch.full_like(q, float("nan"))
    lse = torch.full((U, Hq), float("nan"), device="cuda")
    B.kvc_decode_attn(q, kc, vc, start, length, out, lse, k_new=kn, v_new=vn,
                      max_len=max_len, scale=scale)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    return out, lse


def pool(lens, slack, d, dtype, seed):
    lens = np.asarray(lens)
    start = np.concatenate([[0], np.cumsum(lens + slack)[:-1]]).astype(np.int64)
    rows = int((lens + slack).sum())
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn((rows, d), generator=g).to(dtype)
    vc = torch.randn((rows, d), generator=g).to(dtype)
    return kc, vc, start, lens.astype(np.int32)


@pytest.mark.parametrize("dtype,d,G", [(torch.bfloat16, 128, 4), (torch.float32, 128, 4),
                                       (torch.bfloat16, 64, 2), (torch.float32, 64, 7),
                                       (torch.bfloat16, 128, 8), (torch.bfloat16, 128, 1)])
@pytest.mark.parametrize("append", [True, False])
def test_decode_small(B, dtype, d, G, append):
    U, Hkv = 2, 3
    lens = [0, 1, 511, 512, 513, 2000][: U * Hkv]
    kc, vc, start, lens = pool(lens, 1, d, dtype, 3)
    g = torch.Generator().manual_seed(4)
    q = torch.randn((U, Hkv * G, d), generator=g).to(dtype)
    kn = torch.randn((U, Hkv, d), generator=g).to(dtype) if append else None
    vn = torch.randn((U, Hkv, d), generator=g).to(dtype) if append else None
    scale = d ** -0.5
    kcg, vcg = kc.cuda(), vc.cuda()
    st, ln = torch.from_numpy(start).cuda(), torch.from_numpy(lens).cuda()
    out, lse = run_decode(B, q.cuda(), kcg, vcg, st, ln, None if kn is None else kn.cuda(),
                          None if vn is None else vn.cuda(), int(lens.max()) + 1, scale)
    ro, rl, rkc, rvc, rlen = O.decode_attn(np64(q), kc.float().numpy(), vc.float().numpy(), start,
                                           lens, None if kn is None else np64(kn),
                                           None if vn is None else np64(vn), scale)
    assert row_rel_err(np64(out).reshape(-1, d), ro.reshape(-1, d)) <= TOL[dtype]
    assert lse_err(np64(lse), rl) <= TOL[dtype]
    np.testing.assert_array_equal(ln.cpu().numpy(), rlen)
    if append:
        np.testing.assert_array_equal(kcg.cpu().float().numpy(), rkc)
        np.testing.assert_array_equal(vcg.cpu().float().numpy(), rvc)


def test_decode_steps_c5_sampled(B):
    """256 decode steps over per-head compressed lengths ~ U[0.1, 0.3]*32768,
    batch 64; the oracle follows 2 sampled sequences through every append and
    is compared at steps 0, 1, 127 and 255."""
    w = inputs.WORKLOADS["c5_decode"]
    lens = inputs.head_budgets(w, "cpu")
    kc, vc, start, length = inputs.compressed_pool(w, lens, "cuda")
    max_len = int(lens.max()) + w.decode_steps
    ws = torch.empty(B.kvc_decode_workspace(w.U, w.Hq, w.Hkv, w.d, max_len), dtype=torch.uint8,
                     device="cuda")
    sample_u = [0, 41]
    heads = [u * w.Hkv + g for u in sample_u for g in range(w.Hkv)]
    st_np = start.cpu().numpy()
    ln0 = length.cpu().numpy()
    # the sampled heads' rows, re-based into a small host pool for the oracle
    pk, pv, pstart = [], [], []
    base = 0
    for i in heads:
        rows = slice(int(st_np[i]), int(st_np[i]) + int(ln0[i]) + w.slack)
        pk.append(kc[rows].float().cpu().numpy()); pv.append(vc[rows].float().cpu().numpy())
        pstart.append(base); base += int(ln0[i]) + w.slack
    okc, ovc = np.concatenate(pk), np.concatenate(pv)
    ostart = np.array(pstart, dtype=np.int64)
    olen = ln0[heads].astype(np.int32)
    for step in range(w.decode_steps):
        q, kn, vn = inputs.decode_step_inputs(w, step, "cuda")
        out = torch.empty_like(q)
        lse = torch.empty((w.U, w.Hq), device="cuda")
        B.kvc_decode_attn(q, kc, vc, start, length, out, lse, k_new=kn, v_new=vn,
                          max_len=max_len, scale=w.scale, workspace=ws)
        qs, kns, vns = np64(q[sample_u]), np64(kn[sample_u]), np64(vn[sample_u])
        ro, rl, okc, ovc, olen = O.decode_attn(qs, okc, ovc, ostart, olen, kns, vns, w.scale) \
            if step in (0, 1, 127, 255) else _append_only(qs, okc, ovc, ostart, olen, kns, vns)
        if step in (0, 1, 127, 255):
            got = np64(out[sample_u]).reshape(-1, w.d)
            assert row_rel_err(got, ro.reshape(-1, w.d)) <= 2e-2, step
            assert lse_err(np64(lse[sample_u]), rl) <= 2e-2, step
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    np.testing.assert_array_equal(length.cpu().numpy(), ln0 + w.decode_steps)


def _append_only(q, kc, vc, start, length, kn, vn):
    Hkv = length.size // q.shape[0]
    length = length.copy()
    for u in range(q.shape[0]):
        for g in range(Hkv):
            i = u * Hkv + g
            kc[start[i] + length[i]] = kn[u, g]
            vc[start[i] + length[i]] = vn[u, g]
            length[i] += 1
    return None, None, kc, vc, length


def test_fidelity_kernel(B):
    g = torch.Generator().manual_seed(8)
    for dtype in (torch.float32, torch.bfloat16):
        oc = torch.randn((5, 128), generator=g).to(dtype)
        of = torch.randn((5, 128), generator=g).to(dtype)
        of[2] = oc[2]
        lc = torch.randn(5, generator=g)
        lf = lc + torch.rand(5, generator=g)
        rel = torch.empty(5, device="cuda")
        kl = torch.empty(5, device="cuda")
        B.kvc_fidelity(oc.cuda(), of.cuda(), lc.cuda(), lf.cuda(), rel, kl)
        r_rel, r_kl = O.fidelity(np64(oc), np64(of), np64(lc), np64(lf))
        np.testing.assert_allclose(rel.cpu().numpy(), r_rel, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(kl.cpu().numpy(), r_kl, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("dtype,d,ratio", [(torch.float32, 64, 0.25), (torch.bfloat16, 128, 0.1),
                                           (torch.bfloat16, 128, 1.0)])
def test_pipeline_against_oracle(B, dtype, d, ratio):
    """score -> select -> compact -> decode (+ the fidelity probe against the
    full cache) on the GPU, and the same chain run independently by the
    oracle from the same generated inputs.  Scores agree within tolerance;
    the kept sets may differ only at tokens whose oracle score is within that
    tolerance of the oracle's cut (none do for these seeds); with equal sets
    the outputs, lse and KL agree within tolerance."""
    w = inputs.WORKLOADS["c1_tiny"].with_(d=d, dtype="f32" if dtype == torch.float32 else "bf16",
                                          Hq=16 if d == 128 else 8, W=64 if d == 128 else 32,
                                          T=3000, keep_ratio=ratio)
    tol = TOL[dtype]
    q_win = inputs.window_queries(w, "cuda")
    k, v = inputs.keys_values(w, q_win, "cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn((w.U, w.Hq, d), generator=g, device="cuda").to(dtype)
    kn = torch.randn((w.U, w.Hkv, d), generator=g, device="cuda").to(dtype)
    vn = torch.randn((w.U, w.Hkv, d), generator=g, device="cuda").to(dtype)
    n, slack = w.U * w.Hkv, 1
    # ---- GPU chain
    scores = torch.empty((w.U, w.Hkv, w.T), device="cuda")
    B.kvc_score_attn(q_win, k, scores, w.scale)
    kept = torch.empty((n, w.T), dtype=torch.int32, device="cuda")
    counts = torch.empty(n, dtype=torch.int32, device="cuda")
    offs = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    B.kvc_select(scores, "global", kept, counts, offs, keep_ratio=ratio, n_sink=w.n_sink,
                 n_recent=w.n_recent)
    rows = int(offs[-1].item()) + n * slack
    kc = torch.zeros((rows, d), dtype=dtype, device="cuda")
    vc = torch.zeros_like(kc)
    start = torch.empty(n, dtype=torch.int64, device="cuda")
    length = torch.empty(n, dtype=torch.int32, device="cuda")
    B.kvc_compact(k, v, kept, counts, offs, kc, vc, start, length, slack=slack)
    allk = torch.arange(w.T, dtype=torch.int32, device="cuda").repeat(n, 1).contiguous()
    allc = torch.full((n,), w.T, dtype=torch.int32, device="cuda")
    allo = (torch.arange(n + 1, device="cuda") * w.T).to(torch.int64)
    kf = torch.zeros((n * (w.T + slack), d), dtype=dtype, device="cuda")
    vf = torch.zeros_like(kf)
    sf = torch.empty(n, dtype=torch.int64, device="cuda")
    lf = torch.empty(n, dtype=torch.int32, device="cuda")
    B.kvc_compact(k, v, allk, allc, allo, kf, vf, sf, lf, slack=slack)
    oc, lc = run_decode(B, q, kc, vc, start, length, kn, vn, w.T + 1, w.scale)
    of, lfu = run_decode(B, q, kf, vf, sf, lf, kn, vn, w.T + 1, w.scale)
    rel = torch.empty(w.U * w.Hq, device="cuda")
    kl = torch.empty(w.U * w.Hq, device="cuda")
    B.kvc_fidelity(oc, of, lc, lfu, rel, kl)
    torch.cuda.synchronize()
    # ---- oracle chain, from the generator's inputs only
    kk, vv = np64(k), np64(v)
    ref_s = O.score_attn(np64(q_win), kk, w.scale)
    assert mass_rel_err(np64(scores), ref_s) <= tol
    rs32 = ref_s.astype(np.float32)
    rk, rc, ro = O.select(rs32, "global", keep_ratio=ratio, n_sink=w.n_sink, n_recent=w.n_recent)
    gk, gc = kept.cpu().numpy(), counts.cpu().numpy()
    assert gc.sum() == rc.sum()
    gset = {(i, int(t)) for i in range(n) for t in gk[i, : gc[i]]}
    rset = {(i, int(t)) for i in range(n) for t in rk[i, : rc[i]]}
    diff = gset ^ rset
    if diff:
        # only tokens at the cut may flip: their oracle score is within tol of it
        P = O.protected_mask(w.T, w.n_sink, w.n_recent)
        free = [rs32[0, i, t] for i in range(n) for t in range(w.T) if not P[t] and (i, t) in rset]
        cut = min(free)
        for i, t in diff:
            assert abs(ref_s[0, i, t] - cut) <= 2 * tol * abs(cut), (i, t)
        pytest.skip(f"{len(diff)} near-tie tokens flipped at the cut; outputs not comparable")
    okc, ovc, ost, oln = O.compact(kk, vv, rk, rc, ro, slack)
    ro_c, rl_c, *_ = O.decode_attn(np64(q), okc, ovc, ost, oln, np64(kn), np64(vn), w.scale)
    fkc, fvc, fst, fln = O.compact(kk, vv, np.tile(np.arange(w.T, dtype=np.int32), (n, 1)),
                                   np.full(n, w.T, dtype=np.int32),
                                   np.arange(n + 1, dtype=np.int64) * w.T, slack)
    ro_f, rl_f, *_ = O.decode_attn(np64(q), fkc, fvc, fst, fln, np64(kn), np64(vn), w.scale)
    assert row_rel_err(np64(oc).reshape(-1, d), ro_c.reshape(-1, d)) <= tol
    assert row_rel_err(np64(of).reshape(-1, d), ro_f.reshape(-1, d)) <= tol
    assert lse_err(np64(lc), rl_c) <= tol and lse_err(np64(lfu), rl_f) <= tol
    r_rel, r_kl = O.fidelity(ro_c, ro_f, rl_c, rl_f)
    assert np.abs(kl.cpu().numpy() - r_kl.reshape(-1)).max() <= tol * max(1.0, np.abs(rl_f).max())
    assert (r_kl >= 0).all()
    if ratio == 1.0:
        assert np.abs(kl.cpu().numpy()).max() == 0.0      # same rows, same order: identical
        assert rel.cpu().numpy().max() == 0.0


def test_bounded_wait_times_out_and_context_survives(B):
    B.kvc_selftest_wait_timeout(2_000_000)        # 2 ms on an mbarrier nothing completes
    assert B.kvc_device_status() == -5            # KVC_ERR_TIMEOUT
    assert B.kvc_device_status() == 0
    x = torch.ones(4, device="cuda") * 2          # the context is still usable
    assert x.sum().item() == 8


def test_decode_more_chunks_than_the_combine_stages(B):
    """A head of 280 000 rows has 274 chunks of 1024, more than the combine
    kernel stages in shared memory (256): the second merge path runs."""
    L = 280000
    kc, vc, start, lens = pool([L], 1, 128, torch.bfloat16, 17)
    g = torch.Generator().manual_seed(18)
    q = torch.randn((1, 2, 128), generator=g).to(torch.bfloat16)
    kn = torch.randn((1, 1, 128), generator=g).to(torch.bfloat16)
    vn = torch.randn((1, 1, 128), generator=g).to(torch.bfloat16)
    kcg, vcg = kc.cuda(), vc.cuda()
    st, ln = torch.from_numpy(start).cuda(), torch.from_numpy(lens).cuda()
    out, lse = run_decode(B, q.cuda(), kcg, vcg, st, ln, kn.cuda(), vn.cuda(), L + 1, 128 ** -0.5)
    ro, rl, *_ = O.decode_attn(np64(q), kc.float().numpy(), vc.float().numpy(), start, lens,
                               np64(kn), np64(vn), 128 ** -0.5)
    assert row_rel_err(np64(out).reshape(-1, 128), ro.reshape(-1, 128)) <= 2e-2
    assert lse_err(np64(lse), rl) <= 2e-2


def test_decode_fidelity_c5_sequence_against_oracle(B):
    """The batch-64 decode workload as configured, on one sampled sequence:
    its compressed cache is cut from its full 32k cache (window scores ->
    per-head top-k at its budgets, 4 sinks + 64 recent -> compaction with 256
    slack rows), then 256 decode steps run over the compressed and the full
    cache.  The GPU selection is fed the oracle's scores (the bit-exact
    contract), so both sides hold the same kept tokens; the fidelity of steps
    0 and 255 (rel-L2 output error, KL = lse_full - lse_comp, [Sculpt] §4) is
    compared with the oracle's, which follows every append on its own copies."""
    w = inputs.WORKLOADS["c5_decode"]
    u = 37
    q_all = inputs.window_queries(w, "cuda")
    k_all, v_all = inputs.keys_values(w, q_all, "cuda")
    qw, k, v = q_all[u:u + 1].contiguous(), k_all[u:u + 1].contiguous(), v_all[u:u + 1].contiguous()
    del q_all, k_all, v_all
    torch.cuda.empty_cache()
    n = w.Hkv
    budgets = inputs.head_budgets(w, "cpu")[u * n:(u + 1) * n]
    s_ref = O.score_attn(np64(qw), np64(k), w.scale).astype(np.float32)
    r_kept, r_counts, r_offs = O.select(s_ref, "per_head", head_budget=budgets.numpy(),
                                        n_sink=w.n_sink, n_recent=w.n_recent)
    kept = torch.empty((n, w.T), dtype=torch.int32, device="cuda")
    counts = torch.empty(n, dtype=torch.int32, device="cuda")
    offs = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    B.kvc_select(torch.from_numpy(s_ref).cuda(), "per_head", kept, counts, offs,
                 head_budget=budgets.cuda(), n_sink=w.n_sink, n_recent=w.n_recent)
    np.testing.assert_array_equal(counts.cpu().numpy(), r_counts)
    np.testing.assert_array_equal(offs.cpu().numpy(), r_offs)

    def gpu_pool(kept_, counts_, offs_):
        rows = int(offs_[-1].item()) + n * w.slack
        kc = torch.zeros((rows, w.d), dtype=k.dtype, device="cuda")
        vc = torch.zeros_like(kc)
        st = torch.empty(n, dtype=torch.int64, device="cuda")
        ln = torch.empty(n, dtype=torch.int32, device="cuda")
        B.kvc_compact(k, v, kept_, counts_, offs_, kc, vc, st, ln, slack=w.slack)
        return kc, vc, st, ln

    comp = gpu_pool(kept, counts, offs)
    all_np = np.tile(np.arange(w.T, dtype=np.int32), (n, 1))
    allc_np = np.full(n, w.T, dtype=np.int32)
    allo_np = np.arange(n + 1, dtype=np.int64) * w.T
    full = gpu_pool(torch.from_numpy(all_np).cuda(), torch.from_numpy(allc_np).cuda(),
                    torch.from_numpy(allo_np).cuda())
    # the oracle's own caches, from its own selection
    kh, vh = np64(k), np64(v)
    o_comp = list(O.compact(kh, vh, r_kept, r_counts, r_offs, w.slack))
    o_full = list(O.compact(kh, vh, all_np, allc_np, allo_np, w.slack))
    max_len = w.T + w.decode_steps
    rel = torch.empty(w.Hq, device="cuda")
    kl = torch.empty_like(rel)
    for step in range(w.decode_steps):
        q, kn, vn = inputs.decode_step_inputs(w, step, "cuda")
        q, kn, vn = q[u:u + 1].contiguous(), kn[u:u + 1].contiguous(), vn[u:u + 1].contiguous()
        oc = torch.empty_like(q); of = torch.empty_like(q)
        lc = torch.empty((1, w.Hq), device="cuda"); lf = torch.empty_like(lc)
        B.kvc_decode_attn(q, *comp, oc, lc, k_new=kn, v_new=vn, max_len=max_len, scale=w.scale)
        B.kvc_decode_attn(q, *full, of, lf, k_new=kn, v_new=vn, max_len=max_len, scale=w.scale)
        B.kvc_fidelity(oc, of, lc, lf, rel, kl)
        qs, kns, vns = np64(q), np64(kn), np64(vn)
        if step in (0, w.decode_steps - 1):
            roc, rlc, o_comp[0], o_comp[1], o_comp[3] = O.decode_attn(
                qs, o_comp[0], o_comp[1], o_comp[2], o_comp[3], kns, vns, w.scale)
            rof, rlf, o_full[0], o_full[1], o_full[3] = O.decode_attn(
                qs, o_full[0], o_full[1], o_full[2], o_full[3], kns, vns, w.scale)
            r_rel, r_kl = O.fidelity(roc, rof, rlc, rlf)
            torch.cuda.synchronize()
            assert B.kvc_device_status() == 0
            g_kl, g_rel = np64(kl), np64(rel)
            tol = 2e-2 * np.maximum(1.0, np.abs(rlf.reshape(-1)))
            assert (np.abs(g_kl - r_kl.reshape(-1)) <= tol).all(), step
            assert (r_kl >= -1e-9).all()                     # a subset retains mass <= 1
            assert (np.abs(g_rel - r_rel.reshape(-1)) <= 2e-2 * np.maximum(1.0, r_rel.reshape(-1))).all(), step
        else:
            for arrs in (o_comp, o_full):
                _, _, arrs[0], arrs[1], arrs[3] = _append_only(qs, arrs[0], arrs[1], arrs[2],
                                                               arrs[3], kns, vns)
    np.testing.assert_array_equal(comp[3].cpu().numpy(), r_counts + w.decode_steps)
