"""GPU decode-time threshold pruning ([KVzap] §2.3) through the C ABI against
the CPU oracle: per-row score gather bit for bit; prefill compaction followed
by a stream of decode steps (append, attend, prune) on bf16 and on
group-quantised pools, with every step's lengths, kept rows and per-row
scores bit-exact and the attention outputs within the bf16 tolerance; the
batch-64 compressed caches with the 128-token window, sampled heads against
the oracle and every head's length against the rule.
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
    """Raw bits of a tensor for bit-exact comparison (NaN payloads included)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


def prefill(U, Hkv, T, d, n_sink, window, slack, seed):
    """Seeded prefill: scores, per-head budgets, oracle selection and
    compaction (the inputs of the decode stream)."""
    rng = np.random.default_rng(seed)
    scores = rng.standard_normal((U, Hkv, T)).astype(np.float32)
    budget = rng.integers(n_sink + window, T // 2, U * Hkv).astype(np.int32)
    budget[0] = n_sink + window                       # a head that is all sinks and window
    kept, counts, offsets = O.select(scores, "per_head", head_budget=budget, n_sink=n_sink,
                                     n_recent=window)
    g = torch.Generator().manual_seed(seed)
    k = torch.randn((U, Hkv, T, d), generator=g).to(torch.bfloat16)
    v = torch.randn((U, Hkv, T, d), generator=g).to(torch.bfloat16)
    kc, vc, start, length = O.compact(k.float().numpy(), v.float().numpy(), kept, counts,
                                      offsets, slack=slack)
    return scores, kept, counts, offsets, start, length, kc, vc


def test_gather_scores_bit_exact(B):
    scores, kept, counts, offsets, start, length, kc, _ = prefill(2, 4, 700, 8, 4, 16, 5, 51)
    rows = kc.shape[0]
    rs = torch.full((rows,), float("nan"), device="cuda")
    B.kvc_gather_scores(torch.from_numpy(scores).cuda(), torch.from_numpy(kept).cuda(),
                        torch.from_numpy(counts).cuda(), torch.from_numpy(start).cuda(), rs)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    ref = O.gather_scores(scores, kept, counts, start, rows)
    np.testing.assert_array_equal(bits(rs), ref.view(np.int32))


def step_scores(rng, n, tau):
    s = rng.standard_normal(n).astype(np.float32)
    s[rng.random(n) < 0.1] = np.float32(tau)          # ties with tau stay
    s[rng.random(n) < 0.05] = np.nan                  # NaN goes
    return s


@pytest.mark.parametrize("quantised", [False, True])
def test_decode_prune_stream(B, quantised):
    U, Hkv, G, T, d = 2, 4, 4, 900, 128
    n_sink, window, slack, steps, tau = 4, 16, 48, 40, 0.25
    scores, kept, counts, offsets, start, length, kc, vc = prefill(U, Hkv, T, d, n_sink, window,
                                                                   slack, 52 + quantised)
    rows = kc.shape[0]
    n = U * Hkv
    rs0 = O.gather_scores(scores, kept, counts, start, rows)
    st = torch.from_numpy(start).cuda()
    ln = torch.from_numpy(length).cuda()
    rs = torch.from_numpy(rs0).cuda()
    kc_t = torch.from_numpy(kc).to(torch.bfloat16).cuda()
    vc_t = torch.from_numpy(vc).to(torch.bfloat16).cuda()
    if quantised:
        kq = torch.empty((rows, d), dtype=torch.uint8, device="cuda")
        kp = torch.empty((rows, d // 32, 2), dtype=torch.float16, device="cuda")
        vq, vp = torch.empty_like(kq), torch.empty_like(kp)
        B.kvc_quantize_rows(kc_t, kq, kp)
        B.kvc_quantize_rows(vc_t, vq, vp)
        pools_gpu = [kq, kp, vq, vp]
        rkq, rkp = O.quantize_rows(kc)
        rvq, rvp = O.quantize_rows(vc)
        pools_ref = [rkq, rkp, rvq, rvp]
    else:
        pools_gpu = [kc_t, vc_t]
        pools_ref = [kc, vc]
    ref_len = length.copy()
    rs_ref = rs0.copy()
    rng = np.random.default_rng(54)
    g = torch.Generator().manual_seed(55)
    max_len = int(length.max()) + steps + 1
    dropped_total = 0
    for step in range(steps):
        q = torch.randn((U, Hkv * G, d), generator=g).to(torch.bfloat16)
        kn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16)
        vn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16)
        s_new = step_scores(rng, n, tau)
        out = torch.empty((U, Hkv * G, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((U, Hkv * G), device="cuda")
        if quantised:
            B.kvc_decode_attn_q8(q.cuda(), kq, kp, vq, vp, st, ln, out, lse, k_new=kn.cuda(),
                                 v_new=vn.cuda(), max_len=max_len)
        else:
            B.kvc_decode_attn(q.cuda(), kc_t, vc_t, st, ln, out, lse, k_new=kn.cuda(),
                              v_new=vn.cuda(), max_len=max_len)
        B.kvc_decode_prune(pools_gpu, rs, st, ln, torch.from_numpy(s_new).cuda(), tau, window,
                           n_sink)
        # oracle: append (quantised like the kernel when the pool is), attend, prune
        if quantised:
            akq, akp = O.quantize_rows(kn.float().numpy().reshape(-1, d))
            avq, avp = O.quantize_rows(vn.float().numpy().reshape(-1, d))
            for i in range(n):
                r = int(start[i] + ref_len[i])
                pools_ref[0][r], pools_ref[1][r] = akq[i], akp[i]
                pools_ref[2][r], pools_ref[3][r] = avq[i], avp[i]
            # the kernel attends the new token's exact row and stores it quantised
            kd = O.dequantize_rows(pools_ref[0], pools_ref[1])
            vd = O.dequantize_rows(pools_ref[2], pools_ref[3])
            ro, rl, _, _, _ = O.decode_attn(np64(q), kd, vd, start, ref_len, kn.float().numpy(),
                                            vn.float().numpy(), d ** -0.5)
        else:
            ro, rl, pools_ref[0], pools_ref[1], _ = O.decode_attn(
                np64(q), pools_ref[0], pools_ref[1], start, ref_len, kn.float().numpy(),
                vn.float().numpy(), d ** -0.5)
        ref_len = ref_len + 1
        pools_ref, rs_ref, ref_len, dropped = O.decode_prune(pools_ref, rs_ref, start, ref_len,
                                                             s_new, tau, window, n_sink)
        dropped_total += int(dropped.sum())
        torch.cuda.synchronize()
        assert B.kvc_device_status() == 0
        np.testing.assert_array_equal(ln.cpu().numpy(), ref_len, err_msg=f"step {step}")
        got_pools = [bits(p) for p in pools_gpu]
        got_rs = bits(rs)
        for i in range(n):
            r = slice(int(start[i]), int(start[i] + ref_len[i]))
            for gp, rp in zip(got_pools, pools_ref):
                if rp.dtype == np.float16:
                    np.testing.assert_array_equal(gp[r], rp[r].view(np.int16))
                elif rp.dtype == np.uint8:
                    np.testing.assert_array_equal(gp[r], rp[r])
                else:   # bf16 values held in float32
                    ref_bits = torch.from_numpy(np.ascontiguousarray(rp[r])).to(torch.bfloat16)
                    np.testing.assert_array_equal(gp[r], ref_bits.view(torch.int16).numpy())
            np.testing.assert_array_equal(got_rs[r], rs_ref[r].view(np.int32))
        if step % 8 == 0 or step == steps - 1:
            assert row_rel_err(np64(out).reshape(-1, d), ro.reshape(-1, d)) <= 2e-2, step
            assert lse_err(np64(lse), rl) <= 2e-2, step
    # the stream exercised both outcomes
    assert 0 < dropped_total < steps * n


def test_decode_prune_batch64(B):
    """The batch-64 compressed caches (32 q / 8 kv heads, d = 128, lengths
    ~ U(0.1, 0.3) x 32768): decode with append, linear surrogate scores of the
    new tokens, prune with the 128-token window; four steps."""
    w = inputs.WORKLOADS["c5_decode"]
    window, n_sink, tau, Dh = 128, 4, 0.5, 4096
    lens = inputs.head_budgets(w, "cpu")
    kc, vc, start, length = inputs.compressed_pool(w, lens, "cuda")
    rows = kc.shape[0]
    rs = inputs.row_scores(rows, "cuda", seed=61)
    weight, bias = inputs.decode_surrogate(w, Dh, "cuda")
    max_len = int(lens.max()) + 8
    ws = torch.empty(B.kvc_decode_workspace(w.U, w.Hq, w.Hkv, w.d, max_len), dtype=torch.uint8,
                     device="cuda")
    n = w.U * w.Hkv
    sample = [0, 1, 7, 100, 263, 511]
    st_np = start.cpu().numpy()
    # oracle state of the sampled heads, re-based into small pools
    sub = {}
    for i in sample:
        r = slice(int(st_np[i]), int(st_np[i]) + int(lens[i]) + w.slack)
        sub[i] = [kc[r].float().cpu().numpy(), vc[r].float().cpu().numpy(),
                  rs[r].cpu().numpy(), np.array([int(lens[i])], np.int32)]
    s_new = torch.empty((w.U, w.Hkv, 1), device="cuda")
    for step in range(4):
        q, kn, vn = inputs.decode_step_inputs(w, step, "cuda")
        hidden = inputs.decode_hidden(w, Dh, step, "cuda")
        out = torch.empty_like(q)
        len_before = length.clone()
        rs_before = rs.clone()
        B.kvc_decode_attn(q, kc, vc, start, length, out, k_new=kn, v_new=vn, max_len=max_len,
                          scale=w.scale, workspace=ws)
        B.kvc_score_linear(hidden, weight, bias, s_new)
        B.kvc_decode_prune([kc, vc], rs, start, length, s_new.reshape(-1), tau, window, n_sink)
        torch.cuda.synchronize()
        assert B.kvc_device_status() == 0
        # every head: the length follows the rule on the exiting token's score
        lb = len_before.cpu().numpy().astype(np.int64)
        e = st_np + lb - window          # row of the exiting token (len after append - w - 1)
        se = rs_before.cpu().numpy()[e]
        want = lb + 1 - (~(se >= np.float32(tau))).astype(np.int64)
        np.testing.assert_array_equal(length.cpu().numpy(), want, err_msg=f"step {step}")
        sn = s_new.reshape(-1).cpu().numpy()
        for i in sample:
            ok, ov, ors, ol = sub[i]
            u, gg = divmod(i, w.Hkv)
            ok[ol[0]], ov[ol[0]] = kn[u, gg].float().cpu().numpy(), vn[u, gg].float().cpu().numpy()
            (ok, ov), ors, ol, _ = O.decode_prune([ok, ov], ors, [0], ol + 1, [sn[i]], tau,
                                                  window, n_sink)
            sub[i] = [ok, ov, ors, ol]
            L = int(ol[0])
            assert L == int(length[i])
            r = slice(int(st_np[i]), int(st_np[i]) + L)
            np.testing.assert_array_equal(bits(kc[r]), bits(torch.from_numpy(ok[:L]).to(torch.bfloat16)))
            np.testing.assert_array_equal(bits(vc[r]), bits(torch.from_numpy(ov[:L]).to(torch.bfloat16)))
            np.testing.assert_array_equal(bits(rs[r]), ors[:L].view(np.int32))


def head_rows(pools, rscore, start, length, i):
    """The rows head i holds as a sorted list of byte strings (every pool's
    row bytes and the row's score bits): the content of the head as a set."""
    r = slice(int(start[i]), int(start[i]) + int(length[i]))
    parts = [np.ascontiguousarray(p[r]).reshape(int(length[i]), -1).view(np.uint8) for p in pools]
    parts.append(np.ascontiguousarray(rscore[r]).reshape(-1, 1).view(np.uint8))
    rows = np.concatenate(parts, axis=1)
    return sorted(bytes(x) for x in rows)


@pytest.mark.parametrize("quantised", [False, True])
def test_decode_prune_ring_matches_the_ordered_rule(B, quantised):
    """kvc_decode_prune_ring on a stream of decode steps: the rows every head
    holds (pool rows and their scores, compared as a set) and the lengths
    equal the oracle's token-ordered pruning at every step; a drop moves one
    row, so the order differs."""
    U, Hkv, G, T, d = 2, 4, 4, 900, 128
    n_sink, window, slack, steps, tau = 4, 16, 48, 40, 0.25
    scores, kept, counts, offsets, start, length, kc, vc = prefill(U, Hkv, T, d, n_sink, window,
                                                                   slack, 62 + quantised)
    rows = kc.shape[0]
    n = U * Hkv
    rs0 = O.gather_scores(scores, kept, counts, start, rows)
    st = torch.from_numpy(start).cuda()
    ln = torch.from_numpy(length).cuda()
    rs = torch.from_numpy(rs0).cuda()
    kc_t = torch.from_numpy(kc).to(torch.bfloat16).cuda()
    vc_t = torch.from_numpy(vc).to(torch.bfloat16).cuda()
    if quantised:
        kq = torch.empty((rows, d), dtype=torch.uint8, device="cuda")
        kp = torch.empty((rows, d // 32, 2), dtype=torch.float16, device="cuda")
        vq, vp = torch.empty_like(kq), torch.empty_like(kp)
        B.kvc_quantize_rows(kc_t, kq, kp)
        B.kvc_quantize_rows(vc_t, vq, vp)
        pools_gpu = [kq, kp, vq, vp]
        rkq, rkp = O.quantize_rows(kc)
        rvq, rvp = O.quantize_rows(vc)
        pools_ref = [rkq, rkp, rvq, rvp]
    else:
        pools_gpu = [kc_t, vc_t]
        pools_ref = [kc, vc]
    ring = torch.full((n, window), -1, dtype=torch.int32, device="cuda")
    B.kvc_prune_ring_init(ln, window, T, ring)
    ref_len = length.copy()
    rs_ref = rs0.copy()
    rng = np.random.default_rng(64)
    g = torch.Generator().manual_seed(65)
    max_len = int(length.max()) + steps + 1
    dropped_total = 0
    for step in range(steps):
        q = torch.randn((U, Hkv * G, d), generator=g).to(torch.bfloat16)
        kn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16)
        vn = torch.randn((U, Hkv, d), generator=g).to(torch.bfloat16)
        s_new = step_scores(rng, n, tau)
        out = torch.empty((U, Hkv * G, d), dtype=torch.bfloat16, device="cuda")
        if quantised:
            B.kvc_decode_attn_q8(q.cuda(), kq, kp, vq, vp, st, ln, out, None, k_new=kn.cuda(),
                                 v_new=vn.cuda(), max_len=max_len)
        else:
            B.kvc_decode_attn(q.cuda(), kc_t, vc_t, st, ln, out, None, k_new=kn.cuda(),
                              v_new=vn.cuda(), max_len=max_len)
        B.kvc_decode_prune_ring(pools_gpu, rs, st, ln, ring, T + step,
                                torch.from_numpy(s_new).cuda(), tau, window, n_sink)
        # oracle: append (quantised like the kernel when the pool is), prune in token order
        if quantised:
            akq, akp = O.quantize_rows(kn.float().numpy().reshape(-1, d))
            avq, avp = O.quantize_rows(vn.float().numpy().reshape(-1, d))
            for i in range(n):
                r = int(start[i] + ref_len[i])
                pools_ref[0][r], pools_ref[1][r] = akq[i], akp[i]
                pools_ref[2][r], pools_ref[3][r] = avq[i], avp[i]
        else:
            kf, vf = kn.float().numpy(), vn.float().numpy()
            for i in range(n):
                u, gg = divmod(i, Hkv)
                r = int(start[i] + ref_len[i])
                pools_ref[0][r], pools_ref[1][r] = kf[u, gg], vf[u, gg]
        ref_len = ref_len + 1
        pools_ref, rs_ref, ref_len, dropped = O.decode_prune(pools_ref, rs_ref, start, ref_len,
                                                             s_new, tau, window, n_sink)
        dropped_total += int(dropped.sum())
        torch.cuda.synchronize()
        assert B.kvc_device_status() == 0
        np.testing.assert_array_equal(ln.cpu().numpy(), ref_len, err_msg=f"step {step}")
        got_pools = [bits(p) for p in pools_gpu]
        ref_bits = []
        for rp in pools_ref:
            if rp.dtype == np.float16:
                ref_bits.append(rp.view(np.int16))
            elif rp.dtype == np.uint8:
                ref_bits.append(rp)
            else:   # bf16 values held in float32
                ref_bits.append(torch.from_numpy(np.ascontiguousarray(rp)).to(torch.bfloat16)
                                .view(torch.int16).numpy())
        got_rs, ref_rs = bits(rs), rs_ref.view(np.int32)
        for i in range(n):
            assert head_rows(got_pools, got_rs, start, ref_len, i) == \
                head_rows(ref_bits, ref_rs, start, ref_len, i), (step, i)
    assert 0 < dropped_total < steps * n
