"""Pins for the CPU oracle: it is checked against things other than itself.

* brute force in pure Python (math.exp, explicit loops in another order),
* hand-derived closed forms (tests/golden/closed_forms.json, with citations),
* invariants the definitions imply (rows of a softmax add to one, kept count
  equals the budget, protected tokens always kept, ...),
* independent library routines (scipy softmax, torch SDPA in float64),
* planted mistakes: wrong variants of the oracle must fail these pins.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


# ----------------------------------------------------------- brute force
def brute_score_attn(q, k, scale, head_scale=None, causal=True, aggregation="sum"):
    """Pure-Python attention mass (or maximum attention weight): token-major
    loop, explicit normaliser."""
    U, Hq, W, d = q.shape
    Hkv, T = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = [[[0.0] * T for _ in range(Hkv)] for _ in range(U)]
    for u in range(U):
        for h in range(Hq):
            g = h // G
            c = scale * (1.0 if head_scale is None else float(head_scale[u][h]))
            for w in range(W):
                last = T - W + w if causal else T - 1
                logit = []
                for t in range(last + 1):
                    acc = 0.0
                    for x in range(d):
                        acc += float(q[u][h][w][x]) * float(k[u][g][t][x])
                    logit.append(c * acc)
                mx = max(logit)
                z = sum(math.exp(v - mx) for v in logit)
                for t in range(last + 1):
                    p = math.exp(logit[t] - mx) / z
                    if aggregation == "sum":
                        out[u][g][t] += p
                    else:
                        out[u][g][t] = max(out[u][g][t], p)
    return np.array(out)


def sort_key(score, t, g):
    """(score desc, token asc, head asc) with NaN last, -0 == +0."""
    s = float(score)
    if math.isnan(s):
        return (1, 0.0, t, g)
    return (0, -(s + 0.0), t, g)


def brute_select_global(s, keep_ratio, n_sink, n_recent):
    U, Hkv, T = s.shape
    prot = [t < n_sink or t >= T - n_recent for t in range(T)]
    nP = sum(prot)
    B = math.floor(keep_ratio * (Hkv * T))
    need = min(max(B, Hkv * nP), Hkv * T) - Hkv * nP
    res = []
    for u in range(U):
        cand = [(sort_key(s[u, g, t], t, g), g, t) for t in range(T) for g in range(Hkv)
                if not prot[t]]
        cand.sort()
        chosen = {(g, t) for _, g, t in cand[:need]}
        for g in range(Hkv):
            res.append([t for t in range(T) if prot[t] or (g, t) in chosen])
    return res


def brute_select_per_head(s, budgets, n_sink, n_recent):
    U, Hkv, T = s.shape
    prot = [t < n_sink or t >= T - n_recent for t in range(T)]
    nP = sum(prot)
    res = []
    for u in range(U):
        for g in range(Hkv):
            b = int(budgets[u * Hkv + g])
            need = min(max(b, nP), T) - nP
            cand = sorted((sort_key(s[u, g, t], t, 0), t) for t in range(T) if not prot[t])
            chosen = {t for _, t in cand[:need]}
            res.append([t for t in range(T) if prot[t] or t in chosen])
    return res


def kept_lists(kept, counts):
    return [list(kept[i, : counts[i]]) for i in range(len(counts))]


def rng_arrays(seed, *shapes):
    r = np.random.default_rng(seed)
    return [r.standard_normal(s) for s in shapes]


# -------------------------------------------------------------- scoring
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("with_scale", [True, False])
def test_score_attn_matches_brute_force(causal, with_scale):
    q, k = rng_arrays(1, (2, 4, 3, 5), (2, 2, 9, 5))
    hs = np.random.default_rng(2).uniform(0.5, 2.0, (2, 4)) if with_scale else None
    got = O.score_attn(q, k, 0.7, hs, causal)
    ref = brute_score_attn(q, k, 0.7, hs, causal)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("case", ["score_attn_softmax_row", "score_attn_causal_window"])
def test_score_attn_golden(case):
    c = GOLD[case]
    got = O.score_attn(np.array(c["q_win"]), np.array(c["k"]), c["scale"], None, c["causal"])
    np.testing.assert_allclose(got, np.array(c["score"]), rtol=1e-14)


def test_score_attn_rows_sum_to_one():
    q, k = rng_arrays(3, (3, 8, 16, 16), (3, 2, 200, 16))
    for causal in (True, False):
        s = O.score_attn(q, k, 0.25, None, causal)
        # every window row is a probability distribution -> each kv head
        # collects exactly G*W units of mass
        np.testing.assert_allclose(s.sum(axis=-1), 4 * 16, rtol=1e-12)
        assert (s >= 0).all()


def test_score_attn_single_row_is_textbook_softmax():
    from scipy.special import softmax
    q, k = rng_arrays(4, (1, 1, 1, 8), (1, 1, 50, 8))
    got = O.score_attn(q, k, 0.3, None, causal=False)[0, 0]
    np.testing.assert_allclose(got, softmax(0.3 * (k[0, 0] @ q[0, 0, 0])), rtol=1e-12)


def test_score_attn_identical_keys_give_uniform_rows():
    U, Hq, Hkv, W, T, d = 1, 6, 2, 5, 17, 4
    q = rng_arrays(5, (U, Hq, W, d))[0]
    k = np.tile(rng_arrays(6, (d,))[0], (U, Hkv, T, 1))
    G = Hq // Hkv
    got = O.score_attn(q, k, 1.0, None, causal=True)
    ref = np.zeros(T)
    for w in range(W):
        n = T - W + w + 1           # tokens visible to window row w
        ref[:n] += G / n
    for g in range(Hkv):
        np.testing.assert_allclose(got[0, g], ref, rtol=1e-12)


def test_score_attn_dominant_sink():
    q = np.ones((1, 2, 4, 8))
    k = np.zeros((1, 1, 32, 8))
    k[0, 0, 0] = 10.0                    # logit 80 against 0 for the rest
    s = O.score_attn(q, k, 1.0, None, causal=True)
    assert abs(s[0, 0, 0] - 8.0) < 1e-12 and 0 < s[0, 0, 1:].sum() < 1e-30


# ------------------------------------------- max aggregation ([KVzap] §2.1)
@pytest.mark.parametrize("causal", [True, False])
def test_score_max_matches_brute_force(causal):
    q, k = rng_arrays(11, (2, 4, 3, 5), (2, 2, 9, 5))
    hs = np.random.default_rng(12).uniform(0.5, 2.0, (2, 4))
    got = O.score_attn(q, k, 0.7, hs, causal, aggregation="max")
    ref = brute_score_attn(q, k, 0.7, hs, causal, aggregation="max")
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)


def test_score_max_identical_keys_closed_form():
    """Uniform rows: token t is seen by rows w >= t - (T - W), the one with
    the fewest visible tokens gives it 1 / (T - W + w_min + 1)."""
    U, Hq, Hkv, W, T, d = 1, 6, 2, 5, 17, 4
    q = rng_arrays(13, (U, Hq, W, d))[0]
    k = np.tile(rng_arrays(14, (d,))[0], (U, Hkv, T, 1))
    got = O.score_attn(q, k, 1.0, None, causal=True, aggregation="max")
    ref = np.array([1.0 / (T - W + max(0, t - (T - W)) + 1) for t in range(T)])
    for g in range(Hkv):
        np.testing.assert_allclose(got[0, g], ref, rtol=1e-12)


def test_score_max_bounds_and_single_row():
    q, k = rng_arrays(15, (2, 8, 16, 16), (2, 2, 200, 16))
    G, W = 4, 16
    smax = O.score_attn(q, k, 0.25, None, True, aggregation="max")
    ssum = O.score_attn(q, k, 0.25, None, True)
    assert (smax <= ssum * (1 + 1e-12)).all() and (ssum <= G * W * smax * (1 + 1e-12)).all()
    assert (smax <= 1.0).all() and (smax > 0).all()
    q1, k1 = rng_arrays(16, (1, 1, 1, 8), (1, 1, 50, 8))
    np.testing.assert_allclose(O.score_attn(q1, k1, 0.3, None, False, aggregation="max"),
                               O.score_attn(q1, k1, 0.3, None, False), rtol=1e-14)


def _score_max_first_head_only(q, k, scale, head_scale=None, causal=True):
    """A planted mistake: the maximum over the first query head of each group only."""
    G = q.shape[1] // k.shape[1]
    return O.score_attn(q[:, ::G], k, scale, None, causal, "max")


def test_planted_max_mistake_is_caught():
    q, k = rng_arrays(17, (1, 4, 3, 5), (1, 2, 9, 5))
    ref = brute_score_attn(q, k, 0.7, None, True, aggregation="max")
    assert not np.allclose(_score_max_first_head_only(q, k, 0.7), ref, rtol=1e-6)
    assert not np.allclose(O.score_attn(q, k, 0.7, None, True), ref, rtol=1e-6)


# ------------------------------------------ group quantisation ([KVTC] §2B)
def brute_quantize(x):
    """Element by element with float32 / float16 scalars."""
    rows, d = x.shape
    codes = np.zeros((rows, d), dtype=np.uint8)
    params = np.zeros((rows, d // 32, 2), dtype=np.float16)
    for r in range(rows):
        for gi in range(d // 32):
            grp = [np.float32(v) for v in x[r, gi * 32:(gi + 1) * 32]]
            lo = np.float16(min(grp))
            lo32 = np.float32(lo)
            sc = np.float16(np.float32(max(grp) - lo32) / np.float32(255.0))
            sc32 = np.float32(sc)
            params[r, gi] = (sc, lo)
            for e, v in enumerate(grp):
                if sc32 == 0:
                    c = 0
                else:
                    c = int(min(255.0, max(0.0, float(np.rint(np.float32(v - lo32) / sc32)))))
                codes[r, gi * 32 + e] = c
    return codes, params


def test_quantize_matches_brute_force_and_bound():
    x = (np.random.default_rng(21).standard_normal((6, 128)) *
         np.array([1.0, 8.0, 0.01, 1.0] * 32)).astype(np.float32)
    codes, params = O.quantize_rows(x)
    bc, bp = brute_quantize(x)
    np.testing.assert_array_equal(codes, bc)
    np.testing.assert_array_equal(params.view(np.uint16), bp.view(np.uint16))
    # rounding error of a code is at most half a step, plus the offset's own
    # rounding at the clamped ends
    xr = O.dequantize_rows(codes, params).reshape(6, 4, 32)
    g = x.reshape(6, 4, 32).astype(np.float64)
    sc = params[..., 0].astype(np.float64)[..., None]
    lo_err = np.abs(params[..., 1].astype(np.float64) - g.min(-1))[..., None]
    assert (np.abs(xr - g) <= 0.5 * sc + lo_err + sc * 1e-3 + 1e-12).all()


def test_quantize_closed_forms():
    # integers 0..255 with both ends present: lo = 0, scale = 1, codes = values
    rng = np.random.default_rng(22)
    ints = rng.integers(0, 256, (3, 64)).astype(np.float32)
    ints[:, 0] = 0; ints[:, 31] = 255; ints[:, 32] = 0; ints[:, 63] = 255
    codes, params = O.quantize_rows(ints)
    np.testing.assert_array_equal(codes, ints.astype(np.uint8))
    np.testing.assert_array_equal(O.dequantize_rows(codes, params), ints)
    # half steps round to even: 3.5 -> 4, 2.5 -> 2
    h = ints.copy(); h[0, 5] = 3.5; h[0, 6] = 2.5
    c2, _ = O.quantize_rows(h)
    assert c2[0, 5] == 4 and c2[0, 6] == 2
    # a constant group: scale 0, codes 0, the value back exactly (fp16-representable)
    const = np.full((1, 32), 0.75, dtype=np.float32)
    c3, p3 = O.quantize_rows(const)
    assert (c3 == 0).all() and p3[0, 0, 0] == 0 and O.dequantize_rows(c3, p3)[0, 0] == 0.75


def test_planted_quantize_mistakes_are_caught():
    x = np.random.default_rng(23).standard_normal((2, 64)).astype(np.float32)
    ref, _ = brute_quantize(x)

    def floor_codes(xx):                   # truncation instead of rounding
        xf = xx.reshape(2, 2, 32)
        lo = xf.min(-1).astype(np.float16).astype(np.float32)
        sc = ((xf.max(-1) - lo) / np.float32(255)).astype(np.float16).astype(np.float32)
        return np.clip(np.floor((xf - lo[..., None]) / sc[..., None]), 0, 255).astype(np.uint8).reshape(2, 64)

    def wide_groups(xx):                   # one group of 64
        lo = np.float32(np.float16(xx.min(-1, keepdims=True)))
        sc = np.float32(np.float16((xx.max(-1, keepdims=True) - lo) / np.float32(255)))
        return np.clip(np.rint((xx - lo) / sc), 0, 255).astype(np.uint8)

    assert not np.array_equal(floor_codes(x), ref)
    assert not np.array_equal(wide_groups(x), ref)


def test_score_linear_matches_loops_and_torch():
    h, w, b = rng_arrays(7, (2, 11, 13), (13, 3), (3,))
    got = O.score_linear(h, w, b)
    for u in range(2):
        for g in range(3):
            for t in range(11):
                ref = b[g] + sum(h[u, t, j] * w[j, g] for j in range(13))
                assert abs(got[u, g, t] - ref) < 1e-12
    th = torch.from_numpy(h) @ torch.from_numpy(w) + torch.from_numpy(b)
    np.testing.assert_allclose(got, th.permute(0, 2, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_threshold_keep_fraction_matches_gaussian_tail():
    # linear outputs with weight ~ N(0, 1/Dh) are ~ N(0, 1): P(x >= 0.5) = 0.3085
    from kv_cache_compression_attention_b300 import inputs
    wl = inputs.WORKLOADS["c4_qwen128k"].with_(T=8192, Dh=512)
    hid, wt, bias = inputs.linear_scorer(wl)
    s = O.score_linear(hid.float().numpy(), wt.float().numpy(), bias.numpy())
    kept, counts, _ = O.select(s.astype(np.float32), "threshold", tau=0.5, n_sink=0, n_recent=0)
    frac = counts.sum() / s.size
    assert abs(frac - 0.30854) < 0.01



def test_tiny_workload_keeps_every_needle():
    """Statistical sanity of the sink / needle construction (keys aligned with
    the group's mean window-query direction: 4 sqrt(d) u for the sinks, 3 sqrt(d)
    u + noise for the needles): on the tiny workload at keep ratio 0.25 the
    oracle's global top-k keeps all 16 needles in every kv head, and the
    needles are the highest-scoring tokens after the four sinks.  If this
    fails, the generator does not build the structure the fidelity probe
    relies on ([KVTC] §2A sinks; [KVzap] §2.1 attention-based scores)."""
    from kv_cache_compression_attention_b300 import inputs
    w = inputs.WORKLOADS["c1_tiny"]
    q = inputs.window_queries(w)
    k, _ = inputs.keys_values(w, q)
    s = O.score_attn(q.double().numpy(), k.double().numpy(), w.scale)
    kept, counts, _ = O.select(s.astype(np.float32), "global", keep_ratio=w.keep_ratio,
                               n_sink=w.n_sink, n_recent=w.n_recent)
    pos = inputs.needle_positions(w).numpy()[0]
    assert pos.size == 16
    for g in range(w.Hkv):
        kept_g = set(kept[g, : counts[g]].tolist())
        assert all(int(p) in kept_g for p in pos), g
        order = np.argsort(-s[0, g], kind="stable")
        assert set(order[:4].tolist()) == set(range(4))             # the sinks first
        assert set(order[4:4 + pos.size].tolist()) == set(pos.tolist())   # then the needles

# ------------------------------------------------------------ selection
@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("ties,specials", [(False, False), (True, False), (True, True)])
def test_select_global_matches_brute_force(seed, ties, specials):
    from kv_cache_compression_attention_b300 import inputs
    s = inputs.random_scores((2, 3, 23), seed=seed, ties=ties, specials=specials).numpy()
    for ratio in (0.0, 0.1, 0.37, 0.5, 1.0):
        kept, counts, offs = O.select(s, "global", keep_ratio=ratio, n_sink=2, n_recent=3)
        assert kept_lists(kept, counts) == brute_select_global(s, ratio, 2, 3)
        assert offs[0] == 0 and (np.diff(offs) == counts).all()


@pytest.mark.parametrize("case", ["select_global_with_ties", "select_protected_overrides_budget"])
def test_select_golden(case):
    c = GOLD[case]
    s = np.array(c["scores"], dtype=np.float32)
    for cc in c["cases"]:
        kept, counts, _ = O.select(s, "global", keep_ratio=cc["keep_ratio"],
                                   n_sink=c.get("n_sink", 0), n_recent=c.get("n_recent", 0))
        assert [list(map(int, x)) for x in kept_lists(kept, counts)] == cc["kept"]


@pytest.mark.parametrize("seed", range(3))
def test_select_per_head_matches_brute_force(seed):
    from kv_cache_compression_attention_b300 import inputs
    s = inputs.random_scores((2, 3, 31), seed=10 + seed, ties=True, specials=seed == 2).numpy()
    budgets = np.random.default_rng(seed).integers(-2, 35, size=6)
    kept, counts, _ = O.select(s, "per_head", head_budget=budgets, n_sink=1, n_recent=4)
    assert kept_lists(kept, counts) == brute_select_per_head(s, budgets, 1, 4)


def test_protected_mask_closed_forms():
    """The always-kept tokens: the first n_sink and the last n_recent
    positions, with the two ranges overlapping when they cover T."""
    T_, F_ = True, False
    assert O.protected_mask(10, 2, 3).tolist() == [T_, T_, F_, F_, F_, F_, F_, T_, T_, T_]
    assert O.protected_mask(5, 3, 4).all()
    assert not O.protected_mask(6, 0, 0).any()
    assert O.protected_mask(4, 0, 1).tolist() == [F_, F_, F_, T_]
    assert O.protected_mask(4, 1, 0).tolist() == [T_, F_, F_, F_]


def test_global_budget_one_double_rounding():
    """B = floor(ratio * Hkv * T), the product rounded once in IEEE double:
    0.1 of 8 x 32768 keys is 26214.4 -> 26214; 0.29 * 100 is
    28.999999999999996 in double -> 28 (not 29); exact products stay exact."""
    assert O.global_budget(0.10, 8, 32768) == 26214
    assert O.global_budget(0.25, 4, 1024) == 1024
    assert O.global_budget(0.29, 1, 100) == 28
    assert O.global_budget(0.7, 1, 10) == 7
    assert O.global_budget(0.0, 8, 32768) == 0
    assert O.global_budget(1.0, 8, 32768) == 8 * 32768


def test_select_threshold_exact_set():
    from kv_cache_compression_attention_b300 import inputs
    s = inputs.random_scores((2, 2, 40), seed=3, ties=True, specials=True).numpy()
    tau = 0.5
    kept, counts, _ = O.select(s, "threshold", tau=tau, n_sink=3, n_recent=5)
    got = kept_lists(kept, counts)
    for i in range(4):
        u, g = divmod(i, 2)
        ref = [t for t in range(40)
               if t < 3 or t >= 35 or (not math.isnan(s[u, g, t]) and s[u, g, t] >= tau)]
        assert got[i] == ref


def test_select_invariants_large():
    from kv_cache_compression_attention_b300 import inputs
    U, Hkv, T = 3, 8, 4099
    s = inputs.random_scores((U, Hkv, T), seed=9, ties=True).numpy()
    n_sink, n_recent, ratio = 4, 64, 0.1
    kept, counts, offs = O.select(s, "global", keep_ratio=ratio, n_sink=n_sink, n_recent=n_recent)
    B = math.floor(ratio * Hkv * T)
    P = set(range(n_sink)) | set(range(T - n_recent, T))
    for u in range(U):
        assert counts[u * Hkv:(u + 1) * Hkv].sum() == B
        kept_free, dropped = [], []
        for g in range(Hkv):
            idx = list(kept[u * Hkv + g, : counts[u * Hkv + g]])
            assert idx == sorted(set(idx))                     # ascending, unique
            assert P <= set(idx)                                # protected kept
            ks = set(idx)
            for t in range(T):
                if t in P:
                    continue
                (kept_free if t in ks else dropped).append(sort_key(s[u, g, t], t, g))
        assert max(kept_free) < min(dropped)                  # nothing dropped outranks a kept one
    # heads keep different counts (adaptive per-head budget)
    assert len(set(counts.tolist())) > 1


# ------------------------------------------------------------ compaction
def test_compact_matches_fancy_indexing():
    r = np.random.default_rng(11)
    U, Hkv, T, d = 2, 3, 20, 6
    k = r.standard_normal((U, Hkv, T, d)).astype(np.float32)
    v = r.standard_normal((U, Hkv, T, d)).astype(np.float32)
    s = r.random((U, Hkv, T)).astype(np.float32)
    kept, counts, offs = O.select(s, "global", keep_ratio=0.3, n_sink=1, n_recent=2)
    kc, vc, start, length = O.compact(k, v, kept, counts, offs, slack=2)
    assert kc.shape[0] == offs[-1] + 2 * U * Hkv
    for i in range(U * Hkv):
        u, g = divmod(i, Hkv)
        assert start[i] == offs[i] + 2 * i and length[i] == counts[i]
        idx = kept[i, : counts[i]]
        np.testing.assert_array_equal(kc[start[i]: start[i] + counts[i]], k[u, g][idx])
        np.testing.assert_array_equal(vc[start[i]: start[i] + counts[i]], v[u, g][idx])
        assert not kc[start[i] + counts[i]: start[i] + counts[i] + 2].any()


# ---------------------------------------------------------------- decode
def sdpa_ref(q, kc, vc, start, length, scale, G):
    """torch float64 scaled_dot_product_attention per (unit, head)."""
    U, Hq, d = q.shape
    out = np.zeros((U, Hq, d))
    lse = np.zeros((U, Hq))
    for u in range(U):
        for h in range(Hq):
            i = u * (Hq // G) + h // G
            K = torch.from_numpy(kc[start[i]: start[i] + length[i]].astype(np.float64))
            V = torch.from_numpy(vc[start[i]: start[i] + length[i]].astype(np.float64))
            qq = torch.from_numpy(q[u, h].astype(np.float64))
            o = torch.nn.functional.scaled_dot_product_attention(
                qq[None, None, None], K[None, None], V[None, None], scale=scale)
            out[u, h] = o[0, 0, 0].numpy()
            lse[u, h] = torch.logsumexp(scale * (K @ qq), 0).item()
    return out, lse


def test_decode_matches_sdpa_and_appends():
    r = np.random.default_rng(12)
    U, Hq, Hkv, d, slack = 2, 8, 2, 16, 1
    lens = np.array([5, 17, 1, 40])
    start = np.concatenate([[0], np.cumsum(lens + slack)[:-1]])
    rows = int((lens + slack).sum())
    kc = r.standard_normal((rows, d))
    vc = r.standard_normal((rows, d))
    q = r.standard_normal((U, Hq, d))
    kn = r.standard_normal((U, Hkv, d))
    vn = r.standard_normal((U, Hkv, d))
    out, lse, kc2, vc2, len2 = O.decode_attn(q, kc, vc, start, lens, kn, vn, scale=0.25)
    assert (len2 == lens + 1).all()
    for i in range(U * Hkv):
        u, g = divmod(i, Hkv)
        np.testing.assert_array_equal(kc2[start[i] + lens[i]], kn[u, g])
        np.testing.assert_array_equal(vc2[start[i] + lens[i]], vn[u, g])
    ref_o, ref_l = sdpa_ref(q, kc2, vc2, start, len2, 0.25, Hq // Hkv)
    np.testing.assert_allclose(out, ref_o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12)


def test_decode_golden():
    c = GOLD["decode_append"]
    out, lse, _, _, len2 = O.decode_attn(np.array(c["q"]), np.array(c["kc"]), np.array(c["vc"]),
                                         np.array(c["start"]), np.array(c["len"]),
                                         np.array(c["k_new"]), np.array(c["v_new"]), scale=1.0)
    np.testing.assert_allclose(out, np.array(c["out"]), rtol=1e-14)
    np.testing.assert_allclose(lse, np.array(c["lse"]), rtol=1e-14)
    assert len2[0] == 2


def _full_cache(k, v, slack):
    """Full cache laid out like a compacted one (every token kept)."""
    U, Hkv, T, d = k.shape
    kept = np.tile(np.arange(T, dtype=np.int32), (U * Hkv, 1))
    counts = np.full(U * Hkv, T, dtype=np.int32)
    offs = np.arange(U * Hkv + 1, dtype=np.int64) * T
    return O.compact(k, v, kept, counts, offs, slack)


def test_keep_ratio_one_is_the_full_cache_and_kl_is_zero():
    r = np.random.default_rng(13)
    U, Hq, Hkv, W, T, d = 1, 4, 2, 4, 30, 8
    q_win = r.standard_normal((U, Hq, W, d))
    k = r.standard_normal((U, Hkv, T, d))
    v = r.standard_normal((U, Hkv, T, d))
    s = O.score_attn(q_win, k, 0.3).astype(np.float32)
    kept, counts, offs = O.select(s, "global", keep_ratio=1.0, n_sink=1, n_recent=2)
    kc, vc, st, ln = O.compact(k, v, kept, counts, offs, slack=1)
    kf, vf, sf, lf = _full_cache(k, v, 1)
    np.testing.assert_array_equal(kc, kf)
    q = r.standard_normal((U, Hq, d))
    kn, vn = r.standard_normal((U, Hkv, d)), r.standard_normal((U, Hkv, d))
    oc, lc, *_ = O.decode_attn(q, kc, vc, st, ln, kn, vn, 0.3)
    of, lf2, *_ = O.decode_attn(q, kf, vf, sf, lf, kn, vn, 0.3)
    np.testing.assert_array_equal(oc, of)
    err, kl = O.fidelity(oc, of, lc, lf2)
    assert (err == 0).all() and (kl == 0).all()


def test_kl_is_minus_log_retained_mass():
    r = np.random.default_rng(14)
    U, Hq, Hkv, W, T, d = 1, 4, 2, 4, 60, 8
    q_win = r.standard_normal((U, Hq, W, d))
    k = r.standard_normal((U, Hkv, T, d))
    v = r.standard_normal((U, Hkv, T, d))
    s = O.score_attn(q_win, k, 0.3).astype(np.float32)
    kept, counts, offs = O.select(s, "global", keep_ratio=0.3, n_sink=2, n_recent=4)
    kc, vc, st, ln = O.compact(k, v, kept, counts, offs)
    kf, vf, sf, lf = _full_cache(k, v, 0)
    q = r.standard_normal((U, Hq, d))
    oc, lc, *_ = O.decode_attn(q, kc, vc, st, ln, None, None, 0.3)
    of, lfull, *_ = O.decode_attn(q, kf, vf, sf, lf, None, None, 0.3)
    err, kl = O.fidelity(oc, of, lc, lfull)
    for h in range(Hq):
        g = h // 2
        logits = 0.3 * (k[0, g] @ q[0, h])
        p = np.exp(logits - logits.max())
        p /= p.sum()
        mass = p[kept[g, : counts[g]]].sum()
        assert abs(kl[0, h] + math.log(mass)) < 1e-12
        assert kl[0, h] >= 0 and err[0, h] > 0


def test_fidelity_golden_and_scaling():
    c = GOLD["fidelity_kl"]
    _, kl = O.fidelity(np.ones((1, 1, 2)), np.ones((1, 1, 2)),
                       np.array([[c["lse_comp"]]]), np.array([[c["lse_full"]]]))
    assert abs(kl[0, 0] - c["kl"]) < 1e-15
    o = np.random.default_rng(15).standard_normal((2, 3, 8))
    err, _ = O.fidelity(1.5 * o, o, np.zeros((2, 3)), np.zeros((2, 3)))
    np.testing.assert_allclose(err, 0.5, rtol=1e-14)


# ------------------------------------------------------ planted mistakes
def _score_attn_wrong_gqa(q, k, scale, head_scale=None, causal=True):
    """Planted mistake: query head h read against kv head h % Hkv."""
    q = np.asarray(q, float)
    U, Hq, W, d = q.shape
    Hkv = k.shape[1]
    perm = [(h % Hkv) * (Hq // Hkv) + h // Hkv for h in range(Hq)]
    return O.score_attn(q[:, np.argsort(perm)], k, scale, head_scale, causal)


def _score_attn_no_causal(q, k, scale, head_scale=None, causal=True):
    return O.score_attn(q, k, scale, head_scale, causal=False)


def _score_attn_no_scale(q, k, scale, head_scale=None, causal=True):
    return O.score_attn(q, k, 1.0, head_scale, causal)


@pytest.mark.parametrize("bad", [_score_attn_wrong_gqa, _score_attn_no_causal, _score_attn_no_scale])
def test_planted_score_mistakes_are_caught(bad):
    q, k = rng_arrays(1, (2, 4, 3, 5), (2, 2, 9, 5))
    ref = brute_score_attn(q, k, 0.7, None, True)
    assert not np.allclose(bad(q, k, 0.7, None, True), ref, rtol=1e-6)


def test_planted_tie_break_mistake_is_caught():
    # head-asc before token-asc would pick (t1,g0) before (t0,g1)
    c = GOLD["select_global_with_ties"]
    s = np.array(c["scores"], dtype=np.float32)
    U, Hkv, T = s.shape
    cand = sorted(((-(float(s[0, g, t])), g, t) for g in range(Hkv) for t in range(T)))
    chosen = {(g, t) for _, g, t in cand[:6]}
    wrong = [[t for t in range(T) if (g, t) in chosen] for g in range(Hkv)]
    assert wrong != c["cases"][1]["kept"]


# ------------------------------------- decode-time pruning ([KVzap] §2.3)
def _prune_stream_matches(prune, tau, seed, steps=40, w=6, n_sink=2, T=40, heads=3, slack=48,
                          nan_frac=0.05, tie_frac=0.1):
    """Prefill compaction followed by `steps` decode steps of append + prune.
    After every step each head's rows must be, in token order, the set the
    rule defines without reference to rows: the prefill-kept tokens older
    than the prefill window, the tokens that have left the window since then
    with score >= tau, and the last w tokens.  The pools carry token ids, so
    any misplaced row shows; the per-row scores must follow their rows."""
    rng = np.random.default_rng(seed)
    S = rng.standard_normal((heads, T + steps)).astype(np.float32)
    if np.isfinite(tau):
        S[rng.random(S.shape) < tie_frac] = np.float32(tau)
    S[rng.random(S.shape) < nan_frac] = np.nan
    kept = []
    for i in range(heads):
        mid = [t for t in range(n_sink, T - w) if rng.random() < 0.4]
        kept.append(list(range(n_sink)) + mid + list(range(T - w, T)))
    counts = np.array([len(k) for k in kept])
    start = np.concatenate([[0], np.cumsum(counts + slack)[:-1]]).astype(np.int64)
    rows = int((counts + slack).sum())
    kpool = np.full((rows, 2), -1, dtype=np.int64)      # (token, head)
    vpool = np.full(rows, -1.0)                         # token + 0.5
    rscore = np.full(rows, np.nan, dtype=np.float32)
    for i in range(heads):
        for j, t in enumerate(kept[i]):
            kpool[start[i] + j] = (t, i)
            vpool[start[i] + j] = t + 0.5
            rscore[start[i] + j] = S[i, t]
    length = counts.astype(np.int32)
    for step in range(steps):
        pos = T + step
        for i in range(heads):           # the decode step's append
            kpool[start[i] + length[i]] = (pos, i)
            vpool[start[i] + length[i]] = pos + 0.5
        length = length + 1
        (kpool, vpool), rscore, length, _ = prune([kpool, vpool], rscore, start, length,
                                                  S[:, pos], tau, w, n_sink)
        cur = pos + 1
        for i in range(heads):
            expect = ([t for t in kept[i] if t < T - w] +
                      [t for t in range(T - w, cur - w) if S[i, t] >= np.float32(tau)] +
                      list(range(cur - w, cur)))
            s0, L = int(start[i]), int(length[i])
            got = kpool[s0: s0 + L]
            if L != len(expect) or list(got[:, 0]) != expect or np.any(got[:, 1] != i):
                return False
            if np.any(vpool[s0: s0 + L] != got[:, 0] + 0.5):
                return False
            if rscore[s0: s0 + L].tobytes() != S[i, got[:, 0]].tobytes():
                return False
    return True


@pytest.mark.parametrize("tau", [0.0, 0.7, -1.3])
@pytest.mark.parametrize("seed", [41, 42])
def test_prune_matches_the_set_definition(tau, seed):
    assert _prune_stream_matches(O.decode_prune, tau, seed)


def test_prune_closed_forms():
    # tau = -inf, no NaN: nothing is ever dropped; the cache only grows
    assert _prune_stream_matches(O.decode_prune, -np.inf, 43, nan_frac=0.0)
    # tau = +inf, finite scores: every token leaving the window goes, so the
    # length stays at the prefill count after every step
    pools = [np.arange(30, dtype=np.int64)]
    length = np.array([12], dtype=np.int32)
    rs = np.zeros(30, dtype=np.float32)
    for step in range(10):
        length = length + 1
        pools, rs, length, dropped = O.decode_prune(pools, rs, [0], length, [1.0], np.inf, 5, 2)
        assert length[0] == 12 and dropped[0]
    # sinks are never dropped: 4 sinks, a window of 2, 3 rows before the append
    pools, rs2, L2, dropped = O.decode_prune([np.arange(8)], np.full(8, -5.0, np.float32), [0],
                                             np.array([4], np.int32), [2.5], np.inf, 2, 4)
    assert L2[0] == 4 and not dropped[0] and rs2[3] == np.float32(2.5)
    # no row at all: nothing written, nothing dropped
    _, rs3, L3, d3 = O.decode_prune([np.arange(4)], np.zeros(4, np.float32), [0],
                                    np.array([0], np.int32), [9.0], 0.0, 2, 0)
    assert L3[0] == 0 and not d3[0] and not np.any(rs3)


def test_gather_scores_brute_force():
    rng = np.random.default_rng(44)
    scores = rng.standard_normal((2, 3, 20)).astype(np.float32)
    kept, counts, offsets = O.select(scores, "per_head", head_budget=np.full(6, 7), n_sink=2,
                                     n_recent=3)
    _, _, start, length = O.compact(np.zeros((2, 3, 20, 1)), np.zeros((2, 3, 20, 1)), kept, counts,
                                    offsets, slack=4)
    rs = O.gather_scores(scores, kept, counts, start, int(offsets[-1]) + 6 * 4)
    for u in range(2):
        for g in range(3):
            i = u * 3 + g
            picked = sorted(scores[u, g, t] for t in range(20)
                            if t < 2 or t >= 17 or t in set(kept[i, :counts[i]].tolist()))
            assert sorted(rs[start[i]: start[i] + length[i]].tolist()) == picked
            assert np.all(np.isnan(rs[start[i] + length[i]: start[i] + length[i] + 4]))


def _prune_planted(kind):
    """Planted mistakes in decode-time pruning, each a copy of the rule with
    one thing wrong."""
    def prune(pools, rscore, start, length, s_new, tau, window, n_sink=0):
        pools = [np.array(p, copy=True) for p in pools]
        rs = np.array(rscore, dtype=np.float32, copy=True)
        length = np.array(length, dtype=np.int64, copy=True)
        for i in range(length.size):
            s0, L = int(start[i]), int(length[i])
            rs[s0 + L - (0 if kind == "score_row" else 1)] = np.float32(s_new[i])
            e = L - window - (0 if kind == "exit_row" else 1)
            s = rs[s0 + e]
            if kind == "strict":
                keep = s > np.float32(tau)
            elif kind == "nan_kept":
                keep = not (s < np.float32(tau))
            else:
                keep = s >= np.float32(tau)
            if e < n_sink or keep:
                continue
            for p in pools:
                p[s0 + e: s0 + L - 1] = p[s0 + e + 1: s0 + L].copy()
            if kind != "scores_stay":
                rs[s0 + e: s0 + L - 1] = rs[s0 + e + 1: s0 + L].copy()
            length[i] = L - 1
        return pools, rs, length.astype(np.int32), None
    return prune


@pytest.mark.parametrize("kind", ["score_row", "exit_row", "strict", "nan_kept", "scores_stay"])
def test_planted_prune_mistakes_are_caught(kind):
    assert not all(_prune_stream_matches(_prune_planted(kind), tau, seed)
                   for tau in (0.0, 0.7) for seed in (41, 42))


# --------------------------------------------- VECTOR three-way routing
def _lowrank_kv(rng, Hkv, N, d, r, noise):
    """K and V as linear maps of one shared low-rank state plus noise."""
    h = rng.standard_normal((Hkv, N, r))
    Ak = rng.standard_normal((Hkv, d, r))
    Av = rng.standard_normal((Hkv, d, r))
    k = np.einsum("gnr,gdr->gnd", h, Ak) + noise * rng.standard_normal((Hkv, N, d))
    v = np.einsum("gnr,gdr->gnd", h, Av) + noise * rng.standard_normal((Hkv, N, d))
    return k, v


def test_fit_ols_closed_form_and_lstsq():
    rng = np.random.default_rng(71)
    # exact linear relation v = A k: the fit returns A
    k = rng.standard_normal((2, 40, 6))
    A = rng.standard_normal((2, 6, 6))
    v = np.einsum("gxy,gny->gnx", A, k)
    np.testing.assert_allclose(O.fit_ols(k, v), A, rtol=0, atol=1e-9)
    # noisy: residuals orthogonal to the keys, and equal to an SVD least squares
    k, v = _lowrank_kv(rng, 2, 200, 8, 3, 0.3)
    W = O.fit_ols(k, v)
    for g in range(2):
        res = v[g] - k[g] @ W[g].T
        np.testing.assert_allclose(res.T @ k[g], 0.0, atol=1e-8)
        sol = np.linalg.lstsq(k[g], v[g], rcond=None)[0]      # k @ sol ~ v
        np.testing.assert_allclose(W[g], sol.T, rtol=1e-9, atol=1e-9)


def test_vector_budgets_memory_accounting():
    # K rows for the pool plus V rows for the exact tokens = 2 (1 - p_c) pairs
    for p_c, p_a, Hkv, T in [(0.9, 0.05, 8, 32768), (0.75, 0.1, 4, 1000), (0.5, 0.2, 2, 777)]:
        _, B, A = O.vector_budgets(p_c, p_a, Hkv, T, 4, 64)
        assert abs((B + (B - A)) - 2 * (1 - p_c) * Hkv * T) <= 2
    # the approximated count never reaches into the protected set
    _, B, A = O.vector_budgets(0.5, 0.45, 2, 100, 4, 16)
    assert B - A == 2 * 20


def _vector_case(seed, U=2, Hkv=3, T=40, d=6):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((U, Hkv, T, d))
    v = rng.standard_normal((U, Hkv, T, d))
    W = rng.standard_normal((Hkv, d, d))                      # not symmetric
    scores = rng.standard_normal((U, Hkv, T)).astype(np.float32)
    kept, counts, offsets = O.select(scores, "global", keep_ratio=0.5, n_sink=2, n_recent=3)
    return k, v, W, kept, counts


def test_vector_residual_brute_force():
    k, v, W, kept, counts = _vector_case(72)
    key = O.vector_residual(k, v, W, kept, counts, 2, 3)
    U, Hkv, T, d = k.shape
    for u in range(U):
        for g in range(Hkv):
            i = u * Hkv + g
            for j in range(T):
                if j >= counts[i]:
                    assert np.isnan(key[u, g, j])
                    continue
                t = kept[i, j]
                if t < 2 or t >= T - 3:
                    assert np.isnan(key[u, g, j])
                    continue
                eps = 0.0
                for x in range(d):
                    rec = sum(W[g, x, y] * k[u, g, t, y] for y in range(d))
                    eps += (v[u, g, t, x] - rec) ** 2
                assert key[u, g, j] == np.float32(-eps)
    # v = W k exactly: every error is zero
    v2 = np.einsum("gxy,ugty->ugtx", W, k)
    key2 = O.vector_residual(k, v2, W, kept, counts, 2, 3)
    ok = ~np.isnan(key2)
    assert ok.sum() > 0 and np.all(np.abs(key2[ok]) < 1e-9)


def test_vector_approx_and_compact_invariants():
    k, v, W, kept, counts = _vector_case(73)
    key = O.vector_residual(k, v, W, kept, counts, 2, 3)
    U, Hkv, T, d = k.shape
    A = 15
    pos, cnt = O.vector_approx(key, A)
    for u in range(U):
        heads = range(u * Hkv, (u + 1) * Hkv)
        assert sum(cnt[i] for i in heads) == A
        # every chosen error is <= every eligible unchosen error of the unit
        chosen = [float(-key[u, i - u * Hkv, j]) for i in heads for j in pos[i, :cnt[i]]]
        rest = [float(-key[u, g, j]) for g in range(Hkv) for j in range(T)
                if not np.isnan(key[u, g, j]) and j not in set(pos[u * Hkv + g, :cnt[u * Hkv + g]])]
        assert max(chosen) <= min(rest)
    kc, vc, kstart, klen, vstart, napprox = O.vector_compact(k, v, kept, counts, pos, cnt, slack=2)
    for i in range(U * Hkv):
        u, g = divmod(i, Hkv)
        pool = [int(t) for t in kept[i, :counts[i]]]
        approx_t = [pool[j] for j in pos[i, :cnt[i]]]
        exact_t = [t for t in pool if t not in approx_t]
        assert klen[i] == len(pool) and napprox[i] == len(approx_t)
        np.testing.assert_array_equal(kc[kstart[i]: kstart[i] + napprox[i]], k[u, g, approx_t])
        np.testing.assert_array_equal(kc[kstart[i] + napprox[i]: kstart[i] + klen[i]], k[u, g, exact_t])
        np.testing.assert_array_equal(vc[vstart[i]: vstart[i] + len(exact_t)], v[u, g, exact_t])
        # protected tokens keep exact values
        assert all(t >= 2 and t < T - 3 for t in approx_t)


def test_decode_attn_vector_against_sdpa_and_special_cases():
    k, v, W, kept, counts = _vector_case(74)
    U, Hkv, T, d = k.shape
    key = O.vector_residual(k, v, W, kept, counts, 2, 3)
    pos, cnt = O.vector_approx(key, 12)
    kc, vc, kstart, klen, vstart, napprox = O.vector_compact(k, v, kept, counts, pos, cnt, slack=1)
    rng = np.random.default_rng(75)
    G = 2
    q = rng.standard_normal((U, Hkv * G, d))
    kn = rng.standard_normal((U, Hkv, d))
    vn = rng.standard_normal((U, Hkv, d))
    out, lse, _, _, klen2 = O.decode_attn_vector(q, kc, vc, kstart, klen, vstart, napprox, W,
                                                 kn, vn, 0.4)
    np.testing.assert_array_equal(klen2, klen + 1)
    for i in range(U * Hkv):
        u, g = divmod(i, Hkv)
        pool = [int(t) for t in kept[i, :counts[i]]]
        approx_t = set(pool[j] for j in pos[i, :cnt[i]])
        K = np.concatenate([k[u, g, pool], kn[u, g][None]])
        V = np.concatenate([np.stack([W[g] @ k[u, g, t] if t in approx_t else v[u, g, t]
                                      for t in pool]), vn[u, g][None]])
        for j in range(G):
            h = g * G + j
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[u, h][None, None, None]), torch.from_numpy(K[None, None]),
                torch.from_numpy(V[None, None]), scale=0.4)[0, 0, 0].numpy()
            np.testing.assert_allclose(out[u, h], ref, rtol=1e-10, atol=1e-12)
            logits = 0.4 * (K @ q[u, h])
            assert abs(lse[u, h] - (logits.max() + np.log(np.exp(logits - logits.max()).sum()))) < 1e-12
    # no approximated rows: the plain decode over the same rows
    z = np.zeros_like(napprox)
    kc0, vc0, ks0, kl0, vs0, _ = O.vector_compact(k, v, kept, counts, pos, z, slack=1)
    o1, l1, _, _, _ = O.decode_attn_vector(q, kc0, vc0, ks0, kl0, vs0, z, W, None, None, 0.4)
    o2, l2, _, _, _ = O.decode_attn(q, kc0, vc0, ks0, kl0, None, None, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)


def test_planted_vector_mistakes_are_caught():
    k, v, W, kept, counts = _vector_case(76)
    key = O.vector_residual(k, v, W, kept, counts, 2, 3)
    # transposed predictor: the errors change
    keyT = O.vector_residual(k, v, np.transpose(W, (0, 2, 1)), kept, counts, 2, 3)
    ok = ~np.isnan(key)
    assert not np.allclose(key[ok], keyT[ok])
    # approximating the highest-error tokens instead of the lowest picks others
    pos, cnt = O.vector_approx(key, 10)
    pos_bad, cnt_bad = O.vector_approx(-key, 10)
    assert any(set(pos[i, :cnt[i]]) != set(pos_bad[i, :cnt_bad[i]]) for i in range(len(cnt)))
    # reconstructing with W^T in the decode changes the outputs
    kc, vc, kstart, klen, vstart, napprox = O.vector_compact(k, v, kept, counts, pos, cnt)
    q = np.random.default_rng(77).standard_normal((2, 3, 6))
    o1, _, _, _, _ = O.decode_attn_vector(q, kc, vc, kstart, klen, vstart, napprox, W)
    o2, _, _, _, _ = O.decode_attn_vector(q, kc, vc, kstart, klen, vstart, napprox,
                                          np.transpose(W, (0, 2, 1)))
    assert not np.allclose(o1, o2)


def test_fit_ols_recovers_the_synthetic_predictor():
    """The VECTOR workloads draw the predictor W and values v = W k + noise;
    the oracle's offline OLS fit on such calibration pairs recovers W."""
    from kv_cache_compression_attention_b300 import inputs
    w = inputs.WORKLOADS["c1_tiny"].with_(T=32768)     # sampling error ~ 0.026 relative
    k = torch.randn((w.U, w.Hkv, w.T, w.d), generator=torch.Generator().manual_seed(78))
    W = inputs.vector_predictor(w, "cpu")
    v = inputs.vector_values(w, k, W, "cpu")
    fit = O.fit_ols(k[0].numpy(), v[0].float().numpy())
    Wf = W.float().numpy()
    rel = np.linalg.norm(fit - Wf) / np.linalg.norm(Wf)
    assert rel < 0.05, rel


# ------------------------------------------ MLP surrogate ([KVzap] §2.2)
def test_gelu_special_cases_and_torch():
    z = np.array([0.0, 1.0, -1.0, 8.0, -8.0, 0.5, -3.0])
    g = O.gelu(z)
    assert g[0] == 0.0
    assert abs(g[1] - 0.8413447460685429) < 1e-15          # Phi(1) = 0.841344746...
    assert abs(g[1] - g[2] - 1.0) < 1e-15                  # GELU(z) - GELU(-z) = z
    assert abs(g[3] - 8.0) < 1e-14 and abs(g[4]) < 1e-14
    ref = torch.nn.functional.gelu(torch.from_numpy(z)).numpy()
    np.testing.assert_allclose(g, ref, rtol=1e-15, atol=1e-16)


def test_score_mlp_brute_force():
    rng = np.random.default_rng(79)
    U, T, Dh, Dm, Hkv = 2, 3, 5, 4, 3
    h = rng.standard_normal((U, T, Dh))
    w1, b1 = rng.standard_normal((Dh, Dm)), rng.standard_normal(Dm)
    w2, b2 = rng.standard_normal((Dm, Hkv)), rng.standard_normal(Hkv)
    got = O.score_mlp(h, w1, b1, w2, b2)
    for u in range(U):
        for t in range(T):
            act = []
            for m in range(Dm):
                z = b1[m] + sum(h[u, t, j] * w1[j, m] for j in range(Dh))
                act.append(0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0))))
            for g in range(Hkv):
                ref = b2[g] + sum(act[m] * w2[m, g] for m in range(Dm))
                assert abs(got[u, g, t] - ref) < 1e-12


def test_score_mlp_reduces_to_linear_when_gelu_is_identity():
    # pre-activations far above 0: GELU(z) = z to double precision, so the MLP
    # is the linear surrogate with weight w1 w2 and bias b1 w2 + b2
    rng = np.random.default_rng(80)
    h = rng.standard_normal((1, 6, 4)) * 0.1
    w1, b1 = rng.standard_normal((4, 3)) * 0.1, np.full(3, 40.0)
    w2, b2 = rng.standard_normal((3, 2)), rng.standard_normal(2)
    got = O.score_mlp(h, w1, b1, w2, b2)
    ref = O.score_linear(h, w1 @ w2, b1 @ w2 + b2)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_planted_mlp_mistakes_are_caught():
    rng = np.random.default_rng(81)
    h = rng.standard_normal((1, 8, 6))
    w1, b1 = rng.standard_normal((6, 5)), rng.standard_normal(5)
    w2 = rng.standard_normal((5, 2))
    ref = O.score_mlp(h, w1, b1, w2)
    z = np.einsum("utj,jm->utm", h, w1) + b1
    tanh_gelu = 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))
    relu = np.maximum(z, 0)
    no_bias = O.gelu(np.einsum("utj,jm->utm", h, w1))
    for bad in (tanh_gelu, relu, no_bias):
        out = np.einsum("utm,mg->ugt", bad, w2)
        assert np.abs(out - ref).max() > 1e-5


# -------------------------------------------------- KVzip+ ([KVzap] §2.1)
def test_value_norms_against_an_explicit_projection():
    rng = np.random.default_rng(82)
    U, Hkv, G, T, d, Dm = 1, 2, 2, 7, 4, 6
    v = rng.standard_normal((U, Hkv, T, d))
    WO = rng.standard_normal((Hkv * G, Dm, d))                 # per-head slices of W_O
    gram = np.einsum("hmd,hme->hde", WO, WO)
    got = O.value_norms(v, gram, G)
    for h in range(Hkv * G):
        for t in range(T):
            assert abs(got[0, h, t] - np.linalg.norm(WO[h] @ v[0, h // G, t])) < 1e-12


def test_kvzip_plus_brute_force_and_reductions():
    q, k = rng_arrays(83, (1, 4, 3, 5), (1, 2, 9, 5))
    v = np.random.default_rng(84).standard_normal((1, 2, 9, 5))
    WO = np.random.default_rng(85).standard_normal((4, 7, 5))
    gram = np.einsum("hmd,hme->hde", WO, WO)
    hn = np.array([[2.0, 0.5, 3.0]])
    got = O.score_kvzip_plus(q, k, v, gram, hn, 0.6)
    G, W, T = 2, 3, 9
    for g in range(2):
        for t in range(T):
            best = 0.0
            for i in range(G):
                h = g * G + i
                for w in range(W):
                    if t > T - W + w:
                        continue
                    logits = [0.6 * float(q[0, h, w] @ k[0, g, tt]) for tt in range(T - W + w + 1)]
                    mx = max(logits)
                    den = sum(math.exp(x - mx) for x in logits)
                    a = math.exp(logits[t] - mx) / den
                    best = max(best, a * np.linalg.norm(WO[h] @ v[0, g, t]) / hn[0, w])
            assert abs(got[0, g, t] - best) < 1e-12
    # unit hidden norms and identity Grams on unit-norm values: the KVzip score
    vu = v / np.linalg.norm(v, axis=-1, keepdims=True)
    eye = np.broadcast_to(np.eye(5), (4, 5, 5))
    np.testing.assert_allclose(O.score_kvzip_plus(q, k, vu, eye, np.ones((1, 3)), 0.6),
                               O.score_attn(q, k, 0.6, aggregation="max"), rtol=1e-12)


def test_planted_kvzip_plus_mistakes_are_caught():
    q, k = rng_arrays(86, (1, 4, 3, 5), (1, 2, 9, 5))
    v = np.random.default_rng(87).standard_normal((1, 2, 9, 5))
    WO = np.random.default_rng(88).standard_normal((4, 7, 5))
    gram = np.einsum("hmd,hme->hde", WO, WO)
    hn = np.array([[2.0, 0.5, 3.0]])
    ref = O.score_kvzip_plus(q, k, v, gram, hn, 0.6)
    # the printed division (contribution in the denominator) ranks differently
    vn = O.value_norms(v, gram, 2)
    div = np.zeros_like(ref)
    for g in range(2):
        for i in range(2):
            h = g * 2 + i
            p = O.score_attn(q[:, h:h + 1], k[:, g:g + 1], 0.6, aggregation="max")
            div[0, g] = np.maximum(div[0, g], p[0, 0] / vn[0, h])
    assert not np.allclose(div, ref)
    # one head's Gram for the whole group
    gram_bad = gram.copy()
    gram_bad[1] = gram[0]
    assert not np.allclose(O.score_kvzip_plus(q, k, v, gram_bad, hn, 0.6), ref)
