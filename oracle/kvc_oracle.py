"""CPU oracle for the score -> select -> compact -> decode path (test infrastructure).

This file is test infrastructure.  Only the test-suite, the package smoke
check and the benchmark's CPU-baseline leg may import it; the library's
product path never does.  It shares no code with the CUDA implementation:
plain numpy, float64 arithmetic, one obvious loop per definition, no blocking,
fusion or reordering beyond what each definition states.

Sources (web pages on KV-cache compression; cited by title and section):

* [Sculpt]  "KVSculpt: KV Cache Compression as Distillation"
            §1 (eviction keeps a subset chosen by attention scores),
            §2A (retention zone of the m most recent pairs),
            §2B (loss with the log-sum-exp l of the attention scores),
            §2D (budgets that differ per layer and per KV head).
* [VECTOR]  "A Simple Plug-in for Improving Eviction-Based KV Cache
            Compression", "Énoncé du Problème" (importance eviction: score
            tokens, drop the low-score entries) and "Méthodologie : VECTOR"
            (three-way routing: keys kept, values kept / rebuilt by an OLS
            predictor from the key / evicted).
* [KVTC]    "KV Cache Transform Coding for Compact Storage in LLM Inference" §2A
            (attention sinks and the recent sliding window are kept as is).
* [KVzap]   "KVzap: Fast, Adaptive, and Faithful KV Cache Pruning"
            §1 (the T axis is the one left to compress; GQA on the H axis),
            §2.1 (scores built from the attention weight a token receives),
            §2.2 (linear surrogate h_t in R^{D_h} -> one score per KV head),
            §2.3 (drop tokens whose score is below tau; keep the w most recent).

Readings taken where the pages are silent (each is listed with its reason in
the design notes of the repository):

* attention-mass score = sum over the window rows of the row-softmax weight
  a token receives (sum, not max); causal mask inside the window (window row
  w sits at position T - W + w); no pooling or smoothing;
* GQA: query head h belongs to kv head floor(h / G);
* budget B = floor(keep_ratio * (Hkv * T)) in IEEE double, protected tokens
  counted inside B, and when the protected set alone exceeds B only the
  protected set is kept;
* one pool per unit across its kv heads; order (score desc, token asc,
  head asc), -0 == +0, NaN ranks below everything;
* threshold rule: keep iff score >= tau (NaN never kept);
* decode fidelity: KL(p_comp || p_full) = lse_full - lse_comp, the rel-L2
  output error ||o_comp - o_full|| / ||o_full||.

Parity pins: every function below is checked in ``tests/test_oracle_pins.py``
against brute force on tiny inputs, closed forms, invariants and independent
library routines; none of them is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------- scoring
def score_attn(q_win, k, scale, head_scale=None, causal=True, aggregation="sum"):
    """Attention-based score of every cached token, per (unit, kv head).

    q_win [U, Hq, W, d], k [U, Hkv, T, d] (any float dtype; computed in
    float64).  For query head h of kv head g = h // G and window row w:
        s[(h,w), t] = scale * f[u,h] * <q[u,h,w], k[u,g,t]>,  t <= T-W+w if causal
        p[(h,w), :] = softmax_t(s[(h,w), :])
    aggregation "sum" (attention mass):
        score[u,g,t] = sum_{h in g} sum_w p[(h,w), t]
    aggregation "max" (the largest attention weight the token receives from
    any window row of the group, the KVzip score of [KVzap] §2.1 without its
    KVzip+ normalisation):
        score[u,g,t] = max_{h in g, w} p[(h,w), t]
    The log-sum-exp lse = m + log(sum exp(s - m)) is the row normaliser
    ([Sculpt] §2B); [VECTOR] "Énoncé du Problème" and [Sculpt] §1 rank tokens
    by the attention they receive.  Returns float64 [U, Hkv, T].
    """
    if aggregation not in ("sum", "max"):
        raise ValueError(aggregation)
    q = np.asarray(q_win, dtype=F64)
    kk = np.asarray(k, dtype=F64)
    U, Hq, W, d = q.shape
    _, Hkv, T, _ = kk.shape
    G = Hq // Hkv
    hs = None if head_scale is None else np.asarray(head_scale, dtype=F64)
    out = np.zeros((U, Hkv, T), dtype=F64)
    for u in range(U):
        for g in range(Hkv):
            for i in range(G):
                h = g * G + i
                c = scale * (1.0 if hs is None else hs[u, h])
                logits = c * (q[u, h] @ kk[u, g].T)             # [W, T]
                if causal:
                    for w in range(W):
                        logits[w, T - W + w + 1:] = -np.inf
                m = logits.max(axis=1, keepdims=True)
                lse = m + np.log(np.exp(logits - m).sum(axis=1, keepdims=True))
                p = np.exp(logits - lse)
                if aggregation == "sum":
                    out[u, g] += p.sum(axis=0)
                else:
                    out[u, g] = np.maximum(out[u, g], p.max(axis=0))
    return out


def value_norms(v, gram, G):
    """||W_O^h v_t|| for every query head h and token t, from the Gram
    matrices gram[h] = W_O^h^T W_O^h (d x d) of the output projection's
    per-head slices: sqrt(v^T gram[h] v).  v [U, Hkv, T, d], gram [Hq, d, d],
    query head h reads kv head h // G.  Returns float64 [U, Hq, T]."""
    vv = np.asarray(v, dtype=F64)
    M = np.asarray(gram, dtype=F64)
    U, Hkv, T, d = vv.shape
    out = np.zeros((U, Hkv * G, T), dtype=F64)
    for u in range(U):
        for h in range(Hkv * G):
            x = vv[u, h // G]                                   # [T, d]
            out[u, h] = np.sqrt(np.maximum(np.einsum("td,de,te->t", x, M[h], x), 0.0))
    return out


def score_kvzip_plus(q_win, k, v, gram, hnorm, scale, head_scale=None, causal=True):
    """KVzip+ score ([KVzap] §2.1): the largest attention weight a token
    receives from the window rows, each weighted by the size of the token's
    value contribution to the residual stream relative to the row's hidden
    state.  The printed formula divides a_ji by ||W_O v_i|| / ||h_j||; the
    text (and the normalisation it cites) weights by the contribution, so
    this reads it as
        s+[u,g,t] = max_{h in g, w} p[(h,w), t] * ||W_O^h v_t|| / ||h_w||
    with p the row softmax of score_attn, ||W_O^h v_t|| from value_norms and
    hnorm [U, W] the hidden-state norms of the window positions.
    Returns float64 [U, Hkv, T]."""
    q = np.asarray(q_win, dtype=F64)
    kk = np.asarray(k, dtype=F64)
    U, Hq, W, d = q.shape
    _, Hkv, T, _ = kk.shape
    G = Hq // Hkv
    vn = value_norms(v, gram, G)
    hn = np.asarray(hnorm, dtype=F64)
    hs = None if head_scale is None else np.asarray(head_scale, dtype=F64)
    out = np.zeros((U, Hkv, T), dtype=F64)
    for u in range(U):
        for g in range(Hkv):
            for i in range(G):
                h = g * G + i
                c = scale * (1.0 if hs is None else hs[u, h])
                logits = c * (q[u, h] @ kk[u, g].T)             # [W, T]
                if causal:
                    for w in range(W):
                        logits[w, T - W + w + 1:] = -np.inf
                m = logits.max(axis=1, keepdims=True)
                lse = m + np.log(np.exp(logits - m).sum(axis=1, keepdims=True))
                p = np.exp(logits - lse) / hn[u][:, None]        # a_wt / ||h_w||
                out[u, g] = np.maximum(out[u, g], p.max(axis=0) * vn[u, h])
    return out


def score_linear(hidden, weight, bias=None):
    """Linear surrogate score ([KVzap] §2.2): score[u,g,t] = b_g + h[u,t,:] . W[:,g].

    hidden [U, T, Dh], weight [Dh, Hkv], bias [Hkv] or None.  The raw linear
    output is the score compared with tau (the pages' surrogate predicts a
    log-score; the threshold is applied to that prediction).
    Returns float64 [U, Hkv, T].
    """
    h = np.asarray(hidden, dtype=F64)
    wt = np.asarray(weight, dtype=F64)
    out = np.einsum("utj,jg->ugt", h, wt)
    if bias is not None:
        out = out + np.asarray(bias, dtype=F64)[None, :, None]
    return out


def gelu(z):
    """GELU(z) = z * Phi(z) = z (1 + erf(z / sqrt 2)) / 2 (the exact form)."""
    from scipy.special import erf
    z = np.asarray(z, dtype=F64)
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def score_mlp(hidden, w1, b1, w2, b2=None):
    """Two-layer surrogate score ([KVzap] §2.2, the MLP variant: hidden width
    D_h / 8 with a GELU): for every token t of unit u and kv head g
        z_m = b1_m + sum_j hidden[u,t,j] * w1[j,m]
        score[u,g,t] = b2_g + sum_m GELU(z_m) * w2[m,g]
    hidden [U, T, Dh], w1 [Dh, Dm], b1 [Dm] or None, w2 [Dm, Hkv], b2 [Hkv] or
    None.  As for the linear surrogate, the raw output is compared with tau.
    Returns float64 [U, Hkv, T]."""
    h = np.asarray(hidden, dtype=F64)
    z = np.einsum("utj,jm->utm", h, np.asarray(w1, dtype=F64))
    if b1 is not None:
        z = z + np.asarray(b1, dtype=F64)
    out = np.einsum("utm,mg->ugt", gelu(z), np.asarray(w2, dtype=F64))
    if b2 is not None:
        out = out + np.asarray(b2, dtype=F64)[None, :, None]
    return out


# -------------------------------------------------------------- selection
def protected_mask(T, n_sink, n_recent):
    """Tokens that are always kept: the first n_sink (attention sinks,
    [KVTC] §2A) and the last n_recent (sliding window, [KVzap] §2.3 and the
    retention zone of [Sculpt] §2A)."""
    t = np.arange(T)
    return (t < n_sink) | (t >= T - n_recent)


def global_budget(keep_ratio, Hkv, T):
    """B = floor(keep_ratio * (Hkv*T)) with one IEEE-double rounding."""
    return int(math.floor(float(keep_ratio) * float(Hkv * T)))


def _order_key(scores_f32, t_idx, g_idx):
    """Sort keys for (score desc, token asc, head asc) with NaN last and
    -0 == +0, suitable for np.lexsort (last key is primary)."""
    s = scores_f32.astype(F64)
    isnan = np.isnan(s)
    neg = np.where(isnan, 0.0, -s) + 0.0      # + 0.0 turns -0.0 into +0.0
    return (g_idx, t_idx, neg, isnan)


def select(scores, mode, keep_ratio=0.0, tau=0.0, head_budget=None,
           n_sink=0, n_recent=0):
    """Budget selection over fp32 scores [U, Hkv, T].

    mode "global": per unit, keep the protected set of every head, then fill
    B_eff - Hkv*|P| slots with the highest non-protected (g, t) across heads
    ([KVzap] §2.3 fixed budget; [Sculpt] §2D budgets that differ per head).
    mode "per_head": the same inside each head with budget head_budget[i].
    mode "threshold": keep t iff score >= tau or t protected ([KVzap] §2.3).

    Returns (kept_idx int32 [U*Hkv, T] padded with -1, counts int32 [U*Hkv],
    offsets int64 [U*Hkv + 1]); indices of each head are ascending.
    """
    s = np.asarray(scores, dtype=np.float32)
    U, Hkv, T = s.shape
    n = U * Hkv
    P = protected_mask(T, n_sink, n_recent)
    nP = int(P.sum())
    free_t = np.nonzero(~P)[0]
    kept = np.full((n, T), -1, dtype=np.int32)
    counts = np.zeros(n, dtype=np.int32)

    def emit(i, mask_t):
        idx = np.nonzero(mask_t)[0].astype(np.int32)
        kept[i, : idx.size] = idx
        counts[i] = idx.size

    if mode == "threshold":
        for u in range(U):
            for g in range(Hkv):
                emit(u * Hkv + g, P | (s[u, g] >= np.float32(tau)))
    elif mode == "global":
        B = global_budget(keep_ratio, Hkv, T)
        B_eff = min(max(B, Hkv * nP), Hkv * T)
        need = B_eff - Hkv * nP
        for u in range(U):
            tt, gg = np.meshgrid(free_t, np.arange(Hkv), indexing="ij")
            tt, gg = tt.ravel(), gg.ravel()
            order = np.lexsort(_order_key(s[u, gg, tt], tt, gg))
            take = order[:need]
            chosen = np.zeros((Hkv, T), dtype=bool)
            chosen[gg[take], tt[take]] = True
            for g in range(Hkv):
                emit(u * Hkv + g, P | chosen[g])
    elif mode == "per_head":
        hb = np.asarray(head_budget, dtype=np.int64).reshape(n)
        for u in range(U):
            for g in range(Hkv):
                i = u * Hkv + g
                B_eff = min(max(int(hb[i]), nP), T)
                need = B_eff - nP
                zeros = np.zeros(free_t.size, dtype=np.int64)
                order = np.lexsort(_order_key(s[u, g, free_t], free_t, zeros))
                chosen = np.zeros(T, dtype=bool)
                chosen[free_t[order[:need]]] = True
                emit(i, P | chosen)
    else:
        raise ValueError(mode)
    offsets = np.zeros(n + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts.astype(np.int64))
    return kept, counts, offsets


# ------------------------------------------------------------- compaction
def compact(k, v, kept_idx, counts, offsets, slack=0):
    """Gather the kept rows into one variable-length cache.

    Head i = u*Hkv + g owns rows [start_i, start_i + counts_i + slack) with
    start_i = offsets_i + i*slack; row start_i + j is K[u, g, kept_idx[i, j]]
    (same for V).  Slack rows are left zero.  Byte-exact copy.
    Returns (kc, vc, start int64 [n], length int32 [n]).
    """
    k = np.asarray(k)
    v = np.asarray(v)
    U, Hkv, T, d = k.shape
    n = U * Hkv
    total = int(offsets[n]) + n * slack
    kc = np.zeros((total, d), dtype=k.dtype)
    vc = np.zeros((total, d), dtype=v.dtype)
    start = np.zeros(n, dtype=np.int64)
    for i in range(n):
        u, g = divmod(i, Hkv)
        start[i] = int(offsets[i]) + i * slack
        for j in range(int(counts[i])):
            kc[start[i] + j] = k[u, g, kept_idx[i, j]]
            vc[start[i] + j] = v[u, g, kept_idx[i, j]]
    return kc, vc, start, np.asarray(counts, dtype=np.int32).copy()


# ----------------------------------------------------------------- decode
def decode_attn(q, kc, vc, start, length, k_new=None, v_new=None, scale=1.0):
    """One decode step over a variable-length cache (GQA).

    If k_new/v_new [U, Hkv, d] are given they are first appended at row
    start_i + length_i and length_i grows by one (the caller reserved the
    slack).  Then for query head h of kv head g:
        s_j = scale * <q[u,h], kc[start+j]>, j < length
        lse = log sum_j exp(s_j),  o = sum_j exp(s_j - lse) * vc[start+j]
    The lse is the log-sum-exp of [Sculpt] §2B.  Works on copies; returns
    (out float64 [U, Hq, d], lse float64 [U, Hq], kc, vc, length).
    """
    qq = np.asarray(q, dtype=F64)
    kc = np.array(kc, copy=True)
    vc = np.array(vc, copy=True)
    length = np.array(length, dtype=np.int64, copy=True)
    U, Hq, d = qq.shape
    Hkv = length.size // U
    G = Hq // Hkv
    out = np.zeros((U, Hq, d), dtype=F64)
    lse = np.zeros((U, Hq), dtype=F64)
    for u in range(U):
        for g in range(Hkv):
            i = u * Hkv + g
            s0 = int(start[i])
            if k_new is not None:
                kc[s0 + length[i]] = np.asarray(k_new)[u, g]
                vc[s0 + length[i]] = np.asarray(v_new)[u, g]
                length[i] += 1
            L = int(length[i])
            K = kc[s0: s0 + L].astype(F64)
            V = vc[s0: s0 + L].astype(F64)
            for j in range(G):
                h = g * G + j
                if L == 0:
                    lse[u, h] = -np.inf
                    continue
                logits = scale * (K @ qq[u, h])
                m = logits.max()
                e = np.exp(logits - m)
                l = e.sum()
                lse[u, h] = m + math.log(l)
                out[u, h] = (e / l) @ V
    return out, lse, kc, vc, length.astype(np.int32)


# ---------------------------------------------------- decode-time pruning
def gather_scores(scores, kept_idx, counts, start, rows):
    """Per-row scores of a compacted cache: the score of the token each row
    holds, rscore[start_i + j] = scores[u, g, kept_idx[i, j]] for j < counts_i
    (i = u*Hkv + g).  Rows outside the heads' kept ranges are NaN.
    Returns float32 [rows]."""
    sc = np.asarray(scores, dtype=np.float32)
    U, Hkv, T = sc.shape
    rscore = np.full(int(rows), np.nan, dtype=np.float32)
    for i in range(U * Hkv):
        u, g = divmod(i, Hkv)
        for j in range(int(counts[i])):
            rscore[int(start[i]) + j] = sc[u, g, kept_idx[i, j]]
    return rscore


def decode_prune(pools, rscore, start, length, s_new, tau, window, n_sink=0):
    """Decode-time threshold pruning ([KVzap] §2.3: the `window` most recent
    tokens are always kept, a token whose score is below tau is dropped, and
    the pruning runs after attention, in decoding as in prefilling).

    Runs after a decode step appended one token per head (its row is
    start_i + length_i - 1, length_i already counting it).  Rows of a head
    are in token order; rows [0, length_i - window) have been judged, the
    last `window` rows are the window.  Per head i:
      1. rscore[start_i + length_i - 1] = s_new[i]   (the new token's score);
      2. e = length_i - window - 1 is the row of the token that just left the
         window; if e >= n_sink (sinks are never dropped) and the token's
         score is not >= tau (compared in float32; NaN is dropped), the rows
         e+1 .. length_i-1 of every pool and of rscore move down by one and
         length_i shrinks by one.
    pools: list of arrays indexed by pool row (K and V rows, or their codes
    and group parameters).  Works on copies; rows at or beyond the new
    length are unspecified.  Returns (pools, rscore, length int32, dropped
    bool [n])."""
    pools = [np.array(p, copy=True) for p in pools]
    rs = np.array(rscore, dtype=np.float32, copy=True)
    length = np.array(length, dtype=np.int64, copy=True)
    n = length.size
    dropped = np.zeros(n, dtype=bool)
    tau32 = np.float32(tau)
    for i in range(n):
        s0, L = int(start[i]), int(length[i])
        if L < 1:
            continue
        rs[s0 + L - 1] = np.float32(s_new[i])
        e = L - window - 1
        if e < n_sink or rs[s0 + e] >= tau32:
            continue
        for p in pools:
            p[s0 + e: s0 + L - 1] = p[s0 + e + 1: s0 + L].copy()
        rs[s0 + e: s0 + L - 1] = rs[s0 + e + 1: s0 + L].copy()
        length[i] = L - 1
        dropped[i] = True
    return pools, rs, length.astype(np.int32), dropped


QGROUP = 32     # elements per quantisation group (one row, consecutive along d)


def quantize_rows(x):
    """Group quantisation of cache rows ([KVTC] §2B: coefficients are
    quantised in groups that share a scale and an offset, after the
    Microscaling formats; here applied to the cached K/V rows themselves).

    x [rows, d] with float32-representable values inside the float16 range,
    d a multiple of 32.  For every row and group of 32 consecutive elements,
    in float32 arithmetic (the integer codes are decided in the precision the
    kernel decides them in):
        lo    = fp16(min(group))                      round to nearest even
        scale = fp16((max(group) - lo) / 255)         difference and quotient in fp32
        code  = clamp(rint((x - lo) / scale), 0, 255)  0 for the whole group if scale == 0
    Returns (codes uint8 [rows, d], params float16 [rows, d/32, 2] = (scale, lo)).
    """
    xf = np.asarray(x, dtype=np.float32)
    rows, d = xf.shape
    g = xf.reshape(rows, d // QGROUP, QGROUP)
    lo = g.min(axis=-1).astype(np.float16)
    lo32 = lo.astype(np.float32)
    scale = ((g.max(axis=-1) - lo32) / np.float32(255.0)).astype(np.float16)
    sc32 = scale.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (g - lo32[..., None]) / sc32[..., None]
    codes = np.clip(np.rint(v), 0, 255)
    codes = np.where(sc32[..., None] == 0, 0, codes).astype(np.uint8)
    params = np.stack([scale, lo], axis=-1)
    return codes.reshape(rows, d), params


def dequantize_rows(codes, params):
    """x' = code * scale + lo per group (float64; the product of an 8-bit
    code and a float16 is exact).  Returns float64 [rows, d]."""
    c = np.asarray(codes, dtype=F64)
    rows, d = c.shape
    p = np.asarray(params, dtype=F64)
    return (c.reshape(rows, d // QGROUP, QGROUP) * p[..., 0:1] + p[..., 1:2]).reshape(rows, d)


# ------------------------------------------- VECTOR three-way routing
# [VECTOR] "Méthodologie : VECTOR": keys are kept exactly for every token of
# the candidate pool; values are retained, approximated (dropped and rebuilt
# as W_OLS k from the stored key) or evicted.  Step 1 widens the base
# eviction's pool to 1 - p_c + p_a; step 2 scores each pool token by its
# reconstruction error eps = ||v - W_OLS k||^2; step 3 drops the values of
# the 2 p_a lowest-error tokens and keeps K and V of the rest.  Synthetic
# caches carry no rotary encoding, so the inverse rotation before the
# reconstruction is the identity here.

def fit_ols(k_cal, v_cal):
    """Offline OLS calibration of the K -> V predictor, one matrix per kv
    head: W = argmin_W sum_t ||v_t - W k_t||^2 = (sum_t v_t k_t^T)
    (sum_t k_t k_t^T)^-1 (normal equations).  k_cal, v_cal [Hkv, N, d] with
    N >= d.  Returns float64 [Hkv, d, d] (row = output dimension)."""
    kc = np.asarray(k_cal, dtype=F64)
    vc = np.asarray(v_cal, dtype=F64)
    Hkv, N, d = kc.shape
    W = np.zeros((Hkv, d, d), dtype=F64)
    for g in range(Hkv):
        gram = kc[g].T @ kc[g]             # sum_t k_t k_t^T
        cross = vc[g].T @ kc[g]            # sum_t v_t k_t^T
        W[g] = np.linalg.solve(gram.T, cross.T).T
    return W


def vector_budgets(p_c, p_a, Hkv, T, n_sink, n_recent):
    """Integer budgets of one unit: the pool B_pool = floor((1 - p_c + p_a)
    Hkv T) (raised to the protected set, as in global selection) and the
    approximated count A = floor(2 p_a Hkv T), capped at the pool's
    non-protected tokens (protected tokens keep exact values).  Returns
    (pool keep ratio, B_pool_eff, A)."""
    nP = int(protected_mask(T, n_sink, n_recent).sum())
    ratio = (1.0 - float(p_c)) + float(p_a)
    B = global_budget(ratio, Hkv, T)
    B_eff = min(max(B, Hkv * nP), Hkv * T)
    A = min(global_budget(2.0 * float(p_a), Hkv, T), B_eff - Hkv * nP)
    return ratio, B_eff, A


def vector_residual(k, v, W, kept_idx, counts, n_sink, n_recent):
    """Step 2: reconstruction error of every pool token, as a selection key
    per pool position.  For head i = u*Hkv + g and pool position j < counts_i
    holding token t = kept_idx[i, j]:
        eps = sum_x (v[u,g,t,x] - sum_y W[g,x,y] k[u,g,t,y])^2
    key[u, g, j] = -eps (float32) for tokens that may be approximated; NaN for
    protected tokens (sinks, recent window: their values stay exact) and for
    positions j >= counts_i.  Returns float32 [U, Hkv, T]."""
    kk = np.asarray(k, dtype=F64)
    vv = np.asarray(v, dtype=F64)
    Wm = np.asarray(W, dtype=F64)
    U, Hkv, T, d = kk.shape
    P = protected_mask(T, n_sink, n_recent)
    key = np.full((U, Hkv, T), np.nan, dtype=np.float32)
    for u in range(U):
        for g in range(Hkv):
            i = u * Hkv + g
            for j in range(int(counts[i])):
                t = int(kept_idx[i, j])
                if P[t]:
                    continue
                r = vv[u, g, t] - Wm[g] @ kk[u, g, t]
                key[u, g, j] = np.float32(-(r @ r))
    return key


def vector_approx(key, A):
    """Step 3's choice, per unit: the A pool positions with the lowest
    error, i.e. the highest key, ranked across the unit's heads by (key desc,
    position asc, head asc); NaN keys are never chosen.  Returns (approx_pos
    int32 [U*Hkv, T] padded with -1, ascending per head; counts int32)."""
    kf = np.asarray(key, dtype=np.float32)
    U, Hkv, T = kf.shape
    pos = np.full((U * Hkv, T), -1, dtype=np.int32)
    cnt = np.zeros(U * Hkv, dtype=np.int32)
    for u in range(U):
        cand = [(-float(kf[u, g, j]), j, g) for g in range(Hkv) for j in range(T)
                if not np.isnan(kf[u, g, j])]
        cand.sort()
        chosen = [[] for _ in range(Hkv)]
        for _, j, g in cand[:A]:
            chosen[g].append(j)
        for g in range(Hkv):
            js = sorted(chosen[g])
            pos[u * Hkv + g, :len(js)] = js
            cnt[u * Hkv + g] = len(js)
    return pos, cnt


def vector_compact(k, v, kept_idx, counts, approx_pos, approx_counts, slack=0):
    """Step 3's asymmetric truncation as a cache layout.  Head i keeps the K
    rows of all counts_i pool tokens, the approximated ones first:
      kc rows [kstart_i, kstart_i + counts_i + slack): the napprox_i tokens
        at the chosen pool positions (ascending), then the exact tokens
        (ascending);
      vc rows [vstart_i, vstart_i + nexact_i + slack): the exact tokens' V.
    kstart_i = sum_{h<i} (counts_h + slack), vstart_i = sum_{h<i} (nexact_h +
    slack).  Byte-exact copies.  Returns (kc, vc, kstart int64, klen int32,
    vstart int64, napprox int32)."""
    k = np.asarray(k)
    v = np.asarray(v)
    U, Hkv, T, d = k.shape
    n = U * Hkv
    napprox = np.asarray(approx_counts, dtype=np.int32).copy()
    nexact = np.asarray(counts, dtype=np.int64) - napprox
    kstart = np.zeros(n, dtype=np.int64)
    vstart = np.zeros(n, dtype=np.int64)
    for i in range(1, n):
        kstart[i] = kstart[i - 1] + int(counts[i - 1]) + slack
        vstart[i] = vstart[i - 1] + int(nexact[i - 1]) + slack
    kc = np.zeros((int(kstart[-1] + counts[n - 1] + slack) if n else 0, d), dtype=k.dtype)
    vc = np.zeros((int(vstart[-1] + nexact[n - 1] + slack) if n else 0, d), dtype=v.dtype)
    for i in range(n):
        u, g = divmod(i, Hkv)
        apos = set(int(j) for j in approx_pos[i, :napprox[i]])
        approx_t = [int(kept_idx[i, j]) for j in range(int(counts[i])) if j in apos]
        exact_t = [int(kept_idx[i, j]) for j in range(int(counts[i])) if j not in apos]
        for r, t in enumerate(approx_t + exact_t):
            kc[kstart[i] + r] = k[u, g, t]
        for r, t in enumerate(exact_t):
            vc[vstart[i] + r] = v[u, g, t]
    return kc, vc, kstart, np.asarray(counts, dtype=np.int32).copy(), vstart, napprox


def decode_attn_vector(q, kc, vc, kstart, klen, vstart, napprox, W, k_new=None, v_new=None,
                       scale=1.0):
    """One decode step over a VECTOR cache.  Head i = u*Hkv + g holds klen_i
    keys at kc[kstart_i:]; the value of row j is the reconstruction
    W[g] @ kc[kstart_i + j] for j < napprox_i and vc[vstart_i + j - napprox_i]
    otherwise.  k_new / v_new [U, Hkv, d], if given, are appended as an exact
    row (kc row kstart_i + klen_i, vc row vstart_i + klen_i - napprox_i) and
    klen_i grows by one.  Then, as in decode_attn, lse = log sum_j exp(s_j),
    o = sum_j softmax_j * value_j with s_j = scale <q, k_j>.  Works on copies;
    returns (out float64 [U, Hq, d], lse float64 [U, Hq], kc, vc, klen)."""
    qq = np.asarray(q, dtype=F64)
    Wm = np.asarray(W, dtype=F64)
    kc = np.array(kc, copy=True)
    vc = np.array(vc, copy=True)
    klen = np.array(klen, dtype=np.int64, copy=True)
    U, Hq, d = qq.shape
    Hkv = klen.size // U
    G = Hq // Hkv
    out = np.zeros((U, Hq, d), dtype=F64)
    lse = np.zeros((U, Hq), dtype=F64)
    for u in range(U):
        for g in range(Hkv):
            i = u * Hkv + g
            ks, vs, na = int(kstart[i]), int(vstart[i]), int(napprox[i])
            if k_new is not None:
                kc[ks + klen[i]] = np.asarray(k_new)[u, g]
                vc[vs + klen[i] - na] = np.asarray(v_new)[u, g]
                klen[i] += 1
            L = int(klen[i])
            K = kc[ks: ks + L].astype(F64)
            V = np.concatenate([K[:na] @ Wm[g].T, vc[vs: vs + L - na].astype(F64)])
            for j in range(G):
                h = g * G + j
                if L == 0:
                    lse[u, h] = -np.inf
                    continue
                logits = scale * (K @ qq[u, h])
                m = logits.max()
                e = np.exp(logits - m)
                l = e.sum()
                lse[u, h] = m + math.log(l)
                out[u, h] = (e / l) @ V
    return out, lse, kc, vc, klen.astype(np.int32)


def fidelity(out_comp, out_full, lse_comp, lse_full):
    """Fidelity probe of a compressed cache against the full one.

    rel_err[u,h] = ||o_comp - o_full||_2 / ||o_full||_2 and
    kl[u,h] = KL(p_comp || p_full) = lse_full - lse_comp, which equals
    -log(attention mass the full distribution puts on the kept rows) >= 0.
    Returns float64 arrays (rel_err, kl) of shape [U, Hq].
    """
    oc = np.asarray(out_comp, dtype=F64)
    of = np.asarray(out_full, dtype=F64)
    num = np.sqrt(((oc - of) ** 2).sum(axis=-1))
    den = np.sqrt((of ** 2).sum(axis=-1))
    rel = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    kl = np.asarray(lse_full, dtype=F64) - np.asarray(lse_comp, dtype=F64)
    return rel, kl
