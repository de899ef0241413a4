"""GPU selection and compaction, bit-exact against the oracle on the oracle's
fp32 scores (through the C ABI).

Covers global top-k across heads, per-head budgets and the threshold rule;
ties, -0/+0, +-inf and NaN; protected sinks / recent windows that overlap or
swallow the whole budget; one-token and ragged pools; and the full-size
workloads (32k single layer, 32-layer x batch-4 cache, 128k threshold).
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_compression_attention_b300 import inputs
from oracle import kvc_oracle as O
from tests.kvc_testutil import np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kv_cache_compression_attention_b300 import binding
    binding.lib()
    return binding


def gpu_select(B, scores, mode, **kw):
    U, Hkv, T = scores.shape
    kept = torch.full((U * Hkv, T), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((U * Hkv,), -7, dtype=torch.int32, device="cuda")
    offs = torch.full((U * Hkv + 1,), -7, dtype=torch.int64, device="cuda")
    hb = kw.pop("head_budget", None)
    if hb is not None:
        hb = torch.as_tensor(np.asarray(hb), dtype=torch.int32).cuda()
    B.kvc_select(scores, mode, kept, counts, offs, head_budget=hb, **kw)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    return kept.cpu().numpy(), counts.cpu().numpy(), offs.cpu().numpy()


def check_same(got, ref):
    kept, counts, offs = got
    rk, rc, ro = ref
    np.testing.assert_array_equal(counts, rc)
    np.testing.assert_array_equal(offs, ro)
    for i in range(len(rc)):
        np.testing.assert_array_equal(kept[i, : rc[i]], rk[i, : rc[i]])


@pytest.mark.parametrize("shape", [(1, 4, 1024), (2, 8, 5000), (3, 2, 1), (1, 1, 3), (2, 5, 40001)])
@pytest.mark.parametrize("ties,specials", [(False, False), (True, False), (True, True)])
def test_select_global_small(B, shape, ties, specials):
    s = inputs.random_scores(shape, seed=sum(shape), ties=ties, specials=specials)
    sc = s.numpy()
    for ratio, ns, nr in [(0.25, 4, 32), (0.1, 0, 0), (0.0, 2, 2), (1.0, 4, 4), (0.5, 3000, 3000)]:
        got = gpu_select(B, s.cuda(), "global", keep_ratio=ratio, n_sink=ns, n_recent=nr)
        ref = O.select(sc, "global", keep_ratio=ratio, n_sink=ns, n_recent=nr)
        check_same(got, ref)


def test_select_global_budget_rounds_once_in_double(B):
    """The library's budget is floor(ratio * Hkv * T) with the product
    rounded once in double, as the oracle's: 0.29 of 100 keys is
    28.999999999999996 there, so 28 keys are kept, not 29 (and 0.57 of them
    56.99999999999999: 56 kept)."""
    s = inputs.random_scores((2, 1, 100), seed=29)
    for ratio, want in [(0.29, 28), (0.57, 56), (0.1, 10)]:
        got = gpu_select(B, s.cuda(), "global", keep_ratio=ratio)
        assert (got[1] == want).all()
        check_same(got, O.select(s.numpy(), "global", keep_ratio=ratio))


@pytest.mark.parametrize("shape", [(2, 3, 777), (1, 8, 4096)])
def test_select_per_head_and_threshold_small(B, shape):
    s = inputs.random_scores(shape, seed=5, ties=True, specials=True)
    sc = s.numpy()
    U, Hkv, T = shape
    hb = np.random.default_rng(1).integers(-5, T + 5, size=U * Hkv)
    got = gpu_select(B, s.cuda(), "per_head", head_budget=hb, n_sink=2, n_recent=7)
    check_same(got, O.select(sc, "per_head", head_budget=hb, n_sink=2, n_recent=7))
    for tau in (0.5, -0.0, float("inf"), float("-inf"), float("nan")):
        got = gpu_select(B, s.cuda(), "threshold", tau=tau, n_sink=1, n_recent=3)
        check_same(got, O.select(sc, "threshold", tau=tau, n_sink=1, n_recent=3))


def test_select_all_equal_scores_ties_by_token_then_head(B):
    s = torch.zeros((1, 4, 1000))
    got = gpu_select(B, s.cuda(), "global", keep_ratio=0.3, n_sink=1, n_recent=1)
    check_same(got, O.select(s.numpy(), "global", keep_ratio=0.3, n_sink=1, n_recent=1))


@pytest.mark.parametrize("shape,mode", [
    ((1, 8, 40960), "global"),      # the largest shared-memory pools
    ((1, 8, 65536), "global"),      # 524 288 keys: the streaming kernel
    ((2, 32, 3000), "global"),      # more heads per pool than the registers hold
    ((1, 2, 400000), "per_head"),   # one head of 400 000 tokens
    ((1, 2, 400000), "threshold"),
])
def test_select_large_pools(B, shape, mode):
    """Pools whose keys do not fit one cluster's shared memory, or with more
    than 8 heads, take the streaming kernel: same result, bit for bit."""
    s = inputs.random_scores(shape, seed=sum(shape), ties=True, specials=True)
    sc = s.numpy()
    kw = dict(n_sink=4, n_recent=64)
    if mode == "global":
        kw["keep_ratio"] = 0.1
    elif mode == "per_head":
        kw["head_budget"] = np.array([1000, 250000] * shape[0])
    else:
        kw["tau"] = 1.0
    got = gpu_select(B, s.cuda(), mode, **kw)
    check_same(got, O.select(sc, mode, **kw))


@pytest.mark.parametrize("shape,kind", [
    ((1, 8, 16384), "equal"),        # every key equal: ranked by (token, head) alone
    ((1, 8, 32768), "levels"),       # six distinct values: large tie blocks
    ((1, 3, 70001), "specials"),     # NaN, +-inf, -0 / +0, ragged per-CTA ranges
    ((3, 8, 9000), "specials"),      # three pools in one launch
    ((9, 8, 8192), "random"),        # nine pools in one launch
])
def test_select_global_pools_ties_and_specials(B, shape, kind):
    """Global pools of 65 K - 262 K keys with tie blocks and special values,
    at budgets from nothing to everything, bit-exact against the oracle."""
    if kind == "equal":
        s = torch.full(shape, 0.25)
    elif kind == "levels":
        g = torch.Generator().manual_seed(3)
        s = torch.randint(0, 6, shape, generator=g).float() * 0.5
    else:
        s = inputs.random_scores(shape, seed=sum(shape), ties=kind != "random",
                                 specials=kind == "specials")
    sc = s.numpy()
    for ratio, ns, nr in [(0.1, 4, 64), (0.37, 0, 0), (0.0, 2, 2), (1.0, 1, 1),
                          (0.999, 3, 5)]:
        kw = dict(keep_ratio=ratio, n_sink=ns, n_recent=nr)
        check_same(gpu_select(B, s.cuda(), "global", **kw), O.select(sc, "global", **kw))


def test_select_cross_layer_pool(B):
    """One global budget over every layer and kv head of a sequence (32
    layers x 8 kv heads = 256 heads of 16 384 tokens, 4.2 M keys per pool,
    after KVSculpt's layer-and-head allocation), two sequences; the oracle
    checks one, the other is checked for the invariants."""
    U, H, T = 2, 256, 16384
    s = inputs.random_scores((U, H, T), seed=2026)
    got = gpu_select(B, s.cuda(), "global", keep_ratio=0.2, n_sink=4, n_recent=64)
    ref = O.select(s[:1].numpy(), "global", keep_ratio=0.2, n_sink=4, n_recent=64)
    kept, counts, offs = got
    check_same((kept[:H], counts[:H], offs[:H + 1]), ref)
    assert offs[-1] == U * math.floor(0.2 * H * T)
    assert len(set(counts[:H].tolist())) > 1          # heads keep different counts
    for i in range(H, 2 * H, 37):
        k = kept[i, : counts[i]]
        assert (np.diff(k) > 0).all() and k[:4].tolist() == [0, 1, 2, 3]


def test_select_llama32k_full(B):
    w = inputs.WORKLOADS["c2_llama32k"]
    q = inputs.window_queries(w, "cuda")
    k, _ = inputs.keys_values(w, q, "cuda")
    ref_scores = O.score_attn(np64(q), np64(k), w.scale).astype(np.float32)
    got = gpu_select(B, torch.from_numpy(ref_scores).cuda(), "global", keep_ratio=w.keep_ratio,
                     n_sink=w.n_sink, n_recent=w.n_recent)
    ref = O.select(ref_scores, "global", keep_ratio=w.keep_ratio, n_sink=w.n_sink,
                   n_recent=w.n_recent)
    check_same(got, ref)
    assert got[2][-1] == math.floor(0.10 * 8 * 32768)
    assert len(set(got[1].tolist())) > 1          # heads keep different counts


def test_select_32layer_full_units(B):
    w = inputs.WORKLOADS["c3_32layer"]
    s = inputs.random_scores((w.U, w.Hkv, w.T), seed=33)
    got = gpu_select(B, s.cuda(), "global", keep_ratio=w.keep_ratio, n_sink=w.n_sink,
                     n_recent=w.n_recent)
    ref = O.select(s.numpy(), "global", keep_ratio=w.keep_ratio, n_sink=w.n_sink,
                   n_recent=w.n_recent)
    check_same(got, ref)


def test_select_threshold_qwen128k(B):
    w = inputs.WORKLOADS["c4_qwen128k"]
    g = torch.Generator().manual_seed(4)
    s = torch.randn((w.U, w.Hkv, w.T), generator=g)
    got = gpu_select(B, s.cuda(), "threshold", tau=w.tau, n_sink=w.n_sink, n_recent=w.n_recent)
    check_same(got, O.select(s.numpy(), "threshold", tau=w.tau, n_sink=w.n_sink,
                             n_recent=w.n_recent))


# ------------------------------------------------------------- compaction
def gpu_compact(B, k, v, kept, counts, offs, slack):
    U, Hkv, T, d = k.shape
    n = U * Hkv
    rows = int(offs[-1]) + n * slack
    kc = torch.zeros((max(rows, 1), d), dtype=k.dtype, device="cuda")
    vc = torch.zeros_like(kc)
    start = torch.full((n,), -1, dtype=torch.int64, device="cuda")
    length = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    B.kvc_compact(k, v, torch.as_tensor(kept).cuda(), torch.as_tensor(counts).cuda(),
                  torch.as_tensor(offs).cuda(), kc, vc, start, length, slack=slack)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    return kc[:rows], vc[:rows], start.cpu().numpy(), length.cpu().numpy()


def as_bytes(t):
    return t.cpu().contiguous().view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 128),
                                     (torch.bfloat16, 64), (torch.float32, 64)])
@pytest.mark.parametrize("slack", [0, 3])
def test_compact_bit_exact_small(B, dtype, d, slack):
    U, Hkv, T = 2, 3, 1001
    g = torch.Generator().manual_seed(9)
    k = torch.randn((U, Hkv, T, d), generator=g).to(dtype)
    v = torch.randn((U, Hkv, T, d), generator=g).to(dtype)
    s = inputs.random_scores((U, Hkv, T), seed=2).numpy()
    kept, counts, offs = O.select(s, "global", keep_ratio=0.2, n_sink=4, n_recent=16)
    kc, vc, start, length = gpu_compact(B, k.cuda(), v.cuda(), kept, counts, offs, slack)
    rk, rv, rs, rl = O.compact(k.numpy() if dtype == torch.float32 else k.view(torch.int16).numpy(),
                               v.numpy() if dtype == torch.float32 else v.view(torch.int16).numpy(),
                               kept, counts, offs, slack)
    np.testing.assert_array_equal(start, rs)
    np.testing.assert_array_equal(length, rl)
    kb = as_bytes(kc).reshape(kc.shape[0], -1)
    vb = as_bytes(vc).reshape(vc.shape[0], -1)
    rkb = rk.view(np.uint8).reshape(rk.shape[0], -1)
    rvb = rv.view(np.uint8).reshape(rv.shape[0], -1)
    for i in range(U * Hkv):           # written rows only (slack rows are not the kernel's)
        sl = slice(rs[i], rs[i] + rl[i])
        np.testing.assert_array_equal(kb[sl], rkb[sl])
        np.testing.assert_array_equal(vb[sl], rvb[sl])


def test_compact_llama32k_full(B):
    w = inputs.WORKLOADS["c2_llama32k"]
    q = inputs.window_queries(w, "cuda")
    k, v = inputs.keys_values(w, q, "cuda")
    s = O.score_attn(np64(q), np64(k), w.scale).astype(np.float32)
    kept, counts, offs = O.select(s, "global", keep_ratio=w.keep_ratio, n_sink=w.n_sink,
                                  n_recent=w.n_recent)
    kc, vc, start, length = gpu_compact(B, k, v, kept, counts, offs, 0)
    kh = k.cpu().view(torch.int16).numpy()
    vh = v.cpu().view(torch.int16).numpy()
    rk, rv, rs, rl = O.compact(kh, vh, kept, counts, offs, 0)
    np.testing.assert_array_equal(kc.cpu().view(torch.int16).numpy(), rk)
    np.testing.assert_array_equal(vc.cpu().view(torch.int16).numpy(), rv)


def test_compact_reports_capacity_overflow_without_writing_past(B):
    U, Hkv, T, d = 1, 2, 64, 128
    k = torch.randn((U, Hkv, T, d), device="cuda").to(torch.bfloat16)
    v = torch.randn_like(k)
    kept = np.tile(np.arange(T, dtype=np.int32), (2, 1))
    counts = np.array([T, T], dtype=np.int32)
    offs = np.array([0, T, 2 * T], dtype=np.int64)
    guard = torch.zeros((2 * T + 8, d), dtype=torch.bfloat16, device="cuda")
    kc = guard[: T + 5]                     # too small on purpose: rows >= T+5 must be skipped
    vc = torch.zeros_like(guard)[: T + 5]
    start = torch.empty(2, dtype=torch.int64, device="cuda")
    length = torch.empty(2, dtype=torch.int32, device="cuda")
    B.kvc_compact(k, v, torch.as_tensor(kept).cuda(), torch.as_tensor(counts).cuda(),
                  torch.as_tensor(offs).cuda(), kc, vc, start, length)
    assert B.kvc_device_status() == -6            # KVC_ERR_RANGE
    assert B.kvc_device_status() == 0             # cleared
    assert guard[T + 5:].abs().sum().item() == 0  # nothing written past the capacity


@pytest.mark.parametrize("case", ["first_offset_not_zero", "step_beyond_T", "total_beyond_cache"])
def test_compact_rejects_offsets_that_disagree_with_counts(B, case):
    """Offsets are caller data: rows they place outside a head's count (or
    outside T) are reported as KVC_ERR_RANGE before any index is read, and
    nothing is written outside the stated capacity."""
    U, Hkv, T, d = 1, 2, 64, 128
    k = torch.randn((U, Hkv, T, d), device="cuda").to(torch.bfloat16)
    v = torch.randn_like(k)
    kept = np.tile(np.arange(T, dtype=np.int32), (2, 1))
    counts = np.array([10, 12], dtype=np.int32)
    if case == "first_offset_not_zero":
        offs = np.array([5, 15, 27], dtype=np.int64)       # rows 0..4 belong to no head
    elif case == "step_beyond_T":
        offs = np.array([0, T + 7, T + 19], dtype=np.int64)  # head 0 spans more than T rows
    else:
        offs = np.array([0, 10, 3 * T], dtype=np.int64)      # total above U * Hkv * T
    cap = 40
    guard = torch.zeros((cap + 16, d), dtype=torch.bfloat16, device="cuda")
    vguard = torch.zeros_like(guard)
    start = torch.empty(2, dtype=torch.int64, device="cuda")
    length = torch.empty(2, dtype=torch.int32, device="cuda")
    B.kvc_compact(k, v, torch.as_tensor(kept).cuda(), torch.as_tensor(counts).cuda(),
                  torch.as_tensor(offs).cuda(), guard[:cap], vguard[:cap], start, length)
    assert B.kvc_device_status() == -6            # KVC_ERR_RANGE
    assert B.kvc_device_status() == 0             # cleared
    assert guard[cap:].abs().sum().item() == 0    # nothing written past the capacity
    assert vguard[cap:].abs().sum().item() == 0


# --------------------------------------------------- select + compact in one call
def fused_and_separate(B, s, k, v, mode, slack, workspace=None, **kw):
    """Outputs of kvc_select_compact and of kvc_select + kvc_compact on the same
    inputs, every output buffer pre-filled with the same sentinel."""
    U, Hkv, T = s.shape
    n = U * Hkv
    hb = kw.pop("head_budget", None)
    if hb is not None:
        hb = torch.as_tensor(np.asarray(hb), dtype=torch.int32).cuda()
    cap = n * T + n * slack
    res = []
    for fused in (True, False):
        kept = torch.full((n, T), -7, dtype=torch.int32, device="cuda")
        counts = torch.full((n,), -7, dtype=torch.int32, device="cuda")
        offs = torch.full((n + 1,), -7, dtype=torch.int64, device="cuda")
        kc = torch.full((cap, k.shape[-1]), 3.0, dtype=k.dtype, device="cuda")
        vc = torch.full_like(kc, -3.0)
        start = torch.full((n,), -7, dtype=torch.int64, device="cuda")
        length = torch.full((n,), -7, dtype=torch.int32, device="cuda")
        if fused:
            B.kvc_select_compact(s, mode, k, v, kept, counts, offs, kc, vc, start, length,
                                 head_budget=hb, slack=slack, workspace=workspace, **kw)
        else:
            B.kvc_select(s, mode, kept, counts, offs, head_budget=hb, **kw)
            B.kvc_compact(k, v, kept, counts, offs, kc, vc, start, length, slack=slack)
        torch.cuda.synchronize()
        assert B.kvc_device_status() == 0
        c = counts.cpu().numpy()
        kn = kept.cpu().numpy()
        res.append(([kn[i, : c[i]] for i in range(n)], c, offs.cpu().numpy(),
                    start.cpu().numpy(), length.cpu().numpy(), as_bytes(kc), as_bytes(vc)))
    return res


def assert_same_outputs(a, b):
    for x, y in zip(a[0], b[0]):
        np.testing.assert_array_equal(x, y)
    for x, y in zip(a[1:], b[1:]):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("shape,mode,dtype,d", [
    ((1, 8, 32768), "global", torch.bfloat16, 128),   # the 32k layer's shape: hand-off path
    ((1, 4, 5000), "global", torch.float32, 64),      # ragged ranges
    ((1, 3, 777), "global", torch.bfloat16, 64),
    ((1, 1, 70001), "per_head", torch.bfloat16, 128),
    ((1, 1, 4099), "threshold", torch.float32, 128),
    ((2, 8, 3000), "global", torch.bfloat16, 128),    # two pools: the two calls back to back
    ((1, 8, 65536), "global", torch.bfloat16, 64),    # beyond one cluster: streaming select
])
@pytest.mark.parametrize("ties,specials", [(False, False), (True, True)])
def test_select_compact_equals_the_two_calls(B, shape, mode, dtype, d, ties, specials):
    s = inputs.random_scores(shape, seed=sum(shape) + 3, ties=ties, specials=specials).cuda()
    U, Hkv, T = shape
    g = torch.Generator().manual_seed(11)
    k = torch.randn((U, Hkv, T, d), generator=g).to(dtype).cuda()
    v = torch.randn((U, Hkv, T, d), generator=g).to(dtype).cuda()
    if mode == "global":
        cases = [dict(keep_ratio=r, n_sink=ns, n_recent=nr)
                 for r, ns, nr in [(0.1, 4, 64), (0.0, 2, 2), (1.0, 1, 1), (0.37, 0, 0)]]
    elif mode == "per_head":
        cases = [dict(head_budget=[b] * (U * Hkv), n_sink=4, n_recent=64)
                 for b in (0, 700, 7000, T + 5)]
    else:
        cases = [dict(tau=t, n_sink=1, n_recent=3) for t in (0.5, float("nan"), float("-inf"))]
    for kw in cases:
        for slack in (0, 5):
            a, b = fused_and_separate(B, s, k, v, mode, slack, **dict(kw))
            assert_same_outputs(a, b)


def test_select_compact_llama32k_against_the_oracle(B):
    """The 32k layer through the fused call on the oracle's scores: kept
    indices, counts, offsets and the compacted rows equal the oracle's."""
    w = inputs.WORKLOADS["c2_llama32k"]
    q = inputs.window_queries(w, "cuda")
    k, v = inputs.keys_values(w, q, "cuda")
    s = O.score_attn(np64(q), np64(k), w.scale).astype(np.float32)
    kw = dict(keep_ratio=w.keep_ratio, n_sink=w.n_sink, n_recent=w.n_recent)
    a, _ = fused_and_separate(B, torch.from_numpy(s).cuda(), k, v, "global", 0, **kw)
    rk, rc, ro = O.select(s, "global", **kw)
    np.testing.assert_array_equal(a[1], rc)
    np.testing.assert_array_equal(a[2], ro)
    for i in range(len(rc)):
        np.testing.assert_array_equal(a[0][i], rk[i, : rc[i]])
    kh = k.cpu().view(torch.int16).numpy()
    vh = v.cpu().view(torch.int16).numpy()
    ck, cv, cs, cl = O.compact(kh, vh, rk, rc, ro, 0)
    rows = int(ro[-1])
    np.testing.assert_array_equal(a[3], cs)
    np.testing.assert_array_equal(a[4], cl)
    np.testing.assert_array_equal(a[5].reshape(-1, w.d * 2)[:rows], ck.view(np.uint8).reshape(rows, -1))
    np.testing.assert_array_equal(a[6].reshape(-1, w.d * 2)[:rows], cv.view(np.uint8).reshape(rows, -1))


def test_select_compact_without_workspace_and_capacity_overflow(B):
    U, Hkv, T, d = 1, 2, 640, 128
    s = inputs.random_scores((U, Hkv, T), seed=4).cuda()
    k = torch.randn((U, Hkv, T, d), device="cuda").to(torch.bfloat16)
    v = torch.randn_like(k)
    # no workspace: the two calls, same outputs
    a, b = fused_and_separate(B, s, k, v, "global", 2,
                              workspace=torch.empty(0, dtype=torch.uint8, device="cuda"),
                              keep_ratio=0.3, n_sink=4, n_recent=8)
    assert_same_outputs(a, b)
    # a cache too small: rows past it are skipped and reported
    guard = torch.zeros((2 * T, d), dtype=torch.bfloat16, device="cuda")
    kc = guard[:100]
    vc = torch.zeros_like(guard)[:100]
    kept = torch.empty((2, T), dtype=torch.int32, device="cuda")
    counts = torch.empty(2, dtype=torch.int32, device="cuda")
    offs = torch.empty(3, dtype=torch.int64, device="cuda")
    start = torch.empty(2, dtype=torch.int64, device="cuda")
    length = torch.empty(2, dtype=torch.int32, device="cuda")
    B.kvc_select_compact(s, "global", k, v, kept, counts, offs, kc, vc, start, length,
                         keep_ratio=0.5, n_sink=4, n_recent=8)
    assert B.kvc_device_status() == -6            # KVC_ERR_RANGE
    assert B.kvc_device_status() == 0
    assert guard[100:].abs().sum().item() == 0


@pytest.mark.parametrize("shape,mode", [((1, 8, 32768), "global"), ((2, 3, 777), "global"),
                                        ((1, 1, 4099), "threshold")])
def test_compaction_reads_a_cache_held_in_pinned_host_memory(B, shape, mode):
    """K and V left in pinned host memory (mapped at the same address under
    unified addressing): both compaction calls read only the kept rows across
    the bus and write the same outputs, bit for bit, as from device copies."""
    s = inputs.random_scores(shape, seed=sum(shape) + 17).cuda()
    U, Hkv, T = shape
    g = torch.Generator().manual_seed(19)
    k = torch.randn((U, Hkv, T, 128), generator=g).to(torch.bfloat16)
    v = torch.randn((U, Hkv, T, 128), generator=g).to(torch.bfloat16)
    hk, hv = k.pin_memory(), v.pin_memory()
    kw = dict(keep_ratio=0.1, n_sink=4, n_recent=64) if mode == "global" else dict(tau=0.5)
    on_device = fused_and_separate(B, s, k.cuda(), v.cuda(), mode, 3, **dict(kw))
    on_host = fused_and_separate(B, s, hk, hv, mode, 3, **dict(kw))
    for a, b in zip(on_device, on_host):
        assert_same_outputs(a, b)


def test_compaction_refuses_host_memory_the_device_cannot_read(B):
    """Pageable host memory would fault on the device: both calls refuse it
    on the host (KVC_ERR_INVALID) and launch nothing."""
    shape = (1, 2, 256)
    s = inputs.random_scores(shape, seed=3).cuda()
    n, T = 2, 256
    k = torch.zeros((1, 2, T, 128), dtype=torch.bfloat16)       # pageable
    v_dev = torch.zeros((1, 2, T, 128), dtype=torch.bfloat16, device="cuda")
    kept = torch.zeros((n, T), dtype=torch.int32, device="cuda")
    counts = torch.zeros(n, dtype=torch.int32, device="cuda")
    offs = torch.zeros(n + 1, dtype=torch.int64, device="cuda")
    kc = torch.zeros((n * T, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    start = torch.zeros(n, dtype=torch.int64, device="cuda")
    length = torch.zeros(n, dtype=torch.int32, device="cuda")
    with pytest.raises(B.KvcError) as e:
        B.kvc_compact(k, v_dev, kept, counts, offs, kc, vc, start, length)
    assert e.value.status == -1
    with pytest.raises(B.KvcError) as e:
        B.kvc_select_compact(s, "global", v_dev, k, kept, counts, offs, kc, vc, start, length,
                             keep_ratio=0.5)
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
