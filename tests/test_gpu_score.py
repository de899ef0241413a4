"""GPU parity of the scoring kernels against the CPU oracle (through the C ABI).

Attention-mass scoring: fp32 (SIMT path) and bf16 (tcgen05 path for d = 128,
G*W in {128, 256}; SIMT path otherwise), causal and not, with and without a
per-head temperature, on sizes that span several 128-token tiles and a ragged
tail, then on the full workloads (Llama-3-8B-shaped 32k layer in full; the
32-layer x batch-4 cache on sampled units).  Linear surrogate scoring on
small shapes and on sampled rows of the 128k Qwen-shaped workload.
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_compression_attention_b300 import inputs
from oracle import kvc_oracle as O
from tests.kvc_testutil import TOL, mass_rel_err, np64, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kv_cache_compression_attention_b300 import binding
    binding.lib()
    return binding


def gpu_scores(B, q, k, scale, hs=None, causal=True, aggregation="sum"):
    U, Hkv, T = k.shape[0], k.shape[1], k.shape[2]
    out = torch.full((U, Hkv, T), float("nan"), device="cuda", dtype=torch.float32)
    B.kvc_score_attn(q, k, out, scale, head_scale=hs, causal=causal, aggregation=aggregation)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    return out


def rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (scale * torch.randn(shape, generator=g, device="cuda")).to(dtype)


SHAPES = [
    (torch.float32, 64, 2, 32, 1024),     # the tiny fp32 workload's shape
    (torch.float32, 128, 4, 16, 777),
    (torch.bfloat16, 128, 4, 64, 1000),   # tcgen05, R = 256, ragged tail
    (torch.bfloat16, 128, 2, 64, 1300),   # tcgen05, R = 128
    (torch.bfloat16, 128, 4, 64, 300),    # tcgen05, fewer tiles than cluster ranks
    (torch.bfloat16, 128, 16, 8, 900),    # tcgen05, R = 128 of 8-row query heads
    (torch.bfloat16, 128, 8, 32, 640),    # tcgen05, R = 256, an odd count of whole tiles
    (torch.bfloat16, 64, 4, 16, 500),     # SIMT bf16
]


@pytest.mark.parametrize("dtype,d,G,W,T", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
def test_score_attn_small(B, dtype, d, G, W, T, causal):
    U, Hkv = 2, 2
    q = rand((U, Hkv * G, W, d), dtype, 1)
    k = rand((U, Hkv, T, d), dtype, 2)
    hs = (0.5 + 1.5 * torch.rand((U, Hkv * G), generator=torch.Generator(device="cuda").manual_seed(3),
                                 device="cuda")).float()
    scale = d ** -0.5
    got = np64(gpu_scores(B, q, k, scale, hs, causal))
    ref = O.score_attn(np64(q), np64(k), scale, np64(hs), causal)
    assert mass_rel_err(got, ref) <= TOL[dtype]
    # every window row is a softmax: each kv head collects G*W
    np.testing.assert_allclose(got.sum(-1), G * W, rtol=TOL[dtype])


@pytest.mark.parametrize("dtype,d,G,W,T", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
def test_score_attn_max_small(B, dtype, d, G, W, T, causal):
    """Largest attention weight per token (KVzip's aggregation), both paths."""
    U, Hkv = 2, 2
    q = rand((U, Hkv * G, W, d), dtype, 11)
    k = rand((U, Hkv, T, d), dtype, 12)
    hs = (0.5 + 1.5 * torch.rand((U, Hkv * G), generator=torch.Generator(device="cuda").manual_seed(13),
                                 device="cuda")).float()
    scale = d ** -0.5
    got = np64(gpu_scores(B, q, k, scale, hs, causal, aggregation="max"))
    ref = O.score_attn(np64(q), np64(k), scale, np64(hs), causal, aggregation="max")
    assert mass_rel_err(got, ref) <= TOL[dtype]
    assert (got > 0).all() and (got <= 1 + TOL[dtype]).all()


def test_score_attn_max_llama32k_full(B):
    w = inputs.WORKLOADS["c2_llama32k"]
    q = inputs.window_queries(w, "cuda")
    k, _ = inputs.keys_values(w, q, "cuda")
    got = np64(gpu_scores(B, q, k, w.scale, aggregation="max"))
    ref = O.score_attn(np64(q), np64(k), w.scale, aggregation="max")
    assert mass_rel_err(got, ref) <= 2e-2


def test_score_attn_tiny_workload(B):
    w = inputs.WORKLOADS["c1_tiny"]
    q = inputs.window_queries(w, "cuda")
    k, _ = inputs.keys_values(w, q, "cuda")
    got = np64(gpu_scores(B, q, k, w.scale))
    ref = O.score_attn(np64(q), np64(k), w.scale)
    assert mass_rel_err(got, ref) <= 1e-4


def test_score_attn_llama32k_full(B):
    w = inputs.WORKLOADS["c2_llama32k"]
    q = inputs.window_queries(w, "cuda")
    k, _ = inputs.keys_values(w, q, "cuda")
    got = np64(gpu_scores(B, q, k, w.scale))
    ref = O.score_attn(np64(q), np64(k), w.scale)
    assert mass_rel_err(got, ref) <= 2e-2
    # the sinks and every needle outrank the median token of their head (the
    # positions are drawn on the device the keys were built on)
    pos = inputs.needle_positions(w, "cuda").cpu().numpy()[0]
    med = np.median(got, axis=-1)                     # [U, Hkv]
    assert (got[0, :, :4] > med[0, :, None]).all()
    assert (got[0][:, pos] > med[0, :, None]).all()


def test_score_attn_tiny_workload_keeps_every_needle(B):
    """The GPU scores of the tiny workload, selected at keep 0.25 by the GPU
    top-k, keep all 16 needles in every kv head (the oracle's pin of the same
    structure is a CPU test)."""
    w = inputs.WORKLOADS["c1_tiny"]
    q = inputs.window_queries(w, "cuda")
    k, _ = inputs.keys_values(w, q, "cuda")
    s = gpu_scores(B, q, k, w.scale)
    n = w.U * w.Hkv
    kept = torch.empty((n, w.T), dtype=torch.int32, device="cuda")
    counts = torch.empty(n, dtype=torch.int32, device="cuda")
    offs = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    B.kvc_select(s, "global", kept, counts, offs, keep_ratio=w.keep_ratio, n_sink=w.n_sink,
                 n_recent=w.n_recent)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    pos = set(inputs.needle_positions(w, "cuda").cpu().numpy()[0].tolist())
    kept, counts = kept.cpu().numpy(), counts.cpu().numpy()
    for g in range(n):
        assert pos <= set(kept[g, : counts[g]].tolist()), g


def test_score_attn_32layer_sampled_units(B):
    w = inputs.WORKLOADS["c3_32layer"]
    q = inputs.window_queries(w, "cuda")
    k, _ = inputs.keys_values(w, q, "cuda")
    hs = inputs.head_scale(w, "cuda")
    got = gpu_scores(B, q, k, w.scale, hs)
    for u in (0, 77, 127):
        ref = O.score_attn(np64(q[u:u + 1]), np64(k[u:u + 1]), w.scale, np64(hs[u:u + 1]))
        assert mass_rel_err(np64(got[u:u + 1]), ref) <= 2e-2
    del k


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("U,Hkv,Dh,T", [
    (2, 4, 256, 1000), (2, 8, 128, 1100),     # streaming kernel (weights in shared memory)
    (2, 3, 64, 37), (2, 8, 128, 129),         # few rows: one CTA per row
    (64, 8, 4096, 1),                         # a decode step's new tokens, Llama-3-8B hidden size
    (1, 8, 8192, 1500),                       # weights too large for shared memory, many rows
])
def test_score_linear_small(B, dtype, U, Hkv, Dh, T):
    h = rand((U, T, Dh), dtype, 5)
    wt = rand((Dh, Hkv), dtype, 6, scale=Dh ** -0.5)
    bias = rand((Hkv,), torch.float32, 7)
    out = torch.full((U, Hkv, T), float("nan"), device="cuda")
    B.kvc_score_linear(h, wt, bias, out)
    ref = O.score_linear(np64(h), np64(wt), np64(bias))
    assert row_rel_err(np64(out), ref) <= TOL[dtype]


@pytest.mark.parametrize("U,Hkv,Dh,T", [
    (1, 4, 3584, 4099),    # the 128k layer's width, ragged last stage of whole rows
    (3, 4, 128, 2001),     # one 8-dim chunk per warp slice: most lanes idle
    (1, 2, 6144, 1500),    # two chunks per lane
    (2, 2, 384, 1029),
])
def test_score_linear_streamed_rows(B, U, Hkv, Dh, T):
    """Many bf16 rows of widths from one 128-dim block to 6144, ragged row
    counts; compared with the oracle on every row."""
    h = rand((U, T, Dh), torch.bfloat16, 15)
    wt = rand((Dh, Hkv), torch.bfloat16, 16, scale=Dh ** -0.5)
    bias = rand((Hkv,), torch.float32, 17)
    out = torch.full((U, Hkv, T), float("nan"), device="cuda")
    B.kvc_score_linear(h, wt, bias, out)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    ref = O.score_linear(np64(h), np64(wt), np64(bias))
    assert row_rel_err(np64(out), ref) <= TOL[torch.bfloat16]


def test_score_linear_qwen128k_sampled_rows(B):
    w = inputs.WORKLOADS["c4_qwen128k"]
    hid, wt, bias = inputs.linear_scorer(w, "cuda")
    out = torch.empty((w.U, w.Hkv, w.T), device="cuda")
    B.kvc_score_linear(hid, wt, bias, out)
    rows = torch.cat([torch.arange(0, 512), torch.arange(65536, 66048),
                      torch.arange(w.T - 512, w.T)]).cuda()
    ref = O.score_linear(np64(hid[:, rows]), np64(wt), np64(bias))
    assert row_rel_err(np64(out[:, :, rows]), ref) <= 2e-2
    # outputs ~ N(0,1): about 30.85% of the tokens score >= 0.5
    frac = (out >= 0.5).float().mean().item()
    assert abs(frac - 0.3085) < 0.01


@pytest.mark.parametrize("dtype,d,G,W", [(torch.bfloat16, 128, 4, 64), (torch.float32, 64, 2, 32)])
def test_score_attn_rejects_non_positive_temperature_on_device(B, dtype, d, G, W):
    U, Hkv, T = 1, 2, 300
    q = rand((U, Hkv * G, W, d), dtype, 1)
    k = rand((U, Hkv, T, d), dtype, 2)
    hs = torch.ones((U, Hkv * G), device="cuda")
    hs[0, 3] = 0.0
    out = torch.empty((U, Hkv, T), device="cuda")
    B.kvc_score_attn(q, k, out, d ** -0.5, head_scale=hs)
    assert B.kvc_device_status() == -1            # KVC_ERR_INVALID, recorded on the device
    assert B.kvc_device_status() == 0


@pytest.mark.parametrize("Hkv,Dh,Dm,T", [
    (4, 256, 32, 300), (1, 512, 64, 77), (8, 128, 16, 1000),
    (4, 3584, 448, 257),      # the 128k layer's widths: two MMAs of N = 224, ragged row tile
    (3, 200, 520, 129),       # Dh not a multiple of the 64-wide k-block; two passes of 288
    (8, 1024, 1000, 333),     # two passes of 512 columns, padded rows of W1t
    (2, 256, 64, 50),         # one 128-row tile: a single CTA instead of a pair
])
def test_score_mlp_small(B, Hkv, Dh, Dm, T):
    U = 2
    g = torch.Generator().manual_seed(97 + Hkv)
    h = torch.randn((U, T, Dh), generator=g).to(torch.bfloat16)
    w1 = (torch.randn((Dh, Dm), generator=g) / Dh ** 0.5).to(torch.bfloat16)
    b1 = 0.1 * torch.randn(Dm, generator=g)
    w2 = (torch.randn((Dm, Hkv), generator=g) / Dm ** 0.5).to(torch.bfloat16)
    b2 = torch.randn(Hkv, generator=g)
    out = torch.full((U, Hkv, T), float("nan"), device="cuda")
    B.kvc_score_mlp(h.cuda(), w1.cuda(), b1.cuda(), w2.cuda(), b2.cuda(), out)
    torch.cuda.synchronize()
    ref = O.score_mlp(np64(h), np64(w1), np64(b1), np64(w2), np64(b2))
    assert row_rel_err(np64(out), ref) <= 2e-2


def test_score_mlp_qwen128k_sampled_rows(B):
    """The 128k Qwen-shaped layer (hidden 3584, MLP width 448, 4 kv heads)."""
    w = inputs.WORKLOADS["c4_qwen128k"]
    hid, _, _ = inputs.linear_scorer(w, "cuda")
    w1, b1, w2, b2 = inputs.mlp_scorer(w, "cuda")
    out = torch.empty((w.U, w.Hkv, w.T), device="cuda")
    B.kvc_score_mlp(hid, w1, b1, w2, b2, out)
    torch.cuda.synchronize()
    rows = torch.cat([torch.arange(0, 256), torch.arange(70000, 70256),
                      torch.arange(w.T - 256, w.T)]).cuda()
    ref = O.score_mlp(np64(hid[:, rows]), np64(w1), np64(b1), np64(w2), np64(b2))
    assert row_rel_err(np64(out[:, :, rows]), ref) <= 2e-2
    assert torch.isfinite(out).all()


def test_score_mlp_gelu_against_the_oracle(B):
    """The epilogue's GELU alone: W1 = I (z = h exactly, already bf16), b1 = 0
    and one-hot W2 columns make score[g, t] = GELU(h[t, m_g]); its erf
    (Abramowitz & Stegun 7.1.26, absolute error <= 1.5e-7) against the
    oracle's exact GELU over [-8, 8], zeros and tiny values."""
    U, T, Dh, Hkv = 1, 384, 64, 4
    g = torch.Generator().manual_seed(5)
    h = (16 * torch.rand((U, T, Dh), generator=g) - 8).to(torch.bfloat16)
    h[0, :8, 0] = torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e-3, -1e-3, 8.0, -8.0])
    w1 = torch.eye(Dh).to(torch.bfloat16)
    b1 = torch.zeros(Dh)
    cols = [0, 1, 17, 63]
    w2 = torch.zeros((Dh, Hkv))
    for k, m in enumerate(cols):
        w2[m, k] = 1.0
    out = torch.full((U, Hkv, T), float("nan"), device="cuda")
    B.kvc_score_mlp(h.cuda(), w1.cuda(), b1.cuda(), w2.to(torch.bfloat16).cuda(), None, out)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    ref = O.gelu(np64(h)[0][:, cols].T)                      # [Hkv, T]
    # |error| <= |z| / 2 * (1.5e-7 + two fp32 ulps of 1) <= 1.1e-6 on [-8, 8]
    np.testing.assert_allclose(np64(out)[0], ref, rtol=2e-6, atol=1.5e-6)


def kvzip_case(seed, U, Hq, Hkv, W, T, d=128):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((U, Hq, W, d), generator=g).to(torch.bfloat16)
    k = torch.randn((U, Hkv, T, d), generator=g).to(torch.bfloat16)
    v = torch.randn((U, Hkv, T, d), generator=g).to(torch.bfloat16)
    wo = torch.randn((Hq, 3 * d, d), generator=g) / (3 * d) ** 0.5
    gram = torch.einsum("hmd,hme->hde", wo, wo).to(torch.bfloat16).contiguous()
    hnorm = 0.5 + torch.rand((U, W), generator=g) * 2
    return q, k, v, gram, hnorm


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv,W,T", [
    (8, 2, 16, 300), (4, 4, 8, 77), (16, 2, 32, 513),    # SIMT scoring pass
    (8, 2, 64, 700), (4, 2, 64, 300),                     # tensor-core pass (G*W = 256, 128)
])
def test_score_kvzip_plus_small(B, causal, Hq, Hkv, W, T):
    U = 2
    q, k, v, gram, hnorm = kvzip_case(101 + Hq + T, U, Hq, Hkv, W, T)
    hs = 0.5 + torch.rand((U, Hq), generator=torch.Generator().manual_seed(5))
    out = torch.full((U, Hkv, T), float("nan"), device="cuda")
    B.kvc_score_kvzip_plus(q.cuda(), k.cuda(), v.cuda(), gram.cuda(), hnorm.cuda(), out, 0.09,
                           head_scale=hs.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    ref = O.score_kvzip_plus(np64(q), np64(k), np64(v), np64(gram), np64(hnorm), 0.09,
                             head_scale=np64(hs), causal=causal)
    assert mass_rel_err(np64(out), ref) <= 2e-2


def test_score_kvzip_plus_llama32k_full(B):
    """The 32k Llama-3-8B-shaped layer with a synthetic output projection."""
    w = inputs.WORKLOADS["c2_llama32k"]
    q = inputs.window_queries(w, "cuda")
    k, v = inputs.keys_values(w, q, "cuda")
    gram, hnorm = inputs.kvzip_plus_weights(w, "cuda")
    out = torch.empty((w.U, w.Hkv, w.T), device="cuda")
    B.kvc_score_kvzip_plus(q, k, v, gram, hnorm, out, w.scale)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    ref = O.score_kvzip_plus(np64(q), np64(k), np64(v), np64(gram), np64(hnorm), w.scale)
    assert mass_rel_err(np64(out), ref) <= 2e-2
