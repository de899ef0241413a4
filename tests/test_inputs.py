"""The seeded input generators hold the distributions the design notes state
(and no method arithmetic): same seed -> same bytes; the stated scales of the
later rows' synthetic weights and values."""
import math

import torch

from kv_cache_compression_attention_b300 import inputs


def test_generators_are_deterministic():
    w = inputs.WORKLOADS["c1_tiny"]
    a = inputs.window_queries(w)
    b = inputs.window_queries(w)
    assert torch.equal(a, b)
    k1, v1 = inputs.keys_values(w, a)
    k2, v2 = inputs.keys_values(w, b)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(inputs.vector_predictor(w), inputs.vector_predictor(w))
    assert torch.equal(inputs.row_scores(100, seed=3), inputs.row_scores(100, seed=3))
    assert not torch.equal(inputs.row_scores(100, seed=3), inputs.row_scores(100, seed=4))


def test_vector_values_are_predicted_plus_uniform_noise():
    # v = W k + sigma * N(0, I), sigma ~ U[0, 1]: residual variance E[sigma^2] = 1/3
    w = inputs.WORKLOADS["c1_tiny"].with_(T=4096)
    k = torch.randn((w.U, w.Hkv, w.T, w.d), generator=torch.Generator().manual_seed(1))
    W = inputs.vector_predictor(w)
    v = inputs.vector_values(w, k, W)
    res = v.float() - torch.einsum("ugty,gxy->ugtx", k, W.float())
    assert abs(res.var().item() - 1.0 / 3.0) < 0.02
    # W ~ N(0, 1/d): W k has the scale of k
    assert abs(W.float().var().item() * w.d - 1.0) < 0.05


def test_kvzip_plus_weights_scales():
    w = inputs.WORKLOADS["c1_tiny"]
    gram, hnorm = inputs.kvzip_plus_weights(w)
    assert gram.shape == (w.Hq, w.d, w.d) and hnorm.shape == (w.U, w.W)
    g = gram.float()
    assert torch.allclose(g, g.transpose(1, 2))                      # Gram matrices
    # W_O ~ N(0, 1/(Hq d)) with Hq d rows: the Gram matrices are close to I
    assert abs(torch.diagonal(g, dim1=1, dim2=2).mean().item() - 1.0) < 0.02
    # hidden states ~ N(0, I_{Hq d}): norms near sqrt(Hq d)
    assert abs(hnorm.mean().item() / math.sqrt(w.Hq * w.d) - 1.0) < 0.02


def test_surrogate_weight_scales():
    w = inputs.WORKLOADS["c4_qwen128k"]
    w1, b1, w2, b2 = inputs.mlp_scorer(w)
    assert w1.shape == (w.Dh, w.Dh // 8) and w2.shape == (w.Dh // 8, w.Hkv)
    assert abs(w1.float().var().item() * w.Dh - 1.0) < 0.02
    assert abs(b1.std().item() - 0.1) < 0.01 and torch.count_nonzero(b2) == 0
    wd = inputs.WORKLOADS["c5_decode"]
    ws, bs = inputs.decode_surrogate(wd, 4096)
    assert abs(ws.float().var().item() * 4096 - 1.0) < 0.05 and torch.count_nonzero(bs) == 0
    h = inputs.decode_hidden(wd, 4096, 0)
    assert h.shape == (wd.U, 1, 4096)


def test_vector_pool_layout():
    w = inputs.WORKLOADS["c5_decode"]
    lens = torch.tensor([10, 0, 7], dtype=torch.int32)
    nap = torch.tensor([6, 0, 1], dtype=torch.int32)
    kc, vc, ks, kl, vs, na = inputs.vector_pool(w.with_(U=1, Hkv=3), lens, nap)
    assert ks.tolist() == [0, 10 + w.slack, 10 + 2 * w.slack]
    assert vs.tolist() == [0, 4 + w.slack, 4 + 2 * w.slack]
    assert kc.shape[0] == 17 + 3 * w.slack and vc.shape[0] == 10 + 3 * w.slack
    assert kl.tolist() == [10, 0, 7] and na.tolist() == [6, 0, 1]
