"""Seeded synthetic inputs for the score -> select -> compact -> decode path.

This module is shared by the CUDA path's tests, the oracle's tests and the
benchmark.  It draws random numbers and lays them out; it computes nothing of
the compression method itself (no attention, no scoring, no selection, no
gather).  Everything is drawn with a seeded ``torch.Generator`` on the device
the caller names, so a GPU run and a CPU run of the same seed give different
values: callers that compare two implementations generate once and hand the
same bytes to both.

The five workloads stand in for the long-context evaluations on the pages
(LongBench, RULER, needle-in-a-haystack, AIME25), which are not available
here; only their shapes are reproduced:

* ``c1_tiny``     -- 8 q / 4 kv heads, d 64, T 1024, fp32, W 32, keep 0.25.
* ``c2_llama32k`` -- Llama-3-8B-shaped layer: 32 q / 8 kv, d 128, T 32768,
                     bf16, 4 outlier key channels per kv head (x8), W 64,
                     keep 0.10 (global top-k across heads), 4 sinks + 64 recent.
* ``c3_32layer``  -- 32 layers x batch 4 folded into U = 128 units, T 16384,
                     bf16, per-(layer, kv head) softmax temperature ~ U[0.5, 2],
                     keep 0.20 per unit.
* ``c4_qwen128k`` -- Qwen-shaped 28 q / 4 kv, T 131072, hidden 3584 ~ N(0,1),
                     linear surrogate weight ~ N(0, 1/3584), tau 0.5, 4 sinks +
                     128 recent.
* ``c5_decode``   -- batch 64, 32 q / 8 kv, d 128, per-head compressed lengths
                     ~ floor(U[0.1, 0.3] * 32768), 256 decode steps.

Key construction ("sinks" and "needles"): for every unit u and kv head g the
mean direction of that group's window queries is formed, u_dir = qbar/|qbar|;
sink keys (tokens 0..3) are 4*sqrt(d)*u_dir and needle keys are
3*sqrt(d)*u_dir + N(0, I) at seeded distinct positions in
[n_sink, T - n_recent).  "Scaled x4" is read relative to the typical key
norm sqrt(d): a literal unit-norm reading gives logits near 0.5, i.e. no
sink at all.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

SEED_BASE = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    U: int                  # independent units (batch x layers)
    Hq: int
    Hkv: int
    d: int
    T: int
    W: int                  # observation window (queries per q head)
    dtype: str              # "f32" | "bf16"
    n_sink: int
    n_recent: int
    mode: str               # "global" | "threshold" | "per_head"
    keep_ratio: float = 0.0
    tau: float = 0.0
    needles_per_1024: float = 0.0   # needle density (tokens per 1024)
    n_needles: int = 0              # explicit count (overrides density)
    outlier_channels: int = 0       # per kv head, keys scaled x8
    head_temperature: Optional[tuple] = None   # (lo, hi) factor per (layer, kv head)
    layers: int = 1                 # units = batch * layers, layer = u % layers
    Dh: int = 0                     # hidden size for the linear surrogate
    decode_steps: int = 0
    len_frac: Optional[tuple] = None  # (lo, hi) compressed length / T
    slack: int = 0                  # rows reserved per head for appends
    index: int = 0                  # workload number, used in the seed

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def needles(self) -> int:
        if self.n_needles:
            return self.n_needles
        return int(round(self.needles_per_1024 * self.T / 1024.0))

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "c1_tiny": Workload("c1_tiny", U=1, Hq=8, Hkv=4, d=64, T=1024, W=32, dtype="f32",
                        n_sink=4, n_recent=32, mode="global", keep_ratio=0.25,
                        n_needles=16, index=1),
    "c2_llama32k": Workload("c2_llama32k", U=1, Hq=32, Hkv=8, d=128, T=32768, W=64,
                            dtype="bf16", n_sink=4, n_recent=64, mode="global",
                            keep_ratio=0.10, n_needles=64, outlier_channels=4, index=2),
    "c3_32layer": Workload("c3_32layer", U=128, Hq=32, Hkv=8, d=128, T=16384, W=64,
                           dtype="bf16", n_sink=4, n_recent=64, mode="global",
                           keep_ratio=0.20, needles_per_1024=16.0,
                           head_temperature=(0.5, 2.0), layers=32, index=3),
    "c4_qwen128k": Workload("c4_qwen128k", U=1, Hq=28, Hkv=4, d=128, T=131072, W=0,
                            dtype="bf16", n_sink=4, n_recent=128, mode="threshold",
                            tau=0.5, needles_per_1024=16.0, Dh=3584, index=4),
    "c5_decode": Workload("c5_decode", U=64, Hq=32, Hkv=8, d=128, T=32768, W=64,
                          dtype="bf16", n_sink=4, n_recent=64, mode="per_head",
                          needles_per_1024=16.0, decode_steps=256, len_frac=(0.1, 0.3),
                          slack=256, index=5),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _seed(w: Workload, tensor_id: int, extra: int = 0) -> int:
    return SEED_BASE + 1000 * w.index + tensor_id + 100003 * extra


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def window_queries(w: Workload, device="cpu") -> torch.Tensor:
    """Q_win [U, Hq, W, d] ~ N(0, 1), cast to the workload dtype."""
    g = _gen(device, _seed(w, 1))
    return _randn((w.U, w.Hq, w.W, w.d), g, device).to(w.torch_dtype)


def head_scale(w: Workload, device="cpu") -> Optional[torch.Tensor]:
    """Per-(unit, q head) softmax temperature factor, or None (all ones).

    One factor f ~ U[lo, hi] is drawn per (layer, kv head) and broadcast to the
    G query heads of that kv head and to every batch item of that layer.
    """
    if w.head_temperature is None:
        return None
    lo, hi = w.head_temperature
    g = _gen(device, _seed(w, 4))
    f = lo + (hi - lo) * torch.rand((w.layers, w.Hkv), generator=g, device=device)
    layer_of_unit = torch.arange(w.U, device=device) % w.layers
    per_kv = f[layer_of_unit]                                 # [U, Hkv]
    return per_kv.repeat_interleave(w.G, dim=1).contiguous()  # [U, Hq]


def needle_positions(w: Workload, device="cpu") -> torch.Tensor:
    """[U, n_needles] distinct token positions in [n_sink, T - n_recent)."""
    n = w.needles()
    lo, hi = w.n_sink, w.T - w.n_recent
    if n == 0 or hi - lo < n:
        return torch.zeros((w.U, 0), dtype=torch.long, device=device)
    g = _gen(device, _seed(w, 5))
    out = []
    for _ in range(w.U):
        perm = torch.randperm(hi - lo, generator=g, device=device)[:n] + lo
        out.append(torch.sort(perm).values)
    return torch.stack(out)


def _key_direction(w: Workload, q_win: Optional[torch.Tensor], device) -> torch.Tensor:
    """Unit direction [U, Hkv, d]: mean window-query direction of each group,
    or a seeded random direction when the workload has no window."""
    if q_win is not None and w.W > 0:
        qg = q_win.float().view(w.U, w.Hkv, w.G * w.W, w.d)
        qbar = qg.mean(dim=2)
    else:
        g = _gen(device, _seed(w, 6))
        qbar = _randn((w.U, w.Hkv, w.d), g, device)
    return qbar / qbar.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def keys_values(w: Workload, q_win: Optional[torch.Tensor] = None, device="cpu"):
    """K, V [U, Hkv, T, d] in the workload dtype.

    K, V ~ N(0, 1); optional outlier key channels scaled x8 (seeded channel
    indices per kv head); sink and needle keys aligned with the group's mean
    query direction as described in the module docstring.
    """
    gk = _gen(device, _seed(w, 2))
    gv = _gen(device, _seed(w, 3))
    k = _randn((w.U, w.Hkv, w.T, w.d), gk, device)
    v = _randn((w.U, w.Hkv, w.T, w.d), gv, device)
    if w.outlier_channels:
        go = _gen(device, _seed(w, 7))
        for g_ in range(w.Hkv):
            ch = torch.randperm(w.d, generator=go, device=device)[: w.outlier_channels]
            k[:, g_, :, ch] *= 8.0
    u_dir = _key_direction(w, q_win, device)                  # [U, Hkv, d]
    root_d = math.sqrt(w.d)
    ns = min(w.n_sink, w.T)
    if ns:
        k[:, :, :ns, :] = (4.0 * root_d) * u_dir[:, :, None, :]
    pos = needle_positions(w, device)
    if pos.shape[1]:
        gn = _gen(device, _seed(w, 8))
        noise = _randn((w.U, w.Hkv, pos.shape[1], w.d), gn, device)
        for u in range(w.U):
            k[u, :, pos[u], :] = (3.0 * root_d) * u_dir[u, :, None, :] + noise[u]
    return k.to(w.torch_dtype), v.to(w.torch_dtype)


def linear_scorer(w: Workload, device="cpu"):
    """hidden [U, T, Dh] ~ N(0,1), weight [Dh, Hkv] ~ N(0, 1/Dh), bias zeros [Hkv].

    "N(0, 1/3584)" is read as variance 1/Dh, so each linear output is ~ N(0, 1).
    """
    gh = _gen(device, _seed(w, 9))
    gw = _gen(device, _seed(w, 10))
    hidden = _randn((w.U, w.T, w.Dh), gh, device).to(w.torch_dtype)
    weight = (_randn((w.Dh, w.Hkv), gw, device) / math.sqrt(w.Dh)).to(w.torch_dtype)
    bias = torch.zeros(w.Hkv, dtype=torch.float32, device=device)
    return hidden, weight, bias


def kvzip_plus_weights(w: Workload, device="cpu"):
    """Synthetic model weights for the KVzip+ score: the Gram matrices
    gram[h] = W_O^h^T W_O^h of a random output projection W_O [Hq*d, Hq*d] ~
    N(0, 1/(Hq*d)) split by query head (bf16 [Hq, d, d]), and the norms of
    the window positions' hidden states h ~ N(0, I_{Hq*d}) (fp32 [U, W])."""
    dm = w.Hq * w.d
    g1, g2 = _gen(device, _seed(w, 25)), _gen(device, _seed(w, 26))
    gram = torch.empty((w.Hq, w.d, w.d), dtype=torch.bfloat16, device=device)
    for h in range(w.Hq):
        wo = _randn((dm, w.d), g1, device) / math.sqrt(dm)
        gram[h] = (wo.T @ wo).to(torch.bfloat16)
    hnorm = _randn((w.U, w.W, dm), g2, device).norm(dim=-1)
    return gram, hnorm


def mlp_scorer(w: Workload, device="cpu"):
    """Weights of the two-layer surrogate for workload w (hidden width Dh / 8):
    w1 [Dh, Dh/8] ~ N(0, 1/Dh), w2 [Dh/8, Hkv] ~ N(0, 8/Dh) in the workload
    dtype, biases b1 ~ N(0, 0.1^2) [Dh/8] and b2 zeros [Hkv] in fp32."""
    dm = w.Dh // 8
    g1, g2, g3 = _gen(device, _seed(w, 22)), _gen(device, _seed(w, 23)), _gen(device, _seed(w, 24))
    w1 = (_randn((w.Dh, dm), g1, device) / math.sqrt(w.Dh)).to(w.torch_dtype)
    w2 = (_randn((dm, w.Hkv), g2, device) / math.sqrt(dm)).to(w.torch_dtype)
    b1 = 0.1 * _randn((dm,), g3, device)
    return w1, b1, w2, torch.zeros(w.Hkv, dtype=torch.float32, device=device)


def head_budgets(w: Workload, device="cpu") -> torch.Tensor:
    """Per-(unit, kv head) kept-token budgets floor(U[lo, hi] * T), int32 [U*Hkv]."""
    lo, hi = w.len_frac
    g = _gen(device, _seed(w, 11))
    frac = lo + (hi - lo) * torch.rand((w.U * w.Hkv,), generator=g, device=device,
                                       dtype=torch.float64)
    return torch.floor(frac * w.T).to(torch.int32)


def compressed_pool(w: Workload, lengths: torch.Tensor, device="cpu"):
    """A ready-made variable-length cache: rows ~ N(0,1) laid out per head.

    Head i owns rows [start_i, start_i + lengths_i + slack); the first
    lengths_i rows are filled, the slack rows are left zero for appends.
    Returns (kc, vc, start int64 [n], len int32 [n]).
    """
    n = lengths.numel()
    lens = lengths.to(torch.int64).cpu()
    cap = lens + w.slack
    start = torch.zeros(n, dtype=torch.int64)
    if n > 1:
        start[1:] = torch.cumsum(cap, 0)[:-1]
    total = int(cap.sum().item())
    gk = _gen(device, _seed(w, 12))
    gv = _gen(device, _seed(w, 13))
    kc = _randn((total, w.d), gk, device)
    vc = _randn((total, w.d), gv, device)
    fill = torch.zeros(total, dtype=torch.bool)
    for i in range(n):
        fill[start[i]: start[i] + lens[i]] = True
    fill = fill.to(device)
    kc = torch.where(fill[:, None], kc, torch.zeros_like(kc)).to(w.torch_dtype)
    vc = torch.where(fill[:, None], vc, torch.zeros_like(vc)).to(w.torch_dtype)
    return kc, vc, start.to(device), lengths.to(torch.int32).to(device)


def decode_step_inputs(w: Workload, step: int, device="cpu"):
    """q [U, Hq, d], k_new / v_new [U, Hkv, d] ~ N(0,1) for one decode step."""
    g = _gen(device, _seed(w, 14, extra=step + 1))
    q = _randn((w.U, w.Hq, w.d), g, device).to(w.torch_dtype)
    kn = _randn((w.U, w.Hkv, w.d), g, device).to(w.torch_dtype)
    vn = _randn((w.U, w.Hkv, w.d), g, device).to(w.torch_dtype)
    return q, kn, vn


def decode_surrogate(w: Workload, Dh: int, device="cpu"):
    """weight [Dh, Hkv] ~ N(0, 1/Dh), bias zeros [Hkv]: the linear surrogate that
    scores each decode step's new token (outputs ~ N(0, 1), as in linear_scorer)."""
    g = _gen(device, _seed(w, 15))
    weight = (_randn((Dh, w.Hkv), g, device) / math.sqrt(Dh)).to(w.torch_dtype)
    return weight, torch.zeros(w.Hkv, dtype=torch.float32, device=device)


def decode_hidden(w: Workload, Dh: int, step: int, device="cpu") -> torch.Tensor:
    """hidden [U, 1, Dh] ~ N(0,1) of one decode step's new token."""
    g = _gen(device, _seed(w, 16, extra=step + 1))
    return _randn((w.U, 1, Dh), g, device).to(w.torch_dtype)


def row_scores(rows: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """Per-row scores ~ N(0,1) float32 [rows] for a ready-made compressed pool."""
    return _randn((rows,), _gen(device, seed), device)


def vector_predictor(w: Workload, device="cpu") -> torch.Tensor:
    """The K -> V predictor of the VECTOR workloads, W [Hkv, d, d] bf16 with
    entries ~ N(0, 1/d) (row = output dimension), so W k has the scale of k."""
    g = _gen(device, _seed(w, 17))
    return (_randn((w.Hkv, w.d, w.d), g, device) / math.sqrt(w.d)).to(torch.bfloat16)


def vector_values(w: Workload, k: torch.Tensor, W: torch.Tensor, device="cpu") -> torch.Tensor:
    """Values that K predicts linearly, as when K and V are two projections of
    one hidden state: v_t = W_g k_t + sigma_t * N(0, I) with sigma_t ~ U[0, 1]
    per (unit, kv head, token), so tokens differ in how well v is rebuilt from
    k.  Returns bf16 [U, Hkv, T, d]."""
    gs = _gen(device, _seed(w, 18))
    gn = _gen(device, _seed(w, 19))
    sigma = torch.rand((w.U, w.Hkv, w.T, 1), generator=gs, device=device)
    out = torch.empty((w.U, w.Hkv, w.T, w.d), dtype=torch.bfloat16, device=device)
    for u in range(w.U):
        pred = torch.einsum("gty,gxy->gtx", k[u].float(), W.float())
        noise = _randn((w.Hkv, w.T, w.d), gn, device)
        out[u] = (pred + sigma[u] * noise).to(torch.bfloat16)
    return out


def vector_pool(w: Workload, lengths: torch.Tensor, napprox: torch.Tensor, device="cpu"):
    """A ready-made VECTOR cache: head i holds lengths_i key rows (the first
    napprox_i of them approximated) and lengths_i - napprox_i value rows, rows
    ~ N(0,1), w.slack free rows per head in each pool for appends.
    Returns (kc, vc, kstart int64, klen int32, vstart int64, napprox int32)."""
    lens = lengths.to(torch.int64).cpu()
    na = napprox.to(torch.int64).cpu()
    n = lens.numel()
    kcap, vcap = lens + w.slack, lens - na + w.slack
    kstart = torch.zeros(n, dtype=torch.int64)
    vstart = torch.zeros(n, dtype=torch.int64)
    if n > 1:
        kstart[1:] = torch.cumsum(kcap, 0)[:-1]
        vstart[1:] = torch.cumsum(vcap, 0)[:-1]
    gk = _gen(device, _seed(w, 20))
    gv = _gen(device, _seed(w, 21))
    kc = _randn((int(kcap.sum()), w.d), gk, device).to(w.torch_dtype)
    vc = _randn((int(vcap.sum()), w.d), gv, device).to(w.torch_dtype)
    return (kc, vc, kstart.to(device), lens.to(torch.int32).to(device), vstart.to(device),
            na.to(torch.int32).to(device))


def random_scores(shape, device="cpu", seed: int = 0, ties: bool = False,
                  specials: bool = False) -> torch.Tensor:
    """fp32 score tensors for selection tests.

    ``ties`` quantises values to a coarse grid so that many scores are equal;
    ``specials`` plants -0.0, +0.0, +-inf and NaN at seeded positions.
    """
    g = _gen(device, SEED_BASE + 77 + seed)
    s = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    if ties:
        s = torch.floor(s * 16.0) / 16.0
    if specials:
        flat = s.view(-1)
        n = flat.numel()
        idx = torch.randperm(n, generator=g, device=device)[: max(1, n // 16)]
        vals = torch.tensor([-0.0, 0.0, float("inf"), float("-inf"), float("nan"), -1.0],
                            device=device, dtype=torch.float32)
        flat[idx] = vals[torch.arange(idx.numel(), device=device) % vals.numel()]
    return s
