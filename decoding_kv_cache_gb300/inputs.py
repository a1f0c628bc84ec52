"""Seeded synthetic inputs for the eviction step.

This module is shared by the CPU oracle's tests and by the CUDA path. It holds
no arithmetic of the eviction step itself (no farthest-point sampling, no
scoring, no selection, no compaction). It only plays the part of the model
that fills a KV cache and a query buffer during decoding, with the shapes of
the models the BeaconKV page evaluates (section "实验": R1-Distill-Qwen-7B,
R1-Distill-Llama-8B, Qwen3-4B, Qwen3-14B) and the value structure its
observations describe (section "观察": a few clusters of global queries, early
keys 100-450 that those queries revisit).

One piece of arithmetic that looks like the method's lives here on purpose:
the model's forward pass stores queries and keys *after* rotary position
encoding, so the generator rotates the clustered queries of the
Llama-shaped workload to their own positions and plants keys along the
direction a query of the same cluster takes at the current step.
``_synth_rotate`` does that as a complex multiply; it is written independently
of both the oracle and the kernels, and neither of them calls it.

Every tensor is a pure function of (config, seed, overrides, device): a
``torch.Generator`` on the target device is seeded once and drawn in a fixed
order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

__all__ = ["EvictInputs", "CONFIGS", "make_inputs", "config_names", "EpikvInputs", "EPIKV_CONFIGS",
           "make_epikv_inputs"]


@dataclass
class EvictInputs:
    """One eviction-step problem.

    Layouts (all contiguous):
      K, V      [L, B, Hkv, N, D]   cache, storage dtype (bf16 or f32)
      q_recent  [L, B, Hq, n_r, D]  most recent queries, already rotated to their own positions
      qbuf      [L, B, Hq, qmax, D] pre-RoPE query buffer, oldest entry first
      count     [L, B, Hq] int32    valid rows in qbuf
      budget    [L, B, Hkv] int32   per-head kept total, or None (then ``budget_all``)
    """

    name: str
    dtype: str  # "bf16" | "f32"
    L: int
    B: int
    Hq: int
    Hkv: int
    D: int
    N: int
    n_r: int
    n_b: int
    qmax: int
    t: int
    theta: float
    prefix: int
    recent: int
    budget_all: int
    K: torch.Tensor
    V: torch.Tensor
    q_recent: torch.Tensor
    qbuf: torch.Tensor
    count: torch.Tensor
    budget: Optional[torch.Tensor] = None
    planted: Optional[torch.Tensor] = None  # [L, B, Hkv, n_planted] int64 positions (Llama-shaped workload)
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def heads(self) -> int:
        return self.L * self.B * self.Hkv

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def budgets(self) -> torch.Tensor:
        """Per-head kept totals as an int32 [L, B, Hkv] tensor on the inputs' device."""
        if self.budget is not None:
            return self.budget
        return torch.full((self.L, self.B, self.Hkv), self.budget_all, dtype=torch.int32, device=self.K.device)

    def to(self, device) -> "EvictInputs":
        mv = lambda x: None if x is None else x.to(device)
        return replace(self, K=mv(self.K), V=mv(self.V), q_recent=mv(self.q_recent), qbuf=mv(self.qbuf),
                       count=mv(self.count), budget=mv(self.budget), planted=mv(self.planted))


# The five workloads. Sizes follow the model shapes named for each; the
# eviction ratio 7/8 is the BeaconKV page's dual-threshold budget (section
# "实验": evict one eighth on reaching B_max).
CONFIGS = {
    "tiny": dict(cfg=1, dtype="f32", L=1, B=1, Hq=4, Hkv=2, D=64, N=256, n_r=16, n_b=16, qmax=32,
                 theta=1e4, prefix=4, recent=16, seed=0),
    "qwen3-4b": dict(cfg=2, dtype="bf16", L=36, B=1, Hq=32, Hkv=8, D=128, N=2048, n_r=16, n_b=16, qmax=32,
                     theta=1e6, prefix=4, recent=16, seed=2),
    "llama8b-planted": dict(cfg=3, dtype="bf16", L=32, B=16, Hq=32, Hkv=8, D=128, N=4096, n_r=16, n_b=16,
                            qmax=32, theta=5e5, prefix=4, recent=16, seed=3),
    "qwen7b-reasonalloc": dict(cfg=4, dtype="bf16", L=28, B=8, Hq=28, Hkv=4, D=128, N=8192, n_r=16, n_b=16,
                               qmax=32, theta=1e6, prefix=4, recent=16, seed=4),
    "qwen3-14b-long": dict(cfg=5, dtype="bf16", L=40, B=8, Hq=40, Hkv=8, D=128, N=32768, n_r=16, n_b=32,
                           qmax=64, theta=1e6, prefix=4, recent=16, seed=5),
}


def config_names():
    return list(CONFIGS)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _synth_rotate(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate ``x[..., D]`` to positions ``pos`` (broadcast over the leading dims) the way the
    model's forward pass does before caching: channel i pairs with channel i + D/2 and turns by
    pos * theta**(-2i/D). Written as a complex multiply in float64; input synthesis only."""
    D = x.shape[-1]
    h = D // 2
    i = torch.arange(h, dtype=torch.float64, device=x.device)
    freq = torch.exp(-(2.0 * i / D) * math.log(theta))
    phase = pos.to(torch.float64)[..., None] * freq
    z = torch.complex(x[..., :h].double(), x[..., h:].double()) * torch.polar(torch.ones_like(phase), phase)
    return torch.cat([z.real, z.imag], dim=-1)


def _reasonalloc_budgets(L: int, Hkv: int, N: int, g_cpu: torch.Generator) -> torch.Tensor:
    """Per-(layer, KV head) budgets with a mid-peaked layer profile and a Dirichlet(2) head split.

    Layer profile 1024*(0.5 + sin(pi*l/27)), rescaled to average 1024 over the layers; each layer's
    total Hkv*b_l is split across its heads by one Dirichlet(2,...,2) draw (a normalised pair of
    Erlang(2) variables per head), rounded half-to-even and clamped to [20, N].
    """
    l = torch.arange(L, dtype=torch.float64)
    prof = 1024.0 * (0.5 + torch.sin(math.pi * l / 27.0))
    prof = prof * (1024.0 / prof.mean())
    u = torch.rand((L, Hkv, 2), generator=g_cpu, dtype=torch.float64)
    gam = -torch.log1p(-u).sum(-1)  # Erlang(2, 1): sum of two unit exponentials
    w = gam / gam.sum(-1, keepdim=True)
    b = torch.round(Hkv * prof[:, None] * w)
    return b.clamp(20, N).to(torch.int32)


def make_inputs(name: str, device="cpu", seed: Optional[int] = None, **over) -> EvictInputs:
    """Build the named workload, optionally with smaller sizes (``L=2, N=1000`` ...).

    ``over`` may override any entry of ``CONFIGS[name]`` plus ``keep`` (the uniform kept total,
    default 7/8 of N), ``count`` (valid rows of every query buffer, default full) and, for the
    Llama-shaped workload, ``recent_global=False`` (no clustered queries in the recent window).
    """
    spec = dict(CONFIGS[name])
    keep = over.pop("keep", None)
    recent_global = over.pop("recent_global", True)
    count_over = over.pop("count", None)
    spec.update(over)
    if seed is not None:
        spec["seed"] = seed
    cfg = spec["cfg"]
    L, B, Hq, Hkv, D, N = (spec[k] for k in ("L", "B", "Hq", "Hkv", "D", "N"))
    n_r, n_b, qmax = spec["n_r"], spec["n_b"], spec["qmax"]
    dt = torch.bfloat16 if spec["dtype"] == "bf16" else torch.float32
    device = torch.device(device)
    g = _gen(device, spec["seed"])
    t = N - 1  # the newest cached token's position at the first eviction
    G = Hq // Hkv

    K = torch.empty((L, B, Hkv, N, D), dtype=dt, device=device)
    V = torch.empty((L, B, Hkv, N, D), dtype=dt, device=device)
    planted = None
    meta = {}

    if cfg in (1, 2, 4):
        scale = None
        if cfg == 2:
            scale = 0.5 + 1.5 * torch.rand((L, 1, Hkv, 1, D), generator=g, device=device)
        for l in range(L):
            k = _randn((B, Hkv, N, D), g, device)
            v = _randn((B, Hkv, N, D), g, device)
            if scale is not None:
                k = k * scale[l]
                v = v * scale[l]
            K[l] = k.to(dt)
            V[l] = v.to(dt)
        q_recent = _randn((L, B, Hq, n_r, D), g, device).to(dt)
        qbuf = _randn((L, B, Hq, qmax, D), g, device).to(dt)
    elif cfg == 5:
        # heavy-tailed outlier channels: 4 per (layer, KV head), Student-t with 3 degrees of freedom
        chan = torch.argsort(torch.rand((L, Hkv, D), generator=g, device=device), dim=-1)[..., :4]
        mask = torch.zeros((L, Hkv, D), dtype=torch.bool, device=device)
        mask.scatter_(-1, chan, True)
        for l in range(L):
            k = _randn((B, Hkv, N, D), g, device)
            z3 = _randn((3, B, Hkv, N, D), g, device)
            student = k / torch.sqrt((z3 * z3).sum(0) / 3.0)
            k = torch.where(mask[l][None, :, None, :], student, k)
            K[l] = k.to(dt)
            V[l] = _randn((B, Hkv, N, D), g, device).to(dt)
            del z3, student, k
        q_recent = _randn((L, B, Hq, n_r, D), g, device).to(dt)
        qbuf = _randn((L, B, Hq, qmax, D), g, device).to(dt)
        meta["outlier_channels"] = chan
    elif cfg == 3:
        n_c, frac_c, sig_c = 4, 0.3, 0.1
        n_plant = min(64, max(1, N // 8))
        lo, hi = min(100, N // 4), min(450, N - 1 - spec["recent"])
        centres = _randn((L, B, Hkv, n_c, D), g, device)
        centres = centres / centres.norm(dim=-1, keepdim=True)
        # query stream per query head: qmax buffered (pre-RoPE) then n_r recent (rotated to t-n_r+1..t)
        S = qmax + n_r
        is_c = torch.rand((L, B, Hq, S), generator=g, device=device) < frac_c
        if not recent_global:  # a decoding moment between revisits: the recent window holds local queries only
            is_c[..., qmax:] = False
        which = torch.randint(0, n_c, (L, B, Hq, S), generator=g, device=device)
        kv_of = (torch.arange(Hq, device=device) // G)
        cen_q = centres[:, :, kv_of]  # [L,B,Hq,n_c,D]
        picked = torch.gather(cen_q, 3, which[..., None].expand(L, B, Hq, S, D))
        noise = _randn((L, B, Hq, S, D), g, device)
        stream = torch.where(is_c[..., None], picked + sig_c * noise, noise / math.sqrt(D))
        qbuf = stream[:, :, :, :qmax].to(dt)
        pos = torch.arange(t - n_r + 1, t + 1, device=device)
        q_recent = _synth_rotate(stream[:, :, :, qmax:], pos, spec["theta"]).to(dt)
        # planted keys: distinct positions in [lo, hi], pointing along a centre as seen at step t and
        # of ordinary expected norm (0.6^2 + 0.8^2 = 1 share of sqrt(D)), so only their direction marks them
        planted = torch.argsort(torch.rand((L, B, Hkv, hi - lo + 1), generator=g, device=device), dim=-1)
        planted = (planted[..., :n_plant] + lo).sort(dim=-1).values
        pm = torch.randint(0, n_c, (L, B, Hkv, n_plant), generator=g, device=device)
        cen_k = torch.gather(centres, 3, pm[..., None].expand(L, B, Hkv, n_plant, D))
        plant_dir = 0.6 * math.sqrt(D) * _synth_rotate(cen_k, torch.tensor(t, device=device), spec["theta"]).float()
        for l in range(L):
            k = _randn((B, Hkv, N, D), g, device)
            idx = planted[l][..., None].expand(B, Hkv, n_plant, D)
            k.scatter_(2, idx, 0.8 * torch.gather(k, 2, idx) + plant_dir[l])
            K[l] = k.to(dt)
            V[l] = _randn((B, Hkv, N, D), g, device).to(dt)
        meta["centres"] = centres
        meta["planted_centre"] = pm
    else:
        raise ValueError(f"unknown config {cfg}")

    cnt = qmax if count_over is None else count_over
    count = torch.full((L, B, Hq), cnt, dtype=torch.int32, device=device)
    budget = None
    budget_all = (7 * N) // 8 if keep is None else int(keep)
    if cfg == 4 and keep is None:
        budget = _reasonalloc_budgets(L, Hkv, N, _gen("cpu", spec["seed"] + 1000))
        budget = budget[:, None, :].expand(L, B, Hkv).contiguous().to(device)
        budget_all = 0
    return EvictInputs(name=name, dtype=spec["dtype"], L=L, B=B, Hq=Hq, Hkv=Hkv, D=D, N=N, n_r=n_r, n_b=n_b,
                       qmax=qmax, t=t, theta=float(spec["theta"]), prefix=spec["prefix"], recent=spec["recent"],
                       budget_all=budget_all, K=K, V=V, q_recent=q_recent, qbuf=qbuf, count=count,
                       budget=budget, planted=planted, meta=meta)


# ---------------------------------------------------------------------------
# EPIKV workload: the model shape the EPIKV write-up evaluates (R1-Distill-Llama-8B: 32 layers,
# 8 KV heads of 128, hidden size 4096) with the hidden states of its two band layers (10 and 21).
# ---------------------------------------------------------------------------
EPIKV_CONFIGS = {
    "llama8b-epikv": dict(dtype="bf16", L=32, B=16, Hq=32, Hkv=8, D=128, N=4096, dm=4096, window=128, eps=1e-6,
                          prefix=4, recent=16, seed=6),
}


@dataclass
class EpikvInputs:
    """One EPIKV eviction problem: the cache K, V [L, B, Hkv, N, D] and the hidden states hA, hB
    [B, N, dm] of the two band layers (storage dtype); budget_all kept tokens per sequence."""

    name: str
    dtype: str
    L: int
    B: int
    Hq: int
    Hkv: int
    D: int
    N: int
    dm: int
    window: int
    eps: float
    prefix: int
    recent: int
    budget_all: int
    K: torch.Tensor
    V: torch.Tensor
    hA: torch.Tensor
    hB: torch.Tensor

    @property
    def heads(self) -> int:
        return self.L * self.B * self.Hkv

    def to(self, device) -> "EpikvInputs":
        return replace(self, K=self.K.to(device), V=self.V.to(device), hA=self.hA.to(device), hB=self.hB.to(device))


def _residual_stream(B: int, N: int, dm: int, g: torch.Generator, device, rho: float = 0.9) -> torch.Tensor:
    """A synthetic residual stream: h(t) = rho h(t-1) + s(t) n(t), h(-1) = 0, n ~ N(0, I), with a
    log-normal step size s(t) = exp(0.3 a(t)) (1 + 0.5 t/N) and an occasional large step (p = 0.02,
    x4): steps of uneven size over a positional trend, the structure the EPIKV write-up's z-score
    addresses. The recurrence runs over blocks of 64 tokens: inside a block as one product with the
    lower-triangular matrix of powers of rho, across blocks through the carried last row."""
    a = _randn((B, N), g, device)
    jump = torch.rand((B, N), generator=g, device=device) < 0.02
    pos = torch.arange(N, device=device, dtype=torch.float32) / max(N, 1)
    s = torch.exp(0.3 * a) * (1.0 + 0.5 * pos) * torch.where(jump, 4.0, 1.0)
    h = torch.empty((B, N, dm), dtype=torch.float32, device=device)
    T = 64
    k = torch.arange(T, device=device, dtype=torch.float32)
    expo = k[:, None] - k[None, :]
    A = torch.where(expo >= 0, rho ** expo.clamp(min=0), torch.zeros_like(expo))  # A[i, j] = rho^(i-j), j <= i
    decay = (rho ** (k + 1.0))[None, :, None]                                        # rho^(i+1)
    prev = torch.zeros((B, 1, dm), dtype=torch.float32, device=device)
    for t0 in range(0, N, T):
        n = min(T, N - t0)
        x = s[:, t0:t0 + n, None] * _randn((B, n, dm), g, device)
        blk = torch.matmul(A[:n, :n], x) + decay[:, :n] * prev
        h[:, t0:t0 + n] = blk
        prev = blk[:, -1:]
    return h


def make_epikv_inputs(name: str = "llama8b-epikv", device="cpu", seed: Optional[int] = None, **over) -> EpikvInputs:
    """Build the EPIKV workload, optionally with smaller sizes; ``keep`` overrides the kept total per
    sequence (default 7/8 of N)."""
    spec = dict(EPIKV_CONFIGS[name])
    keep = over.pop("keep", None)
    spec.update(over)
    if seed is not None:
        spec["seed"] = seed
    L, B, Hkv, D, N, dm = (spec[k] for k in ("L", "B", "Hkv", "D", "N", "dm"))
    dt = torch.bfloat16 if spec["dtype"] == "bf16" else torch.float32
    device = torch.device(device)
    g = _gen(device, spec["seed"])
    K = torch.empty((L, B, Hkv, N, D), dtype=dt, device=device)
    V = torch.empty((L, B, Hkv, N, D), dtype=dt, device=device)
    for l in range(L):
        K[l] = _randn((B, Hkv, N, D), g, device).to(dt)
        V[l] = _randn((B, Hkv, N, D), g, device).to(dt)
    hA = _residual_stream(B, N, dm, g, device).to(dt)
    hB = _residual_stream(B, N, dm, g, device).to(dt)
    return EpikvInputs(name=name, dtype=spec["dtype"], L=L, B=B, Hq=spec["Hq"], Hkv=Hkv, D=D, N=N, dm=dm,
                       window=int(spec["window"]), eps=float(spec["eps"]), prefix=spec["prefix"],
                       recent=spec["recent"], budget_all=(7 * N) // 8 if keep is None else int(keep), K=K, V=V,
                       hA=hA, hB=hB)
