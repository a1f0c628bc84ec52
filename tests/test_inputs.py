"""The seeded input generators (decoding_kv_cache_gb300/inputs.py) follow their stated recipes:
the same seed gives the same tensors, the shapes and storage types are the named models', and each
workload's distinguishing structure is present (per-channel key scales, heavy-tailed outlier
channels, planted keys, ReasonAlloc budgets). No GPU; reduced sizes except where a property needs
the full one."""
import math

import pytest
import torch

from decoding_kv_cache_gb300.inputs import CONFIGS, EPIKV_CONFIGS, make_epikv_inputs, make_inputs

SMALL = dict(L=2, B=1, N=600)


def _tensors(inp):
    out = {k: getattr(inp, k) for k in ("K", "V", "q_recent", "qbuf", "count")}
    if inp.budget is not None:
        out["budget"] = inp.budget
    return out


@pytest.mark.parametrize("name", list(CONFIGS))
def test_same_seed_same_inputs_and_named_shapes(name):
    a, b = make_inputs(name, **SMALL), make_inputs(name, **SMALL)
    for k, t in _tensors(a).items():
        assert torch.equal(t, _tensors(b)[k]), k
    c = make_inputs(name, seed=12345, **SMALL)
    assert not torch.equal(a.K, c.K)
    spec = CONFIGS[name]
    dt = torch.bfloat16 if spec["dtype"] == "bf16" else torch.float32
    L, B, N = SMALL["L"], SMALL["B"], SMALL["N"]
    assert a.K.shape == a.V.shape == (L, B, spec["Hkv"], N, spec["D"]) and a.K.dtype == dt
    assert a.q_recent.shape == (L, B, spec["Hq"], spec["n_r"], spec["D"]) and a.q_recent.dtype == dt
    assert a.qbuf.shape == (L, B, spec["Hq"], spec["qmax"], spec["D"])
    assert (a.count == spec["qmax"]).all() and a.t == N - 1
    if spec["cfg"] != 4:
        assert a.budget is None and a.budget_all == 7 * N // 8  # the 7/8 eviction


def test_qwen3_4b_keys_have_per_channel_scales():
    """Keys and values ~ N(0,1) times a per-(layer, KV head, channel) scale drawn from U(0.5, 2)."""
    inp = make_inputs("qwen3-4b", L=1, B=1, N=2048)
    sd = inp.K.float().std(dim=3).flatten()          # per (head, channel), over 2048 tokens
    assert sd.min() > 0.45 and sd.max() < 2.1
    assert sd.min() < 0.7 and sd.max() > 1.8          # the whole range is used
    vs = inp.V.float().std(dim=3).flatten()
    assert torch.allclose(sd, vs, rtol=0.15)          # the same scale multiplies V


def test_qwen3_14b_has_four_heavy_tailed_channels_per_head():
    """Four channels per (layer, KV head) are Student-t with 3 degrees of freedom: their sample
    kurtosis is far above the Gaussian 3 of the others."""
    inp = make_inputs("qwen3-14b-long", L=1, B=1, N=8192)
    k = inp.K.float()[0, 0]                           # [Hkv, N, D]
    kurt = ((k - k.mean(1, keepdim=True)) ** 4).mean(1) / k.var(1, unbiased=False) ** 2  # [Hkv, D]
    chan = inp.meta["outlier_channels"][0]            # [Hkv, 4]
    for h in range(k.shape[0]):
        out = set(chan[h].tolist())
        assert len(out) == 4
        assert all(kurt[h, c] > 6.0 for c in out)
        assert all(abs(kurt[h, c] - 3.0) < 0.6 for c in range(k.shape[2]) if c not in out)


def test_reasonalloc_budgets_follow_the_layer_profile():
    """Layer totals follow 1024 * (0.5 + sin(pi l / 27)) rescaled to average 1024, split over the
    heads by a Dirichlet(2) draw (rounded, clamped to [20, N])."""
    inp = make_inputs("qwen7b-reasonalloc", B=1, N=8192)
    b = inp.budget[:, 0].double()                     # [L, Hkv]
    L, H = b.shape
    prof = torch.tensor([1024.0 * (0.5 + math.sin(math.pi * l / 27.0)) for l in range(L)], dtype=torch.float64)
    prof *= 1024.0 / prof.mean()
    assert ((b >= 20) & (b <= 8192)).all()
    assert (b.sum(1) - H * prof).abs().max() <= H / 2 + 1e-9 + (b == 20).sum(1).max() * 20
    assert abs(b.mean().item() - 1024.0) < 4.0
    assert b.std(1).mean() > 50                        # the split is not uniform


def test_llama_planted_keys_lie_in_their_window():
    """64 planted keys per head at distinct sorted positions in [100, 450]."""
    inp = make_inputs("llama8b-planted", L=1, B=2, N=4096)
    p = inp.planted
    assert p.shape == (1, 2, 8, 64)
    assert (p >= 100).all() and (p <= 450).all()
    assert (p[..., 1:] > p[..., :-1]).all()


@pytest.mark.parametrize("name", list(EPIKV_CONFIGS))
def test_epikv_inputs_are_seeded(name):
    a = make_epikv_inputs(name, L=1, B=2, N=300, dm=256)
    b = make_epikv_inputs(name, L=1, B=2, N=300, dm=256)
    assert torch.equal(a.hA, b.hA) and torch.equal(a.hB, b.hB) and torch.equal(a.K, b.K)
    assert a.hA.shape == (2, 300, 256)
    assert not torch.equal(a.hA[:, 1:], a.hA[:, :-1])  # the residual stream moves between tokens
