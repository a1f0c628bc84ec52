"""Parity of the EPIKV path (hidden-state change, rolling z-score, per-sequence selection,
compaction of every head) with the oracle, through the C ABI.

Tolerances (the arithmetic they come from):
- the signal g: the kernel sums ~dm squared differences in fp32 (bf16 differences are exact in
  fp32), the oracle in fp64: |gpu - oracle| <= 1e-5 |oracle| + 1e-6;
- the score from the GPU's own signal: the kernel forms the window's mean and variance in fp64 from
  prefix sums (the oracle by direct sums; the two agree to ~1e-12), then sigma, g - mu and the
  quotient in fp32 (~3e-7 relative) and z_A - z_B in fp32 (~1e-6 absolute at |z| ~ 10):
  |gpu - z(g_gpu)| <= 2e-6 |z| + 1e-5;
- the score against the oracle's OWN score, element by element: the bound above plus the signal's
  error carried through the z-score. With dg = |g_gpu - g_oracle| per token and m the largest dg
  in the token's window, the window mean moves by at most m and the population deviation by at
  most m (it is 1-Lipschitz in the largest entry change), so per layer
  |dz| <= (dg + m + |z| m) / (sigma + eps), and the score z_A - z_B adds the two layers' bounds;
- kept lists: identical to the oracle's selection applied to the GPU's own fp32 scores (selection
  is exact given the scores); against the oracle's own scores, a swap is allowed only between
  tokens whose oracle scores lie within their two error bounds (as above) of the threshold score.
  That window is the score's propagated fp32 error, which is larger than a gap of 1e-5 relative to
  the threshold: the signal's fp32 sum alone moves z by ~1e-6..1e-5;
- compaction: bit-exact gather of every head of a sequence with that sequence's kept list.
"""
import numpy as np
import pytest
import torch

from decoding_kv_cache_gb300.inputs import make_epikv_inputs
from oracle import oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
G_RTOL, G_ATOL = 1e-5, 1e-6
Z_RTOL, Z_ATOL = 2e-6, 1e-5


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _run_score(hA, hB, window, eps):
    from decoding_kv_cache_gb300 import kvc
    B, N, _ = hA.shape
    g = torch.full((2, B, N), -1.0, device=DEV)
    sc = torch.full((B, N), -7.0, device=DEV)
    kvc.kvc_epikv_score(hA.to(DEV), hB.to(DEV), window, eps, sc, g=g)
    torch.cuda.synchronize()
    return g.cpu().numpy(), sc.cpu().numpy()


def _window_stats(g, window):
    """Per token t >= 1 of g [..., N] (fp64): population deviation of the causal window
    max(1, t-W+1)..t, and the window's first token index; token 0 lies in no window."""
    N = g.shape[-1]
    t = np.arange(N)
    a = np.maximum(1, t - window + 1)
    c1 = np.concatenate([np.zeros(g.shape[:-1] + (1,)), np.cumsum(g, -1)], -1)
    c2 = np.concatenate([np.zeros(g.shape[:-1] + (1,)), np.cumsum(g * g, -1)], -1)
    n = np.maximum(t - a + 1, 1)
    mu = (c1[..., t + 1] - c1[..., a]) / n
    var = np.maximum((c2[..., t + 1] - c2[..., a]) / n - mu * mu, 0.0)
    return np.sqrt(var), a


def _score_error_bound(g, og, osc_layers, window, eps):
    """Element-wise bound on |score_gpu - score_oracle| [B, N] from the signals' error (see the
    module docstring); osc_layers [2, B, N] are the oracle's per-layer z-scores."""
    dg = np.abs(g.astype(np.float64) - og)
    sigma, a = _window_stats(og, window)
    N = g.shape[-1]
    m = np.zeros_like(dg)
    for t in range(1, N):  # largest signal error in the window
        m[..., t] = dg[..., a[t]:t + 1].max(-1)
    z = np.abs(osc_layers)
    per_layer = (dg + m + z * m) / (sigma + eps) + Z_RTOL * z + Z_ATOL
    per_layer[..., 0] = 0.0
    return per_layer.sum(0)


def _oracle_layer_z(og, window, eps):
    """The oracle's per-layer z-scores: z-scores of (g_A, 0) and (0, g_B) give z_A and -z_B."""
    zA = O.epikv_z(np.stack([og[0], np.zeros_like(og[1])]), window, eps)
    zB = -O.epikv_z(np.stack([np.zeros_like(og[0]), og[1]]), window, eps)
    return np.stack([zA, zB])


def _check_scores(hA, hB, window, eps, dtype):
    g, sc = _run_score(hA, hB, window, eps)
    og, osc = O.epikv_score(_bits(hA), _bits(hB), window, eps, dtype)
    np.testing.assert_allclose(g, og, rtol=G_RTOL, atol=G_ATOL)
    z = O.epikv_z(g.astype(np.float64), window, eps)
    np.testing.assert_allclose(sc, z, rtol=Z_RTOL, atol=Z_ATOL)
    # against the oracle's own scores, element by element, within the propagated bound
    bound = _score_error_bound(g, og, _oracle_layer_z(og, window, eps), window, eps)
    err = np.abs(sc.astype(np.float64) - osc)
    assert (err <= bound).all(), f"worst excess {np.max(err - bound)} at {np.unravel_index(np.argmax(err - bound), err.shape)}"
    return g, sc, og, osc, bound


@pytest.mark.parametrize("dtype,dm", [("bf16", 64), ("bf16", 4096), ("bf16", 8192), ("f32", 1024), ("f32", 4096),
                                      ("bf16", 200)])
@pytest.mark.parametrize("window", [1, 16, 128, 5000])
def test_epikv_score_matches_oracle(dtype, dm, window):
    """Ragged token counts (not a multiple of the 32-token blocks nor of the 1024-token scan
    tiles), every register width of the signal kernel, windows from 1 to longer than the cache."""
    inp = make_epikv_inputs(L=1, B=2, N=1100, dm=dm, dtype=dtype, seed=dm + window)
    g, sc, og, osc, _ = _check_scores(inp.hA, inp.hB, window, 1e-6, dtype)
    assert (g[:, :, 0] == 0).all() and (sc[:, 0] == 0).all()
    if window == 1:  # every window holds one token: sigma 0, z 0
        assert (sc == 0).all()


def test_epikv_score_end_to_end_tolerance():
    """Against the oracle's own scores: the fp32 signal's error carried through the z-score stays
    inside its element-wise bound, and that bound is small next to the scores' spread."""
    inp = make_epikv_inputs(L=1, B=3, N=700, dm=1024)
    _, sc, _, osc, bound = _check_scores(inp.hA, inp.hB, inp.window, inp.eps, "bf16")
    assert np.median(bound[:, 1:]) < 1e-4 and np.abs(sc - osc).max() < 1e-3


@pytest.mark.parametrize("over", [dict(L=2, B=3, N=300, dm=256, D=64, Hkv=2, Hq=4),
                                  dict(L=1, B=2, N=1500, dm=512, D=128, Hkv=4, Hq=8, keep=700),
                                  dict(L=2, B=1, N=129, dm=64, D=128, Hkv=1, Hq=2, keep=129)])
def test_epikv_evict_matches_oracle(over):
    from decoding_kv_cache_gb300 import kvc
    inp = make_epikv_inputs(**over)
    g = inp.to(DEV)
    cache = kvc.Cache(g.K, g.V, g.Hq)
    kept_len = torch.full((g.B,), -7, dtype=torch.int32, device=DEV)
    kept_idx = torch.full((g.B, g.N), -7, dtype=torch.int32, device=DEV)
    scores = torch.full((g.B, g.N), -7.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_epikv_evict(cache, g.hA, g.hB, g.window, g.eps, g.prefix, g.recent, kept_len, budget_all=g.budget_all,
                        kept_idx=kept_idx, scores=scores, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sc, kl, ki = scores.cpu().numpy(), kept_len.cpu().numpy(), kept_idx.cpu().numpy()
    og, osc = O.epikv_score(_bits(inp.hA), _bits(inp.hB), inp.window, inp.eps, inp.dtype)
    gg, _ = _run_score(inp.hA, inp.hB, inp.window, inp.eps)
    bound = _score_error_bound(gg, og, _oracle_layer_z(og, inp.window, inp.eps), inp.window, inp.eps)
    K1, V1 = g.K.cpu(), g.V.cpu()
    for b in range(inp.B):
        mine = O.select(sc[b].astype(np.float32), inp.prefix, inp.recent, inp.budget_all)
        assert kl[b] == len(mine) and np.array_equal(ki[b, :kl[b]], mine), f"sequence {b}"
        ref = O.select(osc[b].astype(np.float32), inp.prefix, inp.recent, inp.budget_all)
        if not np.array_equal(mine, ref):
            kmid = inp.budget_all - inp.prefix - inp.recent
            mid = np.arange(inp.prefix, inp.N - inp.recent)
            order = mid[np.lexsort((mid, -osc[b, mid]))]
            jt = order[kmid - 1]  # the token holding the oracle's threshold score
            thr = osc[b, jt]
            sym = np.setxor1d(mine, ref)
            assert (np.abs(osc[b, sym] - thr) <= bound[b, sym] + bound[b, jt]).all(), (b, sym, osc[b, sym], thr)
        idx = torch.from_numpy(mine.astype(np.int64))
        n = len(mine)
        for before, after in ((inp.K, K1), (inp.V, V1)):
            bb = before.view(torch.int16) if before.dtype == torch.bfloat16 else before.view(torch.int32)
            aa = after.view(torch.int16) if after.dtype == torch.bfloat16 else after.view(torch.int32)
            for l in range(inp.L):
                for h in range(inp.Hkv):
                    assert torch.equal(aa[l, b, h, :n], bb[l, b, h, idx]), (l, b, h)
                    assert torch.equal(aa[l, b, h, n:], bb[l, b, h, n:]), (l, b, h)


def test_epikv_full_size_sampled():
    """The R1-Distill-Llama-8B-shaped workload at full size (16 sequences x 4096 tokens, hidden size
    4096) in the launch configuration the benchmark times: signals and scores of three sequences
    against the oracle, the kept lists of every sequence against the oracle's selection on the
    GPU's scores."""
    from decoding_kv_cache_gb300 import kvc
    inp = make_epikv_inputs(device=DEV)
    cache = kvc.Cache(inp.K, inp.V, inp.Hq)
    kept_len = torch.zeros((inp.B,), dtype=torch.int32, device=DEV)
    kept_idx = torch.zeros((inp.B, inp.N), dtype=torch.int32, device=DEV)
    scores = torch.zeros((inp.B, inp.N), device=DEV)
    g = torch.zeros((2, inp.B, inp.N), device=DEV)
    kvc.kvc_epikv_score(inp.hA, inp.hB, inp.window, inp.eps, scores, g=g)
    kvc.kvc_epikv_evict(cache, inp.hA, inp.hB, inp.window, inp.eps, inp.prefix, inp.recent, kept_len,
                        budget_all=inp.budget_all, kept_idx=kept_idx)
    torch.cuda.synchronize()
    gg, sc = g.cpu().numpy(), scores.cpu().numpy()
    for b in (0, 7, inp.B - 1):
        og, osc = O.epikv_score(_bits(inp.hA[b:b + 1]), _bits(inp.hB[b:b + 1]), inp.window, inp.eps, inp.dtype)
        np.testing.assert_allclose(gg[:, b:b + 1], og, rtol=G_RTOL, atol=G_ATOL)
        np.testing.assert_allclose(sc[b:b + 1], O.epikv_z(gg[:, b:b + 1].astype(np.float64), inp.window, inp.eps),
                                   rtol=Z_RTOL, atol=Z_ATOL)
    kl, ki = kept_len.cpu().numpy(), kept_idx.cpu().numpy()
    for b in range(inp.B):
        mine = O.select(sc[b].astype(np.float32), inp.prefix, inp.recent, inp.budget_all)
        assert kl[b] == len(mine) and np.array_equal(ki[b, :kl[b]], mine)
