"""Helpers for comparing the CUDA path (through the C ABI) with the CPU oracle.

Tolerances: scores |gpu - oracle| <= 1e-3 * |oracle| + 1e-30 (every aggregation variant);
normalised entropy |gpu - oracle| <= 1e-4 absolute; kept sets identical except
where both swapped indices' oracle scores lie within 1e-5 (relative) of the oracle's
threshold score; FPS picks identical except at distance near-ties within 1e-5; compacted
K/V bit-exact against a gather with the GPU's own kept indices.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O

SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-30
TIE_RTOL = 1e-5
FPS_TOL = 1e-5
# The entropy is a mean over rows of -sum p log2 p / log2 N, a number in [0, 1]. The kernels
# take p from exp2 of fp32 logits (relative error ~1e-6 in s and lse2 against fp64, ~2^-22 in
# exp2) and sum ~1e5 to 1e7 terms in fp32 per head; 1e-4 absolute covers both with margin.
ENTROPY_ATOL = 1e-4


def storage_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def run_evict(inp, dev, with_scores=True, row_agg="max", group_agg="max", head_budget="given", entropy=False,
              kernel="auto"):
    """kvc_evict on a device copy of ``inp``; returns numpy results and the compacted cache.
    ``entropy=True`` also returns the per-head normalised entropy output."""
    from decoding_kv_cache_gb300 import kvc
    g = inp.to(dev)
    cache = kvc.Cache(g.K, g.V, g.Hq)
    kept_len = torch.full((g.L, g.B, g.Hkv), -7, dtype=torch.int32, device=dev)
    kept_idx = torch.full((g.L, g.B, g.Hkv, g.N), -7, dtype=torch.int32, device=dev)
    scores = torch.full((g.L, g.B, g.Hkv, g.N), -1.0, dtype=torch.float32, device=dev) if with_scores else None
    ent = torch.full((g.L, g.B, g.Hkv), -1.0, dtype=torch.float32, device=dev) if entropy else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvc.kvc_evict(cache, g.q_recent, g.qbuf, g.count, g.n_b, g.t, g.theta, g.prefix, g.recent, kept_len,
                  budget=g.budget, budget_all=g.budget_all, kept_idx=kept_idx, scores=scores, status=status,
                  row_agg=row_agg, group_agg=group_agg, head_budget=head_budget, entropy=ent, kernel=kernel)
    torch.cuda.synchronize()
    return dict(kept_len=kept_len.cpu().numpy(), kept_idx=kept_idx.cpu().numpy(),
                scores=None if scores is None else scores.cpu().numpy(), status=int(status.item()),
                K=g.K.cpu(), V=g.V.cpu(), entropy=None if ent is None else ent.cpu().numpy())


def run_score(inp, dev, row_agg="max", group_agg="max", entropy=False, kernel="auto"):
    from decoding_kv_cache_gb300 import kvc
    g = inp.to(dev)
    cache = kvc.Cache(g.K, g.V, g.Hq)
    scores = torch.full((g.L, g.B, g.Hkv, g.N), -1.0, dtype=torch.float32, device=dev)
    picks = torch.full((g.L, g.B, g.Hq, max(g.n_b, 1)), -7, dtype=torch.int32, device=dev)[..., :g.n_b].contiguous()
    ent = torch.full((g.L, g.B, g.Hkv), -1.0, dtype=torch.float32, device=dev) if entropy else None
    kvc.kvc_score(cache, g.q_recent, g.qbuf, g.count, g.n_b, g.t, g.theta, scores,
                  beacon_picks=picks if g.n_b else None, row_agg=row_agg, group_agg=group_agg, entropy=ent,
                  kernel=kernel)
    torch.cuda.synchronize()
    if entropy:
        return scores.cpu().numpy(), picks.cpu().numpy(), ent.cpu().numpy()
    return scores.cpu().numpy(), picks.cpu().numpy()


def assert_scores_close(gpu: np.ndarray, ora: np.ndarray, what=""):
    assert gpu.shape == ora.shape
    err = np.abs(gpu.astype(np.float64) - ora.astype(np.float64))
    bound = SCORE_RTOL * np.abs(ora.astype(np.float64)) + SCORE_FLOOR
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / np.maximum(bound, 1e-300), 0)), gpu.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} scores out of tolerance; worst at {i}: gpu {gpu[i]!r} "
                             f"oracle {ora[i]!r}")


def check_beacon_picks(inp, gpu_picks: np.ndarray, ora_picks: np.ndarray):
    """Identical picks, or a valid near-tie alternative. Returns True if any differ."""
    differ = False
    L, B, Hq = inp.L, inp.B, inp.Hq
    for l in range(L):
        for b in range(B):
            for hq in range(Hq):
                gp, op = gpu_picks[l, b, hq], ora_picks[l, b, hq]
                if np.array_equal(gp, op):
                    continue
                differ = True
                cnt = int(inp.count[l, b, hq])
                x = storage_to_f64(inp.qbuf[l, b, hq, :cnt])
                sel = gp[gp >= 0]
                assert len(sel) == len(op[op >= 0]), f"beacon count differs at {(l, b, hq)}"
                assert O.fps_check(x, sel, FPS_TOL) == 0, f"GPU beacons at {(l, b, hq)} are not a greedy FPS result"
    return differ


def check_kept(inp, gpu, ora, gpu_scores, budgets=None):
    """Kept lists: invariants against the GPU's own scores (exact) and agreement with the oracle
    up to near-ties. ``budgets`` [L,B,Hkv] overrides the input's (reallocated budgets)."""
    N, P, R = inp.N, inp.prefix, inp.recent
    budgets = inp.budgets().cpu().numpy() if budgets is None else budgets
    L, B, Hkv = inp.L, inp.B, inp.Hkv
    for l in range(L):
        for b in range(B):
            for h in range(Hkv):
                n = int(gpu["kept_len"][l, b, h])
                assert n == int(ora["kept_len"][l, b, h]), f"kept_len differs at {(l, b, h)}"
                gk = gpu["kept_idx"][l, b, h, :n]
                ok = ora["kept_idx"][l, b, h, :n]
                assert (np.diff(gk) > 0).all() and gk[0] >= 0 and gk[-1] < N
                bud = int(budgets[l, b, h])
                if bud >= N or bud < P + R:
                    assert np.array_equal(gk, np.arange(N))
                    continue
                assert set(range(min(P, N))) <= set(gk.tolist()) and set(range(N - R, N)) <= set(gk.tolist())
                s = gpu_scores[l, b, h].view(np.uint32)
                keep = np.zeros(N, bool)
                keep[gk] = True
                mid = np.zeros(N, bool)
                mid[P:N - R] = True
                km, dm = mid & keep, mid & ~keep
                if km.any() and dm.any():
                    assert s[dm].max() <= s[km].min(), f"a dropped score beats a kept one at {(l, b, h)}"
                    t = s[km].min()
                    if s[dm].max() == t:  # ties at the threshold keep the lower indices
                        assert np.flatnonzero(km & (s == t)).max() < np.flatnonzero(dm & (s == t)).min()
                if not np.array_equal(gk, ok):
                    os_ = ora["scores"][l, b, h].astype(np.float64)
                    kmid = bud - P - R
                    thr = np.sort(os_[P:N - R])[::-1][kmid - 1]
                    sym = np.setxor1d(gk, ok)
                    far = np.abs(os_[sym] - thr) > TIE_RTOL * thr
                    assert not far.any(), (f"kept sets differ beyond near-ties at {(l, b, h)}: "
                                           f"{sym[far][:8]} scores {os_[sym[far]][:8]} thr {thr}")


def check_compaction(inp, gpu_after_K, gpu_after_V, kept_idx, kept_len):
    """Bit-exact: rows [0, len) are the gather of the GPU's kept list, rows past it untouched."""
    for before, after in ((inp.K, gpu_after_K), (inp.V, gpu_after_V)):
        bb = before.view(torch.int16) if before.dtype == torch.bfloat16 else before.view(torch.int32)
        aa = after.view(torch.int16) if after.dtype == torch.bfloat16 else after.view(torch.int32)
        for l in range(inp.L):
            for b in range(inp.B):
                for h in range(inp.Hkv):
                    n = int(kept_len[l, b, h])
                    idx = torch.from_numpy(kept_idx[l, b, h, :n].astype(np.int64))
                    assert torch.equal(aa[l, b, h, :n], bb[l, b, h, idx]), f"compacted rows differ at {(l, b, h)}"
                    assert torch.equal(aa[l, b, h, n:], bb[l, b, h, n:]), f"tail rows changed at {(l, b, h)}"


def full_check(inp, dev, heads_subset=None):
    """kvc_evict vs the oracle on every head (or a subset of flat head ids)."""
    gpu = run_evict(inp, dev)
    ora = O.evict(inp, heads=heads_subset)
    return gpu, ora
