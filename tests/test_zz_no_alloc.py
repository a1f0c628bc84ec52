"""kvc_score_static: the scoring entry point for callers that cannot allocate device memory
(a runtime that reserved all memory for weights and its KV pool up front, or code running
where allocation is not allowed). Its scratch is a fixed region the library reserves when
it loads, so it must give the same scores as kvc_score with a caller workspace and as the
oracle, call after call, whatever an earlier call left in the region, and reject problems
too big for the region before launching anything.

Collected last on purpose: if it fails, a run that stops at the first failure has already
run everything else. It passes alone in a fresh process and after the other tests."""
import numpy as np
import pytest
import torch

from decoding_kv_cache_gb300.inputs import make_inputs
from oracle import oracle as O
from parity_util import ENTROPY_ATOL, assert_scores_close, check_beacon_picks

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _scores_with_workspace(kvc, inp, cache):
    out = torch.full((inp.L, inp.B, inp.Hkv, inp.N), -1.0, device=DEV)
    kvc.kvc_score(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, out)
    return out


def _static(kvc, inp, cache, row_agg="max", group_agg="max", entropy=False):
    """One kvc_score_static call; returns scores, beacon picks and (optionally) entropies on the host."""
    out = torch.full((inp.L, inp.B, inp.Hkv, inp.N), -1.0, device=DEV)
    picks = torch.full((inp.L, inp.B, inp.Hq, inp.n_b), -7, dtype=torch.int32, device=DEV)
    ent = torch.full((inp.L, inp.B, inp.Hkv), -1.0, device=DEV) if entropy else None
    kvc.kvc_score_static(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, out,
                         beacon_picks=picks, row_agg=row_agg, group_agg=group_agg, entropy=ent)
    torch.cuda.synchronize()
    return out.cpu().numpy(), picks.cpu().numpy(), None if ent is None else ent.cpu().numpy()


@pytest.mark.parametrize("name,over", [("qwen3-4b", dict(L=2, N=1000)), ("qwen3-14b-long", dict(L=1, B=1, N=700)),
                                       ("tiny", {})])
def test_static_scratch_matches_workspace_path_twice(name, over):
    from decoding_kv_cache_gb300 import kvc
    inp = make_inputs(name, device=DEV, **over)
    cache = kvc.Cache(inp.K, inp.V, inp.Hq)
    ref = _scores_with_workspace(kvc, inp, cache)
    for _ in range(2):  # the region keeps the previous call's contents; results must not depend on them
        got = torch.full_like(ref, -1.0)
        kvc.kvc_score_static(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, got)
        torch.cuda.synchronize()
        assert_scores_close(got.cpu().numpy(), ref.cpu().numpy(), f"static scratch, {name}")


# Consecutive calls on different problems: each checked call finds the region holding another
# problem's observation tiles, exchange words and partials (in the default or the extended
# options' layout), and must still match the oracle.
SEQUENCE = [
    ("qwen3-4b", dict(L=1, N=900, seed=11), dict(row_agg="mean", group_agg="sum", entropy=True)),
    ("qwen3-4b", dict(L=2, N=1000), {}),
    ("qwen3-14b-long", dict(L=1, B=1, N=700, seed=12), {}),
    ("qwen3-4b", dict(L=2, N=1000, seed=13), dict(entropy=True)),
    ("tiny", {}, dict(row_agg="mean")),
    ("tiny", dict(N=500, seed=15), {}),  # the fp32 cluster kernel (no observation tiles in the region)
    ("qwen3-4b", dict(L=1, N=1500, seed=14), {}),
]


def test_static_scratch_matches_oracle_call_after_call():
    from decoding_kv_cache_gb300 import kvc
    for i, (name, over, opts) in enumerate(SEQUENCE):
        cpu = make_inputs(name, **over)
        g = cpu.to(DEV)
        cache = kvc.Cache(g.K, g.V, g.Hq)
        sc, picks, ent = _static(kvc, g, cache, **opts)
        ora_kw = {k: v for k, v in opts.items() if k != "entropy"}
        ora = O.evict(cpu, **ora_kw)
        if check_beacon_picks(cpu, picks, ora["beacon_picks"]):  # a valid near-tie alternative
            ora = O.evict(cpu, forced_picks=picks, **ora_kw)
        assert_scores_close(sc, ora["scores"], f"static scratch call {i}: {name} {opts}")
        if ent is not None:
            np.testing.assert_allclose(ent, ora["entropy"], rtol=0, atol=ENTROPY_ATOL)


def test_static_scratch_rejects_problems_beyond_its_size():
    from decoding_kv_cache_gb300 import kvc
    inp = make_inputs("llama8b-planted", device=DEV, L=8, B=8, N=256)  # 512 KV heads of 32 KB tiles: > 16 MB
    cache = kvc.Cache(inp.K, inp.V, inp.Hq)
    assert kvc.kvc_score_workspace_size(cache, inp.n_r, inp.n_b) > kvc.KVC_STATIC_SCRATCH_BYTES
    out = torch.full((inp.L, inp.B, inp.Hkv, inp.N), -1.0, device=DEV)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_score_static(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, out)
    assert e.value.code == -7
    torch.cuda.synchronize()
    assert (out == -1.0).all()  # nothing was launched
