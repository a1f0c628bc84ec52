"""Full-size workloads, in the launch configuration the benchmark times (one kvc_evict over
the whole cache), checked against the oracle on sampled heads. Inputs are generated on the
device; the sampled heads' inputs are copied to the host before the step runs."""
import dataclasses

import numpy as np
import pytest
import torch

from decoding_kv_cache_gb300.inputs import make_inputs
from oracle import oracle as O
from parity_util import assert_scores_close, check_beacon_picks, check_compaction, check_kept

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _head_problem(inp, l, b, h):
    """The (l, b, h) head of a device-resident problem as a 1x1x1 host problem."""
    G = inp.G
    qs = slice(h * G, (h + 1) * G)
    sub = lambda t: t[l:l + 1, b:b + 1].clone().cpu()
    return dataclasses.replace(
        inp, L=1, B=1, Hkv=1, Hq=G,
        K=inp.K[l:l + 1, b:b + 1, h:h + 1].clone().cpu(), V=inp.V[l:l + 1, b:b + 1, h:h + 1].clone().cpu(),
        q_recent=sub(inp.q_recent)[:, :, qs].contiguous(), qbuf=sub(inp.qbuf)[:, :, qs].contiguous(),
        count=sub(inp.count)[:, :, qs].contiguous(),
        budget=None if inp.budget is None else inp.budget[l:l + 1, b:b + 1, h:h + 1].clone().cpu(),
        planted=None, meta={})


@pytest.mark.parametrize("name", ["qwen3-4b", "llama8b-planted", "qwen7b-reasonalloc", "qwen3-14b-long"])
def test_fullsize_sampled_heads(name):
    from decoding_kv_cache_gb300 import kvc
    torch.cuda.empty_cache()
    inp = make_inputs(name, device=DEV)
    rng = np.random.default_rng(17)
    heads = sorted({0, inp.heads - 1, *rng.integers(0, inp.heads, 2).tolist()})
    locs = [(hd // (inp.B * inp.Hkv), (hd // inp.Hkv) % inp.B, hd % inp.Hkv) for hd in heads]
    probs = [_head_problem(inp, *loc) for loc in locs]

    cache = kvc.Cache(inp.K, inp.V, inp.Hq)
    kept_len = torch.zeros((inp.L, inp.B, inp.Hkv), dtype=torch.int32, device=DEV)
    kept_idx = torch.zeros((inp.L, inp.B, inp.Hkv, inp.N), dtype=torch.int32, device=DEV)
    scores = torch.zeros((inp.L, inp.B, inp.Hkv, inp.N), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_evict(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, inp.prefix, inp.recent,
                  kept_len, budget=inp.budget, budget_all=inp.budget_all, kept_idx=kept_idx, scores=scores,
                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    for (l, b, h), p in zip(locs, probs):
        gpu = dict(kept_len=kept_len[l:l + 1, b:b + 1, h:h + 1].cpu().numpy(),
                   kept_idx=kept_idx[l:l + 1, b:b + 1, h:h + 1].cpu().numpy(),
                   scores=scores[l:l + 1, b:b + 1, h:h + 1].cpu().numpy())
        ora = O.evict(p)
        # the beacons the GPU used for this head's query heads (score path, same inputs)
        sc_probe = torch.zeros((1, 1, 1, p.N), dtype=torch.float32, device=DEV)
        picks = torch.zeros((1, 1, p.Hq, p.n_b), dtype=torch.int32, device=DEV)
        pd = p.to(DEV)
        kvc.kvc_score(kvc.Cache(pd.K, pd.V, pd.Hq), pd.q_recent, pd.qbuf, pd.count, pd.n_b, pd.t, pd.theta,
                      sc_probe, beacon_picks=picks)
        torch.cuda.synchronize()
        gp = picks.cpu().numpy()
        if check_beacon_picks(p, gp, ora["beacon_picks"]):
            ora = O.evict(p, forced_picks=gp)
        assert_scores_close(gpu["scores"], ora["scores"], f"{name} head {(l, b, h)}")
        assert np.array_equal(sc_probe.cpu().numpy(), gpu["scores"]), "one head alone must score as in the batch"
        check_kept(p, gpu, ora, gpu["scores"])
        K_after = inp.K[l:l + 1, b:b + 1, h:h + 1].cpu()
        V_after = inp.V[l:l + 1, b:b + 1, h:h + 1].cpu()
        check_compaction(p, K_after, V_after, gpu["kept_idx"], gpu["kept_len"])
    del inp, cache, kept_idx, scores
    torch.cuda.empty_cache()
