"""Parity of the aggregation variants, the entropy output and the entropy-driven head budgets
(CUDA path through the C ABI) with the CPU oracle.

Cases cover every scoring kernel: the single-read kernel (128-row tiles, and 224-row tiles split
in two), the two-pass kernel (48-row query heads crossing the 128-row boundary, and a 128-row tile
over 50k keys), the fp32 path, a row count that is not a
multiple of 16 (each query head's rows then start on a 16-row boundary) and buffers holding
fewer rows than n_b (query heads with different row counts, so the mean's weights differ).
"""
import numpy as np
import pytest
import torch

from decoding_kv_cache_gb300.inputs import make_inputs
from oracle import oracle as O
from parity_util import (ENTROPY_ATOL, assert_scores_close, check_beacon_picks, check_compaction, check_kept,
                         run_evict, run_score)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    ("qwen3-4b", dict(L=2, N=1000)),                        # single-read kernel
    ("qwen3-4b", dict(L=1, N=700, n_b=8, qmax=16)),         # 24 rows per query head, stride 32
    ("qwen3-4b", dict(L=2, N=600, count=10)),               # 26 valid rows per query head
    ("qwen7b-reasonalloc", dict(L=1, B=2, N=1500)),          # 224 rows: two 128-row tiles
    ("qwen7b-reasonalloc", dict(L=1, B=1, N=5000)),          # two tiles, 20 CTAs per head
    ("qwen3-14b-long", dict(L=1, B=1, N=2100)),              # 48 rows per query head: variants cross
                                                             # tiles (two-pass kernel), max/max is tiled
    ("qwen3-4b", dict(L=1, Hq=4, Hkv=1, N=50000)),           # two-pass kernel, many keys per SM
    ("tiny", dict(N=1000, D=128)),                           # fp32 path
    ("tiny", dict(N=300, count=5)),                          # fp32, short buffers
]
MODES = [("mean", "max"), ("max", "sum"), ("mean", "sum"), ("max", "max")]


def _ids(c):
    return f"{c[0]}-" + "-".join(f"{k}{v}" for k, v in c[1].items())


def _oracle(inp, gpu_picks, **kw):
    ora = O.evict(inp, **kw)
    if check_beacon_picks(inp, gpu_picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=gpu_picks, **kw)
    return ora


@pytest.mark.parametrize("mode", MODES, ids=lambda m: ",".join(m))
@pytest.mark.parametrize("name,over", CASES, ids=[_ids(c) for c in CASES])
def test_variants_match_oracle(name, over, mode):
    inp = make_inputs(name, **over)
    gpu = run_evict(inp, DEV, row_agg=mode[0], group_agg=mode[1], entropy=True)
    _, picks = run_score(inp, DEV)
    ora = _oracle(inp, picks, row_agg=mode[0], group_agg=mode[1])
    assert gpu["status"] == 0
    assert_scores_close(gpu["scores"], ora["scores"], f"{name} {mode}")
    np.testing.assert_allclose(gpu["entropy"], ora["entropy"], rtol=0, atol=ENTROPY_ATOL)
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


def test_score_entry_point_variants_and_entropy():
    inp = make_inputs("qwen3-4b", L=2, N=900)
    for mode in MODES:
        scores, picks, ent = run_score(inp, DEV, row_agg=mode[0], group_agg=mode[1], entropy=True)
        ora = _oracle(inp, picks, row_agg=mode[0], group_agg=mode[1])
        assert_scores_close(scores, ora["scores"], f"kvc_score {mode}")
        np.testing.assert_allclose(ent, ora["entropy"], rtol=0, atol=ENTROPY_ATOL)


def test_default_options_are_the_plain_step():
    """An all-default options struct changes nothing: same scores, bit for bit."""
    inp = make_inputs("qwen3-4b", L=2, N=1000)
    a = run_evict(inp, DEV)
    b = run_evict(inp, DEV, row_agg="max", group_agg="max")
    assert np.array_equal(a["scores"], b["scores"]) and np.array_equal(a["kept_idx"], b["kept_idx"])


@pytest.mark.parametrize("name,over", [
    ("qwen3-4b", dict(L=2, B=2, N=1000)),
    ("qwen7b-reasonalloc", dict(L=2, B=2, N=1500)),  # per-head given budgets (the layer totals)
    ("tiny", dict(L=2, B=3, N=500)),
], ids=lambda x: x if isinstance(x, str) else "-".join(f"{k}{v}" for k, v in x.items()))
def test_entropy_budgets_match_oracle(name, over):
    inp = make_inputs(name, **over)
    gpu = run_evict(inp, DEV, head_budget="entropy", entropy=True)
    _, picks = run_score(inp, DEV)
    ora = _oracle(inp, picks, head_budget="entropy")
    np.testing.assert_allclose(gpu["entropy"], ora["entropy"], rtol=0, atol=ENTROPY_ATOL)
    assert gpu["status"] == 0
    # The oracle's rule applied to the GPU's own fp32 entropies: exactly the GPU's budgets (the
    # integer reallocation after the fixed-point weights is exact arithmetic on both sides).
    forced = _oracle(inp, picks, head_budget="entropy", forced_entropy=gpu["entropy"])
    assert np.array_equal(gpu["kept_len"], np.minimum(forced["budget_used"], inp.N))
    # Against the budgets the oracle takes from its OWN entropies: equal, except in a (layer,
    # sequence) where some head's fixed-point weight floor((1 - entropy) * 2^24) differs between
    # the two entropy sets (both within ENTROPY_ATOL of each other), which is where a rounding
    # difference in an entropy can move a slot from one head to another.
    own = np.minimum(ora["budget_used"], inp.N)
    moved = 0
    for l in range(inp.L):
        for b in range(inp.B):
            if np.array_equal(gpu["kept_len"][l, b], own[l, b]):
                continue
            assert (_weights(gpu["entropy"][l, b]) != _weights(ora["entropy"][l, b])).any(), (
                f"budgets differ at {(l, b)} with identical fixed-point weights")
            assert gpu["kept_len"][l, b].sum() == own[l, b].sum()
            moved += 1
    assert moved <= (inp.L * inp.B) // 2, f"{moved} of {inp.L * inp.B} (layer, sequence) groups differ"
    given = inp.budgets().cpu().numpy()
    assert np.array_equal(gpu["kept_len"].sum(-1), np.minimum(given, inp.N).sum(-1))  # layer totals kept
    assert_scores_close(gpu["scores"], ora["scores"], name)
    check_kept(inp, gpu, forced, gpu["scores"], budgets=forced["budget_used"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])
    # the entropy output is optional: without it the workspace holds the entropies
    gpu2 = run_evict(inp, DEV, head_budget="entropy")
    assert np.array_equal(gpu2["kept_len"], gpu["kept_len"])


def _weights(ent):
    """The head-budget rule's fixed-point utilities floor(clip(1 - entropy, 0, 1) * 2^24), in fp64."""
    u = np.clip(1.0 - np.asarray(ent, dtype=np.float32).astype(np.float64), 0.0, 1.0)
    return np.floor(u * 16777216.0).astype(np.int64)


@pytest.mark.parametrize("seed", range(6))
def test_head_budget_entry_point_is_exact(seed):
    from decoding_kv_cache_gb300 import kvc
    rng = np.random.default_rng(seed)
    L, B, Hkv = 3, 4, int(rng.choice([2, 4, 8, 40]))
    N, P, R = int(rng.integers(100, 5000)), 4, 16
    if seed % 3 == 0:  # ties: equal entropies, equal remainders
        ent = np.repeat(rng.choice([0.3, 0.7, 1.0], (L, B, 1)), Hkv, -1).astype(np.float32)
    else:
        ent = rng.uniform(0.2, 1.0, (L, B, Hkv)).astype(np.float32)
    given = rng.integers(P + R, N + N // 4, (L, B, Hkv)).astype(np.int32)
    if seed == 5:
        given[1, 2, 0] = P + R - 1  # that layer keeps its given budgets and is flagged
    out = torch.full((L, B, Hkv), -7, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_head_budget(torch.from_numpy(ent).to(DEV), N, P, R, out, budget=torch.from_numpy(given).to(DEV),
                        status=status)
    got = out.cpu().numpy()
    for l in range(L):
        for b in range(B):
            want = O.head_budget(ent[l, b], N, P, R, given[l, b])
            assert got[l, b].tolist() == (given[l, b] if want is None else want).tolist(), (l, b)
    assert int(status.item()) == (kvc.KVC_STATUS_BUDGET_RANGE if seed == 5 else 0)
    # a uniform budget and an output aliasing the input
    inplace = torch.from_numpy(given).to(DEV)
    kvc.kvc_head_budget(torch.from_numpy(ent).to(DEV), N, P, R, inplace, budget=inplace)
    assert np.array_equal(inplace.cpu().numpy(), got)
    kvc.kvc_head_budget(torch.from_numpy(ent).to(DEV), N, P, R, out, budget_all=N // 2)
    for l in range(L):
        for b in range(B):
            assert out[l, b].cpu().tolist() == O.head_budget(ent[l, b], N, P, R, [N // 2] * Hkv).tolist()
