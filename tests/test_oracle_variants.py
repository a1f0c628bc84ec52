"""Pins for the oracle's aggregation variants, attention entropy and head-budget reallocation.

Hand-worked cases (tests/golden), closed forms, invariants and brute force, so that a dropped
term, a swapped mode or a wrong index in the oracle fails here. No GPU is needed.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O
from decoding_kv_cache_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MODES = [("max", "max"), ("mean", "max"), ("max", "sum"), ("mean", "sum")]


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# aggregation variants and entropy
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden("agg_entropy_handworked.json")["cases"], ids=lambda c: c["name"])
@pytest.mark.parametrize("mode", MODES, ids=lambda m: ",".join(m))
def test_agg_handworked(case, mode):
    s, ent = O.score_agg(np.array(case["q"]), case["row_head"], case["G"], np.array(case["k"]), *mode)
    want = [float(Fraction(v[0])) for v in case["scores"][",".join(mode)]]
    np.testing.assert_allclose(s, want, rtol=1e-14, atol=0)
    N = len(case["k"])
    np.testing.assert_allclose(ent, np.mean(case["row_entropy_bits"]) / math.log2(N), rtol=1e-13)


def _rand_problem(seed, M=12, G=3, N=40, D=8, scale=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((M, D)) * scale
    k = rng.standard_normal((N, D)) * scale
    rh = np.sort(rng.integers(0, G, M))
    return q, rh, G, k


@pytest.mark.parametrize("seed", range(4))
def test_agg_max_max_is_the_plain_score(seed):
    q, rh, G, k = _rand_problem(seed)
    s, _ = O.score_agg(q, rh, G, k, "max", "max")
    np.testing.assert_array_equal(s, O.score(q, k))


@pytest.mark.parametrize("seed", range(4))
def test_agg_invariants(seed):
    q, rh, G, k = _rand_problem(seed, scale=1.5)
    S = {m: O.score_agg(q, rh, G, k, *m)[0] for m in MODES}
    heads_with_rows = len(set(rh.tolist()))
    # each mean-over-rows head contributes a distribution: the sum over heads sums to #heads
    assert abs(S[("mean", "sum")].sum() - heads_with_rows) < 1e-12
    # a max over heads of distributions: between one distribution's mass and #heads
    assert 1.0 - 1e-12 <= S[("mean", "max")].sum() <= heads_with_rows + 1e-12
    eps = 1e-15
    assert np.all(S[("mean", "max")] <= S[("max", "max")] + eps)
    assert np.all(S[("max", "max")] <= S[("max", "sum")] + eps)
    assert np.all(S[("mean", "sum")] <= S[("max", "sum")] + eps)
    assert np.all(S[("mean", "max")] <= S[("mean", "sum")] + eps)
    # every score of a sum over heads is at most the number of heads; of a max at most 1
    assert S[("max", "sum")].max() <= heads_with_rows and S[("max", "max")].max() <= 1.0


def test_agg_degenerate_cases():
    q, rh, G, k = _rand_problem(7, M=6, G=1)
    # one head: summing over heads is the max over heads
    for r in ("max", "mean"):
        np.testing.assert_array_equal(O.score_agg(q, rh, 1, k, r, "sum")[0], O.score_agg(q, rh, 1, k, r, "max")[0])
    # one row per head: mean over rows is the max over rows
    q1, k1 = q[:3], k
    rh1 = [0, 1, 2]
    for gm in ("max", "sum"):
        np.testing.assert_allclose(O.score_agg(q1, rh1, 3, k1, "mean", gm)[0], O.score_agg(q1, rh1, 3, k1, "max", gm)[0],
                                   rtol=1e-15)
    # identical heads: summing G copies is G times one
    qq = np.concatenate([q[:2]] * 3)
    rr = [0, 0, 1, 1, 2, 2]
    np.testing.assert_allclose(O.score_agg(qq, rr, 3, k, "mean", "sum")[0], 3 * O.score_agg(q[:2], [0, 0], 1, k, "mean",
                                                                                           "max")[0], rtol=1e-14)
    # identical keys get identical scores, heads without rows take no part
    kk = np.repeat(k[:1], 5, axis=0)
    for m in MODES:
        s, _ = O.score_agg(q, rh, 4, kk, *m)
        assert np.all(s == s[0])


def test_agg_is_invariant_to_row_and_head_order():
    q, rh, G, k = _rand_problem(11, M=9, G=3)
    rng = np.random.default_rng(5)
    perm = rng.permutation(len(rh))
    relabel = np.array([2, 0, 1])
    for m in MODES:
        a, ea = O.score_agg(q, rh, G, k, *m)
        b, eb = O.score_agg(q[perm], relabel[rh[perm]], G, k, *m)
        np.testing.assert_allclose(a, b, rtol=1e-13)
        assert abs(ea - eb) < 1e-13


def test_entropy_closed_forms():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((64, 4))
    # zero queries attend uniformly: the normalised entropy is exactly 1
    _, e = O.score_agg(np.zeros((3, 4)), [0, 0, 0], 1, k)
    assert abs(e - 1.0) < 1e-14
    # one key far ahead of the others: the entropy vanishes
    kk = np.zeros((64, 4))
    kk[17, 0] = 1.0
    _, e = O.score_agg(np.array([[4000.0, 0, 0, 0]]), [0], 1, kk)
    assert e < 1e-12
    # m keys tied at the top, the rest far below: entropy = ln m / ln N
    kk = np.zeros((64, 4))
    kk[[3, 9, 40, 41, 63], 0] = 1.0
    _, e = O.score_agg(np.array([[2000.0, 0, 0, 0]]), [0], 1, kk)
    assert abs(e - math.log(5) / math.log(64)) < 1e-12
    # the entropy does not depend on the aggregation mode
    q, rh, G, k = _rand_problem(2)
    es = {O.score_agg(q, rh, G, k, *m)[1] for m in MODES}
    assert len(es) == 1


# ---------------------------------------------------------------------------
# head-budget reallocation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden("head_budget_handworked.json")["cases"], ids=lambda c: c["name"])
def test_head_budget_handworked(case):
    out = O.head_budget(case["entropy"], case["N"], case["prefix"], case["recent"], case["given"])
    if case["budget"] is None:
        assert out is None
    else:
        assert out.tolist() == case["budget"]


def _weights(ent):
    """The rule's utilities as 24-bit fixed point: floor((1 - entropy) * 2^24), clipped to [0, 1]."""
    u = np.clip(1.0 - np.asarray(ent, dtype=np.float32).astype(np.float64), 0.0, 1.0)
    return [int(math.floor(v * 2 ** 24)) for v in u]


def _waterfill(w, E, cap):
    """Exact shares s_h = min(cap, lam * w_h) with sum E, as Fractions: lam from the breakpoints
    (independent of the oracle's iteration); zero-weight heads share what the others leave."""
    H = len(w)
    if sum(w) == 0:
        return [Fraction(E, H)] * H
    # lam is where sum_h min(cap, lam w_h) = E: try the heads capped in order of decreasing weight
    order = sorted(range(H), key=lambda h: -w[h])
    for k in range(H + 1):
        capped = set(order[:k])
        rest = [h for h in range(H) if h not in capped]
        Wr = sum(w[h] for h in rest)
        left = E - cap * k
        if Wr == 0:
            s = [Fraction(cap) if h in capped else Fraction(0) for h in range(H)]
            z = [h for h in rest if w[h] == 0]
            for h in z:
                s[h] = Fraction(left, len(z))
            if all(v <= cap for v in s):
                return s
            continue
        lam = Fraction(left, Wr)
        if all(lam * w[h] <= cap for h in rest) and all(lam * w[h] >= cap for h in capped):
            return [Fraction(cap) if h in capped else lam * w[h] for h in range(H)]
    raise AssertionError("no water level")


@pytest.mark.parametrize("seed", range(30))
def test_head_budget_brute_force(seed):
    """The integer budgets minimise sum (x - s)^2 over all integer vectors with the same total
    and bounds, s being the exact water-filled shares of the fixed-point weights; among
    minimisers the lower heads get the extra slots (lexicographically largest)."""
    rng = np.random.default_rng(seed)
    H = int(rng.integers(2, 5))
    N, P, R = int(rng.integers(24, 34)), 2, 3
    f, cap = P + R, N - P - R
    given = rng.integers(f, N + 3, H)
    ent = rng.choice([0.0, 0.2, 0.5, 0.5, 0.9, 1.0], H) if seed % 3 == 0 else rng.uniform(0, 1, H)
    ent = ent.astype(np.float32)
    out = O.head_budget(ent, N, P, R, given)
    T = int(np.minimum(given, N).sum())
    assert out.sum() == T
    assert np.all(out >= f) and np.all(out <= N)
    if T >= H * N:
        return
    E = T - H * f
    s = _waterfill(_weights(ent), E, cap)
    best, best_x = None, None
    for x in itertools.product(range(cap + 1), repeat=H):
        if sum(x) != E:
            continue
        d = sum((Fraction(xi) - si) ** 2 for xi, si in zip(x, s))
        if best is None or d < best or (d == best and x > best_x):
            best, best_x = d, x
    assert (out - f).tolist() == list(best_x), (ent, given, s)


@pytest.mark.parametrize("seed", range(10))
def test_head_budget_is_monotone_in_entropy(seed):
    rng = np.random.default_rng(100 + seed)
    H = 8
    ent = rng.uniform(0.3, 1.0, H).astype(np.float32)
    given = np.full(H, 1792)
    out = O.head_budget(ent, 2048, 4, 16, given)
    assert out.sum() == given.sum()
    order = np.argsort(ent, kind="stable")
    assert np.all(np.diff(out[order]) <= 0)  # lower entropy, at least as much budget


# ---------------------------------------------------------------------------
# the whole step with the variants
# ---------------------------------------------------------------------------

def _head_rows(inp, l, b, h):
    """Observation rows of one KV head as the oracle builds them, for the restatement below."""
    G = inp.Hq // inp.Hkv
    ev = O.evict(inp, heads=[(l * inp.B + b) * inp.Hkv + h])
    rows, rh = [], []
    for g in range(G):
        hq = h * G + g
        for r in range(inp.n_r):
            rows.append(inp.q_recent[l, b, hq, r].double().numpy())
            rh.append(g)
        for p in ev["beacon_picks"][l, b, hq]:
            if p < 0:
                continue
            x = inp.qbuf[l, b, hq, p].float().numpy()
            rot = O.rope_f32(x, inp.t, inp.theta).astype(np.float64)
            if inp.dtype == "bf16":
                rot = O.bf16_bits_to_f64(O.f64_to_bf16_bits(rot))
            rows.append(rot)
            rh.append(g)
    return np.array(rows), np.array(rh), G


@pytest.mark.parametrize("mode", MODES[1:], ids=lambda m: ",".join(m))
def test_evict_variants_match_restatement(mode):
    inp = make_inputs("tiny", L=1, B=1, N=64, keep=48, seed=21)
    ev = O.evict(inp, row_agg=mode[0], group_agg=mode[1])
    for h in range(inp.Hkv):
        q, rh, G = _head_rows(inp, 0, 0, h)
        k = inp.K[0, 0, h].double().numpy()
        s, e = O.score_agg(q, rh, G, k, *mode)
        np.testing.assert_array_equal(ev["scores"][0, 0, h], s.astype(np.float32))
        assert ev["entropy"][0, 0, h] == np.float32(e)
        kept = O.select(s.astype(np.float32), inp.prefix, inp.recent, inp.budget_all)
        assert ev["kept_idx"][0, 0, h, :len(kept)].tolist() == kept.tolist()


def test_evict_entropy_budgets():
    inp = make_inputs("tiny", L=2, B=2, N=96, keep=64, seed=5)
    ev = O.evict(inp, head_budget="entropy")
    ent = ev["entropy"]
    for l in range(inp.L):
        for b in range(inp.B):
            want = O.head_budget(ent[l, b], inp.N, inp.prefix, inp.recent, [inp.budget_all] * inp.Hkv)
            assert ev["budget_used"][l, b].tolist() == want.tolist()
            assert ev["kept_len"][l, b].sum() == inp.budget_all * inp.Hkv
    # the entropies steer the split: head 0 fully diffuse, head 1 fully focused -> head 1 fills to
    # N and head 0 keeps its windows plus what head 1 could not take (2*64 - 2*20 - 76 = 12)
    forced = np.zeros_like(ent)
    forced[..., 0] = 1.0
    ev2 = O.evict(inp, head_budget="entropy", forced_entropy=forced)
    assert np.all(ev2["budget_used"][..., 1] == inp.N)
    assert np.all(ev2["budget_used"][..., 0] == inp.prefix + inp.recent + 12)
    # a listed head pulls in its layer's other heads for the entropies, but only it is kept
    ev3 = O.evict(inp, heads=[1], head_budget="entropy")
    assert ev3["budget_used"][0, 0, 1] == ev["budget_used"][0, 0, 1] and ev3["kept_len"][0, 0, 0] == 0
