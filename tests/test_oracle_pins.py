"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle step to a hand-worked case, a closed form, an
invariant, a library routine for a special case, or brute force on tiny
inputs, so that a dropped term, a wrong sign or index, or a transposed operand
in the oracle fails here. No GPU is needed.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O
from decoding_kv_cache_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# storage conversion
# ---------------------------------------------------------------------------

def test_bf16_from_f32_matches_torch_rounding():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),  # subnormal range
        (rng.standard_normal(5000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895314e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                  1.0 + 2 ** -8 + 2 ** -20], np.float32),
        # exact ties in f32: mantissa ...1 1000 0000 0000 0000 and ...0 1000 0000 0000 0000
        (np.arange(0x3f800000, 0x3f800000 + (1 << 20), 1 << 15, dtype=np.uint32) | 0x8000).view(np.float32),
    ])
    ours = O.f64_to_bf16_bits(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert O.f64_to_bf16_bits(np.array([np.nan]))[0] & 0x7fc0 == 0x7fc0


def test_bf16_from_f64_is_nearest_even():
    """Direct f64 -> bf16 rounding (not via f32), checked with exact rationals."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal(3000) * np.exp2(rng.integers(-130, 120, 3000))
    # values just above a bf16 tie that a f32 intermediate would round onto the tie
    x = np.concatenate([x, [1.0 + 2 ** -8 + 2 ** -40, -(3.0 + 2 ** -7 + 2 ** -45), 1.0 + 2 ** -8]])
    bits = O.f64_to_bf16_bits(x)
    vals = O.bf16_bits_to_f64(bits)
    for xi, b, v in zip(x, bits, vals):
        fx, fv = Fraction(float(xi)), Fraction(float(v))
        # the two neighbours of v in bf16, by magnitude
        mag, sgn = int(b) & 0x7fff, int(b) & 0x8000
        nbs = [sgn | (mag + d) for d in (1, -1) if 0 <= mag + d < 0x7f80]
        for nbits in nbs:
            nb = O.bf16_bits_to_f64(np.array([nbits], dtype=np.uint16))[0]
            dnb = abs(fx - Fraction(float(nb)))
            assert abs(fx - fv) <= dnb
            if abs(fx - fv) == dnb:
                assert int(b) & 1 == 0, "tie must go to the even mantissa"
    assert O.f64_to_bf16_bits(np.array([1.0 + 2 ** -8 + 2 ** -40]))[0] == 0x3f81


# ---------------------------------------------------------------------------
# farthest-point sampling
# ---------------------------------------------------------------------------

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("fps_handworked.json")["cases"], ids=lambda c: c["name"])
def test_fps_handworked(case):
    picks, order, _ = O.fps(np.array(case["x"]), case["m"], trace=True)
    assert order.tolist() == case["order"]
    assert picks.tolist() == case["picks"]


def _np_cos_dist(x):
    n = np.linalg.norm(x, axis=1, keepdims=True)
    xh = np.divide(x, n, out=np.zeros_like(x), where=n > 0)
    return 1.0 - xh @ xh.T


@pytest.mark.parametrize("seed", range(40))
def test_fps_trace_obeys_greedy_rule(seed):
    """Each step's pick is the lowest-index argmax of the min distance to the chosen set
    (distances recomputed here with numpy, independently of the C code)."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 40))
    D = int(rng.choice([2, 3, 8, 64]))
    x = rng.standard_normal((n, D))
    if seed % 3 == 0:  # duplicated rows and exact ties
        x[n // 2] = x[0] * 3.0
        x[-1] = x[1]
    m = int(rng.integers(1, n + 1))
    picks, order, _ = O.fps(x, m, trace=True)
    dist = _np_cos_dist(x)
    assert order[0] == 0
    chosen = [0]
    for k in range(1, m):
        mind = dist[:, chosen].min(axis=1)
        mind[chosen] = -np.inf
        best = mind.max()
        cand = np.flatnonzero(mind >= best - 1e-12)
        assert order[k] == cand[0] or abs(mind[order[k]] - best) <= 1e-12
        chosen.append(int(order[k]))
    assert sorted(chosen) == picks.tolist()


def _angle_cover(x, S):
    n = np.linalg.norm(x, axis=1, keepdims=True)
    xh = x / n
    ang = np.arccos(np.clip(xh @ xh.T, -1, 1))
    return ang[:, list(S)].min(axis=1).max()


@pytest.mark.parametrize("seed", range(12))
def test_fps_is_two_approx_k_centre(seed):
    """Greedy farthest-point covering is within 2x of the best k-centre cover in angle
    (the angle is a metric and 1 - cos is monotone in it), checked by brute force."""
    rng = np.random.default_rng(100 + seed)
    n, m = 9, int(rng.integers(2, 5))
    x = rng.standard_normal((n, 3))
    picks = O.fps(x, m)
    opt = min(_angle_cover(x, S) for S in itertools.combinations(range(n), m))
    assert _angle_cover(x, picks) <= 2 * opt + 1e-12


def test_fps_scale_invariance_and_check():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((32, 64))
    p = O.fps(x, 16)
    assert np.array_equal(p, O.fps(x * rng.uniform(0.1, 10.0, (32, 1)), 16))
    assert O.fps_check(x, p) == 0
    bad = p.copy()
    bad[-1] = [i for i in range(32) if i not in p][-1]
    bad.sort()
    assert O.fps_check(x, bad) != 0


def test_fps_update_compresses_full_buffers_only():
    rng = np.random.default_rng(3)
    qb = rng.standard_normal((3, 32, 64)).astype(np.float32)
    cnt = np.array([32, 20, 32], np.int32)
    out, c2, picks = O.fps_update(qb, cnt, 32, "f32")
    assert c2.tolist() == [16, 20, 16]
    assert np.array_equal(out[1], qb[1]) and (picks[1] == -1).all()
    for h in (0, 2):
        assert np.array_equal(picks[h], O.fps(qb[h].astype(np.float64), 16))
        assert np.array_equal(out[h, :16], qb[h, picks[h]])
        assert np.array_equal(out[h, 16:], qb[h, 16:])


# ---------------------------------------------------------------------------
# rotary encoding
# ---------------------------------------------------------------------------

def test_rope_identities():
    rng = np.random.default_rng(5)
    for D in (2, 4, 64, 128):
        q, k = rng.standard_normal(D), rng.standard_normal(D)
        for theta in (1e4, 1e6):
            assert np.allclose(O.rope(q, 0, theta), q, rtol=0, atol=0)
            r = O.rope(q, 12345, theta)
            assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12
            a = O.rope(q, 700, theta) @ O.rope(k, 300, theta)
            b = O.rope(q, 1400, theta) @ O.rope(k, 1000, theta)
            assert abs(a - b) < 1e-10


def test_rope_pairing_and_frequencies():
    # D = 2: one pair, frequency theta^0 = 1, a plain rotation by t radians
    t = 3
    r = O.rope(np.array([1.0, 0.0]), t, 1e4)
    assert np.allclose(r, [math.cos(t), math.sin(t)], atol=1e-15)
    # D = 4: pairs (0,2) and (1,3); the second turns by t * theta^(-1/2)
    theta = 1e4
    x = np.array([1.0, 2.0, 3.0, 4.0])
    r = O.rope(x, t, theta)
    a0, a1 = t, t * theta ** -0.5
    exp = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
           3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    assert np.allclose(r, exp, atol=1e-14)


# ---------------------------------------------------------------------------
# scores
# ---------------------------------------------------------------------------

def test_score_matches_library_softmax_max():
    rng = np.random.default_rng(11)
    for M, N, D in ((1, 7, 4), (32, 300, 64), (70, 129, 128)):
        q = rng.standard_normal((M, D)) * 1.5
        k = rng.standard_normal((N, D))
        ours, lse = O.score(q, k, with_lse=True)
        tq, tk = torch.from_numpy(q), torch.from_numpy(k)
        ref = torch.softmax(tq @ tk.T / math.sqrt(D), dim=-1).amax(0).numpy()
        assert np.allclose(ours, ref, rtol=1e-12, atol=0)
        # every row's softmax sums to one with the returned log-sum-exp
        s = (q @ k.T) / math.sqrt(D)
        assert np.allclose(np.exp(s - lse[:, None]).sum(1), 1.0, rtol=1e-12)
        assert np.allclose(lse, torch.logsumexp(tq @ tk.T / math.sqrt(D), -1).numpy(), rtol=1e-13)


def test_score_special_cases():
    rng = np.random.default_rng(12)
    D, N = 16, 50
    q = rng.standard_normal((5, D))
    # all-zero keys: every softmax is uniform
    assert np.allclose(O.score(q, np.zeros((N, D))), 1.0 / N, rtol=1e-14)
    # identical keys get identical scores
    k = rng.standard_normal((N, D))
    k[10] = k[3]
    s = O.score(q, k)
    assert s[10] == s[3]
    # one row: the score is that row's softmax
    s1 = O.score(q[:1], k)
    e = np.exp((q[:1] @ k.T)[0] / math.sqrt(D))
    assert np.allclose(s1, e / e.sum(), rtol=1e-13)
    # max over rows is at least each row's value, and equals one of them
    rows = np.stack([O.score(q[i:i + 1], k) for i in range(5)])
    assert np.allclose(s, rows.max(0), rtol=1e-14)


# ---------------------------------------------------------------------------
# selection
# ---------------------------------------------------------------------------

def _brute_select(s, P, R, budget):
    N = len(s)
    mid = list(range(P, N - R))
    kmid = budget - P - R
    best, best_key = None, None
    for S in itertools.combinations(mid, kmid):
        tot = sum(Fraction(float(s[i])) for i in S)
        key = (-tot, S)  # max score-sum, then lexicographically smallest
        if best_key is None or key < best_key:
            best, best_key = S, key
    return sorted(list(range(P)) + list(best) + list(range(N - R, N)))


@pytest.mark.parametrize("seed", range(25))
def test_select_brute_force(seed):
    rng = np.random.default_rng(200 + seed)
    N = int(rng.integers(4, 15))
    P = int(rng.integers(0, 3))
    R = int(rng.integers(0, 3))
    if P + R >= N:
        P, R = 1, 1
    budget = int(rng.integers(P + R, N))
    s = rng.integers(0, 5, N).astype(np.float32) / 4.0  # many exact ties
    if seed % 2:
        s = rng.random(N).astype(np.float32)
    kept = O.select(s, P, R, budget)
    assert kept.tolist() == _brute_select(s, P, R, budget)


def test_select_invariants_and_edges():
    rng = np.random.default_rng(9)
    N, P, R = 2048, 4, 16
    s = rng.random(N).astype(np.float32)
    for budget in (20, 21, 1000, 1792, 2047):
        kept = O.select(s, P, R, budget)
        assert len(kept) == budget
        assert (np.diff(kept) > 0).all()
        assert set(range(P)) <= set(kept.tolist()) and set(range(N - R, N)) <= set(kept.tolist())
        mid = np.zeros(N, bool)
        mid[P:N - R] = True
        keptm = np.zeros(N, bool)
        keptm[kept] = True
        if (mid & keptm).any() and (mid & ~keptm).any():
            assert s[mid & ~keptm].max() <= s[mid & keptm].min()
    assert O.select(s, P, R, N).tolist() == list(range(N))
    assert O.select(s, P, R, N + 5).tolist() == list(range(N))
    assert O.select(s, P, R, 19) is None


# ---------------------------------------------------------------------------
# the whole step: assembly of observation rows, budgets, compaction
# ---------------------------------------------------------------------------

def _np_rotate(x, pos, theta):
    """Rotary encoding restated with numpy complex numbers (independent of both sides)."""
    D = x.shape[-1]
    h = D // 2
    f = theta ** (-2.0 * np.arange(h) / D)
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * f)
    return np.concatenate([z.real, z.imag], axis=-1)


def _np_rotate_f32(x, pos, theta):
    """The same rotation in binary32 numpy arithmetic: fp64 angle, cos/sin rounded to f32, then
    separately rounded f32 products and sums (numpy never fuses them)."""
    D = x.shape[-1]
    h = D // 2
    ang = pos * theta ** (-2.0 * np.arange(h) / D)
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    a, b = x[..., :h].astype(np.float32), x[..., h:].astype(np.float32)
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def test_rope_f32_matches_f64_rotation_to_single_precision():
    rng = np.random.default_rng(21)
    for D, pos, theta in ((2, 3, 1e4), (64, 255, 1e4), (128, 32767, 1e6), (128, 4095, 5e5)):
        x = rng.standard_normal((6, D)).astype(np.float32)
        r32 = O.rope_f32(x, pos, theta)
        r64 = O.rope(x.astype(np.float64), pos, theta)
        assert np.allclose(r32, r64, rtol=0, atol=4e-6 * np.abs(x).max())
        assert np.array_equal(r32, _np_rotate_f32(x, pos, theta))


def _to_f64(t):
    return t.double().numpy()


def _restated_scores(inp, picks):
    """Scores of every KV head restated with numpy/torch from the inputs and given beacon picks."""
    L, B, Hq, Hkv, N, D = inp.L, inp.B, inp.Hq, inp.Hkv, inp.N, inp.D
    G = Hq // Hkv
    out = np.zeros((L, B, Hkv, N))
    for l in range(L):
        for b in range(B):
            for h in range(Hkv):
                rows = []
                for g in range(G):
                    hq = h * G + g
                    rows.append(_to_f64(inp.q_recent[l, b, hq]))
                    sel = [r for r in picks[l, b, hq] if r >= 0]
                    if sel:
                        rot = _np_rotate_f32(inp.qbuf[l, b, hq, sel].float().numpy(), inp.t, inp.theta)
                        if inp.dtype == "bf16":  # f32 -> bf16 rounding with torch (round to nearest even)
                            rows.append(torch.from_numpy(rot).to(torch.bfloat16).double().numpy())
                        else:
                            rows.append(rot.astype(np.float64))
                Q = torch.from_numpy(np.concatenate(rows))
                Kh = inp.K[l, b, h].double()
                out[l, b, h] = torch.softmax(Q @ Kh.T / math.sqrt(D), -1).amax(0).numpy()
    return out


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("qwen3-4b", dict(L=1, N=300)),
    ("llama8b-planted", dict(L=1, B=1, N=512)),
    ("qwen3-14b-long", dict(L=1, B=1, Hkv=2, Hq=10, N=200)),
])
def test_evict_matches_restatement(name, over):
    inp = make_inputs(name, **over)
    o = O.evict(inp)
    # beacons: FPS of the full buffer, as the oracle's own FPS picks
    L, B, Hq = inp.L, inp.B, inp.Hq
    for l in range(L):
        for b in range(B):
            for hq in range(Hq):
                x = _to_f64(inp.qbuf[l, b, hq, :inp.count[l, b, hq]])
                assert o["beacon_picks"][l, b, hq].tolist() == O.fps(x, inp.n_b).tolist()
    ref = _restated_scores(inp, o["beacon_picks"])
    assert np.allclose(o["scores"], ref.astype(np.float32), rtol=1e-6, atol=1e-30)
    # compaction: gather of the kept rows, bit for bit; tails untouched
    Kb = O._np_storage(inp.K)
    for l in range(L):
        for b in range(B):
            for h in range(inp.Hkv):
                n = o["kept_len"][l, b, h]
                idx = o["kept_idx"][l, b, h, :n]
                assert n == min(inp.budgets()[l, b, h].item(), inp.N)
                assert np.array_equal(o["K_out"][l, b, h, :n], Kb[l, b, h, idx])
                assert np.array_equal(o["K_out"][l, b, h, n:], Kb[l, b, h, n:])


def test_evict_beacon_count_rules():
    """count <= n_b: the buffer's first rows are the beacons; n_b = 0: recent queries only (RPC)."""
    inp = make_inputs("tiny", count=10)
    o = O.evict(inp)
    assert (o["beacon_picks"][..., :10] == np.arange(10)).all() and (o["beacon_picks"][..., 10:] == -1).all()
    ref = _restated_scores(inp, o["beacon_picks"])
    assert np.allclose(o["scores"], ref.astype(np.float32), rtol=1e-6)
    rpc = make_inputs("tiny", n_b=0)
    o2 = O.evict(rpc)
    ref2 = _restated_scores(rpc, np.full((1, 1, 4, 0), -1))
    assert np.allclose(o2["scores"], ref2.astype(np.float32), rtol=1e-6)
    # forced picks reproduce the FPS result when given the FPS result
    o3 = O.evict(inp.__class__(**{**inp.__dict__, "count": torch.full_like(inp.count, 32)}),
                 forced_picks=o["beacon_picks"])
    assert np.array_equal(o3["scores"], o["scores"])


def test_evict_per_head_budgets_and_errors():
    inp = make_inputs("qwen7b-reasonalloc", L=3, B=2, N=256)
    b = inp.budgets().clone()
    b[0, 0, 0] = 19   # below prefix + recent: head left whole, flagged
    b[1, 1, 2] = 256  # = N: keep all
    inp.budget = b
    o = O.evict(inp)
    assert o["error"][0, 0, 0] == -1 and o["kept_len"][0, 0, 0] == 256
    assert o["kept_len"][1, 1, 2] == 256
    ok = o["error"] == 0
    assert (o["kept_len"][ok] == np.minimum(b.numpy()[ok], 256)).all()


def test_reasonalloc_budget_profile():
    inp = make_inputs("qwen7b-reasonalloc", L=28, B=1, N=8192)
    b = inp.budget[:, 0].numpy()  # [L, Hkv]
    layer = b.sum(1) / inp.Hkv
    assert abs(layer.mean() - 1024) < 8          # rescaled to average 1024 (clamping may drift a little)
    assert layer[13] > layer[0] and layer[13] > layer[27]  # mid-peaked
    assert (b >= 20).all() and (b <= 8192).all()


def test_planted_keys_survive_with_beacons():
    """The thought-revisiting pattern (BeaconKV page, section '观察'): keys 100-450 that clustered
    global queries attend survive eviction when beacons are in the observation set, and fare worse
    with recent queries alone when the recent window holds no global query (a revisit is sparse
    and unpredictable, so the window at eviction time often has none)."""
    kw = dict(L=1, B=2, N=1024, keep=256, recent_global=False)
    inp = make_inputs("llama8b-planted", **kw)
    with_b = O.evict(inp)
    rpc = O.evict(make_inputs("llama8b-planted", n_b=0, **kw))

    def retained(o):
        r = []
        for b in range(inp.B):
            for h in range(inp.Hkv):
                kept = set(o["kept_idx"][0, b, h, :o["kept_len"][0, b, h]].tolist())
                r.append(np.mean([p in kept for p in inp.planted[0, b, h].tolist()]))
        return float(np.mean(r))

    assert retained(with_b) > 0.95
    assert retained(with_b) > retained(rpc) + 0.1
