"""Pins for the oracle's per-step append (pre-RoPE buffer with the FPS trigger, recent ring).

A hand-worked fixture, the fill/compress count cycle in closed form, survivors being earlier
appended rows in time order, the ring holding the latest n_r queries, and the rotation path.
No GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit(deg):
    return np.array([math.cos(math.radians(deg)), math.sin(math.radians(deg))], dtype=np.float32)


def test_append_handworked():
    case = json.load(open(os.path.join(GOLDEN, "append_handworked.json")))
    qmax = case["qmax"]
    qb = np.zeros((1, qmax, 2), np.float32)
    cnt = np.zeros(1, np.int32)
    ring = np.zeros((1, 2, 2), np.float32)
    for t, (deg, want) in enumerate(zip(case["appends_deg"], case["steps"])):
        q = _unit(deg)[None]
        qb, cnt, ring, picks, err = O.append(q, q * 10, t, 1e4, qb, cnt, ring, "f32")
        assert err[0] == 0
        assert int(cnt[0]) == want["count"], (t, cnt)
        assert picks[0].tolist() == want["picks"], (t, picks)
        got = qb[0, :want["count"]]
        np.testing.assert_array_equal(got, np.stack([_unit(d) for d in want["buffer_deg"]]))
        np.testing.assert_array_equal(ring[0, t % 2], q[0] * 10)


@pytest.mark.parametrize("qmax,n_r,dtype", [(8, 4, "f32"), (32, 16, "bf16"), (2, 1, "f32")])
def test_append_cycle_survivors_and_ring(qmax, n_r, dtype):
    rng = np.random.default_rng(qmax)
    nq, D, steps = 3, 8, 3 * qmax + 5
    store = (lambda x: O.f64_to_bf16_bits(x)) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    zero = np.zeros((), np.uint16 if dtype == "bf16" else np.float32)
    qb = np.full((nq, qmax, D), zero)
    ring = np.full((nq, n_r, D), zero)
    cnt = np.zeros(nq, np.int32)
    history = []  # appended rows (storage bits), per step
    c_expect = 0
    for t in range(steps):
        q = store(rng.standard_normal((nq, D)))
        post = store(rng.standard_normal((nq, D)))
        history.append(q)
        qb, cnt, ring, picks, err = O.append(q, post, t, 1e4, qb, cnt, ring, dtype)
        assert not err.any()
        # the fill/compress cycle: +1 per step, back to qmax/2 on reaching qmax
        c_expect = c_expect + 1 if c_expect + 1 < qmax else qmax // 2
        assert (cnt == c_expect).all()
        compressed = c_expect == qmax // 2 and t >= qmax - 1
        assert ((picks >= 0).all(axis=1) == compressed).all()
        # every buffer row is an appended row, in append order
        for h in range(nq):
            steps_of = []
            for r in range(c_expect):
                hit = [s for s in range(t + 1) if np.array_equal(history[s][h], qb[h, r])]
                assert hit, (t, h, r)
                steps_of.append(hit[-1])
            assert steps_of == sorted(steps_of) and len(set(steps_of)) == len(steps_of)
            assert steps_of[-1] == t or compressed  # the newest row is kept unless FPS just ran
        np.testing.assert_array_equal(ring[:, t % n_r], post)


def test_append_rotates_when_no_post_rope_query():
    rng = np.random.default_rng(1)
    nq, D, qmax, n_r = 2, 16, 8, 4
    q = O.f64_to_bf16_bits(rng.standard_normal((nq, D)))
    qb = np.zeros((nq, qmax, D), np.uint16)
    ring = np.zeros((nq, n_r, D), np.uint16)
    _, _, ring2, _, _ = O.append(q, None, 1234, 1e6, qb, np.zeros(nq, np.int32), ring, "bf16")
    for h in range(nq):
        want = O.f64_to_bf16_bits(O.rope_f32(O.bf16_bits_to_f64(q[h]).astype(np.float32), 1234, 1e6).astype(np.float64))
        np.testing.assert_array_equal(ring2[h, 1234 % n_r], want)


def test_append_full_on_entry_and_bad_counts():
    rng = np.random.default_rng(2)
    nq, D, qmax = 3, 4, 8
    qb = rng.standard_normal((nq, qmax, D)).astype(np.float32)
    ring = np.zeros((nq, 2, D), np.float32)
    cnt = np.array([qmax, -1, qmax + 1], np.int32)
    q = rng.standard_normal((nq, D)).astype(np.float32)
    qb2, cnt2, ring2, picks, err = O.append(q, q, 5, 1e4, qb, cnt, ring, "f32")
    # a full buffer is compressed before the new row goes in
    assert cnt2[0] == qmax // 2 + 1 and (picks[0] >= 0).all()
    sel = O.fps(qb[0].astype(np.float64), qmax // 2)
    np.testing.assert_array_equal(qb2[0, :qmax // 2], qb[0, sel])
    np.testing.assert_array_equal(qb2[0, qmax // 2], q[0])
    # out-of-range counts: buffer and count untouched, flagged; the ring is still written
    assert err.tolist() == [0, -1, -1]
    np.testing.assert_array_equal(qb2[1:], qb[1:])
    assert cnt2[1:].tolist() == [-1, qmax + 1]
    np.testing.assert_array_equal(ring2[:, 5 % 2], q)
