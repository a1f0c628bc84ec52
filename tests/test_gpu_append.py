"""Parity of kvc_append (the per-step append into the pre-RoPE buffer and the recent ring, with the
FPS trigger) with the oracle's append, step by step, through the C ABI.

Buffers, counts and rings are compared bit for bit after every step (the whole buffer, rows past
the count included: both sides leave them the same way). FPS picks are identical except at
distance near-ties within 1e-5, where the GPU's choice is checked to be a valid greedy result and
the oracle's state then takes the GPU's buffer for that head.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import FPS_TOL

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    return O.bf16_bits_to_f64(bits) if dtype == "bf16" else bits.astype(np.float64)


def _drive(dtype, D, qmax, n_r, nq, steps, post, seed, t0=0, theta=1e4, counts=None):
    """Run `steps` appends on the GPU and the oracle side by side, checking every step."""
    from decoding_kv_cache_gb300 import kvc
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    qb = torch.randn((nq, qmax, D), generator=g).to(dt)
    cnt = torch.zeros(nq, dtype=torch.int32) if counts is None else torch.as_tensor(counts, dtype=torch.int32)
    ring = torch.randn((nq, n_r, D), generator=g).to(dt)
    qb_d, cnt_d, ring_d = qb.to(DEV), cnt.to(DEV), ring.to(DEV)
    ob, oc, orr = _bits(qb), cnt.numpy().copy(), _bits(ring)
    m = qmax // 2
    compressions = 0
    for t in range(t0, t0 + steps):
        q = torch.randn((nq, D), generator=g).to(dt)
        p = torch.randn((nq, D), generator=g).to(dt) if post else None
        picks = torch.full((nq, m), -7, dtype=torch.int32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        kvc.kvc_append(q.to(DEV), qb_d, cnt_d, ring_d if n_r else None, t, theta,
                       q_post=None if p is None else p.to(DEV), picks=picks, status=status)
        prev_b, prev_c = ob.copy(), oc.copy()
        ob, oc, orr, op, err = O.append(_bits(q), None if p is None else _bits(p), t, theta, ob, oc, orr, dtype)
        torch.cuda.synchronize()
        gp = picks.cpu().numpy()
        want_status = 0x2 if err.any() else 0
        assert int(status.item()) == want_status, (t, int(status.item()))
        assert np.array_equal(cnt_d.cpu().numpy(), oc), t
        if n_r:
            assert np.array_equal(_bits(ring_d), orr), f"ring differs at step {t}"
        gb = _bits(qb_d)
        for h in np.flatnonzero((gp != op).any(axis=1)):
            # a near-tie: the GPU's picks must be a valid greedy FPS of the rows it compressed
            assert (op[h] >= 0).all() and (gp[h] >= 0).all(), (t, h, gp[h], op[h])
            c = int(prev_c[h])
            rows = prev_b[h, :qmax].copy() if c == qmax else np.concatenate([prev_b[h, :qmax - 1], _bits(q)[h:h + 1]])
            assert O.fps_check(_f64(rows, dtype), gp[h], FPS_TOL) == 0, (t, h)
            ob[h] = gb[h]
            op[h] = gp[h]
        assert np.array_equal(gp, op), t
        assert np.array_equal(gb, ob), f"buffer differs at step {t}"
        compressions += int((op[:, 0] >= 0).sum())
    return compressions


@pytest.mark.parametrize("dtype,D,qmax,n_r,post", [
    ("bf16", 128, 32, 16, True),
    ("bf16", 128, 32, 16, False),
    ("f32", 64, 8, 4, False),
    ("f32", 128, 16, 16, True),
    ("bf16", 64, 64, 8, False),
    ("bf16", 64, 2, 1, True),
    ("f32", 64, 4, 0, True),
])
def test_append_sequence_matches_oracle(dtype, D, qmax, n_r, post):
    """Several fill/compress cycles from mixed starting counts (empty, filling, one short of full,
    full on entry), with the ring written from the post-RoPE query or by rotation."""
    nq = 70
    rng = np.random.default_rng(qmax + D)
    counts = rng.integers(0, qmax + 1, nq)
    counts[:4] = [0, qmax - 1, qmax, qmax // 2]
    n = _drive(dtype, D, qmax, n_r, nq, 2 * qmax + 3, post, seed=qmax * 7 + D, t0=1000, theta=1e6, counts=counts)
    assert n >= 2 * nq  # every head compressed at least twice


def test_append_bad_counts_are_flagged_and_left():
    """A count outside [0, qmax] sets the status bit and leaves that head's buffer and count; its
    ring row is still written; other heads proceed."""
    counts = [-1, 33, 31, 32, 5]
    _drive("bf16", 128, 32, 16, 5, 1, True, seed=3, t0=77, counts=counts)


def test_append_qwen3_4b_shape():
    """The Qwen3-4B-shaped decode state (36 layers x 32 query heads, D 128, buffer 32, 16 recent,
    theta 1e6) across a compression: 20 steps from counts 20..31 at positions 2048.."""
    nq = 36 * 32
    counts = 20 + np.arange(nq) % 12
    n = _drive("bf16", 128, 32, 16, nq, 20, False, seed=11, t0=2048, theta=1e6, counts=counts)
    assert n >= nq


def test_append_qwen3_14b_shape_trigger():
    """The Qwen3-14B-shaped long-trace state (40 layers x 8 sequences x 40 query heads, buffer 64)
    on the two steps around the trigger: every buffer one short of full, then just compressed."""
    nq = 40 * 8 * 40
    n = _drive("bf16", 128, 64, 16, nq, 2, True, seed=14, t0=32767, theta=1e6, counts=np.full(nq, 63))
    assert n == nq
