"""The in-place compaction against an out-of-place gather on adversarial kept lists.

Every list is valid (strictly increasing, prefix and recent windows kept); they stress the forward
sweep's hazards: a single dropped token right after the prefix (every later row moves by one), a
single dropped token just before the recent window (one row moves), alternating drops (runs of one
row), one long dropped block (the recent window moves far, across many tiles), only the windows
kept, nothing dropped, sparse lists (one kept token in 4 or 9, as with a 1/8 budget: runs of one
row, one bulk copy each), and random lists. Heads of one launch get different lists. Bit-exact.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _lists(N, P, R, rng):
    mid = np.arange(P, N - R)
    full = np.arange(N)
    out = [
        np.delete(full, P),                      # drop only the first middle token
        np.delete(full, N - R - 1),              # drop only the last middle token
        np.concatenate([np.arange(P), mid[::2], np.arange(N - R, N)]),   # alternating drops
        np.concatenate([np.arange(P), mid[:5], mid[-3:], np.arange(N - R, N)]),  # one long dropped block
        np.concatenate([np.arange(P), np.arange(N - R, N)]),  # only the windows
        full,                                    # nothing dropped
        np.concatenate([np.arange(P), mid[1::4], np.arange(N - R, N)]),  # sparse: every 4th middle token
        np.concatenate([np.arange(P), mid[3::9], np.arange(N - R, N)]),  # sparse: every 9th (a 1/8 budget)
    ]
    for _ in range(4):
        k = int(rng.integers(0, len(mid) + 1))
        out.append(np.concatenate([np.arange(P), np.sort(rng.choice(mid, k, replace=False)), np.arange(N - R, N)]))
    return out


@pytest.mark.parametrize("dtype,D,N", [("bf16", 128, 2048), ("bf16", 64, 777), ("f32", 128, 1000), ("f32", 64, 300)])
def test_compact_adversarial_lists(dtype, D, N):
    from decoding_kv_cache_gb300 import kvc
    rng = np.random.default_rng(D + N)
    P, R = 4, 16
    lists = _lists(N, P, R, rng)
    L, B, Hkv = 2, 1, (len(lists) + 1) // 2
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(N)
    K = torch.randn((L, B, Hkv, N, D), generator=g).to(dt)
    V = torch.randn((L, B, Hkv, N, D), generator=g).to(dt)
    ki = torch.full((L, B, Hkv, N), -7, dtype=torch.int32)
    kl = torch.zeros((L, B, Hkv), dtype=torch.int32)
    for i in range(L * B * Hkv):
        lst = lists[i % len(lists)]
        l, h = divmod(i, Hkv)
        ki[l, 0, h, :len(lst)] = torch.from_numpy(lst.astype(np.int32))
        kl[l, 0, h] = len(lst)
    Kd, Vd = K.to(DEV), V.to(DEV)
    cache = kvc.Cache(Kd, Vd, Hkv)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_compact(cache, ki.to(DEV), kl.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    view = (lambda t: t.view(torch.int16)) if dtype == "bf16" else (lambda t: t.view(torch.int32))
    for before, after in ((K, Kd.cpu()), (V, Vd.cpu())):
        bb, aa = view(before), view(after)
        for l in range(L):
            for h in range(Hkv):
                n = int(kl[l, 0, h])
                idx = ki[l, 0, h, :n].long()
                assert torch.equal(aa[l, 0, h, :n], bb[l, 0, h, idx]), (l, h)
                assert torch.equal(aa[l, 0, h, n:], bb[l, 0, h, n:]), (l, h)
