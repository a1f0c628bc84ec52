"""Parity of the CUDA path (called through the C ABI) with the CPU oracle, element by element.

Sizes are small enough for the oracle to finish in seconds yet span several key chunks
with a ragged tail; the full-size workloads are checked on sampled heads in
test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

from decoding_kv_cache_gb300.inputs import make_inputs
from oracle import oracle as O
from parity_util import (assert_scores_close, check_beacon_picks, check_compaction, check_kept, run_evict,
                         run_score, storage_to_f64)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    ("tiny", {}),
    ("tiny", dict(N=1000, D=128)),
    ("qwen3-4b", dict(L=2, N=1000)),
    ("qwen3-4b", dict(L=1, N=129, D=64)),
    ("llama8b-planted", dict(L=1, B=2, N=700)),
    ("qwen7b-reasonalloc", dict(L=2, B=2, N=1500)),
    ("qwen3-14b-long", dict(L=1, B=1, N=2100)),
    # 512 heads over 76 groups of 2 CTAs: 7 rounds, so the exchange slots and TMEM buffers wrap
    ("qwen3-4b", dict(L=8, B=8, N=300, D=64)),
    # a 128-row tile whose keys exceed 256 per SM: the two-pass kernel takes it
    ("qwen3-4b", dict(L=1, Hq=4, Hkv=1, N=50000)),
    # 224 rows as two 128-row tiles over 20 CTAs per head (the wide exchange batch)
    ("qwen7b-reasonalloc", dict(L=1, B=1, N=5000)),
    # per-head budgets over 384 heads (more than one wave of selection-and-compaction CTAs, which
    # take the heads largest budget first)
    ("qwen7b-reasonalloc", dict(L=12, B=8, N=1000)),
]


def _ids(c):
    return f"{c[0]}-" + "-".join(f"{k}{v}" for k, v in c[1].items())


@pytest.mark.parametrize("name,over", CASES, ids=[_ids(c) for c in CASES])
def test_evict_matches_oracle(name, over):
    inp = make_inputs(name, **over)
    gpu = run_evict(inp, DEV)
    _, gpu_picks = run_score(inp, DEV)
    ora = O.evict(inp)
    if check_beacon_picks(inp, gpu_picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=gpu_picks)  # a valid near-tie alternative: score with the GPU's beacons
    assert gpu["status"] == 0
    assert_scores_close(gpu["scores"], ora["scores"], name)
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


@pytest.mark.parametrize("count", [0, 1, 10, 16, 17, 31, 32])
def test_beacon_count_rules(count):
    """count <= n_b uses the buffer as is; more runs FPS down to n_b (non-destructively)."""
    inp = make_inputs("qwen3-4b", L=1, N=300, count=count)
    scores, picks = run_score(inp, DEV)
    ora = O.evict(inp)
    if check_beacon_picks(inp, picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=picks)
    assert_scores_close(scores, ora["scores"], f"count={count}")


def test_recent_only_observation():
    """n_b = 0: scores come from the recent queries alone (the RPC-style observation set)."""
    inp = make_inputs("qwen3-4b", L=1, N=500, n_b=0)
    gpu = run_evict(inp, DEV)
    ora = O.evict(inp)
    assert_scores_close(gpu["scores"], ora["scores"], "n_b=0")
    check_kept(inp, gpu, ora, gpu["scores"])


def test_beacons_only_observation():
    inp = make_inputs("qwen3-4b", L=1, N=500, n_r=0)
    gpu = run_evict(inp, DEV)
    _, picks = run_score(inp, DEV)
    ora = O.evict(inp)
    if check_beacon_picks(inp, picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=picks)
    assert_scores_close(gpu["scores"], ora["scores"], "n_r=0")


@pytest.mark.parametrize("keep", [20, 21, 299, 300, 301])
def test_budget_edges(keep):
    """budget == prefix + recent keeps no middle key; budget >= N keeps everything."""
    inp = make_inputs("qwen3-4b", L=1, N=300, keep=keep)
    gpu = run_evict(inp, DEV)
    ora = O.evict(inp)
    assert_scores_close(gpu["scores"], ora["scores"], f"keep={keep}")
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


def test_per_head_budget_out_of_range_is_flagged_and_left_whole():
    inp = make_inputs("qwen7b-reasonalloc", L=2, B=1, N=400)
    b = inp.budgets().clone()
    b[0, 0, 1] = 5     # < prefix + recent
    b[1, 0, 3] = 400   # == N
    inp.budget = b
    gpu = run_evict(inp, DEV)
    ora = O.evict(inp)
    assert gpu["status"] & 0x1
    assert gpu["kept_len"][0, 0, 1] == 400 and gpu["kept_len"][1, 0, 3] == 400
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


def test_tiny_cache_shorter_than_windows():
    """N = 12 < prefix + recent = 20: a budget >= N keeps everything, a smaller one cannot hold
    the always-kept windows and is rejected before any launch (as the oracle rejects it)."""
    from decoding_kv_cache_gb300 import kvc
    inp = make_inputs("qwen3-4b", L=1, N=12, keep=12)
    gpu = run_evict(inp, DEV)
    assert (gpu["kept_len"] == 12).all()
    assert O.evict(make_inputs("qwen3-4b", L=1, N=12, keep=10))["error"].min() == -1
    with pytest.raises(kvc.KvcError) as e:
        run_evict(make_inputs("qwen3-4b", L=1, N=12, keep=10), DEV)
    assert e.value.code == -4


@pytest.mark.parametrize("N", [1, 2, 31])
def test_one_or_few_token_caches(N):
    """Caches of one, two and 31 tokens: a single ragged key chunk (the key loads zero-fill past
    the cache), windows as long as or longer than the cache. One key: every softmax weight, so
    every score, is 1 (the kernel forms s*c2 - lse2 in fp32, so within a few ulps). With 31 tokens
    a budget of 26 leaves six middle tokens to choose."""
    inp = make_inputs("qwen3-4b", L=1, N=N, keep=20 if N <= 20 else N - 5)
    gpu = run_evict(inp, DEV)
    ora = O.evict(inp)
    assert_scores_close(gpu["scores"], ora["scores"], f"N={N}")
    if N == 1:
        assert np.abs(gpu["scores"].astype(np.float64) - 1.0).max() <= 2.0 ** -20
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


@pytest.mark.parametrize("dtype,D,qmax", [("f32", 64, 32), ("bf16", 128, 32), ("bf16", 128, 64), ("bf16", 64, 16)])
def test_fps_update_matches_oracle(dtype, D, qmax):
    from decoding_kv_cache_gb300 import kvc
    g = torch.Generator().manual_seed(D + qmax)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    nq = 96
    qb = torch.randn((nq, qmax, D), generator=g).to(dt)
    cnt = torch.full((nq,), qmax, dtype=torch.int32)
    cnt[5] = qmax // 2   # not full: untouched
    cnt[7] = qmax + 3    # out of range: flagged, untouched
    bits = qb.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else qb.numpy()
    ob, oc, op = O.fps_update(bits, cnt.numpy(), qmax, dtype)
    qd, cd = qb.to(DEV), cnt.to(DEV)
    picks = torch.full((nq, qmax // 2), -7, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_fps_update(qd, cd, picks=picks, status=status)
    torch.cuda.synchronize()
    gp = picks.cpu().numpy()
    assert int(status.item()) & 0x2
    assert np.array_equal(cd.cpu().numpy(), oc)
    out = qd.cpu()
    for h in range(nq):
        if oc[h] != qmax // 2 or cnt[h] != qmax:
            assert (gp[h] == -1).all() and torch.equal(out[h], qb[h])
            continue
        if not np.array_equal(gp[h], op[h]):
            assert O.fps_check(storage_to_f64(qb[h]), gp[h], 1e-5) == 0
        assert torch.equal(out[h, :qmax // 2], qb[h, torch.from_numpy(gp[h].astype(np.int64))])
        assert torch.equal(out[h, qmax // 2:], qb[h, qmax // 2:])


def test_select_matches_oracle_on_the_same_scores():
    """Selection is exact given the scores: the GPU and the oracle agree bit for bit, including
    many exact ties (quantised scores) and the empty middle."""
    from decoding_kv_cache_gb300 import kvc
    g = torch.Generator().manual_seed(5)
    L, B, Hkv, N, P, R = 3, 2, 4, 3000, 4, 16
    sc = (torch.randint(0, 50, (L, B, Hkv, N), generator=g).float() / 64.0)
    sc[0] = torch.rand((B, Hkv, N), generator=g)
    bud = torch.randint(P + R, N + 50, (L, B, Hkv), generator=g, dtype=torch.int32)
    bud[1, 0, 0] = P + R
    kept_idx = torch.full((L, B, Hkv, N), -7, dtype=torch.int32, device=DEV)
    kept_len = torch.zeros((L, B, Hkv), dtype=torch.int32, device=DEV)
    kvc.kvc_select(sc.to(DEV), P, R, kept_idx, kept_len, budget=bud.to(DEV))
    torch.cuda.synchronize()
    ki, kl = kept_idx.cpu().numpy(), kept_len.cpu().numpy()
    for l in range(L):
        for b in range(B):
            for h in range(Hkv):
                ref = O.select(sc[l, b, h].numpy(), P, R, int(bud[l, b, h]))
                assert kl[l, b, h] == len(ref)
                assert np.array_equal(ki[l, b, h, :len(ref)], ref)


@pytest.mark.parametrize("N,heads", [(3001, 6), (20001, 3), (60001, 2)])
@pytest.mark.parametrize("dist", ["uniform", "quantised", "split", "constant"])
def test_select_sizes_and_distributions(N, heads, dist):
    """Every launch shape of the selection (256 threads with the scores in shared memory, 1024
    threads, and the global-memory path past 51200 tokens), token counts that are not a multiple
    of 4 or of the sweep's groups, and four score laws: distinct values, heavy exact ties, a split
    where the k-th largest score's leading digit holds exactly the kept middle tokens (the digit
    search then stops after its first digit), and one value everywhere (no digit pass at all: the
    lowest-index middle tokens are kept)."""
    from decoding_kv_cache_gb300 import kvc
    g = torch.Generator().manual_seed(N + len(dist))
    P, R = 4, 16
    kmid = (N * 7) // 8 - P - R
    if dist == "uniform":
        sc = torch.rand((heads, N), generator=g)
    elif dist == "quantised":
        sc = torch.randint(0, 40, (heads, N), generator=g).float() / 64.0
    elif dist == "constant":
        sc = torch.full((heads, N), 0.375)
    else:
        sc = 0.25 + torch.rand((heads, N), generator=g) * 0.2
        for h in range(heads):
            mid = torch.randperm(N - P - R, generator=g)[:kmid] + P
            sc[h, mid] = 0.75 + torch.rand(kmid, generator=g) * 0.2
    bud = torch.full((heads,), kmid + P + R, dtype=torch.int32)
    bud[-1] = P + R + 1
    kept_idx = torch.full((1, 1, heads, N), -7, dtype=torch.int32, device=DEV)
    kept_len = torch.zeros((1, 1, heads), dtype=torch.int32, device=DEV)
    kvc.kvc_select(sc.view(1, 1, heads, N).to(DEV), P, R, kept_idx, kept_len, budget=bud.view(1, 1, heads).to(DEV))
    torch.cuda.synchronize()
    ki, kl = kept_idx.cpu().numpy()[0, 0], kept_len.cpu().numpy()[0, 0]
    for h in range(heads):
        ref = O.select(sc[h].numpy(), P, R, int(bud[h]))
        assert kl[h] == len(ref), h
        assert np.array_equal(ki[h, :len(ref)], ref), h


@pytest.mark.parametrize("N", [3001, 20001])
def test_select_ranks_signed_scores_by_value(N):
    """kvc_select takes any finite fp32 score, not only the non-negative ones the scoring kernels
    produce: negative values, -0 next to +0 (equal, so the lower index wins), and +-inf rank as
    their values do, as in the oracle's sort."""
    from decoding_kv_cache_gb300 import kvc
    g = torch.Generator().manual_seed(N)
    P, R, heads = 4, 16, 4
    sc = torch.randn((heads, N), generator=g) * 10.0
    sc[1] = torch.randint(-3, 3, (N,), generator=g).float()       # heavy ties around zero
    zero = torch.rand(N, generator=g) < 0.5
    sc[1][zero & (sc[1] == 0)] = -0.0                               # -0 and +0 mixed
    sc[2] = -torch.rand(N, generator=g)                             # all negative
    sc[3, 100:200] = float("inf")
    sc[3, 300:400] = float("-inf")
    bud = torch.tensor([(N * 7) // 8, N // 2, P + R + 5, (N * 7) // 8], dtype=torch.int32)
    kept_idx = torch.full((1, 1, heads, N), -7, dtype=torch.int32, device=DEV)
    kept_len = torch.zeros((1, 1, heads), dtype=torch.int32, device=DEV)
    kvc.kvc_select(sc.view(1, 1, heads, N).to(DEV), P, R, kept_idx, kept_len, budget=bud.view(1, 1, heads).to(DEV))
    torch.cuda.synchronize()
    ki, kl = kept_idx.cpu().numpy()[0, 0], kept_len.cpu().numpy()[0, 0]
    for h in range(heads):
        ref = O.select(sc[h].numpy(), P, R, int(bud[h]))
        assert kl[h] == len(ref), h
        assert np.array_equal(ki[h, :len(ref)], ref), h


def test_compact_rejects_malformed_lists():
    from decoding_kv_cache_gb300 import kvc
    inp = make_inputs("qwen3-4b", L=1, N=256)
    g = inp.to(DEV)
    cache = kvc.Cache(g.K, g.V, g.Hq)
    ki = torch.arange(256, dtype=torch.int32).repeat(1, 1, 8, 1).contiguous()
    kl = torch.full((1, 1, 8), 200, dtype=torch.int32)
    ki[0, 0, 0, 10] = 9       # not increasing
    ki[0, 0, 1, 5:] += 60     # runs past N
    kl[0, 0, 2] = 300         # longer than N
    ki[0, 0, 3, :200] = torch.arange(56, 256)  # a valid shift
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_compact(cache, ki.to(DEV), kl.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4
    K = g.K.cpu()
    for h in (0, 1, 2):
        assert torch.equal(K[0, 0, h], inp.K[0, 0, h])
    assert torch.equal(K[0, 0, 3, :200], inp.K[0, 0, 3, 56:256])


PATH_CASES = [
    ("qwen7b-reasonalloc", dict(L=1, B=1, N=5000)),   # 224 rows: two row tiles
    ("qwen3-14b-long", dict(L=1, B=1, N=2100)),       # 240 rows, ragged last range
    ("qwen3-4b", dict(L=2, N=1000)),                  # 128 rows
    ("qwen3-4b", dict(L=1, N=129, D=64)),             # D 64, one key past a chunk
    ("llama8b-planted", dict(L=1, B=2, N=4500)),      # 128 rows, several ranges
]


@pytest.mark.parametrize("path", ["resident", "split", "fused", "wide"])
@pytest.mark.parametrize("name,over", PATH_CASES, ids=[_ids(c) for c in PATH_CASES])
def test_each_scoring_kernel_matches_oracle(path, name, over):
    """Every bf16 scoring kernel (single-read, two-pass streaming, two-pass with group exchange,
    two-pass with the keys on the TMEM lanes), forced through kvc_opts.kernel, against the oracle on
    the same inputs (a kernel that does not apply to a shape falls back to the automatic choice)."""
    inp = make_inputs(name, **over)
    gpu = run_evict(inp, DEV, kernel=path)
    _, gpu_picks = run_score(inp, DEV, kernel=path)
    ora = O.evict(inp)
    if check_beacon_picks(inp, gpu_picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=gpu_picks)
    assert gpu["status"] == 0
    assert_scores_close(gpu["scores"], ora["scores"], f"{name} via {path}")
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


F32_CASES = [
    ("tiny", {}),                                     # 8 CTAs of 32 keys per head
    ("tiny", dict(N=1000, D=128)),                    # 8 CTAs of 125 keys, ragged last CTA
    ("tiny", dict(N=33)),                             # 2 CTAs of 17 and 16 keys
    ("tiny", dict(N=1, keep=1)),                      # one key: every score is 1
    ("tiny", dict(L=2, B=3, N=300, Hq=16, Hkv=2)),    # 256 rows, 12 heads
    ("tiny", dict(N=1500)),                           # 188 keys per CTA: the streaming passes
]


@pytest.mark.parametrize("path", ["auto", "split"])
@pytest.mark.parametrize("name,over", F32_CASES, ids=[_ids(c) for c in F32_CASES])
def test_f32_scoring_paths(path, name, over):
    """fp32 caches: the one-launch cluster kernel (short caches, chosen automatically) and the
    streaming passes (forced with kvc_opts.kernel = split, and the automatic choice past 1024 keys)
    against the oracle."""
    inp = make_inputs(name, **over)
    gpu = run_evict(inp, DEV, kernel=path)
    _, gpu_picks = run_score(inp, DEV, kernel=path)
    ora = O.evict(inp)
    if check_beacon_picks(inp, gpu_picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=gpu_picks)
    assert gpu["status"] == 0
    assert_scores_close(gpu["scores"], ora["scores"], f"{name} via {path}")
    if inp.N == 1:
        assert np.abs(gpu["scores"].astype(np.float64) - 1.0).max() <= 2.0 ** -20
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


WIDE_CASES = [
    ("qwen3-14b-long", dict(L=1, B=2, N=4100)),             # 240 rows: 16-column tail granule, ragged range
    ("qwen7b-reasonalloc", dict(L=1, B=1, N=8192)),         # 224 rows: whole granules only, two ranges
    ("qwen7b-reasonalloc", dict(L=1, B=1, N=200, D=64)),    # D 64, one ragged chunk pair
    ("qwen3-14b-long", dict(L=2, B=1, N=129, Hq=24, Hkv=8)),  # 3 query heads: 144 rows, one key past a chunk
]


@pytest.mark.parametrize("name,over", WIDE_CASES, ids=[_ids(c) for c in WIDE_CASES])
def test_wide_kernel_shapes(name, over):
    """The wide kernel's column splits (whole and half granules), ragged chunks and ranges, D 64."""
    inp = make_inputs(name, **over)
    gpu = run_evict(inp, DEV, kernel="wide")
    _, gpu_picks = run_score(inp, DEV, kernel="wide")
    ora = O.evict(inp)
    if check_beacon_picks(inp, gpu_picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=gpu_picks)
    assert gpu["status"] == 0
    assert_scores_close(gpu["scores"], ora["scores"], f"{name} wide")
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


@pytest.mark.parametrize("where", ["late", "first", "long-late"])
def test_wide_kernel_exact_fallback_on_extreme_logits(where):
    """Keys planted along a recent query with a logit ~160 (base 2) above the rest: late in a lane,
    its sum overflows the lane's reference; as a lane's first key, the references spread far beyond
    what one common reference holds. Either way pass 1 lists the item and the exact fallback
    recomputes it; the scores still match the oracle. long-late: a head of 16500 keys, whose items
    are ranges of 64 chunks (the last one ragged), with the planted key in the second range."""
    inp = make_inputs("qwen3-14b-long", L=1, B=1, N=16500 if where == "long-late" else 1500)
    G = inp.Hq // inp.Hkv
    pos = {"late": 700, "first": 5, "long-late": 9000}[where]
    for h in range(inp.Hkv):
        q = inp.q_recent[0, 0, h * G, 0].float()
        inp.K[0, 0, h, pos] = (10.0 * q).to(inp.K.dtype)
    gpu = run_evict(inp, DEV, kernel="wide")
    _, gpu_picks = run_score(inp, DEV, kernel="wide")
    ora = O.evict(inp)
    if check_beacon_picks(inp, gpu_picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=gpu_picks)
    assert gpu["status"] == 0
    assert_scores_close(gpu["scores"], ora["scores"], f"wide fallback ({where})")
    check_kept(inp, gpu, ora, gpu["scores"])


@pytest.mark.parametrize("name,over,launches", [
    ("tiny", {}, 1),                                        # the fp32 cluster kernel
    ("qwen3-4b", dict(L=1, N=1000), 3),                     # observation rows, single-read scoring, select+compact
    ("qwen3-14b-long", dict(L=1, B=1, N=2100), 6),          # + wide pass 1, exact fallback, combine, pass 2
    ("qwen3-4b", dict(L=1, Hq=4, Hkv=1, N=70000), 6),       # two-pass streaming kernel, separate select and compact
])
def test_evict_launch_count(name, over, launches):
    """kvc_evict_launch_count (the benchmark's gpu_launches) names the kernels kvc_evict launches."""
    from decoding_kv_cache_gb300 import kvc
    inp = make_inputs(name, device=DEV, **over)
    cache = kvc.Cache(inp.K, inp.V, inp.Hq)
    assert kvc.kvc_evict_launch_count(cache, inp.n_r, inp.n_b) == launches


def test_f32_per_head_budget_out_of_range_is_flagged_and_left_whole():
    """The fp32 cluster kernel's own selection: a head whose budget is below prefix + recent is kept
    whole and flagged, one whose budget equals N is kept whole without a flag, the rest follow the
    oracle."""
    inp = make_inputs("tiny", L=2, B=2, N=300)
    b = torch.full((inp.L, inp.B, inp.Hkv), 250, dtype=torch.int32)
    b[0, 1, 0] = 5     # < prefix + recent
    b[1, 0, 1] = 300   # == N
    b[1, 1, 0] = 20    # == prefix + recent: no middle key kept
    inp.budget = b
    gpu = run_evict(inp, DEV)
    ora = O.evict(inp)
    assert gpu["status"] & 0x1
    assert gpu["kept_len"][0, 1, 0] == 300 and gpu["kept_len"][1, 0, 1] == 300 and gpu["kept_len"][1, 1, 0] == 20
    assert_scores_close(gpu["scores"], ora["scores"], "tiny per-head budgets")
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])


def test_f32_streaming_per_head_budgets():
    """fp32 heads past the cluster kernel's 1024 keys (the streaming passes, then the selection-and-
    compaction CTAs in largest-budget-first order) with budgets that differ per head: below prefix +
    recent (kept whole, flagged), exactly prefix + recent, N, and values in between."""
    inp = make_inputs("tiny", L=2, B=3, N=1500)
    g = torch.Generator().manual_seed(7)
    b = torch.randint(21, 1500, (inp.L, inp.B, inp.Hkv), generator=g, dtype=torch.int32)
    b[0, 0, 0] = 7      # < prefix + recent
    b[0, 2, 1] = 20     # == prefix + recent
    b[1, 1, 0] = 1500   # == N
    inp.budget = b
    gpu = run_evict(inp, DEV)
    ora = O.evict(inp)
    assert gpu["status"] & 0x1
    assert gpu["kept_len"][0, 0, 0] == 1500 and gpu["kept_len"][0, 2, 1] == 20 and gpu["kept_len"][1, 1, 0] == 1500
    assert_scores_close(gpu["scores"], ora["scores"], "tiny streaming per-head budgets")
    check_kept(inp, gpu, ora, gpu["scores"])
    check_compaction(inp, gpu["K"], gpu["V"], gpu["kept_idx"], gpu["kept_len"])
