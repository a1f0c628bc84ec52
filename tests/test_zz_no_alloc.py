"""kvc_score_static: the scoring entry point for callers that cannot allocate device memory
(a runtime that reserved all memory for weights and its KV pool up front, or code running
where allocation is not allowed). Its scratch is a fixed region the library reserves when
it loads, so it must give the same scores as kvc_score with a caller workspace, call after
call, and reject problems too big for the region before launching anything.

Collected last on purpose: if it fails, a run that stops at the first failure has already
run everything else. It passes alone in a fresh process and after the other tests."""
import numpy as np
import pytest
import torch

from decoding_kv_cache_gb300.inputs import make_inputs
from parity_util import assert_scores_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _scores_with_workspace(kvc, inp, cache):
    out = torch.full((inp.L, inp.B, inp.Hkv, inp.N), -1.0, device=DEV)
    kvc.kvc_score(cache, inp.q_recent, inp.qbuf, inp.count, inp.n_b, inp.t, inp.theta, out)
    return out


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
