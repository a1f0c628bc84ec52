"""Failure detection on the GPU without a fault: a bounded wait is made to run out.

The test-only switch `kvc_debug_fault(1)` makes the first CTA of the single-read scoring kernel
withhold its exchange partials (a word that nothing ever writes). Its group's waits must give up
within their bound, raise KVC_STATUS_TIMEOUT in kvc_evict's status word and let the launch
return; the context must stay usable, and the next call must be exact again.
"""
import time

import pytest

from decoding_kv_cache_gb300.inputs import make_inputs
from oracle import oracle as O
from parity_util import assert_scores_close, check_beacon_picks, check_kept, run_evict, run_score

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_withheld_partials_time_out_and_the_context_survives():
    from decoding_kv_cache_gb300 import kvc
    inp = make_inputs("qwen3-4b", L=2, N=1000)  # 128-row observation tiles: the single-read kernel
    kvc.kvc_debug_fault(1)
    try:
        t0 = time.time()
        bad = run_evict(inp, DEV)
        elapsed = time.time() - t0
    finally:
        kvc.kvc_debug_fault(0)
    assert bad["status"] & kvc.KVC_STATUS_TIMEOUT, bad["status"]
    assert not bad["status"] & kvc.KVC_STATUS_BAD_INDEX  # selection still produced valid lists
    assert elapsed < 30.0

    good = run_evict(inp, DEV)
    assert good["status"] == 0
    _, gpu_picks = run_score(inp, DEV)
    ora = O.evict(inp)
    if check_beacon_picks(inp, gpu_picks, ora["beacon_picks"]):
        ora = O.evict(inp, forced_picks=gpu_picks)
    assert_scores_close(good["scores"], ora["scores"], "after the timeout")
    check_kept(inp, good, ora, good["scores"])

