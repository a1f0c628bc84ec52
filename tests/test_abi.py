"""The C-ABI library loads, exports every symbol include/kvc.h declares, and rejects bad
arguments on the host before any CUDA call (none of these tests needs a GPU)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")


@pytest.fixture(scope="module")
def lib():
    from decoding_kv_cache_gb300 import build, kvc
    build.build()
    return kvc.lib()


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"KVC_API\s+[\w\s\*]+?\b(kvc_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("kvc_fps_update", "kvc_score", "kvc_select", "kvc_compact", "kvc_evict"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from decoding_kv_cache_gb300 import kvc
    out = subprocess.run(["nm", "-D", "--defined-only", kvc.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (kvc_\w+)", out))
    assert set(_declared()) <= exported
    assert set(kvc.EXPORTED) == set(_declared())
    assert lib.kvc_abi_version() == kvc.KVC_ABI_VERSION == 5


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER), "-x",
                        "c", "-"], input='#include "kvc.h"\nint main(void){return 0;}\n', capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr


def test_fault_switch_takes_only_known_modes(lib):
    assert lib.kvc_debug_fault(7) == -1
    assert lib.kvc_debug_fault(-1) == -1
    assert lib.kvc_debug_fault(0) == 0


def test_strerror(lib):
    assert lib.kvc_strerror(0) == b"ok"
    assert b"head dimension" in lib.kvc_strerror(-3)
    assert lib.kvc_strerror(-999) == b"unknown error"


def _cache(kvc, **kw):
    base = dict(dtype=0, L=2, B=1, Hq=8, Hkv=2, D=128, N=1024, pad_=0, ncap=1024)
    base.update(kw)
    ptrs = (C.c_void_p * max(base["L"], 1))(*([0x1000] * max(base["L"], 1)))
    c = kvc.kvc_cache(**base, K=C.cast(ptrs, C.POINTER(C.c_void_p)), V=C.cast(ptrs, C.POINTER(C.c_void_p)))
    return c, ptrs


def test_workspace_size_host_only(lib):
    from decoding_kv_cache_gb300 import kvc
    c, _keep = _cache(kvc)
    ws = lib.kvc_score_workspace_size(C.byref(c), 16, 16)
    assert ws > 0
    # scores and kept indices of every head, and the heads' order for the selection and compaction
    assert lib.kvc_evict_workspace_size(C.byref(c), 16, 16) >= ws + 2 * 2 * 2 * 1024 * 4 + 2 * 2 * 4
    bad, _k2 = _cache(kvc, D=96)
    assert lib.kvc_score_workspace_size(C.byref(bad), 16, 16) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), -3),
    (dict(dtype=7), -2),
    (dict(Hq=7), -5),
    (dict(N=0), -1),
    (dict(ncap=10), -1),
    (dict(L=200), -1),
    (dict(pad_=1), -1),
])
def test_evict_rejects_bad_cache_before_launch(lib, kw, code):
    from decoding_kv_cache_gb300 import kvc
    c, _keep = _cache(kvc, **kw)
    rc = lib.kvc_evict(C.byref(c), 0x1000, 16, 0x1000, 0x1000, 32, 16, 1023, 1e6, 4, 16, None, 896, None, 0x1000,
                       None, None, None, 0x100000, 1 << 40, None)
    assert rc == code


def test_evict_rejects_bad_query_and_budget_args(lib):
    from decoding_kv_cache_gb300 import kvc
    c, _keep = _cache(kvc)
    call = lambda **kw: lib.kvc_evict(
        C.byref(c), kw.get("qr", 0x1000), kw.get("n_r", 16), 0x1000, 0x1000, kw.get("qmax", 32), kw.get("n_b", 16),
        1023, kw.get("theta", 1e6), 4, 16, None, kw.get("budget_all", 896), None, kw.get("kept_len", 0x1000), None,
        None, kw.get("opts"), kw.get("ws", 0x100000), kw.get("wsb", 1 << 40), None)
    assert call(n_b=40) == -1                 # more beacons than the buffer holds
    assert call(qmax=65, n_b=16) == -1         # buffer larger than supported
    assert call(n_r=0, n_b=0) == -1            # no observation rows
    assert call(theta=1.0) == -1
    assert call(kept_len=None) == -1
    assert call(budget_all=19) == -4           # below prefix + recent
    assert call(wsb=16) == -7                  # workspace too small
    assert call(ws=0x100010) == -7             # workspace not 256-byte aligned
    assert call(qr=0x1004) == -8               # misaligned query pointer
    assert call(n_r=64, n_b=32, qmax=64) == -9  # 4 * 96 observation rows > 256
    o = lambda **kw: C.byref(kvc.kvc_opts(**{**dict(row_agg=0, group_agg=0, head_budget=0, kernel=0), **kw}))
    assert call(opts=o(row_agg=2)) == -1        # sum is not a row aggregation
    assert call(opts=o(group_agg=1)) == -1      # nor mean a group aggregation
    assert call(opts=o(head_budget=2)) == -1
    assert call(opts=o(kernel=5)) == -1
    assert call(opts=o(kernel=-1)) == -1
    assert call(opts=o(entropy=0x1002)) == -8   # entropy output not 4-byte aligned
    assert call(opts=o(head_budget=1, entropy=0x1004), wsb=16) == -7  # options fine: reaches the workspace check


def test_variant_row_layout_limit(lib):
    """The variants start each query head's rows on a 16-row boundary: 3 heads of 81 rows fit the
    256-row tile (243) but not once padded (96 + 96 + 81 = 273)."""
    from decoding_kv_cache_gb300 import kvc
    c, _keep = _cache(kvc, Hq=6)
    call = lambda opts: lib.kvc_evict(C.byref(c), 0x1000, 64, 0x1000, 0x1000, 18, 17, 1023, 1e6, 4, 16, None, 896,
                                      None, 0x1000, None, None, opts, 0x100000, 16, None)
    assert call(None) == -7  # accepted up to the (too small) workspace
    o = kvc.kvc_opts(row_agg=1, group_agg=0, head_budget=0, kernel=0, entropy=None)
    assert call(C.byref(o)) == -9
    assert lib.kvc_score_workspace_size(C.byref(c), 64, 17) > 0


def test_head_budget_rejects_bad_args(lib):
    assert lib.kvc_head_budget(None, 1, 1, 4, 100, 4, 16, None, 60, 0x1000, None, None) == -1
    assert lib.kvc_head_budget(0x1000, 1, 1, 65, 100, 4, 16, None, 60, 0x1000, None, None) == -9
    assert lib.kvc_head_budget(0x1000, 1, 1, 4, 100, 4, 16, None, 19, 0x1000, None, None) == -4


def test_select_and_fps_reject_bad_args(lib):
    assert lib.kvc_select(None, 1, 1, 1, 10, 4, 4, None, 8, 0x1000, 0x1000, None, None) == -1
    assert lib.kvc_select(0x1000, 1, 1, 1, 100, 4, 16, None, 19, 0x1000, 0x1000, None, None) == -4
    assert lib.kvc_fps_update(0, 1, 1, 4, 128, 0x1000, 31, 0x1000, None, None, None) == -5
    assert lib.kvc_fps_update(0, 1, 1, 4, 100, 0x1000, 32, 0x1000, None, None, None) == -3
    assert lib.kvc_fps_update(3, 1, 1, 4, 128, 0x1000, 32, 0x1000, None, None, None) == -2
    assert lib.kvc_fps_update(0, 1, 1, 4, 128, 0x1008, 32, 0x1000, None, None, None) == -8


def test_append_rejects_bad_args(lib):
    call = lambda **kw: lib.kvc_append(
        kw.get("dtype", 0), 1, 1, 4, kw.get("D", 128), kw.get("q_pre", 0x1000), kw.get("q_post", None),
        kw.get("t", 5), kw.get("theta", 1e6), kw.get("qbuf", 0x1000), kw.get("qmax", 32), kw.get("count", 0x1000),
        kw.get("ring", 0x1000), kw.get("n_r", 16), None, None, None)
    assert call(qmax=31) == -5               # odd buffer
    assert call(qmax=66) == -1               # larger than supported
    assert call(D=100) == -3
    assert call(dtype=3) == -2
    assert call(q_pre=0x1008) == -8          # misaligned
    assert call(q_post=0x1004) == -8
    assert call(ring=None) == -1             # a ring is needed when n_r > 0
    assert call(theta=1.0) == -1             # rotation needs a base > 1 without q_post
    assert call(t=-1) == -1
    assert call(count=None) == -1
    assert call(n_r=65) == -1


def test_epikv_rejects_bad_args(lib):
    ws = lambda **kw: (kw.get("ws", 0x100000), kw.get("wsb", 1 << 40))
    call = lambda **kw: lib.kvc_epikv_score(kw.get("dtype", 0), kw.get("B", 2), kw.get("N", 100), kw.get("dm", 4096),
                                            kw.get("hA", 0x1000), kw.get("hB", 0x1000), kw.get("W", 128),
                                            kw.get("eps", 1e-6), None, kw.get("sc", 0x1000), *ws(**kw), None)
    assert call(dtype=5) == -2
    assert call(dm=4100) == -3                # not a whole number of 16-byte vectors
    assert call(dm=8200) == -3 or call(dm=8200) == -3
    assert call(dm=16384) == -3               # wider than the kernel's registers hold
    assert call(dtype=1, dm=8192) == -3
    assert call(W=0) == -1
    assert call(eps=0.0) == -1                # a constant window needs eps > 0
    assert call(hA=0x1008) == -8
    assert call(sc=None) == -1
    assert call(wsb=16) == -7
    assert lib.kvc_epikv_workspace_size(2, 100) > 2 * 2 * 100 * 4
    assert lib.kvc_epikv_workspace_size(0, 100) == 0
