"""Thin Python binding over libkvc's C ABI (``include/kvc.h``).

Argument marshalling only: tensors are passed as device pointers, sizes are read from
their shapes, and every launch happens inside libkvc on the current torch stream. There
is no fallback: if ``libkvc.so`` is missing the import of this module's functions fails.
Names and argument order follow the C entry points.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence, Union

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvc.so")

KVC_BF16, KVC_F32 = 0, 1
KVC_STATUS_BUDGET_RANGE, KVC_STATUS_COUNT_RANGE, KVC_STATUS_BAD_INDEX, KVC_STATUS_TIMEOUT = 0x1, 0x2, 0x4, 0x8
KVC_MAX_LAYERS = 128

EXPORTED = ("kvc_fps_update", "kvc_score_workspace_size", "kvc_score", "kvc_select", "kvc_compact",
            "kvc_evict_workspace_size", "kvc_evict", "kvc_evict_launch_count", "kvc_strerror", "kvc_abi_version",
            "kvc_score_static", "kvc_debug_fault", "kvc_head_budget", "kvc_append", "kvc_epikv_workspace_size",
            "kvc_epikv_score", "kvc_epikv_evict")
KVC_ABI_VERSION = 5
KVC_AGG_MAX, KVC_AGG_MEAN, KVC_AGG_SUM = 0, 1, 2
KVC_BUDGET_GIVEN, KVC_BUDGET_ENTROPY = 0, 1
ROW_AGG = {"max": KVC_AGG_MAX, "mean": KVC_AGG_MEAN}
GROUP_AGG = {"max": KVC_AGG_MAX, "sum": KVC_AGG_SUM}
HEAD_BUDGET = {"given": KVC_BUDGET_GIVEN, "entropy": KVC_BUDGET_ENTROPY}
# bf16 scoring kernel (a test and profiling aid; every kernel computes the same scores)
KERNEL = {"auto": 0, "resident": 1, "split": 2, "fused": 3, "wide": 4}
KVC_STATIC_SCRATCH_BYTES = 16 << 20


class KvcError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libkvc error {code}: {msg}")
        self.code = code


class kvc_cache(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("L", C.c_int32), ("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32),
                ("D", C.c_int32), ("N", C.c_int32), ("pad_", C.c_int32), ("ncap", C.c_int64),
                ("K", C.POINTER(C.c_void_p)), ("V", C.POINTER(C.c_void_p))]


class kvc_opts(C.Structure):
    _fields_ = [("row_agg", C.c_int32), ("group_agg", C.c_int32), ("head_budget", C.c_int32),
                ("kernel", C.c_int32), ("entropy", C.c_void_p)]


_lib = None


def lib():
    """Load libkvc.so (built by ``decoding_kv_cache_gb300.build``); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m decoding_kv_cache_gb300.build` "
                          "(or __graft_entry__.build()) first")
    L = C.CDLL(LIB_PATH)
    vp, i32, i64, dbl, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_double, C.c_size_t
    pc = C.POINTER(kvc_cache)
    po = C.POINTER(kvc_opts)
    sig = {
        "kvc_fps_update": (C.c_int, [i32, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp]),
        "kvc_append": (C.c_int, [i32, i32, i32, i32, i32, vp, vp, i64, dbl, vp, i32, vp, vp, i32, vp, vp, vp]),
        "kvc_score_workspace_size": (sz, [pc, i32, i32]),
        "kvc_score": (C.c_int, [pc, vp, i32, vp, vp, i32, i32, i64, dbl, vp, vp, po, vp, sz, vp]),
        "kvc_select": (C.c_int, [vp, i32, i32, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp]),
        "kvc_compact": (C.c_int, [pc, vp, vp, vp, vp]),
        "kvc_evict_workspace_size": (sz, [pc, i32, i32]),
        "kvc_evict": (C.c_int, [pc, vp, i32, vp, vp, i32, i32, i64, dbl, i32, i32, vp, i32, vp, vp, vp, vp, po, vp,
                                sz, vp]),
        "kvc_evict_launch_count": (C.c_int, [pc, i32, i32]),
        "kvc_score_static": (C.c_int, [pc, vp, i32, vp, vp, i32, i32, i64, dbl, vp, vp, po, vp]),
        "kvc_head_budget": (C.c_int, [vp, i32, i32, i32, i32, i32, i32, vp, i32, vp, vp, vp]),
        "kvc_epikv_workspace_size": (sz, [i32, i32]),
        "kvc_epikv_score": (C.c_int, [i32, i32, i32, i32, vp, vp, i32, C.c_float, vp, vp, vp, sz, vp]),
        "kvc_epikv_evict": (C.c_int, [pc, vp, vp, i32, i32, C.c_float, i32, i32, vp, i32, vp, vp, vp, vp, vp, sz, vp]),
        "kvc_strerror": (C.c_char_p, [C.c_int]),
        "kvc_abi_version": (C.c_int, []),
        "kvc_debug_fault": (C.c_int, [i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(rc: int):
    if rc != 0:
        raise KvcError(rc, lib().kvc_strerror(rc).decode())


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libkvc takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libkvc takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KVC_BF16
    if t.dtype == torch.float32:
        return KVC_F32
    raise KvcError(-2, f"unsupported storage type {t.dtype}")


class Cache:
    """A ``kvc_cache`` over torch tensors: K/V either one [L,B,Hkv,ncap,D] tensor each or lists of
    per-layer [B,Hkv,ncap,D] tensors. ``N`` is the number of valid tokens per head (default ncap)."""

    def __init__(self, K: Union[torch.Tensor, Sequence[torch.Tensor]], V, Hq: int, N: Optional[int] = None):
        Ks = list(K.unbind(0)) if isinstance(K, torch.Tensor) else list(K)
        Vs = list(V.unbind(0)) if isinstance(V, torch.Tensor) else list(V)
        if len(Ks) != len(Vs) or not Ks:
            raise ValueError("K and V need the same, non-zero number of layers")
        B, Hkv, ncap, D = Ks[0].shape
        for t in Ks + Vs:
            if tuple(t.shape) != (B, Hkv, ncap, D) or t.dtype != Ks[0].dtype or not t.is_contiguous():
                raise ValueError("every layer of K and V must be a contiguous [B,Hkv,ncap,D] tensor of one dtype")
        self.layers_K, self.layers_V = Ks, Vs
        self._kp = (C.c_void_p * len(Ks))(*[t.data_ptr() for t in Ks])
        self._vp = (C.c_void_p * len(Vs))(*[t.data_ptr() for t in Vs])
        self.c = kvc_cache(dtype=_dtype_code(Ks[0]), L=len(Ks), B=B, Hq=Hq, Hkv=Hkv, D=D,
                           N=ncap if N is None else N, pad_=0, ncap=ncap,
                           K=C.cast(self._kp, C.POINTER(C.c_void_p)), V=C.cast(self._vp, C.POINTER(C.c_void_p)))

    @property
    def ref(self):
        return C.byref(self.c)

    @property
    def heads(self) -> int:
        return self.c.L * self.c.B * self.c.Hkv


def kvc_fps_update(qbuf: torch.Tensor, count: torch.Tensor, picks: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None):
    """Continual-FPS compression of every full [..., qmax, D] buffer in place (see kvc.h).
    ``count`` holds one int32 per buffer; ``picks`` (optional) is [..., qmax/2] int32."""
    qmax, D = qbuf.shape[-2], qbuf.shape[-1]
    nq = qbuf.numel() // (qmax * D)
    _check(lib().kvc_fps_update(_dtype_code(qbuf), 1, 1, nq, D, _p(qbuf), qmax, _p(count), _p(picks), _p(status),
                                _stream(stream)))


def kvc_append(q_pre: torch.Tensor, qbuf: torch.Tensor, count: torch.Tensor, q_recent: Optional[torch.Tensor],
               t: int, rope_theta: float = 1e4, q_post: Optional[torch.Tensor] = None,
               picks: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None, stream=None):
    """One decode step's queries into the observation state (see kvc.h): ``q_pre`` [..., D] joins
    each head's [..., qmax, D] buffer (compressed when full), and ``q_post`` (or ``q_pre`` turned to
    ``t``) joins ring row ``t mod n_r`` of ``q_recent`` [..., n_r, D] (None or n_r = 0: no ring)."""
    qmax, D = qbuf.shape[-2], qbuf.shape[-1]
    nq = qbuf.numel() // (qmax * D)
    if q_pre.numel() != nq * D or (q_post is not None and q_post.numel() != nq * D):
        raise ValueError("q_pre / q_post need one [D] row per buffer")
    n_r = 0 if q_recent is None else q_recent.shape[-2]
    if q_recent is not None and q_recent.numel() != nq * n_r * D:
        raise ValueError("q_recent needs one [n_r, D] ring per buffer")
    _check(lib().kvc_append(_dtype_code(qbuf), 1, 1, nq, D, _p(q_pre), _p(q_post), int(t), float(rope_theta),
                            _p(qbuf), qmax, _p(count), _p(q_recent) if n_r else None, n_r, _p(picks), _p(status),
                            _stream(stream)))


def kvc_score_workspace_size(cache: Cache, n_r: int, n_b: int) -> int:
    return int(lib().kvc_score_workspace_size(cache.ref, n_r, n_b))


def kvc_evict_workspace_size(cache: Cache, n_r: int, n_b: int) -> int:
    return int(lib().kvc_evict_workspace_size(cache.ref, n_r, n_b))


def kvc_evict_launch_count(cache: Cache, n_r: int, n_b: int) -> int:
    return int(lib().kvc_evict_launch_count(cache.ref, n_r, n_b))


def kvc_debug_fault(mode: int) -> None:
    """Test-only fault switch (see include/kvc.h): 1 makes the scoring exchange wait run out."""
    _check(lib().kvc_debug_fault(int(mode)))


def make_opts(row_agg: str = "max", group_agg: str = "max", head_budget: str = "given",
              entropy: Optional[torch.Tensor] = None, kernel: str = "auto"):
    """A ``kvc_opts`` (see kvc.h), or None for the defaults (max/max, budgets as given, no entropy,
    automatic kernel choice)."""
    if row_agg == "max" and group_agg == "max" and head_budget == "given" and entropy is None and kernel == "auto":
        return None
    return kvc_opts(row_agg=ROW_AGG[row_agg], group_agg=GROUP_AGG[group_agg], head_budget=HEAD_BUDGET[head_budget],
                    kernel=KERNEL[kernel], entropy=_p(entropy))


def _opts_ref(o):
    return None if o is None else C.byref(o)


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def kvc_score(cache: Cache, q_recent: torch.Tensor, qbuf: torch.Tensor, count: torch.Tensor, n_b: int, t: int,
              rope_theta: float, scores: torch.Tensor, beacon_picks: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, stream=None, row_agg: str = "max", group_agg: str = "max",
              entropy: Optional[torch.Tensor] = None, kernel: str = "auto"):
    """Scores of every cached key; ``row_agg``/``group_agg``/``entropy``/``kernel`` set kvc_opts."""
    n_r, qmax = q_recent.shape[-2], qbuf.shape[-2]
    ws = _workspace(kvc_score_workspace_size(cache, n_r, n_b), scores.device, workspace)
    o = make_opts(row_agg, group_agg, "given", entropy, kernel)
    _check(lib().kvc_score(cache.ref, _p(q_recent), n_r, _p(qbuf), _p(count), qmax, n_b, int(t), float(rope_theta),
                           _p(scores), _p(beacon_picks), _opts_ref(o), _p(ws), ws.numel() * ws.element_size(),
                           _stream(stream)))


def kvc_score_static(cache: Cache, q_recent: torch.Tensor, qbuf: torch.Tensor, count: torch.Tensor, n_b: int,
                     t: int, rope_theta: float, scores: torch.Tensor, beacon_picks: Optional[torch.Tensor] = None,
                     stream=None, row_agg: str = "max", group_agg: str = "max",
                     entropy: Optional[torch.Tensor] = None, kernel: str = "auto"):
    """kvc_score with the library's fixed scratch region instead of a workspace (allocates nothing;
    see kvc.h for the size limit and the sharing rules)."""
    n_r, qmax = q_recent.shape[-2], qbuf.shape[-2]
    o = make_opts(row_agg, group_agg, "given", entropy, kernel)
    _check(lib().kvc_score_static(cache.ref, _p(q_recent), n_r, _p(qbuf), _p(count), qmax, n_b, int(t),
                                  float(rope_theta), _p(scores), _p(beacon_picks), _opts_ref(o), _stream(stream)))


def kvc_select(scores: torch.Tensor, prefix: int, recent: int, kept_idx: torch.Tensor, kept_len: torch.Tensor,
               budget: Optional[torch.Tensor] = None, budget_all: int = 0, status: Optional[torch.Tensor] = None,
               stream=None):
    L, B, Hkv, N = scores.shape
    _check(lib().kvc_select(_p(scores), L, B, Hkv, N, prefix, recent, _p(budget), int(budget_all), _p(kept_idx),
                            _p(kept_len), _p(status), _stream(stream)))


def kvc_compact(cache: Cache, kept_idx: torch.Tensor, kept_len: torch.Tensor, status: Optional[torch.Tensor] = None,
                stream=None):
    _check(lib().kvc_compact(cache.ref, _p(kept_idx), _p(kept_len), _p(status), _stream(stream)))


def kvc_evict(cache: Cache, q_recent: torch.Tensor, qbuf: torch.Tensor, count: torch.Tensor, n_b: int, t: int,
              rope_theta: float, prefix: int, recent: int, kept_len: torch.Tensor,
              budget: Optional[torch.Tensor] = None, budget_all: int = 0, kept_idx: Optional[torch.Tensor] = None,
              scores: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, stream=None, row_agg: str = "max", group_agg: str = "max",
              head_budget: str = "given", entropy: Optional[torch.Tensor] = None, kernel: str = "auto"):
    """The whole eviction step (beacons, scores, selection, in-place compaction) on one stream.
    ``row_agg``/``group_agg``/``head_budget``/``entropy``/``kernel`` set kvc_opts."""
    n_r, qmax = q_recent.shape[-2], qbuf.shape[-2]
    ws = _workspace(kvc_evict_workspace_size(cache, n_r, n_b), kept_len.device, workspace)
    o = make_opts(row_agg, group_agg, head_budget, entropy, kernel)
    _check(lib().kvc_evict(cache.ref, _p(q_recent), n_r, _p(qbuf), _p(count), qmax, n_b, int(t), float(rope_theta),
                           prefix, recent, _p(budget), int(budget_all), _p(kept_idx), _p(kept_len), _p(scores),
                           _p(status), _opts_ref(o), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def kvc_head_budget(entropy: torch.Tensor, N: int, prefix: int, recent: int, budget_out: torch.Tensor,
                    budget: Optional[torch.Tensor] = None, budget_all: int = 0, status: Optional[torch.Tensor] = None,
                    stream=None):
    """Each (layer, sequence)'s budgets reallocated over its heads by entropy (see kvc.h)."""
    L, B, Hkv = entropy.shape
    _check(lib().kvc_head_budget(_p(entropy), L, B, Hkv, int(N), int(prefix), int(recent), _p(budget),
                                 int(budget_all), _p(budget_out), _p(status), _stream(stream)))


def kvc_epikv_workspace_size(B: int, N: int) -> int:
    return int(lib().kvc_epikv_workspace_size(B, N))


def kvc_epikv_score(hA: torch.Tensor, hB: torch.Tensor, window: int, eps: float, scores: torch.Tensor,
                    g: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """EPIKV scores [B, N] from two layers' hidden states [B, N, dm] (see kvc.h); ``g`` [2, B, N]
    optionally receives the two layers' signals."""
    B, N, dm = hA.shape
    if tuple(hB.shape) != (B, N, dm) or hB.dtype != hA.dtype:
        raise ValueError("hA and hB must be [B, N, dm] tensors of one dtype")
    ws = _workspace(kvc_epikv_workspace_size(B, N), hA.device, workspace)
    _check(lib().kvc_epikv_score(_dtype_code(hA), B, N, dm, _p(hA), _p(hB), int(window), float(eps), _p(g),
                                 _p(scores), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def kvc_epikv_evict(cache: Cache, hA: torch.Tensor, hB: torch.Tensor, window: int, eps: float, prefix: int,
                    recent: int, kept_len: torch.Tensor, budget: Optional[torch.Tensor] = None, budget_all: int = 0,
                    kept_idx: Optional[torch.Tensor] = None, scores: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Eviction by the EPIKV score: one kept list per sequence compacts all its layers and heads."""
    B, N, dm = hA.shape
    ws = _workspace(kvc_epikv_workspace_size(B, N), hA.device, workspace)
    _check(lib().kvc_epikv_evict(cache.ref, _p(hA), _p(hB), dm, int(window), float(eps), int(prefix), int(recent),
                                 _p(budget), int(budget_all), _p(kept_idx), _p(kept_len), _p(scores), _p(status),
                                 _p(ws), ws.numel() * ws.element_size(), _stream(stream)))
