"""Python access to the CPU oracle (``kvc_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the benchmark's CPU-baseline leg. The product path never imports it.

The oracle is plain C with fp64 arithmetic; this module only builds it with
gcc, marshals numpy/torch CPU arrays into it and hands results back. See the
C file's header for which passage of the pages each step follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_LIB = os.path.join(_HERE, "libkvc_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: it must build on x86 and Arm alike)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-o", tmp,
                        _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("L", C.c_int32), ("B", C.c_int32), ("Hq", C.c_int32),
                ("Hkv", C.c_int32), ("D", C.c_int32), ("N", C.c_int32), ("n_r", C.c_int32),
                ("n_b", C.c_int32), ("qmax", C.c_int32), ("prefix", C.c_int32), ("recent", C.c_int32),
                ("budget_all", C.c_int32), ("t", C.c_int64), ("theta", C.c_double),
                ("K", C.c_void_p), ("V", C.c_void_p), ("q_recent", C.c_void_p), ("qbuf", C.c_void_p),
                ("count", C.c_void_p), ("budget", C.c_void_p), ("forced_picks", C.c_void_p),
                ("row_agg", C.c_int32), ("group_agg", C.c_int32), ("head_budget", C.c_int32), ("pad_", C.c_int32),
                ("forced_entropy", C.c_void_p)]


class _Outputs(C.Structure):
    _fields_ = [("scores", C.c_void_p), ("kept_idx", C.c_void_p), ("kept_len", C.c_void_p),
                ("K_out", C.c_void_p), ("V_out", C.c_void_p), ("beacon_picks", C.c_void_p),
                ("error", C.c_void_p), ("entropy", C.c_void_p), ("budget_used", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        L.oracle_f64_to_bf16.restype = C.c_uint16
        L.oracle_f64_to_bf16.argtypes = [C.c_double]
        L.oracle_fps_f64.restype = C.c_int
        L.oracle_fps_f64.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
        L.oracle_fps_check_f64.restype = C.c_int
        L.oracle_fps_check_f64.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_double]
        L.oracle_rope_f64.restype = None
        L.oracle_rope_f64.argtypes = [C.c_void_p, C.c_int, C.c_longlong, C.c_double, C.c_void_p]
        L.oracle_rope_f32.restype = None
        L.oracle_rope_f32.argtypes = [C.c_void_p, C.c_int, C.c_longlong, C.c_double, C.c_void_p]
        L.oracle_score_f64.restype = None
        L.oracle_score_f64.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.oracle_score_agg_f64.restype = C.c_int
        L.oracle_score_agg_f64.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_int,
                                           C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.oracle_head_budget.restype = C.c_int
        L.oracle_head_budget.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.oracle_select.restype = C.c_int
        L.oracle_select.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p]
        L.oracle_evict.restype = C.c_int
        L.oracle_evict.argtypes = [C.POINTER(_Problem), C.POINTER(_Outputs), C.c_void_p, C.c_int64]
        L.oracle_fps_update.restype = C.c_int
        L.oracle_fps_update.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                        C.c_void_p]
        L.oracle_append.restype = C.c_int
        L.oracle_append.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_double,
                                    C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]
        L.oracle_epikv_score.restype = C.c_int
        L.oracle_epikv_score.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32,
                                         C.c_double, C.c_void_p, C.c_void_p]
        L.oracle_epikv_z.restype = C.c_int
        L.oracle_epikv_z.argtypes = [C.c_int32, C.c_int32, C.c_void_p, C.c_int32, C.c_double, C.c_void_p]
        L.oracle_set_threads.restype = C.c_int
        L.oracle_set_threads.argtypes = [C.c_int]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def set_threads(n: int = 0) -> int:
    """Set (n > 0) and return the oracle's OpenMP thread count."""
    return lib().oracle_set_threads(int(n))


# ---------------------------------------------------------------------------
# Single steps, on plain fp64 numpy arrays
# ---------------------------------------------------------------------------

def f64_to_bf16_bits(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    f = lib().oracle_f64_to_bf16
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def fps(x, m: int, trace: bool = False):
    """Greedy FPS of m rows of x [n, D]; returns ascending picks (and order, gaps if trace)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    n, D = x.shape
    picks = np.zeros(m, dtype=np.int32)
    order = np.zeros(m, dtype=np.int32)
    gaps = np.zeros(m, dtype=np.float64)
    rc = lib().oracle_fps_f64(_ptr(x), n, D, m, _ptr(picks), _ptr(order), _ptr(gaps))
    if rc:
        raise ValueError("oracle_fps_f64: bad sizes")
    return (picks, order, gaps) if trace else picks


def fps_check(x, picks, tol: float = 1e-5) -> int:
    """0 if ascending ``picks`` is a greedy FPS result of x up to near-ties within ``tol``."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    p = np.ascontiguousarray(picks, dtype=np.int32)
    return lib().oracle_fps_check_f64(_ptr(x), x.shape[0], x.shape[1], _ptr(p), len(p), float(tol))


def rope(x, pos: int, theta: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    flat_in = x.reshape(-1, x.shape[-1])
    flat_out = out.reshape(-1, x.shape[-1])
    for i in range(flat_in.shape[0]):
        lib().oracle_rope_f64(_ptr(flat_in[i]), x.shape[-1], int(pos), float(theta), _ptr(flat_out[i]))
    return out


def rope_f32(x, pos: int, theta: float) -> np.ndarray:
    """The binary32 beacon rotation (the one whose result is rounded to the storage type)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    flat_in = x.reshape(-1, x.shape[-1])
    flat_out = out.reshape(-1, x.shape[-1])
    for i in range(flat_in.shape[0]):
        lib().oracle_rope_f32(_ptr(flat_in[i]), x.shape[-1], int(pos), float(theta), _ptr(flat_out[i]))
    return out


def score(q, k, with_lse: bool = False):
    """max over rows of softmax(q k^T / sqrt(D)) per key, fp64."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    M, D = q.shape
    N = k.shape[0]
    out = np.zeros(N, dtype=np.float64)
    lse = np.zeros(max(M, 1), dtype=np.float64)
    lib().oracle_score_f64(_ptr(q), M, _ptr(k), N, D, _ptr(out), _ptr(lse))
    return (out, lse[:M]) if with_lse else out


ROW_AGG = {"max": 0, "mean": 1}
GROUP_AGG = {"max": 0, "sum": 2}
HEAD_BUDGET = {"given": 0, "entropy": 1}


def score_agg(q, row_head, G: int, k, row_agg: str = "max", group_agg: str = "max"):
    """Scores under the aggregation variants and the normalised entropy, fp64.

    q [M, D] rows, row_head [M] query head of each row (0..G-1), k [N, D] keys. Returns
    (scores [N], entropy) where entropy = mean over rows of H_r / ln N."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    rh = np.ascontiguousarray(row_head, dtype=np.int32)
    M, D = q.shape
    N = k.shape[0]
    out = np.zeros(N, dtype=np.float64)
    ent = np.zeros(1, dtype=np.float64)
    rc = lib().oracle_score_agg_f64(_ptr(q), _ptr(rh), M, G, _ptr(k), N, D, ROW_AGG[row_agg], GROUP_AGG[group_agg],
                                    _ptr(out), _ptr(ent))
    if rc:
        raise ValueError("oracle_score_agg_f64: bad mode or row_head")
    return out, float(ent[0])


def head_budget(entropy, N: int, prefix: int, recent: int, given):
    """Budgets of one layer's heads reallocated by entropy (see oracle_head_budget), or None when a
    given budget is below prefix + recent."""
    e = np.ascontiguousarray(entropy, dtype=np.float32)
    g = np.ascontiguousarray(given, dtype=np.int32)
    out = np.zeros(len(e), dtype=np.int32)
    rc = lib().oracle_head_budget(_ptr(e), len(e), int(N), int(prefix), int(recent), _ptr(g), _ptr(out))
    return None if rc else out


def select(scores, prefix: int, recent: int, budget: int):
    """Kept indices (ascending) or None when the budget cannot hold prefix + recent."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    kept = np.zeros(len(s), dtype=np.int32)
    n = lib().oracle_select(_ptr(s), len(s), prefix, recent, int(budget), _ptr(kept))
    return None if n < 0 else kept[:n].copy()


# ---------------------------------------------------------------------------
# The whole step on an EvictInputs (torch CPU tensors)
# ---------------------------------------------------------------------------

def _np_storage(t):
    """torch CPU tensor -> numpy array of its stored bits (bf16 as uint16)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.int32:
        return t.numpy()
    raise TypeError(t.dtype)


def evict(inp, heads: Optional[Sequence[int]] = None, forced_picks=None, threads: int = 0, row_agg: str = "max",
          group_agg: str = "max", head_budget: str = "given", forced_entropy=None):
    """Run the oracle's eviction step on ``inp`` (an ``EvictInputs`` with CPU tensors).

    Returns a dict of numpy arrays: scores [L,B,Hkv,N] f32, kept_idx [L,B,Hkv,N] (-1 past kept_len),
    kept_len [L,B,Hkv], K_out/V_out (storage bits, compacted copies), beacon_picks [L,B,Hq,n_b],
    error [L,B,Hkv], entropy [L,B,Hkv] (normalised attention entropy), budget_used [L,B,Hkv].
    ``heads`` restricts the work to flat head ids (others stay zero / copied). ``row_agg`` /
    ``group_agg`` pick the aggregation variant, ``head_budget="entropy"`` reallocates each layer's
    budget over its heads by entropy (``forced_entropy`` [L,B,Hkv] replaces the oracle's entropies
    in that decision).
    """
    if threads:
        set_threads(threads)
    K = _np_storage(inp.K)
    V = _np_storage(inp.V)
    qr = _np_storage(inp.q_recent)
    qb = _np_storage(inp.qbuf)
    cnt = _np_storage(inp.count.to(dtype=__import__("torch").int32))
    bud = None if inp.budget is None else _np_storage(inp.budget.to(dtype=__import__("torch").int32))
    fp = None if forced_picks is None else np.ascontiguousarray(forced_picks, dtype=np.int32)
    fe = None if forced_entropy is None else np.ascontiguousarray(forced_entropy, dtype=np.float32)
    L, B, Hq, Hkv, N = inp.L, inp.B, inp.Hq, inp.Hkv, inp.N
    p = _Problem(dtype=0 if inp.dtype == "bf16" else 1, L=L, B=B, Hq=Hq, Hkv=Hkv, D=inp.D, N=N,
                 n_r=inp.n_r, n_b=inp.n_b, qmax=inp.qmax, prefix=inp.prefix, recent=inp.recent,
                 budget_all=inp.budget_all, t=inp.t, theta=inp.theta, K=_ptr(K).value, V=_ptr(V).value,
                 q_recent=_ptr(qr).value, qbuf=_ptr(qb).value, count=_ptr(cnt).value,
                 budget=None if bud is None else _ptr(bud).value,
                 forced_picks=None if fp is None else _ptr(fp).value, row_agg=ROW_AGG[row_agg],
                 group_agg=GROUP_AGG[group_agg], head_budget=HEAD_BUDGET[head_budget], pad_=0,
                 forced_entropy=None if fe is None else _ptr(fe).value)
    out = dict(scores=np.zeros((L, B, Hkv, N), np.float32), kept_idx=np.full((L, B, Hkv, N), -1, np.int32),
               kept_len=np.zeros((L, B, Hkv), np.int32), K_out=K.copy(), V_out=V.copy(),
               beacon_picks=np.full((L, B, Hq, inp.n_b), -1, np.int32), error=np.zeros((L, B, Hkv), np.int32),
               entropy=np.zeros((L, B, Hkv), np.float32), budget_used=np.zeros((L, B, Hkv), np.int32))
    o = _Outputs(**{k: _ptr(v).value for k, v in out.items()})
    hv = None if heads is None else np.ascontiguousarray(heads, dtype=np.int64)
    rc = lib().oracle_evict(C.byref(p), C.byref(o), None if hv is None else _ptr(hv), 0 if hv is None else len(hv))
    if rc:
        raise ValueError("oracle_evict: bad sizes")
    return out


def fps_update(qbuf_bits: np.ndarray, count: np.ndarray, qmax: int, dtype: str, threads: int = 0):
    """Continual-FPS compression of full buffers; returns (qbuf, count, picks) as new arrays."""
    if threads:
        set_threads(threads)
    qb = np.ascontiguousarray(qbuf_bits).copy()
    cnt = np.ascontiguousarray(count, dtype=np.int32).copy()
    nq = cnt.size
    D = qb.shape[-1]
    picks = np.full((nq, qmax // 2), -1, np.int32)
    rc = lib().oracle_fps_update(0 if dtype == "bf16" else 1, nq, D, _ptr(qb), qmax, _ptr(cnt), _ptr(picks))
    if rc < 0:
        raise ValueError("oracle_fps_update: bad sizes")
    return qb, cnt, picks.reshape(count.shape + (qmax // 2,))


def append(q_pre_bits: np.ndarray, q_post_bits, t: int, theta: float, qbuf_bits: np.ndarray, count: np.ndarray,
           q_recent_bits: np.ndarray, dtype: str, threads: int = 0):
    """One decode step's append (see oracle_append) on copies; returns (qbuf, count, q_recent, picks,
    error). Arrays hold storage bits (uint16 for bf16), flattened over query heads in front:
    q_pre [nq, D], q_post [nq, D] or None, qbuf [nq, qmax, D], count [nq], q_recent [nq, n_r, D]."""
    if threads:
        set_threads(threads)
    qb = np.ascontiguousarray(qbuf_bits).copy()
    cnt = np.ascontiguousarray(count, dtype=np.int32).copy()
    qr = np.ascontiguousarray(q_recent_bits).copy()
    qp = np.ascontiguousarray(q_pre_bits)
    qo = None if q_post_bits is None else np.ascontiguousarray(q_post_bits)
    nq, qmax, D = qb.shape[0], qb.shape[1], qb.shape[2]
    n_r = qr.shape[1]
    picks = np.full((nq, qmax // 2), -1, np.int32)
    err = np.zeros(nq, np.int32)
    rc = lib().oracle_append(0 if dtype == "bf16" else 1, nq, D, _ptr(qp), _ptr(qo), int(t), float(theta), _ptr(qb),
                             qmax, _ptr(cnt), _ptr(qr), n_r, _ptr(picks), _ptr(err))
    if rc < 0:
        raise ValueError("oracle_append: bad sizes")
    return qb, cnt, qr, picks, err


def epikv_score(hA_bits: np.ndarray, hB_bits: np.ndarray, window: int, eps: float, dtype: str, threads: int = 0):
    """EPIKV signal and score (see oracle_epikv_score): hA, hB [B, N, dm] as storage bits (uint16 for
    bf16, float32 otherwise). Returns (g [2, B, N], score [B, N]) in fp64."""
    if threads:
        set_threads(threads)
    a = np.ascontiguousarray(hA_bits)
    b = np.ascontiguousarray(hB_bits)
    if a.shape != b.shape or a.ndim != 3:
        raise ValueError("hA and hB must be [B, N, dm] of one shape")
    B, N, dm = a.shape
    g = np.zeros((2, B, N), np.float64)
    sc = np.zeros((B, N), np.float64)
    rc = lib().oracle_epikv_score(0 if dtype == "bf16" else 1, B, N, dm, _ptr(a), _ptr(b), int(window), float(eps),
                                  _ptr(g), _ptr(sc))
    if rc < 0:
        raise ValueError("oracle_epikv_score: bad sizes")
    return g, sc


def epikv_z(g: np.ndarray, window: int, eps: float):
    """The z-score half of epikv_score from given signals g [2, B, N] (any float type, used as fp64)."""
    gg = np.ascontiguousarray(g, dtype=np.float64)
    _, B, N = gg.shape
    sc = np.zeros((B, N), np.float64)
    if lib().oracle_epikv_z(B, N, _ptr(gg), int(window), float(eps), _ptr(sc)) < 0:
        raise ValueError("oracle_epikv_z: bad sizes")
    return sc
