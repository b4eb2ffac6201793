"""fp64 CPU oracle for diagonal-aware sparse decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use this package; the library under
``kv_cache_serving_gb300`` never imports it, and it imports nothing from there.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64, one (request, head)
at a time); this module compiles it with gcc and marshals arguments.  See the
C file's header for the page sections each function follows.

Functions whose parity is pinned by ``tests/test_oracle_pins.py``:
``kept_set``, ``mask_matrix``, ``sparsity``, ``attend_rows``, ``decode``,
``multi``, ``mass``, ``evictable_pages``.  ``top_mass_keep_mask`` lives with the input generators (it is a
selection rule, not the method's arithmetic).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
PAGE = 16


class Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_pages", ctypes.c_int32), ("max_window", ctypes.c_int32),
        ("mask_words", ctypes.c_int32), ("q_dtype", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
        ("prompt_len", ctypes.c_void_p), ("window", ctypes.c_void_p),
        ("grid_w", ctypes.c_void_p), ("keep_mask", ctypes.c_void_p),
        ("scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into oracle/_build/liboracle.so (gcc, -O2, no FMA contraction)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        os.makedirs(_BUILD, exist_ok=True)
        tmp = f"{_LIB}.{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32, p, d = ctypes.c_int32, ctypes.c_void_p, ctypes.c_double
        lib.oracle_kept_set.argtypes = [i32, i32, i32, p, p]
        lib.oracle_kept_set.restype = i32
        lib.oracle_evictable_pages.argtypes = [i32, i32, i32, p]
        lib.oracle_evictable_pages.restype = i32
        lib.oracle_mask_matrix.argtypes = [i32, i32, i32, i32, p]
        lib.oracle_mask_matrix.restype = None
        lib.oracle_sparsity.argtypes = [i32, p]
        lib.oracle_sparsity.restype = d
        lib.oracle_attend_rows.argtypes = [i32, p, p, p, i32, d, p, p]
        lib.oracle_attend_rows.restype = None
        lib.oracle_decode.argtypes = [ctypes.POINTER(Problem), i32, p, i32, p, p, i32]
        lib.oracle_decode.restype = i32
        lib.oracle_mass.argtypes = [ctypes.POINTER(Problem), i32, i32, p, i32, p, p, i32]
        lib.oracle_mass.restype = i32
        lib.oracle_multi.argtypes = [ctypes.POINTER(Problem), p, i32, p, p, i32]
        lib.oracle_multi.restype = i32
        _lib = lib
    return _lib


def _np(a, dtype):
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def kept_set(L: int, P: int, W: int, mask_words) -> np.ndarray:
    """Ascending kept logical rows of one decode query at i = L-1."""
    lib = _load()
    mask = _np(mask_words, np.uint32)
    need = (W + 31) // 32
    if mask.size < need:
        raise ValueError("mask has fewer words than the window needs")
    out = np.zeros(max(L, 1), dtype=np.int32)
    n = lib.oracle_kept_set(L, P, W, _ptr(mask), _ptr(out))
    if n < 0:
        raise ValueError(f"oracle_kept_set rejected L={L} P={P} W={W}")
    return out[:n].copy()


def evictable_pages(L: int, P: int, W: int) -> np.ndarray:
    """bool[ceil(L/16)]: pages of a request that no later decode step reads."""
    lib = _load()
    flags = np.zeros(max((L + 15) // 16, 1), dtype=np.uint8)
    n = lib.oracle_evictable_pages(L, P, W, _ptr(flags))
    if n < 0:
        raise ValueError(f"oracle_evictable_pages rejected L={L} P={P} W={W}")
    return flags[:(L + 15) // 16].astype(bool)


def mask_matrix(N: int, W: int, B: int, causal: bool = False) -> np.ndarray:
    """The summary's literal N x N band mask (uint8)."""
    lib = _load()
    M = np.zeros((N, N), dtype=np.uint8)
    lib.oracle_mask_matrix(N, W, B, int(causal), _ptr(M))
    return M


def sparsity(M: np.ndarray) -> float:
    lib = _load()
    M = _np(M, np.uint8)
    assert M.ndim == 2 and M.shape[0] == M.shape[1]
    return float(lib.oracle_sparsity(M.shape[0], _ptr(M)))


def attend_rows(q, k, v, scale: float):
    """Softmax attention of one query q[D] over rows k[n][D], v[n][D] (fp64)."""
    lib = _load()
    q = _np(q, np.float64)
    k = _np(k, np.float64).reshape(-1, q.size)
    v = _np(v, np.float64).reshape(-1, q.size)
    out = np.zeros(q.size, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib.oracle_attend_rows(q.size, _ptr(q), _ptr(k), _ptr(v), k.shape[0], float(scale),
                           _ptr(out), _ptr(lse))
    return out, float(lse[0])


def _raw(t: torch.Tensor):
    """(numpy view of the stored bits, dtype code) of a CPU tensor, no rounding."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy(), F32
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


class _Bound:
    """Keeps the numpy buffers alive while the C struct points at them."""

    def __init__(self, inp: dict, scale: float | None):
        q, qd = _raw(inp["q"])
        k, kd = _raw(inp["k_pages"])
        v, vd = _raw(inp["v_pages"])
        assert kd == vd
        self.keep = [q, k, v]
        # q is [B][Hq][D] (one query per request) or [B][Q][Hq][D] (several)
        B, Hq, D = inp["q"].shape[0], inp["q"].shape[-2], inp["q"].shape[-1]
        num_pages, page, Hkv, D2 = inp["k_pages"].shape
        assert page == PAGE and D2 == D
        pt = _np(inp["page_table"], np.int32)
        L = _np(inp["seq_len"], np.int32)
        P = _np(inp["prompt_len"], np.int32)
        W = _np(inp["window"], np.int32)
        gw = _np(inp.get("grid_w", np.ones(B)), np.int32)
        self.max_window = int(inp["max_window"])
        if inp.get("keep_mask") is None:      # attention mass reads no mask
            words = int(inp.get("mask_words", max(1, (self.max_window + 31) // 32)))
            mask = np.zeros((B, Hkv, words), dtype=np.uint32)
        else:
            mask = _np(inp["keep_mask"], np.uint32)
        self.keep += [pt, L, P, W, gw, mask]
        self.pr = Problem(
            batch=B, hq=Hq, hkv=Hkv, head_dim=D, num_pages=num_pages,
            max_pages=pt.shape[1], max_window=self.max_window, mask_words=mask.shape[-1],
            q_dtype=qd, kv_dtype=kd,
            q=q.ctypes.data, k_pages=k.ctypes.data, v_pages=v.ctypes.data,
            page_table=pt.ctypes.data, seq_len=L.ctypes.data, prompt_len=P.ctypes.data,
            window=W.ctypes.data, grid_w=gw.ctypes.data, keep_mask=mask.ctypes.data,
            scale=float(scale if scale is not None else 1.0 / np.sqrt(D)))


def _bh_array(bh):
    if bh is None:
        return None, 0
    arr = _np(bh, np.int32).reshape(-1, 2)
    return arr, arr.shape[0]


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def decode(inp: dict, sparse: bool, bh=None, scale: float | None = None,
           nthreads: int | None = None):
    """fp64 decode attention.  Returns (out[n][D], lse[n]) for the listed (b, h)
    pairs, or for all B*Hq pairs in (b, h) order when bh is None."""
    lib = _load()
    bound = _Bound(inp, scale)
    arr, n = _bh_array(bh)
    if arr is None:
        n = bound.pr.batch * bound.pr.hq
    out = np.zeros((n, bound.pr.head_dim), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = lib.oracle_decode(ctypes.byref(bound.pr), int(sparse),
                           None if arr is None else _ptr(arr), n, _ptr(out), _ptr(lse),
                           nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_decode failed with status {rc}")
    return out, lse


def multi(inp: dict, q_len, scale: float | None = None, nthreads: int | None = None):
    """fp64 attention of several query tokens per request under the mask:
    inp["q"] is [B][Q][Hq][D]; the q_len[b] query tokens of request b are its
    last cache rows L-q_len .. L-1, each attending over its own kept set.
    Returns (out [B][Q][Hq][D], lse [B][Q][Hq]); slots t >= q_len[b] are NaN."""
    lib = _load()
    bound = _Bound(inp, scale)
    B, Q, Hq, D = inp["q"].shape
    ql = _np(q_len, np.int32)
    assert ql.shape == (B,)
    out = np.full((B, Q, Hq, D), np.nan, dtype=np.float64)
    lse = np.full((B, Q, Hq), np.nan, dtype=np.float64)
    rc = lib.oracle_multi(ctypes.byref(bound.pr), _ptr(ql), Q, _ptr(out), _ptr(lse),
                          nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_multi failed with status {rc}")
    return out, lse


def mass(inp: dict, r_local: int = 2, r_diag: int = 2, bh=None, scale: float | None = None,
         nthreads: int | None = None, with_offsets: bool = True):
    """fp64 attention-mass bins [n][4] (prompt, local, diagonal, other) and the
    per-offset mass [n][max_window+1]."""
    lib = _load()
    bound = _Bound(inp, scale)
    arr, n = _bh_array(bh)
    if arr is None:
        n = bound.pr.batch * bound.pr.hq
    m4 = np.zeros((n, 4), dtype=np.float64)
    om = np.zeros((n, bound.max_window + 1), dtype=np.float64) if with_offsets else None
    rc = lib.oracle_mass(ctypes.byref(bound.pr), r_local, r_diag,
                         None if arr is None else _ptr(arr), n, _ptr(m4),
                         None if om is None else _ptr(om), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_mass failed with status {rc}")
    return m4, om
