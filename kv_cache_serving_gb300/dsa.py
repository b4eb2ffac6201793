"""Thin ctypes binding of libdsa (include/dsa.h): argument marshalling only.

Every function has the name of its C entry point, takes torch CUDA tensors
(or None where the C argument may be NULL), passes their device pointers and
the current CUDA stream, and raises DSAError on a non-OK status.  All compute
runs in the library's CUDA kernels; there is no fallback of any kind: if the
library cannot be built or loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_DEVICE, \
    DSA_ERR_TIMEOUT, DSA_ERR_SCRATCH_LIMIT = range(7)
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
DSA_F32, DSA_BF16 = 0, 1
DEV_ERRORS = {0: "OK", 1: "BAD_SEQ_LEN", 2: "BAD_PROMPT", 3: "BAD_WINDOW", 4: "BAD_PAGE",
              5: "BAD_INDEX", 6: "BAD_COUNT", 7: "TIMEOUT", 8: "BAD_GRID_W", 9: "BAD_ORDER",
              10: "FREE_LIST_FULL", 11: "BAD_QLEN"}
PAGE = 16


class DSAError(RuntimeError):
    def __init__(self, status: int, what: str, dev_code: int | None = None):
        self.status = status
        self.dev_code = dev_code
        msg = f"{what}: {status_name(status)}"
        if dev_code is not None:
            msg += f" (device code {dev_code} {DEV_ERRORS.get(dev_code, '?')})"
        super().__init__(msg)


class dsa_dims(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "batch", "hq", "hkv", "head_dim", "page_size", "num_pages", "max_pages_per_req",
        "max_window", "mask_words", "max_kept", "q_dtype", "kv_dtype")]


class dsa_host_io(ctypes.Structure):
    _fields_ = [("host_in", ctypes.c_void_p), ("dev_in", ctypes.c_void_p),
                ("in_bytes", ctypes.c_size_t), ("dev_out", ctypes.c_void_p),
                ("host_out", ctypes.c_void_p), ("out_bytes", ctypes.c_size_t)]


_lib = None
_lib_path = None


def library_path() -> str:
    """Path of the loaded libdsa.so (building it first if needed)."""
    _load()
    return _lib_path


def _load():
    global _lib, _lib_path
    if _lib is not None:
        return _lib
    path = os.environ.get("DSA_LIBRARY")
    if not path:
        from . import build as _build
        path = _build.build()
    lib = ctypes.CDLL(path)
    P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(dsa_dims)
    sig = {
        "dsa_version": ([], I32),
        "dsa_status_string": ([I32], ctypes.c_char_p),
        "dsa_workspace_size": ([D], SZ),
        "dsa_build_index": ([D, P, P, P, P, P, P, P, P], I32),
        "dsa_decode_sparse": ([D, P, P, P, P, P, P, P, F32, P, P, P, P], I32),
        "dsa_evict_pages": ([D, P, P, P, P, P, P, I32, P, P], I32),
        "dsa_decode_sparse_masked": ([D, P, P, P, P, P, P, P, P, P, P, P, F32, P, P, P, P], I32),
        "dsa_decode_sparse_masked_io": ([ctypes.POINTER(dsa_host_io), D, P, P, P, P, P, P, P, P,
                                         P, P, P, F32, P, P, P, P], I32),
        "dsa_decode_dense": ([D, P, P, P, P, P, F32, P, P, P, P], I32),
        "dsa_prefill_sparse": ([D, I32, P, P, P, P, P, P, P, P, P, P, F32, P, P, P, P], I32),
        "dsa_attention_mass": ([D, P, P, P, P, P, P, P, I32, I32, F32, P, P, P, P], I32),
        "dsa_decode_plan": ([D, I32, ctypes.POINTER(I32), ctypes.POINTER(I32),
                             ctypes.POINTER(I32), ctypes.POINTER(I32), ctypes.POINTER(I32)],
                            I32),
        "dsa_decode_sparse_noalloc": ([D, P, P, P, P, P, P, P, F32, P, P, P, P], I32),
        "dsa_graph_begin": ([P], I32),
        "dsa_graph_end": ([P, ctypes.POINTER(P)], I32),
        "dsa_graph_launch": ([P, P], I32),
        "dsa_graph_destroy": ([P], I32),
        "dsa_set_sparse_cluster": ([I32], I32),
        "dsa_get_sparse_cluster": ([], I32),
        "dsa_prefill_plan": ([D, I32] + [ctypes.POINTER(I32)] * 6, I32),
        "dsa_set_prefill_split": ([I32], I32),
        "dsa_get_prefill_split": ([], I32),
        "dsa_get_device_error": ([P, P, ctypes.POINTER(I32)], I32),
        "dsa_clear_device_error": ([P, P], I32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib, _lib_path = lib, path
    return lib


def status_name(status: int) -> str:
    try:
        return _load().dsa_status_string(int(status)).decode()
    except OSError:
        return f"status {status}"


def dsa_version() -> int:
    return _load().dsa_version()


def dsa_status_string(status: int) -> str:
    return _load().dsa_status_string(int(status)).decode()


def make_dims(batch, hq, hkv, head_dim, num_pages, max_pages_per_req, max_window, mask_words,
              max_kept, q_dtype, kv_dtype, page_size=PAGE) -> dsa_dims:
    def code(dt):
        if isinstance(dt, int):
            return dt
        return {torch.float32: DSA_F32, torch.bfloat16: DSA_BF16, "f32": DSA_F32,
                "bf16": DSA_BF16}[dt]
    return dsa_dims(batch, hq, hkv, head_dim, page_size, num_pages, max_pages_per_req,
                    max_window, mask_words, max_kept, code(q_dtype), code(kv_dtype))


def _ptr(t, dtype=None, what="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{what} has dtype {t.dtype}, expected {dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != DSA_OK:
        raise DSAError(status, what)


def dsa_workspace_size(dims: dsa_dims) -> int:
    return int(_load().dsa_workspace_size(ctypes.byref(dims)))


def alloc_workspace(dims: dsa_dims, device=None) -> torch.Tensor:
    """A zero-filled workspace of dsa_workspace_size(dims) bytes (torch owns it)."""
    n = dsa_workspace_size(dims)
    if n == 0:
        raise DSAError(DSA_ERR_INVALID_ARG, "dsa_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


_I32 = torch.int32
_MASK = (torch.int32, getattr(torch, "uint32", torch.int32))
_QKV = (torch.float32, torch.bfloat16)


def dsa_build_index(dims, seq_len, prompt_len, window, keep_mask, kept_idx, kept_cnt, ws,
                    stream=None):
    _check(_load().dsa_build_index(
        ctypes.byref(dims), _ptr(seq_len, _I32, "seq_len"), _ptr(prompt_len, _I32, "prompt_len"),
        _ptr(window, _I32, "window"), _ptr(keep_mask, _MASK, "keep_mask"),
        _ptr(kept_idx, _I32, "kept_idx"), _ptr(kept_cnt, _I32, "kept_cnt"), _ptr(ws), _stream(stream)),
        "dsa_build_index")


def dsa_evict_pages(dims, seq_len, prompt_len, window, page_table, freed_pages, freed_count, ws,
                    stream=None):
    """Unmap (set to -1) the page-table entries no later decode step reads and
    append their page ids to freed_pages (int32 CUDA tensor) from freed_count
    (one-element int32 CUDA tensor) on."""
    cap = 0 if freed_pages is None else int(freed_pages.numel())
    _check(_load().dsa_evict_pages(
        ctypes.byref(dims), _ptr(seq_len, _I32, "seq_len"), _ptr(prompt_len, _I32, "prompt_len"),
        _ptr(window, _I32, "window"), _ptr(page_table, _I32, "page_table"),
        _ptr(freed_pages, _I32, "freed_pages"), _ptr(freed_count, _I32, "freed_count"), cap,
        _ptr(ws), _stream(stream)), "dsa_evict_pages")


def dsa_decode_sparse(dims, q, k_pages, v_pages, page_table, seq_len, kept_idx, kept_cnt, scale,
                      out, lse, ws, stream=None):
    _check(_load().dsa_decode_sparse(
        ctypes.byref(dims), _ptr(q, _QKV, "q"), _ptr(k_pages, _QKV, "k_pages"),
        _ptr(v_pages, _QKV, "v_pages"), _ptr(page_table, _I32, "page_table"),
        _ptr(seq_len, _I32, "seq_len"), _ptr(kept_idx, _I32, "kept_idx"),
        _ptr(kept_cnt, _I32, "kept_cnt"), float(scale), _ptr(out, torch.float32, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(ws), _stream(stream)), "dsa_decode_sparse")


def dsa_decode_sparse_masked(dims, q, k_pages, v_pages, page_table, seq_len, prompt_len, window,
                             keep_mask, scale, out, lse, ws, stream=None, request_order=None,
                             k_new=None, v_new=None):
    """dsa_build_index + dsa_decode_sparse in one call: the kernels read each
    (request, kv head)'s kept set from the mask themselves.  request_order
    (int32 [batch] CUDA tensor or None) is the order requests are scheduled in;
    k_new / v_new ([batch, hkv, head_dim] CUDA tensors or None) append the query
    token's K/V row to the cache in the same call."""
    _check(_load().dsa_decode_sparse_masked(
        ctypes.byref(dims), _ptr(q, _QKV, "q"), _ptr(k_pages, _QKV, "k_pages"),
        _ptr(v_pages, _QKV, "v_pages"), _ptr(page_table, _I32, "page_table"),
        _ptr(seq_len, _I32, "seq_len"), _ptr(prompt_len, _I32, "prompt_len"),
        _ptr(window, _I32, "window"), _ptr(keep_mask, _MASK, "keep_mask"),
        _ptr(request_order, _I32, "request_order"), _ptr(k_new, _QKV, "k_new"),
        _ptr(v_new, _QKV, "v_new"), float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _ptr(ws),
        _stream(stream)), "dsa_decode_sparse_masked")


class Prepared:
    """One C call with its arguments marshalled once; calling the object issues
    it again with the same pointers (the tensors must stay alive and in place)."""

    def __init__(self, name: str, args: tuple, keep: tuple = ()):
        self._fn = getattr(_load(), name)
        self._name = name
        self._args = args
        self._keep = keep  # objects the marshalled pointers refer to

    def __call__(self):
        status = self._fn(*self._args)
        if status != DSA_OK:
            raise DSAError(status, self._name)


def host_io(host_in, dev_in, dev_out, host_out) -> dsa_host_io:
    """dsa_host_io over two host tensors (pinned, CPU) and two CUDA tensors:
    host_in -> dev_in before the call, dev_out -> host_out after it."""
    for t, cuda, what in ((host_in, False, "host_in"), (dev_in, True, "dev_in"),
                          (dev_out, True, "dev_out"), (host_out, False, "host_out")):
        if not isinstance(t, torch.Tensor) or t.is_cuda != cuda or not t.is_contiguous():
            raise TypeError(f"{what} must be a contiguous {'CUDA' if cuda else 'host'} tensor")
    nin = host_in.numel() * host_in.element_size()
    nout = dev_out.numel() * dev_out.element_size()
    if dev_in.numel() * dev_in.element_size() != nin or \
            host_out.numel() * host_out.element_size() != nout:
        raise ValueError("host_io: the two buffers of a copy differ in size")
    return dsa_host_io(host_in.data_ptr(), dev_in.data_ptr(), nin, dev_out.data_ptr(),
                       host_out.data_ptr(), nout)


def dsa_decode_sparse_masked_io(io, dims, q, k_pages, v_pages, page_table, seq_len, prompt_len,
                                window, keep_mask, scale, out, lse, ws, stream=None,
                                request_order=None, k_new=None, v_new=None, prepare=False):
    """dsa_decode_sparse_masked with the step's host copies in the same call: io
    (a dsa_host_io, see host_io) is uploaded before the attention and downloaded
    after it, on the same stream.  With prepare=True nothing is issued: the
    return value is a Prepared call that issues it each time it is called."""
    if not isinstance(io, dsa_host_io):
        raise TypeError("io must be a dsa_host_io")
    args = (ctypes.byref(io), ctypes.byref(dims), _ptr(q, _QKV, "q"),
            _ptr(k_pages, _QKV, "k_pages"), _ptr(v_pages, _QKV, "v_pages"),
            _ptr(page_table, _I32, "page_table"), _ptr(seq_len, _I32, "seq_len"),
            _ptr(prompt_len, _I32, "prompt_len"), _ptr(window, _I32, "window"),
            _ptr(keep_mask, _MASK, "keep_mask"), _ptr(request_order, _I32, "request_order"),
            _ptr(k_new, _QKV, "k_new"), _ptr(v_new, _QKV, "v_new"), float(scale),
            _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _ptr(ws),
            _stream(stream))
    call = Prepared("dsa_decode_sparse_masked_io", args,
                    (io, dims, q, k_pages, v_pages, page_table, seq_len, prompt_len, window,
                     keep_mask, request_order, k_new, v_new, out, lse, ws, stream))
    if prepare:
        return call
    call()
    return None


def dsa_graph_begin(stream):
    """Start recording libdsa calls on `stream` (a torch.cuda.Stream, not the
    legacy default stream)."""
    _check(_load().dsa_graph_begin(_stream(stream)), "dsa_graph_begin")


def dsa_graph_end(stream) -> "Graph":
    """End the recording on `stream`; returns the recorded calls as a Graph."""
    h = ctypes.c_void_p()
    _check(_load().dsa_graph_end(_stream(stream), ctypes.byref(h)), "dsa_graph_end")
    return Graph(h)


def dsa_graph_launch(graph: "Graph", stream=None):
    _check(_load().dsa_graph_launch(graph.handle, _stream(stream)), "dsa_graph_launch")


def dsa_graph_destroy(graph: "Graph"):
    graph.close()


class Graph:
    """Owner of a dsa_graph handle; launch() replays it, close() (or garbage
    collection) frees it.  Objects a recorded call points into can be attached
    with keep() so that they live as long as the graph."""

    def __init__(self, handle: ctypes.c_void_p):
        self.handle = handle
        self._keep = []
        self._lib = _load()

    def keep(self, *objs):
        self._keep.extend(objs)
        return self

    def launch(self, stream=None):
        status = self._lib.dsa_graph_launch(self.handle, _stream(stream))
        if status != DSA_OK:
            raise DSAError(status, "dsa_graph_launch")

    def close(self):
        if self.handle:
            _check(self._lib.dsa_graph_destroy(self.handle), "dsa_graph_destroy")
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dsa_decode_sparse_noalloc(dims, q, k_pages, v_pages, page_table, seq_len, kept_idx,
                              kept_cnt, scale, out, lse, dev_error=None, stream=None):
    """dsa_decode_sparse with the library's own fixed scratch instead of a caller
    workspace, for callers that cannot allocate device memory.  dev_error (a
    one-element int32 CUDA tensor, or None) receives the call's device error code."""
    _check(_load().dsa_decode_sparse_noalloc(
        ctypes.byref(dims), _ptr(q, _QKV, "q"), _ptr(k_pages, _QKV, "k_pages"),
        _ptr(v_pages, _QKV, "v_pages"), _ptr(page_table, _I32, "page_table"),
        _ptr(seq_len, _I32, "seq_len"), _ptr(kept_idx, _I32, "kept_idx"),
        _ptr(kept_cnt, _I32, "kept_cnt"), float(scale), _ptr(out, torch.float32, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(dev_error, _I32, "dev_error"), _stream(stream)),
        "dsa_decode_sparse_noalloc")


def dsa_decode_dense(dims, q, k_pages, v_pages, page_table, seq_len, scale, out, lse, ws,
                     stream=None):
    _check(_load().dsa_decode_dense(
        ctypes.byref(dims), _ptr(q, _QKV, "q"), _ptr(k_pages, _QKV, "k_pages"),
        _ptr(v_pages, _QKV, "v_pages"), _ptr(page_table, _I32, "page_table"),
        _ptr(seq_len, _I32, "seq_len"), float(scale), _ptr(out, torch.float32, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(ws), _stream(stream)), "dsa_decode_dense")


def dsa_prefill_sparse(dims, q, k_pages, v_pages, page_table, seq_len, q_len, prompt_len,
                       window, keep_mask, scale, out, lse, ws, stream=None, request_order=None):
    """Several query tokens per request under the mask: q is [batch, max_q, hq,
    head_dim] bf16; the q_len[b] query tokens of request b are its last cache
    rows.  out [batch, max_q, hq, head_dim] f32, lse [batch, max_q, hq] f32 or None;
    request_order [batch] int32 (device) or None: the order requests are handed
    to the GPU."""
    if q.dim() != 4:
        raise ValueError("q must be [batch, max_q, hq, head_dim]")
    _check(_load().dsa_prefill_sparse(
        ctypes.byref(dims), int(q.shape[1]), _ptr(q, torch.bfloat16, "q"),
        _ptr(k_pages, torch.bfloat16, "k_pages"), _ptr(v_pages, torch.bfloat16, "v_pages"),
        _ptr(page_table, _I32, "page_table"), _ptr(seq_len, _I32, "seq_len"),
        _ptr(q_len, _I32, "q_len"), _ptr(prompt_len, _I32, "prompt_len"),
        _ptr(window, _I32, "window"), _ptr(keep_mask, _MASK, "keep_mask"),
        _ptr(request_order, _I32, "request_order"), float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _ptr(ws),
        _stream(stream)), "dsa_prefill_sparse")


def dsa_attention_mass(dims, q, k_pages, page_table, seq_len, prompt_len, window, grid_w,
                       r_local, r_diag, scale, mass, offset_mass, ws, stream=None):
    _check(_load().dsa_attention_mass(
        ctypes.byref(dims), _ptr(q, _QKV, "q"), _ptr(k_pages, _QKV, "k_pages"),
        _ptr(page_table, _I32, "page_table"), _ptr(seq_len, _I32, "seq_len"),
        _ptr(prompt_len, _I32, "prompt_len"), _ptr(window, _I32, "window"),
        _ptr(grid_w, _I32, "grid_w"), int(r_local), int(r_diag), float(scale),
        _ptr(mass, torch.float32, "mass"), _ptr(offset_mass, torch.float32, "offset_mass"),
        _ptr(ws), _stream(stream)), "dsa_attention_mass")


PLAN_DENSE, PLAN_SPARSE, PLAN_MASKED = 0, 1, 2


def dsa_decode_plan(dims, mode: int):
    """(rows per CTA, max CTAs per (request, kv head), kernel launches per call,
    warps per CTA, rows per tile) on the current device for dsa_decode_dense
    (mode 0), dsa_decode_sparse (1) or dsa_decode_sparse_masked (2); calls with
    the same plan sum in the same order."""
    v = [ctypes.c_int32() for _ in range(5)]
    _check(_load().dsa_decode_plan(ctypes.byref(dims), int(mode),
                                   *[ctypes.byref(x) for x in v]), "dsa_decode_plan")
    return tuple(x.value for x in v)


def dsa_set_sparse_cluster(ctas: int) -> None:
    """CTAs per (request, kv head) cluster of sparse decode (1 = no cluster,
    0 = chosen per call from the batch size)."""
    _check(_load().dsa_set_sparse_cluster(int(ctas)), "dsa_set_sparse_cluster")


def dsa_get_sparse_cluster() -> int:
    return int(_load().dsa_get_sparse_cluster())


def dsa_prefill_plan(dims, max_q: int):
    """(warps per CTA, units, units run whole, parts per split unit, resident CTAs
    per SM, CTAs launched) of dsa_prefill_sparse on the current device."""
    v = [ctypes.c_int32() for _ in range(6)]
    _check(_load().dsa_prefill_plan(ctypes.byref(dims), int(max_q),
                                    *[ctypes.byref(x) for x in v]), "dsa_prefill_plan")
    return tuple(x.value for x in v)


def dsa_set_prefill_split(parts: int) -> None:
    """CTAs per unit of dsa_prefill_sparse (1 = never split, 0 = the units of a
    last partial wave, or of a batch below one wave, split per call)."""
    _check(_load().dsa_set_prefill_split(int(parts)), "dsa_set_prefill_split")


def dsa_get_prefill_split() -> int:
    return int(_load().dsa_get_prefill_split())



def dsa_get_device_error(ws, stream=None) -> int:
    """Synchronising read of the workspace error word; returns the DSA_DEV_* code."""
    code = ctypes.c_int32(0)
    st = _load().dsa_get_device_error(_ptr(ws), _stream(stream), ctypes.byref(code))
    if st == DSA_ERR_CUDA:
        raise DSAError(st, "dsa_get_device_error")
    return int(code.value)


def dsa_clear_device_error(ws, stream=None):
    _check(_load().dsa_clear_device_error(_ptr(ws), _stream(stream)), "dsa_clear_device_error")


def check_device_error(ws, what="libdsa", stream=None):
    """Raise DSAError if the kernels flagged invalid data since the last clear."""
    code = dsa_get_device_error(ws, stream)
    if code != 0:
        raise DSAError(DSA_ERR_TIMEOUT if code == 7 else DSA_ERR_DEVICE, what, code)
