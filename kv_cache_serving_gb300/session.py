"""Device-resident batch for the libdsa calls: tensors, dims and workspace.

``DecodeBatch.from_workload`` copies a batch drawn by ``workloads.generate`` to
the GPU once; its methods are one-line calls of the C ABI through the ctypes
binding.  PyTorch provides the device memory and the stream, nothing else.
"""
from __future__ import annotations

import copy
import math

import numpy as np
import torch

from . import dsa


def _i32(x, device):
    return torch.as_tensor(np.ascontiguousarray(x, dtype=np.int32)).to(device)


def estimated_kept_rows(lengths) -> np.ndarray:
    """Upper estimate of each request's kept rows, min(P,L) + min(W, L-1-min(P,L)) + 1,
    from host arrays (seq_len, prompt_len, window)."""
    L, P, W = (np.asarray(x, dtype=np.int64) for x in lengths)
    npr = np.minimum(P, L)
    return npr + np.minimum(np.maximum(L - 1 - npr, 0), W) + 1


def longest_first_order(lengths) -> np.ndarray:
    """int32 permutation of the requests by decreasing estimated kept rows (ties
    by index)."""
    return np.argsort(-estimated_kept_rows(lengths), kind="stable").astype(np.int32)


def schedule_order(lengths, spread: float = 1.25):
    """The request_order a serving host would pass: longest first when the
    estimated kept rows of the batch vary (max > spread * mean), else None
    (batch order; an order costs each CTA one dependent load)."""
    est = estimated_kept_rows(lengths)
    if est.size == 0 or est.max() <= spread * est.mean():
        return None
    return longest_first_order(lengths)


class PackedIO:
    """One pinned host buffer and one device buffer per direction, so that a
    step's inputs go up in one copy and its results come back in one.  The
    batch's tensors become views into the device buffers."""

    def __init__(self, inputs: dict, outputs: dict, device):
        def layout(tensors):
            offs, at = {}, 0
            for name, t in tensors.items():
                offs[name] = at
                at += (t.numel() * t.element_size() + 255) // 256 * 256
            return offs, max(at, 256)
        self._in_off, n_in = layout(inputs)
        self._out_off, n_out = layout(outputs)
        self.dev_in = torch.empty(n_in, dtype=torch.uint8, device=device)
        self.dev_out = torch.empty(n_out, dtype=torch.uint8, device=device)
        self.host_in = torch.empty(n_in, dtype=torch.uint8).pin_memory()
        self.host_out = torch.empty(n_out, dtype=torch.uint8).pin_memory()
        self.dev, self.host = {}, {}
        for offs, dbuf, hbuf, tensors in ((self._in_off, self.dev_in, self.host_in, inputs),
                                          (self._out_off, self.dev_out, self.host_out, outputs)):
            for name, t in tensors.items():
                nb = t.numel() * t.element_size()
                o = offs[name]
                self.dev[name] = dbuf[o:o + nb].view(t.dtype).view(t.shape)
                self.host[name] = hbuf[o:o + nb].view(t.dtype).view(t.shape)
                self.dev[name].copy_(t)
                self.host[name].copy_(t.cpu())
        self.h2d_bytes = n_in
        self.d2h_bytes = n_out

    def upload(self):
        self.dev_in.copy_(self.host_in, non_blocking=True)

    def download(self):
        self.host_out.copy_(self.dev_out, non_blocking=True)

    def descriptor(self) -> dsa.dsa_host_io:
        """The two copies as a dsa_host_io, for the calls that issue them
        themselves (dsa_decode_sparse_masked_io)."""
        return dsa.host_io(self.host_in, self.dev_in, self.dev_out, self.host_out)


class DecodeBatch:
    def __init__(self, *, q, k_pages, v_pages, page_table, seq_len, prompt_len, window,
                 grid_w, keep_mask, max_window, mask_words, max_kept, device="cuda"):
        self.device = torch.device(device)
        self.q = q.to(self.device).contiguous()
        self.k_pages = k_pages.to(self.device).contiguous()
        self.v_pages = v_pages.to(self.device).contiguous()
        self.page_table = _i32(page_table, self.device)
        self.seq_len = _i32(seq_len, self.device)
        self.prompt_len = _i32(prompt_len, self.device)
        self.window = _i32(window, self.device)
        self.grid_w = _i32(grid_w, self.device)
        self._host_lengths = tuple(np.array(x, dtype=np.int32, copy=True)
                                   for x in (seq_len, prompt_len, window))
        B, Hq, D = self.q.shape
        num_pages, page, Hkv, _ = self.k_pages.shape
        self.batch, self.hq, self.hkv, self.head_dim = B, Hq, Hkv, D
        if keep_mask is None:
            keep_mask = np.zeros((B, Hkv, mask_words), dtype=np.uint32)
        self.keep_mask = torch.as_tensor(
            np.ascontiguousarray(keep_mask, dtype=np.uint32).view(np.int32)).to(self.device)
        self.dims = dsa.make_dims(B, Hq, Hkv, D, num_pages, self.page_table.shape[1], max_window,
                                  mask_words, max_kept, self.q.dtype, self.k_pages.dtype)
        self.scale = 1.0 / math.sqrt(D)
        self.ws = dsa.alloc_workspace(self.dims, self.device)
        self.kept_idx = torch.zeros((B, Hkv, max_kept), dtype=torch.int32, device=self.device)
        self.kept_cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=self.device)
        self.out = torch.empty((B, Hq, D), dtype=torch.float32, device=self.device)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=self.device)

    @classmethod
    def from_workload(cls, w: dict, device="cuda", keep_mask=None):
        return cls(q=w["q"], k_pages=w["k_pages"], v_pages=w["v_pages"],
                   page_table=w["page_table"], seq_len=w["seq_len"], prompt_len=w["prompt_len"],
                   window=w["window"], grid_w=w["grid_w"],
                   keep_mask=w["keep_mask"] if keep_mask is None else keep_mask,
                   max_window=w["max_window"], mask_words=w["mask_words"],
                   max_kept=w["max_kept"], device=device)

    def replicate(self) -> "DecodeBatch":
        """A second slot for the same batch shape: the KV cache is shared (not
        copied); the step inputs, kept lists, outputs and workspace are its own
        copies, so that two steps can be in flight at once (double-buffered
        host I/O: one slot's copies overlap the other's kernels)."""
        other = copy.copy(self)
        for name in ("q", "page_table", "seq_len", "prompt_len", "window", "grid_w", "keep_mask",
                     "kept_idx", "kept_cnt", "out", "lse", "ws"):
            setattr(other, name, getattr(self, name).clone())
        other._host_lengths = tuple(x.copy() for x in self._host_lengths)
        return other

    def set_keep_mask(self, keep_mask):
        self.keep_mask.copy_(torch.as_tensor(
            np.ascontiguousarray(keep_mask, dtype=np.uint32).view(np.int32)))

    # -- the C ABI calls --------------------------------------------------
    def build_index(self, stream=None):
        dsa.dsa_build_index(self.dims, self.seq_len, self.prompt_len, self.window, self.keep_mask,
                            self.kept_idx, self.kept_cnt, self.ws, stream)

    def evict_pages(self, capacity=None, stream=None):
        """Unmap the pages no later step reads; returns (freed page ids tensor,
        count tensor) -- the ids are valid up to min(count, capacity)."""
        cap = self.page_table.numel() if capacity is None else capacity
        freed = torch.full((max(cap, 1),), -1, dtype=torch.int32, device=self.device)
        count = torch.zeros(1, dtype=torch.int32, device=self.device)
        dsa.dsa_evict_pages(self.dims, self.seq_len, self.prompt_len, self.window, self.page_table,
                            freed[:cap] if cap > 0 else None, count, self.ws, stream)
        return freed, count

    def decode_sparse(self, out=None, lse=None, stream=None):
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        dsa.dsa_decode_sparse(self.dims, self.q, self.k_pages, self.v_pages, self.page_table,
                              self.seq_len, self.kept_idx, self.kept_cnt, self.scale, out, lse,
                              self.ws, stream)
        return out, lse

    def decode_sparse_masked(self, out=None, lse=None, stream=None, request_order=None,
                             k_new=None, v_new=None):
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        dsa.dsa_decode_sparse_masked(self.dims, self.q, self.k_pages, self.v_pages,
                                     self.page_table, self.seq_len, self.prompt_len, self.window,
                                     self.keep_mask, self.scale, out, lse, self.ws, stream,
                                     request_order, k_new, v_new)
        return out, lse

    def decode_step_io(self, io: PackedIO, request_order=None, stream=None, k_pages=None,
                       v_pages=None, prepare=False):
        """One step from host memory in one C call: io's inputs up, the fused
        sparse decode, out and lse back into io.host.  The batch must have been
        packed by pack_io(io); k_pages / v_pages default to the batch's cache.
        With prepare=True returns a dsa.Prepared that issues the step per call."""
        return dsa.dsa_decode_sparse_masked_io(
            io.descriptor(), self.dims, self.q, self.k_pages if k_pages is None else k_pages,
            self.v_pages if v_pages is None else v_pages, self.page_table, self.seq_len,
            self.prompt_len, self.window, self.keep_mask, self.scale, self.out, self.lse, self.ws,
            stream, request_order, prepare=prepare)

    def record_step_io(self, io: PackedIO, stream, request_order=None, k_pages=None,
                       v_pages=None) -> dsa.Graph:
        """decode_step_io recorded once as a dsa.Graph on `stream` (a non-default
        torch.cuda.Stream): each graph.launch(stream) uploads io's inputs, runs
        the fused decode and downloads out and lse, for one host launch."""
        dsa.dsa_graph_begin(stream)
        try:
            self.decode_step_io(io, request_order, stream, k_pages, v_pages)
        except BaseException:
            try:  # end the recording so that the stream is usable again
                dsa.dsa_graph_end(stream).close()
            except dsa.DSAError:
                pass
            raise
        graph = dsa.dsa_graph_end(stream)
        return graph.keep(io, request_order, k_pages, v_pages, self)

    def longest_first_order(self):
        """Requests by decreasing estimated kept rows: the request_order that
        shortens the tail of a mixed batch (host-side; the serving host knows
        these lengths when it builds the batch)."""
        return longest_first_order(self._host_lengths)

    def schedule_order(self):
        """longest_first_order() when the batch's lengths vary, else None."""
        return schedule_order(self._host_lengths)

    def pack_io(self, order=None) -> tuple:
        """Move the step's inputs (q, lengths, masks, page table, order) and
        results (out, lse) into packed buffers; returns the PackedIO and the
        device order tensor (or None)."""
        inputs = {"q": self.q, "seq_len": self.seq_len, "prompt_len": self.prompt_len,
                  "window": self.window, "keep_mask": self.keep_mask,
                  "page_table": self.page_table}
        if order is not None:
            inputs["order"] = torch.as_tensor(np.asarray(order, dtype=np.int32))
        io = PackedIO(inputs, {"out": self.out, "lse": self.lse}, self.device)
        self.q, self.seq_len, self.prompt_len = io.dev["q"], io.dev["seq_len"], io.dev["prompt_len"]
        self.window, self.keep_mask = io.dev["window"], io.dev["keep_mask"]
        self.page_table = io.dev["page_table"]
        self.out, self.lse = io.dev["out"], io.dev["lse"]
        return io, io.dev.get("order")

    def decode_dense(self, out=None, lse=None, stream=None):
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        dsa.dsa_decode_dense(self.dims, self.q, self.k_pages, self.v_pages, self.page_table,
                             self.seq_len, self.scale, out, lse, self.ws, stream)
        return out, lse

    def attention_mass(self, r_local=2, r_diag=2, with_offsets=True, stream=None):
        mass = torch.empty((self.batch, self.hq, 4), dtype=torch.float32, device=self.device)
        om = None
        if with_offsets:
            om = torch.empty((self.batch, self.hq, self.dims.max_window + 1), dtype=torch.float32,
                             device=self.device)
        dsa.dsa_attention_mass(self.dims, self.q, self.k_pages, self.page_table, self.seq_len,
                               self.prompt_len, self.window, self.grid_w, r_local, r_diag,
                               self.scale, mass, om, self.ws, stream)
        return mass, om

    def device_error(self) -> int:
        return dsa.dsa_get_device_error(self.ws)

    def check(self, what="libdsa"):
        dsa.check_device_error(self.ws, what)
