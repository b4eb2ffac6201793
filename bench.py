#!/usr/bin/env python3
"""Sparse decode-attention benchmark on GB300: tokens/s and effective KV GB/s.

One step = one decode token for every request of the batch through the hot
path as one call, dsa_decode_sparse_masked: each decode CTA reads its kept set
from the keep mask (index compaction), gathers the kept K/V rows, runs the
online softmax and PV, and (when rows are split) the LSE merge follows.  The
same step as two calls, dsa_build_index (kept lists to HBM) + dsa_decode_sparse,
and that decode alone are timed beside it.  Inputs are synthetic (seeded),
shaped like the mixed serving batch by default (--workload mixed-serving: 128
requests, GQA group 4, head_dim 128, lengths up to P+4096, the largest
single-GPU workload); others: --workload janus-pro-7b | llamagen-xl | emu3-8b.
The dense causal decode of the same batch and the attention-mass pass are timed
beside it, and (one GPU, unless --no-other-workloads) every other workload gets
a compact line of its own under "workloads": fused step, roofline fraction,
dense step, speedup and kept fraction.

Timing: W eager warm-up steps, then K steps captured in one CUDA graph and
replayed once between CUDA events (per-step = elapsed / K).  Consecutive steps
rotate through R copies of the KV pool, R chosen so that the rows touched by R
steps exceed 4x the L2, so every step streams its rows from HBM.  nvidia-smi
samples clocks over a busy window that encloses the timed replay.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, replicas
only: the path has no exchange step); the timed region is bracketed by
barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import csv
import glob
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from kv_cache_serving_gb300 import dsa  # noqa: E402
from kv_cache_serving_gb300 import workloads as wl  # noqa: E402
from kv_cache_serving_gb300.session import DecodeBatch  # noqa: E402

METRIC = "sparse decode-attn tokens/s and effective KV GB/s (% of GB300 HBM peak)"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# step's decode kernel, per workload, from one ncu capture of
# `bench.py --workload NAME --profile masked --warmup 2 --steps 1` (the same launch
# on the same batch; the summaries are under profiles/).  They describe the
# decode-kernel sources whose digest is `digest` and are reported as null
# otherwise.
NCU_TRAFFIC = {
    "digest": "9f7d16093e2dc428",
    "bytes": {
        "mixed-serving-gqa4": 167971840,
        "janus-pro-7b-like-32x32": 316328960,
        "llamagen-xl-like-24x24": 21440768,
        "emu3-8b-like-90x90-gqa4": 3281408,
    },
}

# Sources the timed decode kernel (and its launch plan) is built from.
DECODE_SOURCES = ("common.cuh", "decode.cuh", "warp_attn.cuh", "mma.cuh", "internal.h",
                  "decode_bf16.cu", "decode_bf16_list.cu", "decode_bf16_mask.cu", "decode_f32.cu",
                  "dsa_api.cu")


def kernel_digest() -> str:
    """sha256 over the sources of the timed decode kernel and the public header."""
    h = hashlib.sha256()
    files = [os.path.join(ROOT, "kv_cache_serving_gb300", "csrc", f) for f in DECODE_SOURCES]
    files.append(os.path.join(ROOT, "include", "dsa.h"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    if kernel_digest() != NCU_TRAFFIC["digest"]:
        return None
    return NCU_TRAFFIC["bytes"].get(workload)


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default="mixed-serving",
                   choices=["mixed-serving", "janus-pro-7b", "llamagen-xl", "emu3-8b"])
    p.add_argument("--no-other-workloads", action="store_true",
                   help="skip the compact per-workload measurements of the other workloads")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU time budget of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--busy-seconds", type=float, default=1.5,
                   help="GPU busy time around the timed region for clock sampling")
    p.add_argument("--profile", choices=["index", "sparse", "masked", "dense", "mass", "prefill"],
                   help="no timing: run W + K eager launches of one call on one KV pool "
                        "(a small, self-contained case for ncu) and exit")
    p.add_argument("--sparse-cluster", type=int, default=-1,
                   help="CTAs per thread-block cluster of sparse decode (0: chosen per call, "
                        "default: the library's setting)")
    p.add_argument("--sweep-sparsity", action="store_true",
                   help="no headline line: time the fused sparse step against dense decode "
                        "over a range of windows and mask densities (one JSON line each)")
    p.add_argument("--batch", type=int, default=0,
                   help="with --profile: override the workload's batch size")
    return p.parse_args()


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    return rank, world, local


def rank_seed(cfg, rank: int) -> int:
    """Each rank draws its own batch (weak scaling: the per-GPU work is fixed)."""
    return cfg.seed + 1000 * rank


def max_over_ranks(values, device):
    """Element-wise max of a list of floats over all ranks (the job's time is
    its slowest rank's); identity without a process group."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return list(values)
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
            return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.file.read())) if len(r) >= 9]
        self.file.close()
        os.unlink(self.file.name)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4)
                          if r[5 + k].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def step_bytes(w, kept_idx, kept_cnt):
    """Bytes a sparse step must move at minimum, and the dense decode's."""
    B, Hq, Hkv, D = w["batch"], w["hq"], w["hkv"], w["head_dim"]
    elt = 2 if w["dtype"] == "bf16" else 4
    q_elt = 2 if w["dtype"] == "bf16" else 4
    L = w["seq_len"].astype(np.int64)
    rows = int(kept_cnt.sum())
    pages = 0
    for b in range(B):
        touched = set()
        for hk in range(Hkv):
            touched.update((kept_idx[b, hk, :kept_cnt[b, hk]] >> 4).tolist())
        pages += len(touched)
    q_b = B * Hq * D * q_elt
    out_b = B * Hq * D * 4 + B * Hq * 4
    sparse_decode = rows * 2 * D * elt + q_b + out_b + 4 * rows + 4 * pages + 4 * B * Hkv
    mask_in = B * Hkv * w["mask_words"] * 4 + 3 * 4 * B
    index = mask_in + 4 * rows + 4 * B * Hkv
    # one call that builds the kept set in the kernel: no kept list in HBM
    masked = sparse_decode - 4 * rows - 4 * B * Hkv + mask_in
    dense_rows = int(L.sum()) * Hkv
    dense = dense_rows * 2 * D * elt + q_b + out_b + 4 * int(((L + 15) // 16).sum())
    return dict(kv=rows * 2 * D * elt, sparse_decode=sparse_decode, index=index,
                step=sparse_decode + index, masked=masked, dense=dense, rows=rows,
                dense_rows=dense_rows)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def graph_of(fn, steps, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(steps):
            fn(k)
    return g


def time_graph(g, stream):
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3  # seconds


def busy(g, seconds, per_replay):
    n = max(1, int(seconds / max(per_replay, 1e-6)))
    for _ in range(n):
        g.replay()
    torch.cuda.synchronize()


def cpu_oracle_sample(w_cpu, seconds, sparse=True, threads=None):
    """Time the fp64 oracle on a bounded sample of the step: a random subset of
    (request, head) pairs when a full step is slow, or the full step repeated
    while under the budget when it is fast, for about `seconds` of wall time,
    on `threads` threads (default: every host core).
    Returns (tokens/s for the full step, description, threads)."""
    import oracle
    B, Hq = w_cpu["batch"], w_cpu["hq"]
    rng = np.random.default_rng(0)
    allp = [(b, h) for b in range(B) for h in range(Hq)]
    order = rng.permutation(len(allp))
    threads = threads or oracle.default_threads()
    n0 = min(len(allp), max(threads, 16))
    t = time.perf_counter()
    oracle.decode(w_cpu, sparse=sparse, bh=[allp[i] for i in order[:n0]], nthreads=threads)
    per_pair = (time.perf_counter() - t) / n0
    n = int(min(len(allp), max(n0, seconds / max(per_pair, 1e-9))))
    sel = [allp[i] for i in order[:n]]
    reps = 0
    t = time.perf_counter()
    while True:
        oracle.decode(w_cpu, sparse=sparse, bh=sel, nthreads=threads)
        reps += 1
        dt = time.perf_counter() - t
        if dt >= seconds or n < len(allp):
            break
    step_s = dt / reps * len(allp) / n
    what = (f"fp64 C oracle, sparse decode of {n} of {len(allp)} (request, head) pairs"
            + (f", {reps} repetitions" if reps > 1 else "")
            + f", {dt:.1f} s on {threads} thread{'s' if threads > 1 else ''},"
            " scaled to the full step")
    return B / step_s, what, threads


def to_cpu_workload(w, bt):
    c = dict(w)
    c["q"] = bt.q.cpu()
    c["k_pages"] = bt.k_pages.cpu()
    c["v_pages"] = bt.v_pages.cpu()
    c["keep_mask"] = bt.keep_mask.cpu().numpy().view(np.uint32)
    return c


def kv_replicas(bt, kv_bytes, device, cap=64):
    """The batch's KV pool plus copies, so that the rows R consecutive steps touch
    exceed 4x the L2 (or as many copies as half the free memory holds)."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    pool = bt.k_pages.numel() * bt.k_pages.element_size() * 2
    free, _ = torch.cuda.mem_get_info(device)
    R = max(1, math.ceil(4 * l2 / max(kv_bytes, 1)))
    R = int(max(1, min(R, cap, (0.5 * free) // pool)))
    return [(bt.k_pages, bt.v_pages)] + [(bt.k_pages.clone(), bt.v_pages.clone())
                                         for _ in range(R - 1)], l2


def measure_compact(name, K, W, device, stream, peak):
    """One workload's fused sparse step, two-call decode and dense decode, each a
    K-step CUDA graph over rotating KV copies (as the headline), as a compact
    dict."""
    cfg = wl.WORKLOADS[name]
    w = wl.generate(cfg, device=str(device))
    bt = DecodeBatch.from_workload(w, device=device)
    if cfg.mask == "top_mass":
        _, om = bt.attention_mass(r_local=2, r_diag=2)
        w["keep_mask"] = wl.top_mass_keep_mask(om.cpu().numpy(), w["window"], w["hkv"],
                                               w["mask_words"], band=cfg.band,
                                               frac=cfg.top_mass_frac)
        bt.set_keep_mask(w["keep_mask"])
    order = bt.schedule_order()
    order = None if order is None else torch.as_tensor(order).to(device)
    bt.build_index()
    torch.cuda.synchronize()
    bt.check(f"{name}: build_index")
    by = step_bytes(w, bt.kept_idx.cpu().numpy(), bt.kept_cnt.cpu().numpy())
    pools, l2 = kv_replicas(bt, by["kv"], device)
    R, d = len(pools), bt.dims
    out_2, lse_2 = torch.empty_like(bt.out), torch.empty_like(bt.lse)
    out_d, lse_d = torch.empty_like(bt.out), torch.empty_like(bt.lse)

    def fused(k):
        kp, vp = pools[k % R]
        dsa.dsa_decode_sparse_masked(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.prompt_len,
                                     bt.window, bt.keep_mask, bt.scale, bt.out, bt.lse, bt.ws,
                                     stream, order)

    def decode_only(k):
        kp, vp = pools[k % R]
        dsa.dsa_decode_sparse(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.kept_idx,
                              bt.kept_cnt, bt.scale, out_2, lse_2, bt.ws, stream)

    def dense(k):
        kp, vp = pools[k % R]
        dsa.dsa_decode_dense(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.scale, out_d, lse_d,
                             bt.ws, stream)

    for k in range(W):
        fused(k)
        decode_only(k)
        dense(k)
    torch.cuda.synchronize()
    bt.check(f"{name}: warm-up")
    graphs = [graph_of(f, K, stream) for f in (fused, decode_only, dense)]
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    t_f, t_d, t_x = (time_graph(g, stream) / K for g in graphs)
    bt.check(f"{name}: timed")
    res = {
        "workload": cfg.name, "batch": w["batch"], "hq": w["hq"], "hkv": w["hkv"],
        "head_dim": w["head_dim"],
        "step_us": 1e6 * t_f, "tokens_per_s": w["batch"] / t_f, "bytes": by["masked"],
        "gbs": by["masked"] / t_f / 1e9, "frac": by["masked"] / t_f / 1e9 / peak,
        "decode_only_us": 1e6 * t_d, "decode_only_frac": by["sparse_decode"] / t_d / 1e9 / peak,
        "dense_us": 1e6 * t_x, "dense_frac": by["dense"] / t_x / 1e9 / peak,
        "speedup": t_x / t_f, "kept_fraction": by["rows"] / by["dense_rows"],
        "ideal_speedup": by["dense_rows"] / max(by["rows"], 1),
        "kv_copies": R,
    }
    del graphs, pools, bt, w
    torch.cuda.empty_cache()
    return res


def prefill_inputs(w, q_len, device):
    """q [B, Q, Hq, D] bf16 (seeded) and the device q_len for a chunk of the
    last q_len rows of every request."""
    B, Hq, D = w["batch"], w["hq"], w["head_dim"]
    gen = torch.Generator(device=device).manual_seed(w["seed"] + 77)
    q = torch.randn((B, q_len, Hq, D), generator=gen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    ql = torch.full((B,), q_len, dtype=torch.int32, device=device)
    return q, ql


def prefill_order(w, q_len):
    """Requests by decreasing rows their chunk scans (prompt rows, then the
    window range of the chunk's queries), ties by index."""
    L, P, W = (np.asarray(w[k], np.int64) for k in ("seq_len", "prompt_len", "window"))
    n = np.minimum(q_len, L)
    nA = np.minimum(P, L)
    return np.argsort(-(nA + np.minimum(W + n, L - nA)), kind="stable")


def prefill_bytes(w, q_len, dense=False):
    """Algorithmic bytes of one chunk: the union over the chunk's queries of their
    kept rows (each read once per (request, kv head)), q, out and lse; and the
    flops of the kept (query, row) pairs."""
    import itertools
    B, Hq, Hkv, D = w["batch"], w["hq"], w["hkv"], w["head_dim"]
    g = Hq // Hkv
    rows = pairs = 0
    for b, hk in itertools.product(range(B), range(Hkv)):
        L, P, W = (int(w[k][b]) for k in ("seq_len", "prompt_len", "window"))
        n = min(q_len, L)
        if dense:
            rows += L
            pairs += sum(L - n + t + 1 for t in range(n))
            continue
        bits = w["keep_mask"][b, hk]
        offs = [o for o in range(1, W + 1) if (int(bits[(o - 1) >> 5]) >> ((o - 1) & 31)) & 1]
        union = set()
        for t in range(n):
            i = L - n + t
            kept = set(range(min(P, i + 1))) | {i} | {i - o for o in offs if i - o >= P}
            pairs += len(kept)
            union |= kept
        rows += len(union)
    qb = B * q_len * Hq * D * 2
    ob = B * q_len * Hq * (D + 1) * 4
    return rows * 2 * D * 2 + qb + ob, 4 * D * pairs * g


def measure_prefill(name, q_len, K, W, device, stream, peak):
    """dsa_prefill_sparse on one workload, the last q_len rows of every request
    as the query chunk, against the same kernel with every row kept (dense
    causal), each a K-step CUDA graph over rotating KV copies."""
    cfg = wl.WORKLOADS[name]
    w = wl.generate(cfg, device=str(device))
    bt = DecodeBatch.from_workload(w, device=device)
    if cfg.mask == "top_mass":
        _, om = bt.attention_mass(r_local=2, r_diag=2)
        w["keep_mask"] = wl.top_mass_keep_mask(om.cpu().numpy(), w["window"], w["hkv"],
                                               w["mask_words"], band=cfg.band,
                                               frac=cfg.top_mass_frac)
        bt.set_keep_mask(w["keep_mask"])
    q, ql = prefill_inputs(w, q_len, device)
    order = torch.as_tensor(prefill_order(w, q_len), dtype=torch.int32, device=device)
    order_d = torch.as_tensor(np.argsort(-w["seq_len"], kind="stable"), dtype=torch.int32,
                              device=device)
    out = torch.empty(tuple(q.shape), dtype=torch.float32, device=device)
    lse = torch.empty(tuple(q.shape[:3]), dtype=torch.float32, device=device)
    by, flops = prefill_bytes(w, q_len)
    by_d, flops_d = prefill_bytes(w, q_len, dense=True)
    pools, _ = kv_replicas(bt, by, device)
    R = len(pools)
    # dense causal: every earlier row kept (window past every length, all bits set)
    Lmax = int(w["seq_len"].max())
    words = wl.mask_words_for(Lmax)
    dd = dsa.make_dims(w["batch"], w["hq"], w["hkv"], w["head_dim"], w["num_pages"],
                       w["max_pages"], Lmax, words, w["max_kept"], "bf16", "bf16")
    win_d = torch.as_tensor(w["seq_len"]).to(device)
    mask_d = torch.full((w["batch"], w["hkv"], words), -1, dtype=torch.int32, device=device)
    ws_d = dsa.alloc_workspace(dd, device)

    def sparse(k):
        kp, vp = pools[k % R]
        dsa.dsa_prefill_sparse(bt.dims, q, kp, vp, bt.page_table, bt.seq_len, ql, bt.prompt_len,
                               bt.window, bt.keep_mask, bt.scale, out, lse, bt.ws, stream,
                               request_order=order)

    def dense(k):
        kp, vp = pools[k % R]
        dsa.dsa_prefill_sparse(dd, q, kp, vp, bt.page_table, bt.seq_len, ql, bt.prompt_len,
                               win_d, mask_d, bt.scale, out, lse, ws_d, stream,
                               request_order=order_d)

    for k in range(W):
        sparse(k)
        dense(k)
    torch.cuda.synchronize()
    bt.check("prefill warm-up")
    dsa.check_device_error(ws_d, "prefill warm-up (dense)")
    gs, gd = graph_of(sparse, K, stream), graph_of(dense, K, stream)
    gs.replay()
    gd.replay()
    torch.cuda.synchronize()
    ts, td = time_graph(gs, stream) / K, time_graph(gd, stream) / K
    bt.check("prefill timed")
    res = {
        "call": "dsa_prefill_sparse: the last q_len rows of every request as query tokens, "
                "each over its own kept set; requests handed to the GPU by decreasing scanned "
                "rows (dense: by length)",
        "workload": cfg.name, "batch": w["batch"], "q_len": q_len,
        "us": 1e6 * ts, "query_tokens_per_s": w["batch"] * q_len / ts,
        "bytes": by, "gbs": by / ts / 1e9, "frac_hbm": by / ts / 1e9 / peak,
        "tflops": flops / ts / 1e12,
        "dense_causal_us": 1e6 * td, "dense_gbs": by_d / td / 1e9,
        "speedup": td / ts, "kv_copies": R,
    }
    del gs, gd, pools, bt, w
    torch.cuda.empty_cache()
    return res


def measure_evicted_batch(cfg, batch_after, K, device, stream, peak):
    """The memory side of the mask: after eviction a request keeps only its
    prompt, its window and a partial page resident, so the KV pool that held
    the batch before eviction holds batch_after requests.  Draw a batch of
    that size, evict its pages, and time the fused step on it (CUDA graph,
    K steps)."""
    w = wl.generate(wl.scaled(cfg, batch=batch_after), device=str(device))
    bt = DecodeBatch.from_workload(w, device=device)
    if cfg.mask == "top_mass":
        _, om = bt.attention_mass(r_local=2, r_diag=2)
        bt.set_keep_mask(wl.top_mass_keep_mask(om.cpu().numpy(), w["window"], w["hkv"],
                                               w["mask_words"], band=cfg.band,
                                               frac=cfg.top_mass_frac))
    _, nfree = bt.evict_pages()
    order = bt.schedule_order()
    order = None if order is None else torch.as_tensor(order).to(device)
    mapped = int((w["page_table"] >= 0).sum())

    def fused(k):
        bt.decode_sparse_masked(request_order=order, stream=stream)

    for k in range(3):
        fused(k)
    torch.cuda.synchronize()
    bt.check("evicted batch")
    g = graph_of(fused, K, stream)
    g.replay()
    torch.cuda.synchronize()
    t = time_graph(g, stream) / K
    bt.check("evicted batch timed")
    page_bytes = 16 * w["hkv"] * w["head_dim"] * 2 * 2
    res = {"batch_after": batch_after, "step_us_after": 1e6 * t,
           "tokens_per_s_after": batch_after / t,
           "resident_kv_bytes_at_batch_after": (mapped - int(nfree.item())) * page_bytes,
           "note": "the same steady-state KV pool (the batch's pages before eviction) holds "
                   "batch_after requests once pages no later step reads are evicted; the "
                   "step is timed on that batch after its own eviction (one KV copy, its "
                   "kept rows exceed 4x L2)"}
    del g, bt, w
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    if args.sparse_cluster >= 0:
        dsa.dsa_set_sparse_cluster(args.sparse_cluster)
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    # one non-default stream for everything (graph capture needs one)
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    peak, peak_src = hbm_peak()
    others = []
    if world == 1 and not args.no_other_workloads:
        for name in wl.WORKLOADS:
            if name not in (args.workload, "tiny-fp32"):
                others.append(measure_compact(name, max(10, min(args.steps, 50)),
                                              max(3, min(args.warmup, 5)), device, stream, peak))
    prefill = None
    if world == 1 and not args.no_other_workloads:
        prefill = measure_prefill("janus-pro-7b", 32, max(10, min(args.steps, 50)),
                                  max(3, min(args.warmup, 5)), device, stream, peak)
    cfg = wl.WORKLOADS[args.workload]
    w = wl.generate(cfg, seed=rank_seed(cfg, rank), device=str(device))
    bt = DecodeBatch.from_workload(w, device=device)
    torch.cuda.synchronize()

    mass_ms = None
    if cfg.mask == "top_mass":
        # per-head masks from this batch's measured attention mass (our kernel)
        mass, om = bt.attention_mass(r_local=2, r_diag=2)
        mask = wl.top_mass_keep_mask(om.cpu().numpy(), w["window"], w["hkv"], w["mask_words"],
                                     band=cfg.band, frac=cfg.top_mass_frac)
        bt.set_keep_mask(mask)
        w["keep_mask"] = mask
    # request order for the fused call (most kept rows first when the lengths
    # vary), from the host-side lengths a serving host has when it builds the
    # batch; the step's inputs and results live in packed buffers so that the
    # end-to-end run moves them in one copy each way
    packed, order = bt.pack_io(bt.schedule_order())
    bt.build_index()
    torch.cuda.synchronize()
    bt.check("build_index")
    kept_idx = bt.kept_idx.cpu().numpy()
    kept_cnt = bt.kept_cnt.cpu().numpy()
    by = step_bytes(w, kept_idx, kept_cnt)

    # KV replicas so that consecutive steps never find their rows in L2
    pools, l2 = kv_replicas(bt, by["kv"], device)
    R = len(pools)
    d = bt.dims
    K, W = args.steps, args.warmup


    def step(k):
        """The hot path as one call: kept sets read from the masks inside the
        decode kernel (index compaction fused), gather, softmax, PV, merge."""
        kp, vp = pools[k % R]
        dsa.dsa_decode_sparse_masked(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.prompt_len,
                                     bt.window, bt.keep_mask, bt.scale, bt.out, bt.lse, bt.ws,
                                     stream, order)

    out_2 = torch.empty_like(bt.out)
    lse_2 = torch.empty_like(bt.lse)

    def two_call_step(k):
        kp, vp = pools[k % R]
        dsa.dsa_build_index(d, bt.seq_len, bt.prompt_len, bt.window, bt.keep_mask, bt.kept_idx,
                            bt.kept_cnt, bt.ws, stream)
        dsa.dsa_decode_sparse(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.kept_idx,
                              bt.kept_cnt, bt.scale, out_2, lse_2, bt.ws, stream)

    def decode_only(k):
        kp, vp = pools[k % R]
        dsa.dsa_decode_sparse(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.kept_idx,
                              bt.kept_cnt, bt.scale, out_2, lse_2, bt.ws, stream)

    out_dense = torch.empty_like(bt.out)
    lse_dense = torch.empty_like(bt.lse)

    def dense_step(k):
        kp, vp = pools[k % R]
        dsa.dsa_decode_dense(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.scale, out_dense,
                             lse_dense, bt.ws, stream)

    # warm-up: W eager steps of each kind
    for k in range(W):
        step(k)
        two_call_step(k)
        dense_step(k)
    torch.cuda.synchronize()
    bt.check("warm-up")
    plan_m = dsa.dsa_decode_plan(d, dsa.PLAN_MASKED)
    plan_s = dsa.dsa_decode_plan(d, dsa.PLAN_SPARSE)
    same_plan = ((plan_m[0], plan_m[1], plan_m[3], plan_m[4]) ==
                 (plan_s[0], plan_s[1], plan_s[3], plan_s[4]))
    same_bits = bool(torch.equal(bt.out, out_2) and torch.equal(bt.lse, lse_2))

    g_step = graph_of(step, K, stream)
    g_two = graph_of(two_call_step, K, stream)
    g_dec = graph_of(decode_only, K, stream)
    g_dense = graph_of(dense_step, K, stream)
    for g in (g_step, g_two, g_dec, g_dense):
        g.replay()  # graph upload + one more untimed pass
    torch.cuda.synchronize()

    probe = time_graph(g_step, stream)
    sampler = ClockSampler(local)
    sampler.start()
    busy(g_step, args.busy_seconds, probe)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_step = time_graph(g_step, stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    busy(g_step, args.busy_seconds / 3, probe)
    clocks = sampler.stop()

    t_two = time_graph(g_two, stream)
    t_dec = time_graph(g_dec, stream)
    t_dense = time_graph(g_dense, stream)
    torch.cuda.synchronize()
    bt.check("timed region")

    t_step, t_two, t_dec, t_dense = max_over_ranks([t_step, t_two, t_dec, t_dense], device)

    # end-to-end through the API with host buffers; every step uploads its
    # packed inputs from pinned host memory, runs the fused decode and
    # downloads out and lse.  Direct: one C call per step
    # (dsa_decode_sparse_masked_io).  Recorded: that call recorded once per KV
    # copy as a dsa_graph, one dsa_graph_launch per step.  Two slots (the
    # headline): a second slot with its own inputs, outputs, workspace and
    # stream, step k in slot k % 2, so that one slot's copies overlap the
    # other's kernels (double-buffered host I/O).
    h2d, d2h = packed.h2d_bytes, packed.d2h_bytes
    e2e_calls = [bt.decode_step_io(packed, order, stream, kp, vp, prepare=True)
                 for kp, vp in pools]
    e2e_graphs = [bt.record_step_io(packed, stream, order, kp, vp) for kp, vp in pools]
    bt_b = bt.replicate()
    packed_b, order_b = bt_b.pack_io(None if order is None else order.cpu().numpy())
    stream_b = torch.cuda.Stream(device)
    e2e_graphs_b = [bt_b.record_step_io(packed_b, stream_b, order_b, kp, vp) for kp, vp in pools]
    torch.cuda.synchronize()

    def time_e2e(run_step):
        for k in range(min(W, 3) * 2):
            run_step(k)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        stream_b.wait_stream(stream)
        h0 = time.perf_counter()
        for k in range(K):
            run_step(k)
        host = time.perf_counter() - h0
        stream.wait_stream(stream_b)
        e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3
        (t, host) = max_over_ranks([t, host], device)
        return t, host

    def two_slots(k):
        if k % 2 == 0:
            e2e_graphs[k % R].launch(stream)
        else:
            e2e_graphs_b[k % R].launch(stream_b)

    # the same two slots with inputs resident (no copies): how much of the
    # two-slot gain is the overlap of consecutive kernels rather than of copies
    def record(call, st):
        dsa.dsa_graph_begin(st)
        call()
        return dsa.dsa_graph_end(st)

    dev_graphs = [[record(lambda b=b_, s_=s_, o=o_, kp=kp, vp=vp: dsa.dsa_decode_sparse_masked(
                      d, b.q, kp, vp, b.page_table, b.seq_len, b.prompt_len, b.window,
                      b.keep_mask, b.scale, b.out, b.lse, b.ws, s_, o), s_)
                   for kp, vp in pools]
                  for b_, s_, o_ in ((bt, stream, order), (bt_b, stream_b, order_b))]

    def two_slots_device(k):
        if k % 2 == 0:
            dev_graphs[0][k % R].launch(stream)
        else:
            dev_graphs[1][k % R].launch(stream_b)

    t_e2e_direct, host_direct = time_e2e(lambda k: e2e_calls[k % R]())
    t_e2e_rec, host_rec = time_e2e(lambda k: e2e_graphs[k % R].launch(stream))
    t_e2e, host_e2e = time_e2e(two_slots)
    t_two_dev, _ = time_e2e(two_slots_device)
    bt.check("end-to-end steps")
    bt_b.check("end-to-end steps (second slot)")

    # attention-mass pass (the characterisation kernel), timed alone
    if K > 0:
        m_out = torch.empty((w["batch"], w["hq"], 4), dtype=torch.float32, device=device)
        om_out = torch.empty((w["batch"], w["hq"], w["max_window"] + 1), dtype=torch.float32,
                             device=device)

        def mass_step(k):
            kp, _ = pools[k % R]
            dsa.dsa_attention_mass(d, bt.q, kp, bt.page_table, bt.seq_len, bt.prompt_len,
                                   bt.window, bt.grid_w, 2, 2, bt.scale, m_out, om_out, bt.ws,
                                   stream)
        for k in range(3):
            mass_step(k)
        g_mass = graph_of(mass_step, min(K, 50), stream)
        g_mass.replay()
        mass_ms = 1e3 * time_graph(g_mass, stream) / min(K, 50)

    # memory side: pages no later step reads, unmapped on a copy of the table
    freed = torch.empty(bt.page_table.numel(), dtype=torch.int32, device=device)
    nfreed = torch.zeros(1, dtype=torch.int32, device=device)
    pt_copy = bt.page_table.clone()
    dsa.dsa_evict_pages(d, bt.seq_len, bt.prompt_len, bt.window, pt_copy, freed, nfreed, bt.ws,
                        stream)  # warm-up (first launch of the kernel)
    pt_copy.copy_(bt.page_table)
    nfreed.zero_()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    dsa.dsa_evict_pages(d, bt.seq_len, bt.prompt_len, bt.window, pt_copy, freed, nfreed, bt.ws,
                        stream)
    e1.record(stream)
    e1.synchronize()
    bt.check("evict_pages")
    page_bytes = 16 * w["hkv"] * w["head_dim"] * (2 if w["dtype"] == "bf16" else 4) * 2
    mapped = int((w["page_table"] >= 0).sum())
    evicted = int(nfreed.item())
    eviction = {"pages_mapped": mapped, "pages_evicted": evicted,
                "resident_kv_bytes_before": mapped * page_bytes,
                "resident_kv_bytes_after": (mapped - evicted) * page_bytes,
                "evict_us": 1e3 * e0.elapsed_time(e1)}
    if world == 1 and not args.no_other_workloads and w["dtype"] == "bf16" and evicted > 0:
        # requests of this workload that the same pool holds once evicted pages are reused
        batch_after = min(int(w["batch"] * mapped / max(mapped - evicted, 1)), 16 * w["batch"])
        eviction.update(measure_evicted_batch(cfg, batch_after, max(10, min(K, 50)), device,
                                              stream, peak))
        eviction["tokens_per_s_before"] = world * w["batch"] / (t_step / K)

    # attention mass: every K row of every request (no V), q, the bins and the
    # per-offset weights (written as raw scores, then normalised by the merge)
    elt = 2 if w["dtype"] == "bf16" else 4
    om_bytes = w["batch"] * w["hq"] * (w["max_window"] + 1) * 4
    mass_bytes = (int(w["seq_len"].astype(np.int64).sum()) * w["hkv"] * w["head_dim"] * elt
                  + w["batch"] * w["hq"] * w["head_dim"] * elt + w["batch"] * w["hq"] * 16
                  + 3 * om_bytes)

    B = w["batch"]
    step_s = t_step / K
    tokens = world * B / step_s
    chunk, nch, launches, warps, tile_rows = dsa.dsa_decode_plan(d, dsa.PLAN_MASKED)
    launches_two = dsa.dsa_decode_plan(d, dsa.PLAN_SPARSE)[2]
    achieved = by["masked"] / step_s / 1e9
    kernel = "decode_kernel, kept set read from the keep mask (dsa_decode_sparse_masked)"
    if launches > 1:
        kernel += " + LSE merge kernel"

    result = {
        "metric": METRIC,
        "value": tokens,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": 1e3 * step_s,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage_dtype": w["dtype"],
        "data": "synthetic",
        "config": {
            "workload": cfg.name, "batch": B, "hq": w["hq"], "hkv": w["hkv"],
            "head_dim": w["head_dim"], "page_size": 16, "mask": cfg.mask,
            "seq_len_mean": float(np.mean(w["seq_len"])),
            "kept_rows_per_head_mean": by["rows"] / (B * w["hkv"]),
            "l2": f"inputs larger than L2: {R} rotating KV pool copies, "
                  f"{R * by['kv'] / 1e6:.0f} MB of kept rows per rotation (L2 {l2 / 1e6:.0f} MB)",
            "parallelism": f"replicas x{world}",
            "step": "dsa_decode_sparse_masked: index compaction + gather + softmax + PV "
                    "(+ merge) in one call",
            "request_order": "longest first" if order is not None else "batch order",
            "decode_chunk_rows": chunk, "decode_chunks_max": nch,
            "sparse_cluster": nch if launches == 1 else 1,
            "warps_per_cta": warps, "tile_rows": tile_rows,
        },
        "effective_kv_gbs": by["masked"] / step_s / 1e9,
        "pct_of_hbm_peak": 100.0 * by["masked"] / step_s / 1e9 / peak,
        "step_bytes": by["masked"],
        "roofline": {
            "kernel": kernel,
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_src == "measured" else "fallback 6.8 TB/s",
            "traffic": ncu_traffic(cfg.name),
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch of "
                              "this kernel on this workload (null once the kernel changed)",
            "bytes_per_launch": by["masked"], "launch_us": 1e6 * step_s,
        },
        "two_call_step": {
            "calls": "dsa_build_index + dsa_decode_sparse (kept lists through HBM)",
            "ms_per_step": 1e3 * t_two / K,
            "tokens_per_s": world * B / (t_two / K),
            "bytes": by["step"],
            "gbs": by["step"] / (t_two / K) / 1e9,
            "decode_only_us": 1e6 * t_dec / K,
            "decode_only_gbs": by["sparse_decode"] / (t_dec / K) / 1e9,
            "decode_only_frac": by["sparse_decode"] / (t_dec / K) / 1e9 / peak,
            "launches_per_step": 1 + launches_two,
            "same_bits_as_fused": same_bits if same_plan else None,
        },
        "sparse_vs_dense": {
            "dense_ms_per_step": 1e3 * t_dense / K,
            "dense_tokens_per_s": world * B / (t_dense / K),
            "speedup": t_dense / t_step,
            "kept_fraction": by["rows"] / by["dense_rows"],
            "dense_bytes": by["dense"],
            "dense_gbs": by["dense"] / (t_dense / K) / 1e9,
        },
        "attention_mass_ms": mass_ms,
        "attention_mass_roofline": None if mass_ms is None else {
            "bound": "hbm", "bytes": mass_bytes, "achieved": mass_bytes / (mass_ms * 1e-3) / 1e9,
            "peak": peak, "unit": "GB/s", "frac": mass_bytes / (mass_ms * 1e-3) / 1e9 / peak},
        "eviction": eviction,
        "e2e": {"value": world * B / (t_e2e_direct / K), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": 1e3 * t_e2e_direct / K,
                "host_us_per_step": 1e6 * host_direct / K,
                "call": "dsa_decode_sparse_masked_io per step, one batch at a time: one C call "
                        "uploads the packed inputs from pinned host memory, runs the fused "
                        "decode and downloads out and lse",
                "one_slot_graph": {"tokens_per_s": world * B / (t_e2e_rec / K),
                                   "ms_per_step": 1e3 * t_e2e_rec / K,
                                   "host_us_per_step": 1e6 * host_rec / K,
                                   "call": "the same call recorded once as a dsa_graph, one "
                                           "dsa_graph_launch per step, one batch at a time"},
                "two_slot_pipeline": {"tokens_per_s": world * B / (t_e2e / K),
                                      "ms_per_step": 1e3 * t_e2e / K,
                                      "host_us_per_step": 1e6 * host_e2e / K,
                                      "call": "two micro-batches in flight: two slots with their "
                                              "own buffers and streams, step k in slot k % 2 "
                                              "(recorded dsa_graph per slot), so one slot's copies "
                                              "and kernel overlap the other's"}},
        "two_slots_device": {
            "tokens_per_s": world * B / (t_two_dev / K), "ms_per_step": 1e3 * t_two_dev / K,
            "note": "inputs resident, no copies; the two slots of the e2e run on two streams, "
                    "so consecutive steps' kernels overlap each other's ramp and tail"},
        "gpu_launches": K * launches,
        "clocks": clocks,
    }
    if others:
        result["workloads"] = others
    if prefill is not None:
        result["prefill"] = prefill

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w_cpu = to_cpu_workload(w, bt)
        tps, what, threads = cpu_oracle_sample(w_cpu, args.cpu_seconds)
        tps1, what1, _ = cpu_oracle_sample(w_cpu, args.cpu_seconds / 4, threads=1)
        result["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": threads,
                                  "kind": "oracle", "sample": what,
                                  "one_core": {"value": tps1, "sample": what1}}
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# ---------------------------------------------------------------------------
# the reference arm: the fp64 CPU oracle, timed as it stands
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    cfg = wl.WORKLOADS[args.workload]
    w = wl.generate(cfg)
    if cfg.mask == "top_mass":
        # the same selection rule as the GPU arm, applied to the oracle's mass
        _, om = oracle.mass(w)
        om = om.reshape(w["batch"], w["hq"], -1)
        w["keep_mask"] = wl.top_mass_keep_mask(om, w["window"], w["hkv"], w["mask_words"],
                                               band=cfg.band, frac=cfg.top_mass_frac)
    B, Hq = w["batch"], w["hq"]
    allp = [(b, h) for b in range(B) for h in range(Hq)]
    rng = np.random.default_rng(0)
    threads = oracle.default_threads()
    budget = max(0.05, 90.0 / (args.steps + args.warmup))
    n = min(len(allp), max(threads, 16))
    t = time.perf_counter()
    oracle.decode(w, sparse=True, bh=[allp[i] for i in rng.permutation(len(allp))[:n]])
    per_pair = (time.perf_counter() - t) / n
    n = int(min(len(allp), max(1, budget / per_pair)))
    for k in range(args.warmup):
        sel = [allp[i] for i in rng.permutation(len(allp))[:n]]
        oracle.decode(w, sparse=True, bh=sel, nthreads=threads)
    total = 0.0
    for k in range(args.steps):
        sel = [allp[i] for i in rng.permutation(len(allp))[:n]]
        t = time.perf_counter()
        oracle.decode(w, sparse=True, bh=sel, nthreads=threads)
        total += time.perf_counter() - t
    step_s = total / args.steps * len(allp) / n
    tps = B / step_s
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * step_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": B, "hq": Hq, "hkv": w["hkv"],
                   "head_dim": w["head_dim"]},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: fp64 C oracle sparse decode of {n} of {len(allp)} "
                                   f"(request, head) pairs, scaled to the full step"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile(args):
    """W + K eager launches of one library call on one KV pool, for a profiler
    to capture (launch j of the call is the j-th launch of its kernel)."""
    if args.sparse_cluster >= 0:
        dsa.dsa_set_sparse_cluster(args.sparse_cluster)
    device = torch.device("cuda", 0)
    cfg = wl.WORKLOADS[args.workload]
    if args.batch > 0:
        cfg = wl.scaled(cfg, batch=args.batch)
    w = wl.generate(cfg, device=str(device))
    bt = DecodeBatch.from_workload(w, device=device)
    if cfg.mask == "top_mass":
        _, om = bt.attention_mass(r_local=2, r_diag=2)
        bt.set_keep_mask(wl.top_mass_keep_mask(om.cpu().numpy(), w["window"], w["hkv"],
                                               w["mask_words"], band=cfg.band,
                                               frac=cfg.top_mass_frac))
    bt.build_index()
    order = bt.schedule_order()
    order = None if order is None else torch.as_tensor(order).to(device)
    q4, ql = prefill_inputs(w, 32, device)
    o4 = torch.empty(tuple(q4.shape), dtype=torch.float32, device=device)
    l4 = torch.empty(tuple(q4.shape[:3]), dtype=torch.float32, device=device)
    porder = torch.as_tensor(prefill_order(w, 32), dtype=torch.int32, device=device)

    def prefill_call():
        dsa.dsa_prefill_sparse(bt.dims, q4, bt.k_pages, bt.v_pages, bt.page_table, bt.seq_len, ql,
                               bt.prompt_len, bt.window, bt.keep_mask, bt.scale, o4, l4, bt.ws,
                               request_order=porder)
    call = {"prefill": prefill_call, "index": bt.build_index, "sparse": bt.decode_sparse,
            "masked": lambda: bt.decode_sparse_masked(request_order=order),
            "dense": bt.decode_dense,
            "mass": lambda: bt.attention_mass(r_local=2, r_diag=2)}[args.profile]
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    bt.check(args.profile)
    print(json.dumps({"profile": args.profile, "workload": cfg.name, "batch": cfg.batch,
                      "launches": args.warmup + args.steps}), flush=True)


def run_sparsity_sweep(args):
    """Speedup of the sparse step over dense decode as the kept fraction varies.

    The Janus-Pro-7B-like batch (64 requests, 32 heads, head_dim 128, prompt 256,
    L = P + U[64, 1024]) with per-(request, head) random masks: the band 1..8
    always kept, every other window offset kept with probability p; the window
    W and p are swept.  Each point: the fused step and the dense decode of the
    same batch, CUDA-graph timed over KV copies larger than 4x L2."""
    device = torch.device("cuda", 0)
    base = wl.WORKLOADS["janus-pro-7b"]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    K = max(10, min(args.steps, 100))
    for W in (32, 96, 256, 512, 1024):
        for p in (0.0, 0.25, 1.0):
            cfg = wl.scaled(base, window_rows=None, window=W, random_frac=(p, p),
                            seed=base.seed + 17)
            w = wl.generate(cfg, device=str(device))
            bt = DecodeBatch.from_workload(w, device=device)
            bt.build_index()
            torch.cuda.synchronize()
            kept = bt.kept_cnt.cpu().numpy()
            by = step_bytes(w, bt.kept_idx.cpu().numpy(), kept)
            dense_bytes = by["dense"]
            pool = bt.k_pages.numel() * bt.k_pages.element_size() * 2
            free, _ = torch.cuda.mem_get_info(device)
            R = int(max(1, min(math.ceil(4 * l2 / max(by["kv"], 1)), 32, (0.5 * free) // pool)))
            pools = [(bt.k_pages, bt.v_pages)] + [(bt.k_pages.clone(), bt.v_pages.clone())
                                                  for _ in range(R - 1)]
            d = bt.dims
            out_d = torch.empty_like(bt.out)
            lse_d = torch.empty_like(bt.lse)

            def fused(k):
                kp, vp = pools[k % R]
                dsa.dsa_decode_sparse_masked(d, bt.q, kp, vp, bt.page_table, bt.seq_len,
                                             bt.prompt_len, bt.window, bt.keep_mask, bt.scale,
                                             bt.out, bt.lse, bt.ws, stream)

            def dense(k):
                kp, vp = pools[k % R]
                dsa.dsa_decode_dense(d, bt.q, kp, vp, bt.page_table, bt.seq_len, bt.scale,
                                     out_d, lse_d, bt.ws, stream)

            for k in range(3):
                fused(k)
                dense(k)
            torch.cuda.synchronize()
            bt.check("sweep warm-up")
            gf, gd = graph_of(fused, K, stream), graph_of(dense, K, stream)
            gf.replay()
            gd.replay()
            tf = time_graph(gf, stream) / K
            td = time_graph(gd, stream) / K
            bt.check("sweep")
            frac = by["rows"] / by["dense_rows"]
            print(json.dumps({
                "sweep": "sparsity", "workload": cfg.name, "window": W, "keep_p": p,
                "kept_fraction": frac, "fused_us": 1e6 * tf, "dense_us": 1e6 * td,
                "speedup": td / tf, "ideal_speedup": 1.0 / frac,
                "fused_gbs": by["masked"] / tf / 1e9, "dense_gbs": dense_bytes / td / 1e9,
            }), flush=True)
            del pools, bt, w, gf, gd
            torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.sweep_sparsity:
        run_sparsity_sweep(args)
    elif args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
