"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Bars (written here, derived in the design notes):
  kept-index lists and counts: bit-exact;
  fp32 inputs: max |gpu - oracle| <= 1e-5 on outputs;
  bf16 q/KV (fp32 accumulation): max <= 2e-2 and mean <= 2e-3 on outputs;
  lse: max <= 1e-4; attention-mass bins and per-offset weights: max <= 1e-5.
Every oracle input comes from the seeded generators; config-5 masks come from
the oracle's own attention mass.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from kv_cache_serving_gb300 import dsa
from kv_cache_serving_gb300 import workloads as wl
from kv_cache_serving_gb300.session import DecodeBatch

pytestmark = pytest.mark.gpu

F32_MAX = 1e-5
BF16_MAX, BF16_MEAN = 2e-2, 2e-3
LSE_MAX = 1e-4
MASS_MAX = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.init()


def assert_outputs(gpu, ref, fp32):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(ref.shape)
    assert np.isfinite(gpu).all()
    err = np.abs(gpu - ref)
    if fp32:
        assert err.max() <= F32_MAX, err.max()
    else:
        assert err.max() <= BF16_MAX, err.max()
        assert err.mean() <= BF16_MEAN, err.mean()


def oracle_kept(w, mask=None):
    mask = w["keep_mask"] if mask is None else mask
    res = {}
    for b in range(w["batch"]):
        for hk in range(w["hkv"]):
            res[b, hk] = oracle.kept_set(int(w["seq_len"][b]), int(w["prompt_len"][b]),
                                         int(w["window"][b]), mask[b, hk])
    return res


def check_index(bt, w, mask=None):
    bt.build_index()
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    cnt = bt.kept_cnt.cpu().numpy()
    idx = bt.kept_idx.cpu().numpy()
    for (b, hk), want in oracle_kept(w, mask).items():
        assert cnt[b, hk] == len(want), (b, hk)
        assert np.array_equal(idx[b, hk, :cnt[b, hk]], want), (b, hk)


def oracle_inputs(w, mask=None):
    d = dict(w)
    if mask is not None:
        d["keep_mask"] = mask
    return d


def same_plan(bt):
    """True when the two sparse calls split rows into the same chunks over the
    same warps, so that they sum in the same order."""
    ps = dsa.dsa_decode_plan(bt.dims, dsa.PLAN_SPARSE)
    pm = dsa.dsa_decode_plan(bt.dims, dsa.PLAN_MASKED)
    return (ps[0], ps[1], ps[3], ps[4]) == (pm[0], pm[1], pm[3], pm[4])


def run_both(w, mask=None, bh=None):
    """GPU sparse (kept lists, and in-kernel from the mask) + dense vs oracle on
    all (or the listed) (b, h) pairs."""
    bt = DecodeBatch.from_workload(w, keep_mask=mask)
    check_index(bt, w, mask)
    fp32 = w["dtype"] == "f32"
    inp = oracle_inputs(w, mask)
    listed = None
    for mode in ("sparse", "masked", "dense"):
        out, lse = {"sparse": bt.decode_sparse, "masked": bt.decode_sparse_masked,
                    "dense": bt.decode_dense}[mode]()
        torch.cuda.synchronize()
        assert bt.device_error() == 0
        o = out.cpu().numpy().reshape(-1, w["head_dim"])
        l = lse.cpu().numpy().reshape(-1)
        if mode == "sparse":
            listed = o.copy(), l.copy()
        elif mode == "masked":
            if same_plan(bt):
                # same kept set, same order, same chunks: the same bits
                assert np.array_equal(o, listed[0]) and np.array_equal(l, listed[1])
            # the request order changes only the schedule
            order = torch.as_tensor(bt.longest_first_order()[::-1].copy()).to(bt.device)
            o2, l2 = bt.decode_sparse_masked(out=torch.empty_like(out),
                                             lse=torch.empty_like(lse), request_order=order)
            torch.cuda.synchronize()
            assert bt.device_error() == 0
            assert torch.equal(o2, out) and torch.equal(l2, lse)
        ref_o, ref_l = oracle.decode(inp, sparse=mode != "dense", bh=bh)
        if bh is not None:
            sel = [b * w["hq"] + h for b, h in bh]
            o, l = o[sel], l[sel]
        assert_outputs(o, ref_o, fp32)
        assert np.abs(l - ref_l).max() <= LSE_MAX
        if mode == "sparse":
            ref_sparse = ref_o, ref_l
    # sparse decode with clusters off (rows split into chunks of separate CTAs,
    # merged by merge_kernel) and split over thread-block clusters (merged in
    # shared memory)
    saved = dsa.dsa_get_sparse_cluster()
    try:
        for ctas in (1, 2, 4):
            dsa.dsa_set_sparse_cluster(ctas)
            o1, l1 = [t.clone() for t in bt.decode_sparse()]
            o2, l2 = bt.decode_sparse_masked()
            torch.cuda.synchronize()
            assert bt.device_error() == 0
            if same_plan(bt):   # same rows, same split, same warps: same bits
                assert torch.equal(o1, o2) and torch.equal(l1, l2)
            o = o2.cpu().numpy().reshape(-1, w["head_dim"])
            l = l2.cpu().numpy().reshape(-1)
            if bh is not None:
                o, l = o[sel], l[sel]
            assert_outputs(o, ref_sparse[0], fp32)
            assert np.abs(l - ref_sparse[1]).max() <= LSE_MAX
    finally:
        dsa.dsa_set_sparse_cluster(saved)
    return bt


def small_cfg(D, G, dtype, batch=5, hkv=2, Lmax=700, Pmax=100, W=64, seed=0, mask="random"):
    return wl.Config(f"t-{D}-{G}-{dtype}", batch, hkv * G, hkv, D, dtype, (0, Pmax), (8,), None,
                     W, ("abs", 1, Lmax), mask, band=2, seed=seed)


# ---------------------------------------------------------------------------
# small problems: every built (head_dim, group, dtype), several tiles, ragged
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_small_parity(D, G, dtype):
    w = wl.generate(small_cfg(D, G, dtype, seed=D + G), spare_pages=3)
    run_both(w)


@pytest.mark.parametrize("D,G", [(64, 1), (128, 4)])
def test_mixed_q_dtype(D, G):
    w = wl.generate(small_cfg(D, G, "bf16", seed=7))
    w["q"] = torch.randn(w["q"].shape, generator=torch.Generator().manual_seed(70))
    run_both(w)   # q fp32, KV bf16


def test_many_units_single_chunk_path():
    # many short requests: each (request, kv head) fits one chunk, so the decode
    # kernel writes the final output itself.
    w = wl.generate(small_cfg(128, 1, "bf16", batch=96, hkv=8, Lmax=60, Pmax=20, W=32, seed=3))
    run_both(w)


# ---------------------------------------------------------------------------
# the workloads
# ---------------------------------------------------------------------------

def test_tiny_fp32_every_decode_step():
    cfg = wl.scaled(wl.WORKLOADS["tiny-fp32"], seq=("abs", 80, 80))
    w = wl.generate(cfg)
    golden = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_fp32_kept_sets.txt")) as f:
        for ln in f:
            ln = ln.split("#")[0].strip()
            if ln:
                L, rows = ln.split(":")
                golden[int(L)] = rows.split()
    for L in range(17, 81):
        w["seq_len"] = np.array([L], np.int32)
        bt = run_both(w)
        if L in golden:
            from test_oracle_pins import expand_ranges
            n = int(bt.kept_cnt[0, 0])
            assert bt.kept_idx[0, 0, :n].cpu().tolist() == expand_ranges(golden[L])


@pytest.mark.parametrize("name", ["llamagen-xl", "janus-pro-7b", "emu3-8b"])
def test_workload_reduced_batch(name):
    cfg = wl.WORKLOADS[name]
    w = wl.generate(wl.scaled(cfg, batch=3 if name == "emu3-8b" else 6))
    run_both(w)


def top_mass_masks_from_oracle(w):
    _, om = oracle.mass(w, r_local=2, r_diag=2)
    om = om.reshape(w["batch"], w["hq"], -1)
    return wl.top_mass_keep_mask(om, w["window"], w["hkv"], w["mask_words"],
                                 band=w["config"].band, frac=w["config"].top_mass_frac)


def test_mixed_serving_reduced_batch():
    w = wl.generate(wl.scaled(wl.WORKLOADS["mixed-serving"], batch=6))
    run_both(w, mask=top_mass_masks_from_oracle(w))


@pytest.mark.parametrize("name", ["llamagen-xl", "janus-pro-7b", "emu3-8b", "mixed-serving"])
def test_workload_full_size(name):
    """Full-size batches in the launch configuration the benchmark uses (its
    builds, request order, waves and tails): kept lists and the outputs of every
    (request, head) pair compared with the oracle, sparse and dense."""
    w = wl.generate(wl.WORKLOADS[name])
    mask = None
    if name == "mixed-serving":
        _, om = oracle.mass(w, bh=None, with_offsets=True)
        om = om.reshape(w["batch"], w["hq"], -1)
        mask = wl.top_mass_keep_mask(om, w["window"], w["hkv"], w["mask_words"])
    run_both(w, mask=mask)


@pytest.mark.parametrize("name,batch", [("mixed-serving", 64), ("janus-pro-7b", 20),
                                        ("llamagen-xl", 24)])
def test_small_batch_build(name, batch):
    """Batches that need two waves of the default build: the small-batch build
    (5 warps, one stage) where it fits them in one wave, kept lists and the
    fused call, every pair vs the oracle."""
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    mask = top_mass_masks_from_oracle(w) if w["keep_mask"] is None else None
    bt = DecodeBatch.from_workload(w, keep_mask=mask)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = dsa.dsa_decode_plan(bt.dims, dsa.PLAN_MASKED)
    if sms == 152 and w["hq"] == w["hkv"]:
        # CUDA-core engine, 480-640 units: two waves of 3 CTAs/SM, one of the small
        # build (on the tensor-core engine it holds no more CTAs, so the plan keeps
        # the default build there)
        assert plan[3] == 5, plan
    run_both(w, mask=mask)


def test_batch_past_the_schedule_limit():
    """1100 requests: more than dsa_build_index schedules (1024), so no schedule
    is written and dsa_decode_sparse runs in batch order; every path still
    matches the oracle on every pair (many short units, several waves)."""
    w = wl.generate(small_cfg(128, 4, "bf16", batch=1100, hkv=1, Lmax=120, Pmax=30, W=48,
                              seed=77))
    run_both(w)


def test_request_schedule_changes_no_bits():
    """dsa_build_index leaves a longest-first request schedule in the workspace;
    dsa_decode_sparse on it must give the bits it gives on a workspace without
    one (a zero-filled copy: no schedule tag), and a schedule written for
    another batch size must be ignored."""
    w = wl.generate(wl.scaled(wl.WORKLOADS["mixed-serving"], batch=24))
    mask = top_mass_masks_from_oracle(w)
    bt = DecodeBatch.from_workload(w, keep_mask=mask)
    bt.build_index()
    with_sched = [t.clone() for t in bt.decode_sparse()]
    fresh = torch.zeros_like(bt.ws)
    out = torch.empty_like(bt.out)
    lse = torch.empty_like(bt.lse)
    dsa.dsa_decode_sparse(bt.dims, bt.q, bt.k_pages, bt.v_pages, bt.page_table, bt.seq_len,
                          bt.kept_idx, bt.kept_cnt, bt.scale, out, lse, fresh)
    torch.cuda.synchronize()
    assert bt.device_error() == 0 and dsa.dsa_get_device_error(fresh) == 0
    assert torch.equal(out, with_sched[0]) and torch.equal(lse, with_sched[1])
    # the first 12 requests alone, decoded on the workspace that holds the
    # 24-request schedule: the tag does not match, batch order is used
    d12 = dsa.make_dims(12, w["hq"], w["hkv"], w["head_dim"], w["num_pages"], w["max_pages"],
                        w["max_window"], w["mask_words"], w["max_kept"], "bf16", "bf16")
    o12 = torch.empty_like(bt.out[:12])
    l12 = torch.empty_like(bt.lse[:12])
    dsa.dsa_decode_sparse(d12, bt.q[:12].contiguous(), bt.k_pages, bt.v_pages,
                          bt.page_table[:12].contiguous(), bt.seq_len[:12].contiguous(),
                          bt.kept_idx[:12].contiguous(), bt.kept_cnt[:12].contiguous(), bt.scale,
                          o12, l12, bt.ws)
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    ref, ref_lse = oracle.decode(oracle_inputs(w, mask), sparse=True,
                                 bh=[(b, h) for b in range(12) for h in range(w["hq"])])
    assert_outputs(o12.cpu().numpy().reshape(-1, w["head_dim"]), ref, fp32=False)
    assert np.abs(l12.cpu().numpy().reshape(-1) - ref_lse).max() <= LSE_MAX


def test_wide_build_for_small_batches():
    """At most one (request, kv head) per SM: one 8-warp CTA per unit (automatic
    cluster setting), checked against the oracle; forcing clusters of 2 falls
    back to the cluster split."""
    w = wl.generate(wl.scaled(wl.WORKLOADS["emu3-8b"], batch=4))
    bt = DecodeBatch.from_workload(w)
    saved = dsa.dsa_get_sparse_cluster()
    try:
        dsa.dsa_set_sparse_cluster(0)
        plan = dsa.dsa_decode_plan(bt.dims, dsa.PLAN_MASKED)
        assert plan[1] == 1 and plan[2] == 1 and plan[3] == 8, plan
        dsa.dsa_set_sparse_cluster(2)
        assert dsa.dsa_decode_plan(bt.dims, dsa.PLAN_MASKED)[3] != 8
    finally:
        dsa.dsa_set_sparse_cluster(saved)
    run_both(w)


# ---------------------------------------------------------------------------
# invariants and edge cases
# ---------------------------------------------------------------------------

def test_skipped_rows_are_never_read():
    w = wl.generate(wl.scaled(wl.WORKLOADS["janus-pro-7b"], batch=4), spare_pages=5)
    kept = oracle_kept(w)
    bt = DecodeBatch.from_workload(w)
    bt.build_index()
    base = bt.decode_sparse()[0].clone()
    for value in (float("nan"), float("inf"), 1e30):
        p = wl.poison_unread(w, lambda b, hk: kept[b, hk], value)
        bp = DecodeBatch.from_workload(p)
        bp.build_index()
        out = bp.decode_sparse()[0].clone()
        out_m = bp.decode_sparse_masked()[0]
        torch.cuda.synchronize()
        assert torch.equal(out, base)
        if same_plan(bp):
            assert torch.equal(out_m, base)
        else:
            assert torch.isfinite(out_m).all()


def test_batch_zero_is_a_no_op():
    w = wl.generate(small_cfg(64, 1, "bf16", batch=1))
    bt = DecodeBatch.from_workload(w)
    bt.dims.batch = 0
    bt.build_index()
    bt.decode_sparse()
    bt.decode_dense()
    torch.cuda.synchronize()
    assert bt.device_error() == 0


def test_first_token_and_prompt_only():
    w = wl.generate(small_cfg(128, 2, "f32", batch=4, seed=9))
    w["seq_len"] = np.array([1, 1, 5, 30], np.int32)
    w["prompt_len"] = np.array([0, 3, 10, 30], np.int32)   # L <= P for the last two
    run_both(w)


def test_window_zero_and_empty_or_full_masks():
    w = wl.generate(small_cfg(64, 4, "bf16", batch=4, seed=11, W=40))
    w["window"] = np.array([0, 40, 40, 40], np.int32)
    m = w["keep_mask"].copy()
    m[1] = 0
    m[2] = 0xFFFFFFFF
    run_both(w, mask=m)


def test_all_ones_mask_covering_sequence_equals_dense():
    w = wl.generate(small_cfg(128, 1, "bf16", batch=3, Lmax=200, W=256, seed=12))
    w["window"] = np.full(3, 256, np.int32)
    m = np.full_like(w["keep_mask"], 0xFFFFFFFF)
    bt = run_both(w, mask=m)
    dense_ref, _ = oracle.decode(w, sparse=False)
    out, _ = bt.decode_sparse()
    assert_outputs(out.cpu().numpy().reshape(dense_ref.shape), dense_ref, fp32=False)


def test_large_window_many_mask_words():
    w = wl.generate(small_cfg(128, 8, "bf16", batch=3, Lmax=3000, Pmax=50, W=1000, seed=13))
    run_both(w)


@pytest.mark.parametrize("name,batch", [("llamagen-xl", 6), ("mixed-serving", 8),
                                        ("janus-pro-7b", 4)])
def test_fused_append_of_the_query_row(name, batch):
    """k_new / v_new: the call attends with the new row and stores it in the
    cache.  Reference: the same batch whose cache already holds the row (the
    oracle's input) -- same outputs bit for bit, and the cache afterwards
    equals that reference cache."""
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    if w["keep_mask"] is None:
        w["keep_mask"] = top_mass_masks_from_oracle(w)
    ref_bt = DecodeBatch.from_workload(w)
    ref_out, ref_lse = [t.clone() for t in ref_bt.decode_sparse_masked()]
    # the new rows, then a cache whose rows L-1 hold garbage
    B, Hkv, D = w["batch"], w["hkv"], w["head_dim"]
    k_new = torch.empty((B, Hkv, D), dtype=ref_bt.k_pages.dtype, device="cuda")
    v_new = torch.empty_like(k_new)
    bt = DecodeBatch.from_workload(w)
    for b in range(B):
        j = int(w["seq_len"][b]) - 1
        pg, slot = int(w["page_table"][b, j // 16]), j % 16
        k_new[b] = bt.k_pages[pg, slot]
        v_new[b] = bt.v_pages[pg, slot]
        bt.k_pages[pg, slot] = float("nan")
        bt.v_pages[pg, slot] = 1e30
    out, lse = bt.decode_sparse_masked(k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    assert torch.equal(bt.k_pages, ref_bt.k_pages) and torch.equal(bt.v_pages, ref_bt.v_pages)
    ref_o, ref_l = oracle.decode(w, sparse=True)
    assert_outputs(out.cpu().numpy(), ref_o, fp32=False)


@pytest.mark.parametrize("name,batch", [("llamagen-xl", 6), ("mixed-serving", 12)])
def test_host_io_step(name, batch):
    """dsa_decode_sparse_masked_io: a q written only into the pinned host buffer
    goes up with the call, and out / lse come back into the host buffer with
    the bits of the device-only call on the uploaded inputs; a prepared call
    issued again gives them again; the oracle on the new q agrees."""
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    if w["keep_mask"] is None:
        w["keep_mask"] = top_mass_masks_from_oracle(w)
    bt = DecodeBatch.from_workload(w)
    io, order = bt.pack_io(bt.longest_first_order())
    gen = torch.Generator().manual_seed(11)
    q_new = torch.randn(tuple(bt.q.shape), generator=gen).to(bt.q.dtype)
    io.host["q"].copy_(q_new)
    io.host["out"].fill_(float("nan"))
    io.host["lse"].fill_(float("nan"))
    step = bt.decode_step_io(io, order, prepare=True)
    step()
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    assert torch.equal(bt.q.cpu(), q_new)
    host_out, host_lse = io.host["out"].clone(), io.host["lse"].clone()
    out2, lse2 = bt.decode_sparse_masked(out=torch.empty_like(bt.out), lse=torch.empty_like(bt.lse),
                                         request_order=order)
    torch.cuda.synchronize()
    assert torch.equal(out2.cpu(), host_out) and torch.equal(lse2.cpu(), host_lse)
    io.host["out"].zero_()
    step()
    torch.cuda.synchronize()
    assert torch.equal(io.host["out"], host_out)
    ref_o, ref_l = oracle.decode(dict(w, q=q_new), sparse=True)
    assert_outputs(host_out.numpy().reshape(-1, w["head_dim"]), ref_o, fp32=False)
    assert np.abs(host_lse.numpy().reshape(-1) - ref_l).max() <= LSE_MAX
    # pageable (not page-locked) host buffers: the copies take the copy engine
    # instead of the copy kernel, with the same bytes moved
    page_in = torch.empty(io.host_in.shape, dtype=io.host_in.dtype)
    page_in.copy_(io.host_in)
    page_out = torch.full(io.host_out.shape, 255, dtype=io.host_out.dtype)
    assert not page_in.is_pinned() and not page_out.is_pinned()
    desc = dsa.host_io(page_in, io.dev_in, io.dev_out, page_out)
    dsa.dsa_decode_sparse_masked_io(desc, bt.dims, bt.q, bt.k_pages, bt.v_pages, bt.page_table,
                                    bt.seq_len, bt.prompt_len, bt.window, bt.keep_mask, bt.scale,
                                    bt.out, bt.lse, bt.ws, None, order)
    torch.cuda.synchronize()
    assert torch.equal(page_out, io.host_out)


@pytest.mark.parametrize("name,batch", [("llamagen-xl", 6), ("emu3-8b", 4)])
def test_recorded_host_io_step(name, batch):
    """A dsa_graph of dsa_decode_sparse_masked_io: every replay uploads the q then
    in the pinned host buffer and downloads the results of that q (the bits of
    the direct call on it); three replays with three different q."""
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    bt = DecodeBatch.from_workload(w)
    io, order = bt.pack_io(bt.longest_first_order())
    stream = torch.cuda.Stream()
    graph = bt.record_step_io(io, stream, order)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(5)
    for rep in range(3):
        q_new = torch.randn(tuple(bt.q.shape), generator=gen).to(bt.q.dtype)
        io.host["q"].copy_(q_new)
        io.host["out"].fill_(float("nan"))
        graph.launch(stream)
        stream.synchronize()
        assert bt.device_error() == 0
        assert torch.equal(bt.q.cpu(), q_new)
        got_o, got_l = io.host["out"].clone(), io.host["lse"].clone()
        with torch.cuda.stream(stream):
            o2, l2 = bt.decode_sparse_masked(out=torch.empty_like(bt.out),
                                             lse=torch.empty_like(bt.lse), stream=stream,
                                             request_order=order)
        stream.synchronize()
        assert torch.equal(o2.cpu(), got_o) and torch.equal(l2.cpu(), got_l), rep
        if rep == 0:
            ref_o, ref_l = oracle.decode(dict(w, q=q_new), sparse=True)
            assert_outputs(got_o.numpy().reshape(-1, w["head_dim"]), ref_o, fp32=False)
    # two slots in flight at once on two streams (shared KV cache, own inputs,
    # outputs and workspaces): each slot gets the results of its own q
    bt_b = bt.replicate()
    io_b, order_b = bt_b.pack_io(bt_b.longest_first_order())
    stream_b = torch.cuda.Stream()
    graph_b = bt_b.record_step_io(io_b, stream_b, order_b)
    torch.cuda.synchronize()
    qa = torch.randn(tuple(bt.q.shape), generator=gen).to(bt.q.dtype)
    qb = torch.randn(tuple(bt.q.shape), generator=gen).to(bt.q.dtype)
    io.host["q"].copy_(qa)
    io_b.host["q"].copy_(qb)
    for _ in range(2):
        graph.launch(stream)
        graph_b.launch(stream_b)
    torch.cuda.synchronize()
    assert bt.device_error() == 0 and bt_b.device_error() == 0
    for q_in, host in ((qa, io.host), (qb, io_b.host)):
        ref_o, ref_l = oracle.decode(dict(w, q=q_in), sparse=True)
        assert_outputs(host["out"].numpy().reshape(-1, w["head_dim"]), ref_o, fp32=False)
        assert np.abs(host["lse"].numpy().reshape(-1) - ref_l).max() <= LSE_MAX
    graph.close()
    graph_b.close()


@pytest.mark.parametrize("name,batch", [("emu3-8b", 8), ("mixed-serving", 24),
                                        ("llamagen-xl", 8)])
def test_evict_pages_then_decode_unchanged(name, batch):
    """dsa_evict_pages unmaps exactly the pages the oracle marks, hands back
    exactly their ids, frees nothing more when repeated, and the sparse decode
    calls give the same bits on the evicted cache (they never read those rows)."""
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    if w["keep_mask"] is None:
        w["keep_mask"] = top_mass_masks_from_oracle(w)
    bt = DecodeBatch.from_workload(w)
    bt.build_index()
    before = [t.clone() for t in bt.decode_sparse()] + \
             [t.clone() for t in bt.decode_sparse_masked(out=torch.empty_like(bt.out),
                                                         lse=torch.empty_like(bt.lse))]
    table0 = bt.page_table.cpu().numpy().copy()
    freed, count = bt.evict_pages()
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    table1 = bt.page_table.cpu().numpy()
    want_ids = []
    for b in range(batch):
        flags = oracle.evictable_pages(int(w["seq_len"][b]), int(w["prompt_len"][b]),
                                       int(w["window"][b]))
        npg = len(flags)
        assert np.array_equal(table1[b, :npg] == -1, flags), b
        assert np.array_equal(table1[b, npg:], table0[b, npg:])
        want_ids += table0[b, :npg][flags].tolist()
    n = int(count.item())
    assert n == len(want_ids)
    assert sorted(freed[:n].cpu().tolist()) == sorted(want_ids)
    # again: nothing left to free
    freed2, count2 = bt.evict_pages()
    torch.cuda.synchronize()
    assert int(count2.item()) == 0 and bt.device_error() == 0
    # decode on the evicted cache: same bits
    bt.build_index()
    after = [t.clone() for t in bt.decode_sparse()] + \
            [t.clone() for t in bt.decode_sparse_masked(out=torch.empty_like(bt.out),
                                                        lse=torch.empty_like(bt.lse))]
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    for x, y in zip(before, after):
        assert torch.equal(x, y)


def test_evict_pages_free_list_full():
    w = wl.generate(wl.scaled(wl.WORKLOADS["emu3-8b"], batch=4))
    bt = DecodeBatch.from_workload(w)
    total = sum(int(oracle.evictable_pages(int(w["seq_len"][b]), int(w["prompt_len"][b]),
                                           int(w["window"][b])).sum()) for b in range(4))
    cap = total // 2
    freed, count = bt.evict_pages(capacity=cap)
    torch.cuda.synchronize()
    assert bt.device_error() == 10
    assert int(count.item()) == total                  # every candidate took a ticket
    assert int((bt.page_table == -1).sum()) - int((torch.as_tensor(w["page_table"]) == -1).sum()) == cap
    assert (freed[:cap] >= 0).all()


# ---------------------------------------------------------------------------
# attention mass
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,batch,r_local,r_diag", [("llamagen-xl", 4, 2, 2),
                                                       ("emu3-8b", 2, 1, 2),
                                                       ("mixed-serving", 5, 2, 1),
                                                      ("tiny-fp32", 1, 2, 1)])
def test_attention_mass_parity(name, batch, r_local, r_diag):
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    bt = DecodeBatch.from_workload(w)
    mass, om = bt.attention_mass(r_local=r_local, r_diag=r_diag)
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    ref_m, ref_om = oracle.mass(w, r_local=r_local, r_diag=r_diag)
    m = mass.cpu().numpy().reshape(-1, 4)
    assert np.abs(m - ref_m).max() <= MASS_MAX
    assert np.abs(m.sum(axis=1) - 1).max() <= 1e-5
    assert np.abs(om.cpu().numpy().reshape(ref_om.shape) - ref_om).max() <= MASS_MAX


@pytest.mark.parametrize("D,G,dtype", [(64, 1, "bf16"), (64, 2, "bf16"), (64, 8, "bf16"),
                                       (128, 2, "bf16"), (128, 8, "bf16"), (128, 4, "f32"),
                                       (64, 4, "mixed")])
def test_attention_mass_every_engine(D, G, dtype):
    """Both score engines (tensor cores for bf16 q and K with G >= 2, CUDA
    cores otherwise), several tiles per chunk and ragged tails."""
    w = wl.generate(small_cfg(D, G, "f32" if dtype == "f32" else "bf16", batch=4, Lmax=1500,
                              W=40, seed=30 + D + G))
    if dtype == "mixed":
        w["q"] = torch.randn(w["q"].shape, generator=torch.Generator().manual_seed(31))
    bt = DecodeBatch.from_workload(w)
    mass, om = bt.attention_mass(r_local=2, r_diag=1)
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    ref_m, ref_om = oracle.mass(w, r_local=2, r_diag=1)
    m = mass.cpu().numpy().reshape(-1, 4)
    assert np.abs(m - ref_m).max() <= MASS_MAX
    assert np.abs(om.cpu().numpy().reshape(ref_om.shape) - ref_om).max() <= MASS_MAX


# ---------------------------------------------------------------------------
# invalid per-request data: flagged on the device, no fault
# ---------------------------------------------------------------------------

def test_device_errors_are_flagged():
    w = wl.generate(small_cfg(64, 2, "bf16", batch=4, seed=21, Lmax=300))
    bt = DecodeBatch.from_workload(w)

    # seq_len 0 for request 1: dense output of that request is NaN, others fine
    bt.seq_len[1] = 0
    bt.decode_dense()
    torch.cuda.synchronize()
    assert bt.device_error() == 1
    assert torch.isnan(bt.out[1]).all()
    ref, _ = oracle.decode(w, sparse=False, bh=[(0, h) for h in range(w["hq"])])
    assert_outputs(bt.out[0].cpu().numpy(), ref, fp32=False)
    bt.seq_len[1] = int(w["seq_len"][1])
    bt.ws.zero_()

    # a page id outside the pool
    bt.page_table[2, 0] = w["num_pages"] + 7
    bt.decode_dense()
    torch.cuda.synchronize()
    assert bt.device_error() == 4
    bt.page_table[2, 0] = int(w["page_table"][2, 0])
    bt.ws.zero_()

    # a window above max_window: build_index flags it and stores count 0,
    # then decode_sparse flags the count
    bt.window[3] = w["max_window"] + 1
    bt.build_index()
    torch.cuda.synchronize()
    assert bt.device_error() == 3
    assert int(bt.kept_cnt[3].max()) == 0
    bt.ws.zero_()
    bt.decode_sparse()
    torch.cuda.synchronize()
    assert bt.device_error() == 6
    # the in-kernel kept set flags the window itself; request 3 is NaN, the rest exact
    bt.ws.zero_()
    bt.decode_sparse_masked()
    torch.cuda.synchronize()
    assert bt.device_error() == 3
    assert torch.isnan(bt.out[3]).all() and torch.isnan(bt.lse[3]).all()
    ref, _ = oracle.decode(w, sparse=True, bh=[(b, h) for b in range(3) for h in range(w["hq"])])
    assert_outputs(bt.out[:3].cpu().numpy(), ref, fp32=False)
    bt.window[3] = int(w["window"][3])
    bt.ws.zero_()

    # masked: a negative prompt length, then more kept rows than max_kept
    bt.prompt_len[0] = -1
    bt.decode_sparse_masked()
    torch.cuda.synchronize()
    assert bt.device_error() == 2
    assert torch.isnan(bt.out[0]).all()
    bt.prompt_len[0] = int(w["prompt_len"][0])
    bt.ws.zero_()
    # a request order entry outside the batch
    bad = torch.tensor([0, 1, 2, 7], dtype=torch.int32, device=bt.device)
    bt.decode_sparse_masked(request_order=bad)
    torch.cuda.synchronize()
    assert bt.device_error() == 9
    bt.ws.zero_()
    small = DecodeBatch.from_workload(dict(w, max_kept=2))
    small.decode_sparse_masked()
    torch.cuda.synchronize()
    assert small.device_error() == 6
    g = w["hq"] // w["hkv"]
    out = small.out.cpu()
    for (b, hk), rows in oracle_kept(w).items():
        heads = out[b, hk * g:(hk + 1) * g]
        assert bool(torch.isnan(heads).all() if len(rows) > 2 else torch.isfinite(heads).all())
    bt.ws.zero_()

    # a kept index past the end of the sequence
    bt.build_index()
    bt.kept_idx[0, 1, 0] = int(w["seq_len"][0]) + 3
    bt.decode_sparse()
    torch.cuda.synchronize()
    assert bt.device_error() == 5
    bt.ws.zero_()

    # everything valid again: clean run
    run_both(w)
