"""Parity of dsa_prefill_sparse (several query tokens per request under the
mask) with the fp64 CPU oracle, through the C ABI.

Bars as for decode (bf16 q/KV, fp32 accumulation): max |gpu - oracle| <= 2e-2,
mean <= 2e-3 over every written element; lse max <= 1e-4.  Slots past q_len
must be left untouched.  Rows that no query of the chunk keeps are never read:
NaN / huge values there change nothing, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_serving_gb300 import dsa
from kv_cache_serving_gb300 import workloads as wl
from kv_cache_serving_gb300.session import DecodeBatch

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-4
SENTINEL = -12345.0


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.init()


def chunk_inputs(w, qmax, seed, q_len=None):
    """q [B, qmax, Hq, D] bf16 and q_len [B] (ragged, at most min(L, qmax))."""
    rng = np.random.default_rng(seed)
    B, Hq, D = w["batch"], w["hq"], w["head_dim"]
    L = w["seq_len"]
    if q_len is None:
        q_len = np.array([int(rng.integers(0, min(qmax, int(L[b])) + 1)) for b in range(B)],
                         np.int32)
        q_len[0] = min(qmax, int(L[0]))
    q = torch.randn(B, qmax, Hq, D, generator=torch.Generator().manual_seed(seed)).to(
        torch.bfloat16)
    return q, np.asarray(q_len, np.int32)


def run_prefill(bt, q, q_len, check_error=True):
    dev = bt.device
    out = torch.full(tuple(q.shape), SENTINEL, dtype=torch.float32, device=dev)
    lse = torch.full(tuple(q.shape[:3]), SENTINEL, dtype=torch.float32, device=dev)
    ql = torch.as_tensor(q_len).to(dev)
    dsa.dsa_prefill_sparse(bt.dims, q.to(dev), bt.k_pages, bt.v_pages, bt.page_table, bt.seq_len,
                           ql, bt.prompt_len, bt.window, bt.keep_mask, bt.scale, out, lse, bt.ws)
    torch.cuda.synchronize()
    if check_error:
        assert bt.device_error() == 0
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def compare(w, q, q_len, out, lse, mask=None):
    inp = dict(w, q=q)
    if mask is not None:
        inp["keep_mask"] = mask
    ref, ref_lse = oracle.multi(inp, q_len)
    B = w["batch"]
    for b in range(B):
        n = int(q_len[b])
        assert (out[b, n:] == SENTINEL).all() and (lse[b, n:] == SENTINEL).all(), b
    written = ~np.isnan(ref)
    assert np.isfinite(out[written]).all()
    err = np.abs(out[written] - ref[written])
    if err.size:
        assert err.max() <= BF16_MAX, err.max()
        assert err.mean() <= BF16_MEAN, err.mean()
    lw = ~np.isnan(ref_lse)
    if lw.any():
        assert np.abs(lse[lw] - ref_lse[lw]).max() <= LSE_MAX
    return ref, ref_lse


def small_cfg(D, G, batch=5, hkv=2, Lmax=400, Pmax=100, W=64, seed=0):
    return wl.Config(f"mq-{D}-{G}", batch, hkv * G, hkv, D, "bf16", (0, Pmax), (8,), None, W,
                     ("abs", 1, Lmax), "random", band=2, seed=seed)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_small_every_build(D, G):
    """Every (head_dim, group): ragged q_len spanning several query tiles and
    row blocks, prompt-only and window queries, shuffled pages."""
    w = wl.generate(small_cfg(D, G, seed=10 * D + G), spare_pages=3)
    bt = DecodeBatch.from_workload(w)
    qmax = 2 * dsa_queries_per_cta(G) + 5
    q, ql = chunk_inputs(w, qmax, seed=D + G)
    out, lse = run_prefill(bt, q, ql)
    compare(w, q, ql, out, lse)


def dsa_queries_per_cta(G):
    return 64 // G


@pytest.mark.parametrize("name,batch,qmax", [("janus-pro-7b", 6, 64), ("llamagen-xl", 8, 24),
                                             ("emu3-8b", 2, 40), ("mixed-serving", 6, 48)])
def test_prefill_workload_shapes(name, batch, qmax):
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    mask = None
    if w["keep_mask"] is None:
        _, om = oracle.mass(w, r_local=2, r_diag=2)
        mask = wl.top_mass_keep_mask(om.reshape(w["batch"], w["hq"], -1), w["window"], w["hkv"],
                                     w["mask_words"], band=w["config"].band,
                                     frac=w["config"].top_mass_frac)
    bt = DecodeBatch.from_workload(w, keep_mask=mask)
    q, ql = chunk_inputs(w, qmax, seed=batch)
    out, lse = run_prefill(bt, q, ql)
    compare(w, q, ql, out, lse, mask)


def test_prefill_whole_sequences_and_edges():
    """q_len = L (every row a query, prompt queries included), q_len = 0, a
    window of 0, an empty mask and an all-ones mask in one batch."""
    cfg = small_cfg(128, 4, batch=6, Lmax=150, Pmax=40, W=64, seed=5)
    w = wl.generate(cfg)
    L = w["seq_len"]
    w["window"][1] = 0
    w["keep_mask"][2] = 0
    w["keep_mask"][3] = 0xFFFFFFFF
    qmax = int(L.max())
    ql = np.array([int(L[0]), 0, int(L[2]), min(int(L[3]), 17), 1, int(L[5])], np.int32)
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, qmax, seed=6, q_len=ql)
    out, lse = run_prefill(bt, q, ql)
    compare(w, q, ql, out, lse)


def test_prefill_window_past_1024_offsets():
    """Windows longer than the fused decode's limit (1024 offsets): 47 mask words
    in shared memory, kept offsets spread over all of them."""
    cfg = small_cfg(128, 2, batch=3, Lmax=2200, Pmax=60, W=1500, seed=11)
    w = wl.generate(cfg)
    assert w["mask_words"] == 47
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, 40, seed=12)
    out, lse = run_prefill(bt, q, ql)
    compare(w, q, ql, out, lse)


def test_prefill_single_query_is_a_decode_step():
    """q_len = 1 is a decode step: within the bars of the decode oracle."""
    w = wl.generate(wl.scaled(wl.WORKLOADS["janus-pro-7b"], batch=4))
    bt = DecodeBatch.from_workload(w)
    q4 = w["q"].view(w["batch"], 1, w["hq"], w["head_dim"]).contiguous()
    ql = np.ones(w["batch"], np.int32)
    out, lse = run_prefill(bt, q4, ql)
    ref, ref_lse = oracle.decode(w, sparse=True)
    err = np.abs(out.reshape(ref.shape) - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN
    assert np.abs(lse.reshape(-1) - ref_lse).max() <= LSE_MAX


def test_prefill_skipped_rows_are_never_read():
    w = wl.generate(wl.scaled(wl.WORKLOADS["janus-pro-7b"], batch=4), spare_pages=5)
    q, ql = chunk_inputs(w, 40, seed=9)
    bt = DecodeBatch.from_workload(w)
    base, lbase = run_prefill(bt, q, ql)

    def kept(b, hk):
        L, P, W = (int(w[k][b]) for k in ("seq_len", "prompt_len", "window"))
        rows = set()
        for t in range(int(ql[b])):
            rows.update(oracle.kept_set(L - int(ql[b]) + t + 1, P, W,
                                        w["keep_mask"][b, hk]).tolist())
        return sorted(rows)

    for value in (float("nan"), 1e30):
        p = wl.poison_unread(w, kept, value)
        bt2 = DecodeBatch.from_workload(p)
        out, lse = run_prefill(bt2, q, ql)
        assert np.array_equal(out, base) and np.array_equal(lse, lbase)


def test_prefill_invalid_q_len_is_flagged():
    w = wl.generate(wl.scaled(wl.WORKLOADS["llamagen-xl"], batch=3))
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, 8, seed=3)
    ql = ql.copy()
    ql[1] = int(w["seq_len"][1]) + 1          # more queries than rows
    out, lse = run_prefill(bt, q, ql, check_error=False)
    assert bt.device_error() == 11            # DSA_DEV_BAD_QLEN
    assert np.isnan(out[1]).all() and np.isnan(lse[1]).all()
    dsa.dsa_clear_device_error(bt.ws)


@pytest.mark.parametrize("parts", [1, 2, 3, 8])
@pytest.mark.parametrize("D,G", [(128, 4), (64, 1)])
def test_prefill_split_parts(D, G, parts):
    """Every unit split into `parts` CTAs along its scanned rows (1: none), the
    partial states merged by the unit's last part: vs the oracle, with parts that
    get no block at all among them; a repeat on the same workspace gives the same
    bits (the arrival counters are back at zero after each call)."""
    w = wl.generate(small_cfg(D, G, batch=5, Lmax=600, Pmax=100, W=200, seed=20 + D + G))
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, 40, seed=22)
    saved = dsa.dsa_get_prefill_split()
    try:
        dsa.dsa_set_prefill_split(parts)
        out, lse = run_prefill(bt, q, ql)
        compare(w, q, ql, out, lse)
        out2, lse2 = run_prefill(bt, q, ql)
        assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    finally:
        dsa.dsa_set_prefill_split(saved)


@pytest.mark.parametrize("name,qmax", [("janus-pro-7b", 32), ("mixed-serving", 16)])
def test_prefill_full_size_chunk(name, qmax):
    """The benchmark's launch at full size: every request's last qmax rows as
    its chunk, requests in the benchmark's order (decreasing scanned rows), the
    automatic split (the units of a last, partial wave of resident CTAs split and
    merged in the kernel): every slot vs the oracle."""
    import bench
    w = wl.generate(wl.WORKLOADS[name])
    mask = None
    if w["keep_mask"] is None:
        _, om = oracle.mass(w, r_local=2, r_diag=2)
        mask = wl.top_mass_keep_mask(om.reshape(w["batch"], w["hq"], -1), w["window"], w["hkv"],
                                     w["mask_words"], band=w["config"].band,
                                     frac=w["config"].top_mass_frac)
        w["keep_mask"] = mask
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, qmax, seed=31,
                         q_len=np.minimum(qmax, w["seq_len"]).astype(np.int32))
    order = torch.as_tensor(bench.prefill_order(w, qmax), dtype=torch.int32, device=bt.device)
    warps, units, whole, parts, per_sm, ctas = dsa.dsa_prefill_plan(bt.dims, qmax)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    slots = per_sm * sms
    assert units == w["batch"] * w["hkv"] * -(-qmax * (w["hq"] // w["hkv"]) // (16 * warps))
    assert ctas == whole + (units - whole) * parts
    # the units of a last partial wave run split into up to 4 parts (one wave of parts)
    rem = units % slots if units >= slots else units
    want = min(4, slots // rem) if rem else 1
    if want >= 2:
        assert (whole, parts) == (units - rem, want), (units, slots, whole, parts)
    else:
        assert (whole, parts) == (units, 1), (units, slots, whole, parts)
    dev = bt.device
    out = torch.full(tuple(q.shape), SENTINEL, dtype=torch.float32, device=dev)
    lse = torch.full(tuple(q.shape[:3]), SENTINEL, dtype=torch.float32, device=dev)
    dsa.dsa_prefill_sparse(bt.dims, q.to(dev), bt.k_pages, bt.v_pages, bt.page_table, bt.seq_len,
                           torch.as_tensor(ql).to(dev), bt.prompt_len, bt.window, bt.keep_mask,
                           bt.scale, out, lse, bt.ws, request_order=order)
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    compare(w, q, ql, out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))


def test_prefill_split_without_lse_and_in_a_graph():
    """Split units with lse = NULL (the merge writes out only), and the chunk
    captured in a CUDA graph and replayed: every replay gives the eager call's
    bits (the arrival counters return to zero inside each replay)."""
    w = wl.generate(small_cfg(128, 2, batch=4, Lmax=500, Pmax=80, W=120, seed=41))
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, 24, seed=42)
    dev = bt.device
    qd, qld = q.to(dev), torch.as_tensor(ql).to(dev)
    saved = dsa.dsa_get_prefill_split()
    try:
        dsa.dsa_set_prefill_split(3)
        ref, _ = run_prefill(bt, q, ql)
        out = torch.full(tuple(q.shape), SENTINEL, dtype=torch.float32, device=dev)
        dsa.dsa_prefill_sparse(bt.dims, qd, bt.k_pages, bt.v_pages, bt.page_table, bt.seq_len,
                               qld, bt.prompt_len, bt.window, bt.keep_mask, bt.scale, out, None,
                               bt.ws)
        torch.cuda.synchronize()
        assert bt.device_error() == 0
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)
        stream = torch.cuda.Stream(dev)
        gout = torch.full(tuple(q.shape), SENTINEL, dtype=torch.float32, device=dev)
        glse = torch.full(tuple(q.shape[:3]), SENTINEL, dtype=torch.float32, device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            dsa.dsa_prefill_sparse(bt.dims, qd, bt.k_pages, bt.v_pages, bt.page_table,
                                   bt.seq_len, qld, bt.prompt_len, bt.window, bt.keep_mask,
                                   bt.scale, gout, glse, bt.ws, stream)
        for _ in range(3):
            gout.fill_(SENTINEL)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(gout.cpu().numpy().astype(np.float64), ref)
        assert bt.device_error() == 0
    finally:
        dsa.dsa_set_prefill_split(saved)


def test_prefill_request_order():
    """A request order (a permutation) only changes which CTA runs which unit:
    results within the oracle's bars; an entry outside 0..batch-1 is flagged
    (DSA_DEV_BAD_ORDER) and the other requests are still computed."""
    w = wl.generate(small_cfg(64, 4, batch=6, Lmax=500, Pmax=90, W=96, seed=51))
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, 20, seed=52)
    dev = bt.device
    perm = np.random.default_rng(53).permutation(w["batch"]).astype(np.int32)

    def run(order):
        out = torch.full(tuple(q.shape), SENTINEL, dtype=torch.float32, device=dev)
        lse = torch.full(tuple(q.shape[:3]), SENTINEL, dtype=torch.float32, device=dev)
        dsa.dsa_prefill_sparse(bt.dims, q.to(dev), bt.k_pages, bt.v_pages, bt.page_table,
                               bt.seq_len, torch.as_tensor(ql).to(dev), bt.prompt_len, bt.window,
                               bt.keep_mask, bt.scale, out, lse, bt.ws,
                               request_order=torch.as_tensor(order).to(dev))
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)

    out, lse = run(perm)
    assert bt.device_error() == 0
    compare(w, q, ql, out, lse)
    bad = perm.copy()
    skipped = int(bad[2])
    bad[2] = w["batch"] + 3
    out2, lse2 = run(bad)
    assert bt.device_error() == 9               # DSA_DEV_BAD_ORDER
    dsa.dsa_clear_device_error(bt.ws)
    keep = [b for b in range(w["batch"]) if b != skipped]
    assert np.array_equal(out2[keep], out[keep])  # the same units in the same CTAs
    assert (out2[skipped] == SENTINEL).all()


@pytest.mark.parametrize("qmax,warps", [(16, 2), (30, 4), (70, 4)])
def test_prefill_each_warp_count(qmax, warps):
    """The 2- and 4-warp builds (chunks of up to 32 and of more (query, head)
    rows per kv head) against the oracle, the last over three query tiles."""
    w = wl.generate(small_cfg(128, 2, batch=5, Lmax=700, Pmax=120, W=150, seed=60 + qmax))
    bt = DecodeBatch.from_workload(w)
    assert dsa.dsa_prefill_plan(bt.dims, qmax)[0] == warps
    q, ql = chunk_inputs(w, qmax, seed=61)
    out, lse = run_prefill(bt, q, ql)
    compare(w, q, ql, out, lse)


def test_prefill_forced_split_clipped_by_the_workspace():
    """Every unit asked to split in 8 on the full Janus-like chunk: the
    workspace's partial rows hold only some of them, so the last units run
    split and the rest whole (the plan says which); every slot vs the oracle."""
    w = wl.generate(wl.WORKLOADS["janus-pro-7b"])
    bt = DecodeBatch.from_workload(w)
    q, ql = chunk_inputs(w, 32, seed=71, q_len=np.full(w["batch"], 32, np.int32))
    saved = dsa.dsa_get_prefill_split()
    try:
        dsa.dsa_set_prefill_split(8)
        warps, units, whole, parts, per_sm, ctas = dsa.dsa_prefill_plan(bt.dims, 32)
        assert parts == 8 and 0 < whole < units, (units, whole, parts)
        rows_cap = (dsa.dsa_workspace_size(bt.dims) - 256) // ((w["head_dim"] + 2) * 4)
        assert (units - whole) * parts * 16 * warps <= rows_cap
        out, lse = run_prefill(bt, q, ql)
        compare(w, q, ql, out, lse)
    finally:
        dsa.dsa_set_prefill_split(saved)
