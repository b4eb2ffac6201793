"""dsa_decode_sparse_noalloc: the sparse decode for callers that cannot allocate
device memory (a plugin whose host owns the whole memory pool, a real-time loop
that must not synchronise on cudaMalloc, a program that is only lent buffers).

It must give the results of dsa_decode_sparse -- same kernels, scratch in a
fixed array inside the library instead of a caller workspace -- call after call,
and refuse, before touching the GPU, batches whose scratch would not fit.
This file is collected last on purpose: a run that stops at the first failure
has run every other test before reaching it.
"""
import ctypes

import numpy as np
import pytest
import torch

from kv_cache_serving_gb300 import dsa
from kv_cache_serving_gb300 import workloads as wl

BF16_MAX, BF16_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-4


def test_noalloc_rejects_batches_beyond_its_scratch():
    # Host-side check only: the pointers are never dereferenced, because a
    # batch of 200000 x 32 heads needs far more than the fixed scratch.
    d = dsa.make_dims(200000, 32, 8, 128, 1000, 300, 192, 6, 705, "bf16", "bf16")
    need = 200000 * 32 * (128 + 2) * 4
    assert need > dsa.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    st = dsa._load().dsa_decode_sparse_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake,
                                                fake, fake, 0.1, fake, None, None, None)
    assert st == dsa.DSA_ERR_SCRATCH_LIMIT
    assert dsa.dsa_status_string(st) == "DSA_ERR_SCRATCH_LIMIT"


def _batch(name, batch):
    from kv_cache_serving_gb300.session import DecodeBatch
    w = wl.generate(wl.scaled(wl.WORKLOADS[name], batch=batch))
    mask = w["keep_mask"]
    if mask is None:   # mixed-serving masks: band plus a fixed pattern of offsets
        mask = np.zeros((w["batch"], w["hkv"], w["mask_words"]), np.uint32)
        for b in range(w["batch"]):
            offs = list(range(1, 9)) + list(range(9, int(w["window"][b]) + 1, 3))
            mask[b, :] = wl.offsets_to_bits(offs, int(w["window"][b]), w["mask_words"])
    w = dict(w, keep_mask=mask)
    bt = DecodeBatch.from_workload(w)
    bt.build_index()
    return w, bt


def _check_two_calls(w, bt):
    """Two no-alloc calls in a row give the bits of dsa_decode_sparse on the same
    plan, and both stay within the bf16 bars of the fp64 oracle."""
    import oracle
    ref_out, ref_lse = [t.clone() for t in bt.decode_sparse()]
    torch.cuda.synchronize()
    assert bt.device_error() == 0
    chunks = dsa.dsa_decode_plan(bt.dims, dsa.PLAN_SPARSE)[1]
    assert 256 + w["batch"] * w["hq"] * chunks * (w["head_dim"] + 2) * 4 <= \
        dsa.NOALLOC_SCRATCH_BYTES
    want, want_lse = oracle.decode(w, sparse=True)
    for call in range(2):   # the scratch keeps the previous call's contents
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        dsa.dsa_decode_sparse_noalloc(bt.dims, bt.q, bt.k_pages, bt.v_pages, bt.page_table,
                                      bt.seq_len, bt.kept_idx, bt.kept_cnt, bt.scale, out, lse,
                                      err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, call
        # same kernels, same plan, same summation order: the same bits
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), call
        diff = np.abs(out.cpu().numpy().reshape(want.shape).astype(np.float64) - want)
        assert np.isfinite(diff).all()
        assert diff.max() <= BF16_MAX and diff.mean() <= BF16_MEAN, call
        assert np.abs(lse.cpu().numpy().reshape(-1) - want_lse).max() <= LSE_MAX, call
    return chunks


@pytest.mark.gpu
@pytest.mark.parametrize("name,batch", [("janus-pro-7b", 12), ("mixed-serving", 16)])
def test_noalloc_matches_workspace_entry_point(name, batch):
    assert torch.cuda.is_available()
    w, bt = _batch(name, batch)
    _check_two_calls(w, bt)


@pytest.mark.gpu
def test_noalloc_split_rows_merge_through_the_fixed_scratch():
    """Clusters off and a batch small enough that each (request, kv head) is cut
    into several chunks: the chunk partials go through the fixed scratch array
    and are combined by the merge kernel, call after call."""
    assert torch.cuda.is_available()
    saved = dsa.dsa_get_sparse_cluster()
    try:
        dsa.dsa_set_sparse_cluster(1)
        w, bt = _batch("janus-pro-7b", 2)
        plan = dsa.dsa_decode_plan(bt.dims, dsa.PLAN_SPARSE)
        assert plan[1] > 1 and plan[2] == 2, plan   # several chunks, merge launch
        cnt = bt.kept_cnt.cpu().numpy()
        assert (cnt > plan[0]).all()                # every unit really is split
        _check_two_calls(w, bt)
    finally:
        dsa.dsa_set_sparse_cluster(saved)
