"""Host-side logic: the seeded workload generators and the top-mass selection rule."""
import numpy as np
import pytest

from kv_cache_serving_gb300 import workloads as wl


def test_offset_bits_roundtrip():
    bits = wl.offsets_to_bits([1, 2, 32, 33, 64, 65, 90], 70, 3)
    assert wl.bits_to_offsets(bits) == [1, 2, 32, 33, 64, 65]   # 90 > W dropped
    assert bits[0] == (1 | 2 | (1 << 31))


def test_config_masks_match_their_descriptions():
    # LlamaGen-XL-like: band 4 plus {24, 48} +- 1 inside W = 48 (49 dropped)
    w2 = wl.generate(wl.scaled(wl.WORKLOADS["llamagen-xl"], batch=3), with_kv=False)
    assert wl.bits_to_offsets(w2["keep_mask"][0, 0]) == [1, 2, 3, 4, 23, 24, 25, 47, 48]
    # Emu3-like: band 16 plus 91k +- 2, k = 1..3, all inside W = 360
    w4 = wl.generate(wl.scaled(wl.WORKLOADS["emu3-8b"], batch=2), with_kv=False)
    offs = wl.bits_to_offsets(w4["keep_mask"][1, 3])
    assert offs == list(range(1, 17)) + [89, 90, 91, 92, 93, 180, 181, 182, 183, 184,
                                         271, 272, 273, 274, 275]
    # Janus-like: band 8 always kept, 25-50% of the other offsets on average
    w3 = wl.generate(wl.scaled(wl.WORKLOADS["janus-pro-7b"], batch=8), with_kv=False)
    fr = []
    for b in range(8):
        for hk in range(32):
            o = wl.bits_to_offsets(w3["keep_mask"][b, hk])
            assert o[:8] == list(range(1, 9)) and max(o) <= 96
            fr.append((len(o) - 8) / 88)
    assert 0.25 < np.mean(fr) < 0.5


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_generated_shapes_and_page_tables(name):
    cfg = wl.WORKLOADS[name]
    w = wl.generate(wl.scaled(cfg, batch=min(cfg.batch, 6)), with_kv=False)
    L, P, W, t = w["seq_len"], w["prompt_len"], w["window"], w["page_table"]
    assert (L >= 1).all() and (P >= 0).all() and (W <= w["max_window"]).all()
    used = []
    for b in range(len(L)):
        n = (int(L[b]) + 15) // 16
        assert (t[b, :n] >= 0).all() and (t[b, n:] == -1).all()
        used += list(t[b, :n])
    assert sorted(used) == list(range(w["num_pages"]))      # each page used once
    assert w["max_kept"] >= max(min(int(L[b]), int(P[b]) + int(W[b]) + 1) for b in range(len(L)))
    if name == "emu3-8b":
        assert (L >= 8000).all() and (L <= 8250).all()
    if name == "mixed-serving":
        assert set(np.unique(w["grid_w"])) <= {24, 32, 64} and (W == 3 * w["grid_w"]).all()


def test_generation_is_seeded():
    a = wl.generate(wl.scaled(wl.WORKLOADS["llamagen-xl"], batch=2))
    b = wl.generate(wl.scaled(wl.WORKLOADS["llamagen-xl"], batch=2))
    assert np.array_equal(a["page_table"], b["page_table"])
    assert (a["k_pages"].float() == b["k_pages"].float()).all()


def test_top_mass_rule_hand_example():
    # one request, W = 16, frac 0.375 -> ceil(6) = 6 offsets; band 1..2 forced;
    # then the 4 largest of offsets 3..16, ties to the smaller offset.
    om = np.zeros((1, 2, 17))
    om[0, 0, [5, 9, 12, 13, 14]] = [0.3, 0.2, 0.2, 0.1, 0.2]
    om[0, 1, [5, 9, 12, 13, 14]] = [0.3, 0.2, 0.2, 0.3, 0.2]
    # group mean: 5 -> .3, 9 -> .2, 12 -> .2, 13 -> .2, 14 -> .2  => 5, then 9, 12, 13
    m = wl.top_mass_keep_mask(om, np.array([16]), hkv=1, words=1, band=2, frac=0.375)
    assert wl.bits_to_offsets(m[0, 0]) == [1, 2, 5, 9, 12, 13]


def test_prefill_request_order_by_scanned_rows():
    """The benchmark's multi-query order: a permutation of the batch by
    decreasing rows a chunk scans -- the prompt rows min(P, L), then the window
    range of its queries min(W + q_len, L - min(P, L)) -- ties by index."""
    import bench
    w = {"seq_len": np.array([10, 300, 300, 50, 5000, 40]),
         "prompt_len": np.array([20, 100, 100, 0, 10, 40]),
         "window": np.array([8, 64, 64, 16, 96, 8])}
    # scanned rows with q_len 16: 10, 100+80, 100+80, 0+32, 10+112, 40+0
    assert bench.prefill_order(w, 16).tolist() == [1, 2, 4, 5, 3, 0]
    big = wl.generate(wl.scaled(wl.WORKLOADS["mixed-serving"], batch=40), with_kv=False)
    order = bench.prefill_order(big, 16)
    assert sorted(order.tolist()) == list(range(40))
    L, P, W = big["seq_len"], big["prompt_len"], big["window"]
    nA = np.minimum(P, L)
    rows = (nA + np.minimum(W + np.minimum(16, L), L - nA))[order]
    assert (np.diff(rows) <= 0).all()
