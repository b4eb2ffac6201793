"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each check is a value printed on
the page "Understanding and Exploiting Diagonal Attention Sparsity in
Autoregressive Image Generation" (paper-daily summary, worked example and core
formula), a closed form, a hand-derived fixture under tests/golden/, a library
routine (torch's scaled_dot_product_attention / softmax in float64), or an
invariant of masked softmax attention.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from kv_cache_serving_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def expand_ranges(tokens):
    rows = []
    for t in tokens:
        if "-" in t:
            a, b = t.split("-")
            rows += list(range(int(a), int(b) + 1))
        else:
            rows.append(int(t))
    return rows


# ---------------------------------------------------------------------------
# worked example N=8, W=4, B=2, query 6
# ---------------------------------------------------------------------------

def test_worked_example_literal_row_and_reads():
    g = read_kv("worked_example_n8_w4_b2.txt")
    N, W, B, i = (int(g[k][0]) for k in ("N", "W", "B", "query"))
    M = oracle.mask_matrix(N, W, B)
    assert list(np.nonzero(M[i])[0]) == [int(x) for x in g["literal_row"]]
    assert M.shape[1] == int(g["dense_reads"][0])
    assert int(M[i].sum()) == int(g["sparse_reads"][0])


def test_worked_example_decode_kept_set():
    g = read_kv("worked_example_n8_w4_b2.txt")
    W, B, i = int(g["W"][0]), int(g["B"][0]), int(g["query"][0])
    bits = wl.offsets_to_bits(range(1, B + 1), W, 1)
    kept = oracle.kept_set(L=i + 1, P=0, W=W, mask_words=bits)
    assert list(kept) == [int(x) for x in g["decode_kept"]]
    dense = oracle.kept_set(L=i + 1, P=i + 1, W=0, mask_words=np.zeros(1, np.uint32))
    assert len(dense) == int(g["decode_dense_reads"][0])


def test_worked_example_sparsity():
    g = read_kv("worked_example_n8_w4_b2.txt")
    N, W, B = int(g["N"][0]), int(g["W"][0]), int(g["B"][0])
    lit = oracle.mask_matrix(N, W, B)
    cau = oracle.mask_matrix(N, W, B, causal=True)
    assert int(lit.sum()) == int(g["literal_sum"][0])
    assert int(cau.sum()) == int(g["causal_sum"][0])
    assert oracle.sparsity(lit) == float(g["literal_sparsity"][0])
    assert oracle.sparsity(cau) == float(g["causal_sparsity"][0])


def test_worked_example_softmax_of_printed_scores():
    g = read_kv("worked_example_n8_w4_b2.txt")
    s = [float(x) for x in g["scores"]]
    n = len(s)
    # q = e0 and k_j = s_j e0 with scale 1 make the scores exactly s_j;
    # one-hot values v_j = e_j make the output equal to the weights.
    q = np.zeros(n)
    q[0] = 1.0
    k = np.zeros((n, n))
    k[:, 0] = s
    v = np.eye(n)
    out, lse = oracle.attend_rows(q, k, v, scale=1.0)
    want = np.array([float(x) for x in g["softmax_of_scores"]])
    assert np.max(np.abs(out - want)) < 1e-9
    assert abs(lse - float(g["logsumexp_of_scores"][0])) < 1e-9
    # The printed weights are garbled: the oracle must not reproduce them.
    printed = np.array([float(x) for x in g["printed_weights"]])
    assert np.max(np.abs(out - printed)) > 0.05


# ---------------------------------------------------------------------------
# the literal mask matrix and the sparsity formula
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [2, 3, 8, 17, 40])
def test_band_sum_closed_forms(N):
    for B in range(0, N):
        for W in range(B, N + 2):
            lit = oracle.mask_matrix(N, W, B)
            cau = oracle.mask_matrix(N, W, B, causal=True)
            assert int(lit.sum()) == N * (2 * B + 1) - B * (B + 1)
            assert int(cau.sum()) == N * (B + 1) - B * (B + 1) // 2
            assert oracle.sparsity(lit) == pytest.approx(
                1 - (N * (2 * B + 1) - B * (B + 1)) / N ** 2, abs=1e-15)


def test_window_narrower_than_band_cuts_lower_side_only():
    # With W < B the condition j >= i-W cuts the band below the diagonal only:
    # the matrix is then the union of the upper band of width B and the lower
    # band of width W.
    N = 12
    for B in range(1, 6):
        for W in range(0, B):
            M = oracle.mask_matrix(N, W, B)
            upper = oracle.mask_matrix(N, N, B) * np.triu(np.ones((N, N), np.uint8))
            lower = oracle.mask_matrix(N, N, W) * np.tril(np.ones((N, N), np.uint8))
            assert np.array_equal(M, np.maximum(upper, lower))


# ---------------------------------------------------------------------------
# kept sets
# ---------------------------------------------------------------------------

def test_kept_set_equals_causal_rows_of_literal_band():
    N = 30
    for B in range(0, 6):
        for W in range(B, 12):
            cau = oracle.mask_matrix(N, W, B, causal=True)
            bits = wl.offsets_to_bits(range(1, B + 1), W, wl.mask_words_for(W))
            for i in range(N):
                kept = oracle.kept_set(L=i + 1, P=0, W=W, mask_words=bits)
                assert list(kept) == list(np.nonzero(cau[i])[0])


def test_kept_set_tiny_fp32_golden():
    cfg = wl.WORKLOADS["tiny-fp32"]
    P, W, w = cfg.prompt[0], cfg.window, cfg.grid_w[0]
    offs = wl.band_row_offsets(cfg.band, w, cfg.row_ks, cfg.row_r)
    bits = wl.offsets_to_bits(offs, W, 1)
    assert wl.bits_to_offsets(bits) == [1, 2, 7, 8, 9, 15, 16]
    with open(os.path.join(GOLDEN, "tiny_fp32_kept_sets.txt")) as f:
        lines = [ln.split("#")[0].strip() for ln in f]
    checked = 0
    for ln in lines:
        if not ln:
            continue
        L, rows = ln.split(":")
        kept = oracle.kept_set(L=int(L), P=P, W=W, mask_words=bits)
        assert list(kept) == expand_ranges(rows.split()), ln
        checked += 1
    assert checked == 9


def test_kept_set_random_vs_set_union():
    rng = np.random.default_rng(7)
    for _ in range(400):
        L = int(rng.integers(1, 200))
        P = int(rng.integers(0, 80))
        W = int(rng.integers(0, 100))
        words = wl.mask_words_for(W)
        offs = [o for o in range(1, W + 1) if rng.random() < rng.uniform(0, 1)]
        bits = wl.offsets_to_bits(offs, W, words)
        i = L - 1
        want = set(range(min(P, L))) | {i} | {i - o for o in offs if i - o >= 0}
        kept = oracle.kept_set(L=L, P=P, W=W, mask_words=bits)
        assert list(kept) == sorted(want)


def test_kept_set_special_cases():
    z = np.zeros(4, np.uint32)
    ones = np.full(4, 0xFFFFFFFF, np.uint32)
    assert list(oracle.kept_set(10, 10, 0, z)) == list(range(10))        # L <= P
    assert list(oracle.kept_set(10, 25, 5, z)) == list(range(10))        # L < P
    assert list(oracle.kept_set(10, 3, 0, z)) == [0, 1, 2, 9]            # W = 0
    assert list(oracle.kept_set(50, 0, 100, ones)) == list(range(50))    # all ones, W >= i
    assert list(oracle.kept_set(1, 0, 0, z)) == [0]                      # first token
    assert list(oracle.kept_set(50, 0, 20, z)) == [49]                   # empty mask
    with pytest.raises(ValueError):
        oracle.kept_set(0, 0, 0, z)


# ---------------------------------------------------------------------------
# attention: library routine, closed forms, invariants
# ---------------------------------------------------------------------------

def logical_problem(seed, B=3, Hq=4, Hkv=2, D=16, dtype="f32", Lmax=90, Wmax=40,
                    shuffle=True):
    """Random logical K/V sequences, scattered into a shuffled page pool by the
    test itself (independently of the oracle's page walk)."""
    rng = np.random.default_rng(seed)
    L = rng.integers(1, Lmax + 1, size=B).astype(np.int32)
    P = rng.integers(0, 30, size=B).astype(np.int32)
    W = rng.integers(0, Wmax + 1, size=B).astype(np.int32)
    words = wl.mask_words_for(Wmax)
    table, num_pages = wl.make_page_table(L, shuffle, rng, spare_pages=2)
    g = torch.Generator().manual_seed(seed)
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    q = torch.randn(B, Hq, D, generator=g).to(dt)
    klog = [torch.randn(int(L[b]), Hkv, D, generator=g).to(dt) for b in range(B)]
    vlog = [torch.randn(int(L[b]), Hkv, D, generator=g).to(dt) for b in range(B)]
    kp = torch.randn(num_pages, 16, Hkv, D, generator=g).to(dt)
    vp = torch.randn(num_pages, 16, Hkv, D, generator=g).to(dt)
    for b in range(B):
        for j in range(int(L[b])):
            kp[table[b, j // 16], j % 16] = klog[b][j]
            vp[table[b, j // 16], j % 16] = vlog[b][j]
    mask = np.zeros((B, Hkv, words), np.uint32)
    offs = {}
    for b in range(B):
        for hk in range(Hkv):
            o = [x for x in range(1, int(W[b]) + 1) if rng.random() < 0.4]
            offs[b, hk] = o
            mask[b, hk] = wl.offsets_to_bits(o, int(W[b]), words)
    inp = dict(q=q, k_pages=kp, v_pages=vp, page_table=table, seq_len=L, prompt_len=P,
               window=W, keep_mask=mask, max_window=Wmax, grid_w=np.full(B, 5, np.int32))
    return inp, klog, vlog, offs


def sdpa_rows(q, k, v, allowed, scale):
    """torch SDPA in float64 for one query row with a boolean key mask."""
    qq = q.double().view(1, 1, 1, -1)
    kk = k.double().view(1, 1, k.shape[0], -1)
    vv = v.double().view(1, 1, v.shape[0], -1)
    am = torch.as_tensor(allowed, dtype=torch.bool).view(1, 1, 1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=am, scale=scale)
    s = (kk[0, 0] @ qq[0, 0, 0]) * scale
    lse = torch.logsumexp(s[am.view(-1)], dim=0)
    return o.view(-1).numpy(), float(lse)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_matches_torch_sdpa(dtype, seed):
    inp, klog, vlog, offs = logical_problem(seed, dtype=dtype)
    B, Hq, D = inp["q"].shape
    Hkv = inp["k_pages"].shape[2]
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    out_s, lse_s = oracle.decode(inp, sparse=True, nthreads=3)
    out_d, lse_d = oracle.decode(inp, sparse=False, nthreads=2)
    for b in range(B):
        L, P = int(inp["seq_len"][b]), int(inp["prompt_len"][b])
        i = L - 1
        for h in range(Hq):
            hk = h // g
            k, v = klog[b][:, hk], vlog[b][:, hk]
            keep = set(range(min(P, L))) | {i} | {i - o for o in offs[b, hk] if i - o >= 0}
            allowed = [j in keep for j in range(L)]
            o_ref, l_ref = sdpa_rows(inp["q"][b, h], k, v, allowed, scale)
            t = b * Hq + h
            assert np.max(np.abs(out_s[t] - o_ref)) < 1e-12
            assert abs(lse_s[t] - l_ref) < 1e-12
            o_ref, l_ref = sdpa_rows(inp["q"][b, h], k, v, [True] * L, scale)
            assert np.max(np.abs(out_d[t] - o_ref)) < 1e-12
            assert abs(lse_d[t] - l_ref) < 1e-12


def test_decode_selected_pairs_match_full_run():
    inp, *_ = logical_problem(5)
    Hq = inp["q"].shape[1]
    out, lse = oracle.decode(inp, sparse=True)
    bh = [(2, 3), (0, 0), (1, 2)]
    o2, l2 = oracle.decode(inp, sparse=True, bh=bh)
    for n, (b, h) in enumerate(bh):
        assert np.array_equal(o2[n], out[b * Hq + h]) and l2[n] == lse[b * Hq + h]


def test_sparse_equals_dense_when_everything_is_kept():
    inp, *_ = logical_problem(11, Wmax=100)
    B = inp["q"].shape[0]
    full = dict(inp)
    full["window"] = np.full(B, 100, np.int32)
    full["keep_mask"] = np.full_like(inp["keep_mask"], 0xFFFFFFFF)
    a, la = oracle.decode(full, sparse=True)
    d, ld = oracle.decode(full, sparse=False)
    assert np.array_equal(a, d) and np.array_equal(la, ld)
    allprompt = dict(inp)
    allprompt["prompt_len"] = inp["seq_len"].copy()
    a, la = oracle.decode(allprompt, sparse=True)
    assert np.array_equal(a, d) and np.array_equal(la, ld)


def test_skipped_rows_have_no_effect():
    inp, klog, vlog, offs = logical_problem(3, dtype="bf16")
    g = inp["q"].shape[1] // inp["k_pages"].shape[2]
    base, lbase = oracle.decode(inp, sparse=True)

    def kept(b, hk):
        return oracle.kept_set(int(inp["seq_len"][b]), int(inp["prompt_len"][b]),
                               int(inp["window"][b]), inp["keep_mask"][b, hk])

    for value in (float("nan"), 1e30, -3.0):
        p = wl.poison_unread(inp, kept, value)
        out, lse = oracle.decode(p, sparse=True)
        assert np.array_equal(out, base) and np.array_equal(lse, lbase)
    assert g == 2


def test_closed_forms_equal_and_one_hot_scores():
    D = 8
    rng = np.random.default_rng(0)
    v = rng.standard_normal((7, D))
    q = rng.standard_normal(D)
    out, lse = oracle.attend_rows(q, np.zeros((7, D)), v, scale=0.3)
    assert np.max(np.abs(out - v.mean(axis=0))) < 1e-15          # equal scores
    assert abs(lse - math.log(7)) < 1e-15
    k = np.zeros((7, D))
    k[4] = 1e4 * q / np.dot(q, q)                                  # one huge score
    out, _ = oracle.attend_rows(q, k, v, scale=1.0)
    assert np.array_equal(out, v[4])
    out, _ = oracle.attend_rows(q, rng.standard_normal((7, D)), np.ones((7, D)), scale=0.5)
    assert np.max(np.abs(out - 1.0)) < 1e-15                       # weights sum to 1


# ---------------------------------------------------------------------------
# several query tokens per request (chunked prefill under the same mask)
# ---------------------------------------------------------------------------

def test_multi_worked_example_all_queries_at_once():
    """The worked example's eight queries as one chunk (P = 0, band B = 2, W = 4):
    with equal scores and one-hot values the output of query t is its attention
    weights, 1/count on the hand-derived band rows max(0, t-2) .. t."""
    g = read_kv("worked_example_n8_w4_b2.txt")
    N, W, B = int(g["N"][0]), int(g["W"][0]), int(g["B"][0])
    counts = [int(x) for x in g["prefill_kept_counts"]]
    assert sum(counts) == int(g["causal_sum"][0])
    D = N
    k = torch.zeros(1, 16, 1, D)
    v = torch.zeros(1, 16, 1, D)
    v[0, :N, 0, :] = torch.eye(N)                       # v_j = e_j
    inp = dict(q=torch.randn(1, N, 1, D, generator=torch.Generator().manual_seed(8)),
               k_pages=k, v_pages=v, page_table=np.array([[0]], np.int32),
               seq_len=np.array([N], np.int32), prompt_len=np.array([0], np.int32),
               window=np.array([W], np.int32),
               keep_mask=wl.offsets_to_bits(range(1, B + 1), W, 1).reshape(1, 1, 1),
               max_window=W)
    out, lse = oracle.multi(inp, q_len=[N])
    for t in range(N):
        want = np.zeros(D)
        want[max(0, t - B):t + 1] = 1.0 / counts[t]
        assert np.max(np.abs(out[0, t, 0] - want)) < 1e-15, t
        assert abs(lse[0, t, 0] - math.log(counts[t])) < 1e-15


def multi_problem(seed, dtype="f32", B=3, Hq=4, Hkv=2, D=16, Qmax=7):
    inp, klog, vlog, offs = logical_problem(seed, B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype)
    rng = np.random.default_rng(seed + 1)
    L = inp["seq_len"]
    ql = np.array([int(rng.integers(0, min(Qmax, int(L[b])) + 1)) for b in range(B)], np.int32)
    ql[0] = min(Qmax, int(L[0]))                         # at least one full chunk
    g = torch.Generator().manual_seed(seed + 2)
    dt = inp["q"].dtype
    inp["q"] = torch.randn(B, Qmax, Hq, D, generator=g).to(dt)
    return inp, klog, vlog, offs, ql


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_multi_vs_torch_sdpa_boolean_mask(dtype):
    """Every query token of every request against torch float64 SDPA over the
    test's own logical sequence, with a boolean [q_len, L] mask built from the
    drawn offsets (not from the bit encoding)."""
    for seed in (31, 32, 33):
        inp, klog, vlog, offs, ql = multi_problem(seed, dtype)
        B, Q, Hq, D = inp["q"].shape
        g = Hq // inp["k_pages"].shape[2]
        out, lse = oracle.multi(inp, q_len=ql)
        scale = 1.0 / math.sqrt(D)
        for b in range(B):
            L, P, W = (int(inp[k][b]) for k in ("seq_len", "prompt_len", "window"))
            n = int(ql[b])
            assert np.isnan(out[b, n:]).all() and np.isnan(lse[b, n:]).all()
            for t in range(n):
                i = L - n + t
                for h in range(Hq):
                    keep = set(offs[b, h // g])
                    allowed = [j <= i and (j < P or i == j or (i - j <= W and (i - j) in keep))
                               for j in range(L)]
                    o, l = sdpa_rows(inp["q"][b, t, h], klog[b][:, h // g], vlog[b][:, h // g],
                                     allowed, scale)
                    assert np.max(np.abs(out[b, t, h] - o)) < 1e-12
                    assert abs(lse[b, t, h] - l) < 1e-12


def test_multi_all_kept_is_causal_attention():
    """An all-ones mask with W >= L keeps every earlier row: the chunk's queries
    then see the bottom-right-aligned causal mask over the whole sequence."""
    inp, klog, vlog, offs, ql = multi_problem(34, "f32")
    B, Q, Hq, D = inp["q"].shape
    g = Hq // inp["k_pages"].shape[2]
    inp["window"] = np.full(B, inp["max_window"], np.int32)
    inp["prompt_len"] = np.zeros(B, np.int32)
    inp["keep_mask"] = np.full_like(inp["keep_mask"], 0xFFFFFFFF)
    inp["seq_len"] = np.minimum(inp["seq_len"], inp["max_window"]).astype(np.int32)
    ql = np.minimum(ql, inp["seq_len"]).astype(np.int32)
    out, lse = oracle.multi(inp, q_len=ql)
    for b in range(B):
        L, n = int(inp["seq_len"][b]), int(ql[b])
        if n == 0:
            assert np.isnan(out[b]).all()
            continue
        causal = torch.ones(n, L, dtype=torch.bool).tril(diagonal=L - n)
        for h in range(Hq):
            qq = inp["q"][b, :n, h].double().view(1, 1, n, D)
            kk = klog[b][:L, h // g].double().view(1, 1, L, D)
            vv = vlog[b][:L, h // g].double().view(1, 1, L, D)
            o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=causal)
            assert np.max(np.abs(out[b, :n, h] - o[0, 0].numpy())) < 1e-12


def test_multi_skipped_rows_have_no_effect():
    """Rows no query of the chunk keeps may hold anything (NaN, huge, negative)."""
    inp, klog, vlog, offs, ql = multi_problem(35, "bf16")
    base, lbase = oracle.multi(inp, q_len=ql)
    g = inp["q"].shape[2] // inp["k_pages"].shape[2]

    def kept(b, hk):
        L, P, W = (int(inp[k][b]) for k in ("seq_len", "prompt_len", "window"))
        rows = set()
        for t in range(int(ql[b])):
            rows.update(oracle.kept_set(L - int(ql[b]) + t + 1, P, W,
                                        inp["keep_mask"][b, hk]).tolist())
        return sorted(rows)

    for value in (float("nan"), 1e30, -3.0):
        p = wl.poison_unread(inp, kept, value)
        out, lse = oracle.multi(p, q_len=ql)
        assert np.array_equal(out, base, equal_nan=True)
        assert np.array_equal(lse, lbase, equal_nan=True)
    assert g == 2


# ---------------------------------------------------------------------------
# attention mass
# ---------------------------------------------------------------------------

def test_mass_equal_scores_hand_counts():
    # L=20, P=5, W=10, w=4, r_local=1, r_diag=0 with all-zero keys: every weight
    # is 1/20.  Rows: prompt j<5 -> 5; local o in {0,1} -> 2; diagonal o in
    # {4, 8} (multiples of w inside W) -> 2; other -> 11.
    D = 4
    inp = dict(q=torch.randn(1, 1, D), k_pages=torch.zeros(2, 16, 1, D),
               v_pages=torch.zeros(2, 16, 1, D), page_table=np.array([[1, 0]], np.int32),
               seq_len=np.array([20], np.int32), prompt_len=np.array([5], np.int32),
               window=np.array([10], np.int32), grid_w=np.array([4], np.int32),
               keep_mask=np.zeros((1, 1, 1), np.uint32), max_window=12)
    m4, om = oracle.mass(inp, r_local=1, r_diag=0)
    assert np.max(np.abs(m4[0] - np.array([5, 2, 2, 11]) / 20)) < 1e-15
    want = np.zeros(13)
    want[:11] = 1 / 20
    assert np.max(np.abs(om[0] - want)) < 1e-15


def read_mass_cases():
    cases = []
    with open(os.path.join(GOLDEN, "mass_diagonal_bins.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            head, rest = line.split(":")
            counts, diag = rest.split("|")
            name, *nums = head.split()
            cases.append((name, *(int(x) for x in nums), [int(x) for x in counts.split()],
                          expand_ranges(diag.split())))
    return cases


@pytest.mark.parametrize("case", read_mass_cases(), ids=lambda c: c[0])
def test_mass_diagonal_bin_hand_counts(case):
    """Equal scores (all keys zero) with r_diag >= 1: every bin is its hand-counted
    number of rows / L, including bands k*w +- r that cross the window edge, the
    local band or the prompt (fixture mass_diagonal_bins.txt)."""
    name, L, P, W, w, r_local, r_diag, counts, diag = case
    assert sum(counts) == L and len(diag) == counts[2]
    D = 4
    pages = (L + 15) // 16
    gen = torch.Generator().manual_seed(L)
    inp = dict(q=torch.randn(1, 1, D, generator=gen),
               k_pages=torch.zeros(pages + 1, 16, 1, D), v_pages=torch.zeros(pages + 1, 16, 1, D),
               page_table=np.array([list(range(pages, 0, -1))], np.int32),
               seq_len=np.array([L], np.int32), prompt_len=np.array([P], np.int32),
               window=np.array([W], np.int32), grid_w=np.array([w], np.int32),
               keep_mask=np.zeros((1, 1, 1), np.uint32), max_window=W + 3)
    m4, om = oracle.mass(inp, r_local=r_local, r_diag=r_diag)
    assert np.max(np.abs(m4[0] - np.array(counts) / L)) < 1e-15
    want = np.zeros(W + 4)
    want[:min(W, L - 1) + 1] = 1 / L
    assert np.max(np.abs(om[0] - want)) < 1e-15


def test_mass_diagonal_and_other_bins_vs_torch_softmax():
    """Random scores: the diagonal bin is the torch softmax weight summed over the
    offsets {k*w + r : k >= 1, |r| <= r_diag} (enumerated as a set) that lie in
    (r_local, W] and below the prompt boundary; other is the remainder."""
    inp, klog, vlog, offs = logical_problem(23, B=4, Hq=2, Hkv=1, D=16)
    B, Hq, D = inp["q"].shape
    inp["grid_w"] = np.array([3, 5, 7, 4], np.int32)
    for r_local, r_diag in ((0, 1), (2, 2), (1, 3)):
        m4, _ = oracle.mass(inp, r_local=r_local, r_diag=r_diag, with_offsets=False)
        for b in range(B):
            L, P, W, w = (int(inp[k][b]) for k in ("seq_len", "prompt_len", "window", "grid_w"))
            i = L - 1
            near = {k * w + r for k in range(1, W // w + 2) for r in range(-r_diag, r_diag + 1)}
            diag_o = [o for o in near if r_local < o <= W and 0 <= i - o and i - o >= P]
            for h in range(Hq):
                s = (klog[b][:, 0].double() @ inp["q"][b, h].double()) / math.sqrt(D)
                a = torch.softmax(s, dim=0).numpy()
                t = b * Hq + h
                want_diag = sum(a[i - o] for o in diag_o)
                assert abs(m4[t, 2] - want_diag) < 1e-12, (b, h, r_local, r_diag)
                assert abs(m4[t, 3] - (1.0 - m4[t, :3].sum())) < 1e-12


def test_mass_vs_torch_softmax():
    inp, klog, vlog, offs = logical_problem(21, B=3, Hq=4, Hkv=2, D=16)
    B, Hq, D = inp["q"].shape
    g = Hq // inp["k_pages"].shape[2]
    m4, om = oracle.mass(inp, r_local=2, r_diag=1)
    for b in range(B):
        L, P, W = (int(inp[k][b]) for k in ("seq_len", "prompt_len", "window"))
        i = L - 1
        for h in range(Hq):
            s = (klog[b][:, h // g].double() @ inp["q"][b, h].double()) / math.sqrt(D)
            a = torch.softmax(s, dim=0).numpy()
            t = b * Hq + h
            assert abs(m4[t].sum() - 1.0) < 1e-12
            assert abs(m4[t, 0] - a[:min(P, L)].sum()) < 1e-12
            local = a[max(P, i - 2):i + 1].sum()
            assert abs(m4[t, 1] - local) < 1e-12
            for o in range(inp["max_window"] + 1):
                want = a[i - o] if (o <= W and o <= i) else 0.0
                assert abs(om[t, o] - want) < 1e-12


# ---------------------------------------------------------------------------
# evictable pages: rows no later decode step can read
# ---------------------------------------------------------------------------

def test_evictable_pages_against_future_kept_sets():
    """A page is evictable exactly when no kept set of the current or any later
    query (i' = L-1, L, ..., with every window bit set: the largest kept set)
    contains one of its rows -- checked by brute force over later queries."""
    rng = np.random.default_rng(41)
    for _ in range(150):
        L = int(rng.integers(1, 700))
        P = int(rng.integers(0, 300))
        W = int(rng.integers(0, 200))
        ones = np.full((W + 31) // 32 + 1, 0xFFFFFFFF, dtype=np.uint32)
        read_again = set()
        for Lf in range(L, L + W + 40):
            read_again.update(oracle.kept_set(Lf, P, W, ones).tolist())
        want = np.array([not any(j in read_again for j in range(16 * p, 16 * p + 16))
                         for p in range((L + 15) // 16)], dtype=bool)
        assert np.array_equal(oracle.evictable_pages(L, P, W), want), (L, P, W)


@pytest.mark.parametrize("L,P,W", [(100, 20, 30), (8100, 64, 360), (16, 0, 0), (500, 600, 10),
                                   (1, 0, 5), (257, 0, 0)])
def test_evictable_page_count_closed_form(L, P, W):
    """Pages strictly after the prompt's last page and ending before row L-1-W:
    max(0, floor((L-1-W)/16) - ceil(P/16))."""
    want = max(0, (L - 1 - W) // 16 - (P + 15) // 16)
    assert int(oracle.evictable_pages(L, P, W).sum()) == want
