"""Seeded synthetic inputs for diagonal-aware sparse decode attention.

This module is shared by the CUDA path and by the CPU oracle, so it holds no
attention arithmetic: it draws random tensors, lays them out in a paged KV
pool, and encodes keep masks as bits.  The workloads stand in for the model
runs behind "Understanding and Exploiting Diagonal Attention Sparsity in
Autoregressive Image Generation" (LlamaGen, Janus-Pro and Emu3 shapes; the
weights, prompts and image datasets are not available), see ``WORKLOADS``.

Layouts (all row-major, all sizes in elements):
  q           [B, Hq, D]                    f32 or bf16
  k_pages     [num_pages, 16, Hkv, D]       f32 or bf16  (v_pages alike)
  page_table  [B, max_pages]  int32; entries past ceil(L_b/16) are -1
  seq_len, prompt_len, window, grid_w  [B] int32
  keep_mask   [B, Hkv, mask_words] uint32; bit (o-1) keeps window offset o
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

PAGE = 16


@dataclass(frozen=True)
class Config:
    """One synthetic workload.  Ranges are inclusive."""

    name: str
    batch: int
    hq: int
    hkv: int
    head_dim: int
    dtype: str                      # "f32" or "bf16" (q, K and V)
    prompt: tuple                   # (lo, hi) prompt length
    grid_w: tuple                   # choices of image grid width w
    window_rows: int | None         # W = window_rows * w when set ...
    window: int | None              # ... else this fixed W
    seq: tuple                      # ("abs", lo, hi) or ("after_prompt", lo, hi)
    mask: str                       # "offsets" | "random" | "top_mass"
    band: int = 0                   # band offsets 1..band always kept
    row_ks: tuple = ()              # row-aligned offsets k*w + r, |r| <= row_r
    row_r: int = 0
    random_frac: tuple = (0.25, 0.5)
    top_mass_frac: float = 0.375
    shuffle_pages: bool = True
    seed: int = 0
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    # Tiny fp32 check: 16 prompt tokens, an 8x8 image decoded step by step.
    "tiny-fp32": Config("tiny-fp32-8x8", 1, 2, 2, 64, "f32", (16, 16), (8,), None, 16,
              ("abs", 17, 80), "offsets", band=2, row_ks=(1, 2), row_r=1, seed=1),
    # LlamaGen-XL-like: 24x24 grid, W = 2 rows.
    "llamagen-xl": Config("llamagen-xl-like-24x24", 32, 20, 20, 64, "bf16", (120, 120), (24,), 2, None,
              ("after_prompt", 1, 576), "offsets", band=4, row_ks=(1, 2), row_r=1, seed=2),
    # Janus-Pro-7B-like: 32x32 grid, W = 3 rows, per-head random masks.
    "janus-pro-7b": Config("janus-pro-7b-like-32x32", 64, 32, 32, 128, "bf16", (256, 256), (32,), 3, None,
              ("after_prompt", 64, 1024), "random", band=8, seed=3),
    # Emu3-8B-like GQA: 90x90 grid plus one row-end token per row (w = 91), W = 360.
    "emu3-8b": Config("emu3-8b-like-90x90-gqa4", 8, 32, 8, 128, "bf16", (64, 64), (91,), None, 360,
              ("abs", 8000, 8250), "offsets", band=16, row_ks=(1, 2, 3), row_r=2, seed=4),
    # Mixed serving batch, GQA, shuffled pages, masks from the top-mass rule.
    "mixed-serving": Config("mixed-serving-gqa4", 128, 32, 8, 128, "bf16", (32, 512), (24, 32, 64), 3, None,
              ("after_prompt", 1, 4096), "top_mass", band=8, seed=5),
}


def scaled(cfg: Config, **over) -> Config:
    """A copy of cfg with some fields replaced (smaller batches for tests)."""
    return replace(cfg, **over)


# ---------------------------------------------------------------------------
# keep-mask encodings
# ---------------------------------------------------------------------------

def mask_words_for(max_window: int) -> int:
    return max(1, (max_window + 31) // 32)


def offsets_to_bits(offsets, window: int, words: int) -> np.ndarray:
    """uint32[words] with bit (o-1) set for each offset 1 <= o <= window."""
    bits = np.zeros(words, dtype=np.uint32)
    for o in offsets:
        o = int(o)
        if 1 <= o <= window:
            bits[(o - 1) >> 5] |= np.uint32(1 << ((o - 1) & 31))
    return bits


def bits_to_offsets(bits) -> list:
    out = []
    for wi, word in enumerate(np.asarray(bits, dtype=np.uint32)):
        for t in range(32):
            if (int(word) >> t) & 1:
                out.append(wi * 32 + t + 1)
    return out


def band_row_offsets(band: int, w: int, row_ks, row_r: int) -> list:
    """Offsets 1..band plus k*w + r for k in row_ks, |r| <= row_r (unfiltered)."""
    offs = set(range(1, band + 1))
    for k in row_ks:
        for r in range(-row_r, row_r + 1):
            if k * w + r >= 1:
                offs.add(k * w + r)
    return sorted(offs)


def top_mass_keep_mask(offset_mass: np.ndarray, window: np.ndarray, hkv: int, words: int,
                       band: int = 8, frac: float = 0.375) -> np.ndarray:
    """Selection rule for masks derived from measured attention mass.

    offset_mass is [B, Hq, max_window+1] (mass at window offset o, o = 0..).
    For each (b, kv head): the band offsets 1..band are kept, then the offsets
    band+1..W_b with the largest mass, averaged over the query heads of the
    group, until ceil(frac * W_b) offsets are kept.  Ties go to the smaller
    offset.  Returns uint32 [B, hkv, words].
    """
    om = np.asarray(offset_mass, dtype=np.float64)
    B, Hq, _ = om.shape
    g = Hq // hkv
    out = np.zeros((B, hkv, words), dtype=np.uint32)
    for b in range(B):
        W = int(window[b])
        n_total = int(math.ceil(frac * W))
        for hk in range(hkv):
            score = om[b, hk * g:(hk + 1) * g, :].mean(axis=0)
            keep = [o for o in range(1, min(band, W) + 1)]
            rest = list(range(band + 1, W + 1))
            rest.sort(key=lambda o: (-score[o], o))
            keep += rest[:max(0, n_total - len(keep))]
            out[b, hk] = offsets_to_bits(keep, W, words)
    return out


# ---------------------------------------------------------------------------
# the generator
# ---------------------------------------------------------------------------

def _torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def draw_requests(cfg: Config, rng: np.random.Generator):
    """Per-request prompt length, grid width, window and sequence length."""
    B = cfg.batch
    P = rng.integers(cfg.prompt[0], cfg.prompt[1] + 1, size=B).astype(np.int32)
    w = rng.choice(np.asarray(cfg.grid_w, dtype=np.int32), size=B).astype(np.int32)
    if cfg.window_rows is not None:
        W = (cfg.window_rows * w).astype(np.int32)
    else:
        W = np.full(B, cfg.window, dtype=np.int32)
    kind, lo, hi = cfg.seq
    if kind == "abs":
        L = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    else:
        L = (P + rng.integers(lo, hi + 1, size=B)).astype(np.int32)
    return P, w, W, L


def make_page_table(seq_len: np.ndarray, shuffle: bool, rng: np.random.Generator,
                    spare_pages: int = 0, max_pages: int | None = None):
    """Pages for each request (ceil(L/16) of them), drawn from a pool of
    sum(ceil(L/16)) + spare_pages pages, in shuffled order when asked."""
    need = [(int(L) + PAGE - 1) // PAGE for L in seq_len]
    mp = max(need) if max_pages is None else max_pages
    assert mp >= max(need)
    num_pages = sum(need) + spare_pages
    ids = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    table = np.full((len(seq_len), mp), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = ids[at:at + n]
        at += n
    return table, num_pages


def generate(cfg: Config, seed: int | None = None, device: str = "cpu",
             spare_pages: int = 0, with_kv: bool = True) -> dict:
    """Draw one batch.  q/k/v ~ N(0,1) from torch.Generator(seed); the integer
    structure (lengths, page order, masks) from numpy's default_rng(seed).

    Returns a dict with the tensors listed in the module docstring plus the
    sizes the C ABI needs (max_window, mask_words, max_kept, max_pages...).
    keep_mask is None for the "top_mass" workload: it is derived from measured
    attention mass by top_mass_keep_mask().
    """
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    P, w, W, L = draw_requests(cfg, rng)
    table, num_pages = make_page_table(L, cfg.shuffle_pages, rng, spare_pages)
    max_window = int(W.max())
    words = mask_words_for(max_window)
    B, Hq, Hkv, D = cfg.batch, cfg.hq, cfg.hkv, cfg.head_dim

    if cfg.mask == "offsets":
        mask = np.zeros((B, Hkv, words), dtype=np.uint32)
        for b in range(B):
            offs = band_row_offsets(cfg.band, int(w[b]), cfg.row_ks, cfg.row_r)
            mask[b, :] = offsets_to_bits(offs, int(W[b]), words)
    elif cfg.mask == "random":
        mask = np.zeros((B, Hkv, words), dtype=np.uint32)
        for b in range(B):
            for hk in range(Hkv):
                p = rng.uniform(cfg.random_frac[0], cfg.random_frac[1])
                extra = [o for o in range(cfg.band + 1, int(W[b]) + 1) if rng.random() < p]
                mask[b, hk] = offsets_to_bits(list(range(1, cfg.band + 1)) + extra,
                                              int(W[b]), words)
    else:
        mask = None

    out = dict(
        config=cfg, seed=seed, batch=B, hq=Hq, hkv=Hkv, head_dim=D, dtype=cfg.dtype,
        seq_len=L, prompt_len=P, window=W, grid_w=w, page_table=table,
        num_pages=num_pages, max_pages=table.shape[1], max_window=max_window,
        mask_words=words, keep_mask=mask,
        max_kept=int(max(min(int(L[b]), int(P[b]) + int(W[b]) + 1) for b in range(B))),
    )
    if with_kv:
        dt = _torch_dtype(cfg.dtype)
        gen = torch.Generator(device=device).manual_seed(seed)
        out["q"] = torch.randn((B, Hq, D), generator=gen, device=device,
                               dtype=torch.float32).to(dt)
        shape = (num_pages, PAGE, Hkv, D)
        out["k_pages"] = torch.randn(shape, generator=gen, device=device,
                                     dtype=torch.float32).to(dt)
        out["v_pages"] = torch.randn(shape, generator=gen, device=device,
                                     dtype=torch.float32).to(dt)
    return out


def poison_unread(inp: dict, kept_rows_of, value: float = float("nan")) -> dict:
    """A copy of inp whose K/V rows outside `kept_rows_of(b, hk)` (and every
    slot no request uses) are set to `value`.  kept_rows_of returns the logical
    rows that must stay; it is supplied by the caller."""
    k = inp["k_pages"].clone()
    v = inp["v_pages"].clone()
    keep = torch.zeros(k.shape[:3], dtype=torch.bool)
    table = inp["page_table"]
    B, _, Hkv = inp["q"].shape[0], None, k.shape[2]
    for b in range(B):
        for hk in range(Hkv):
            for j in kept_rows_of(b, hk):
                keep[int(table[b, j // PAGE]), j % PAGE, hk] = True
    k[~keep] = value
    v[~keep] = value
    res = dict(inp)
    res["k_pages"], res["v_pages"] = k, v
    return res
