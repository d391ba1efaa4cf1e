"""Seeded synthetic inputs for the low-bit dual-path MLA cache (shared by tests, smoke and bench).

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic (no quantization, packing or attention), so both the CUDA path and the oracle can
consume the very same arrays.

Recipe (numpy PCG64, one generator per workload, seeded):
  - outlier k_R channels: ``rng.choice(64, n_outliers, replace=False)`` drawn first;
  - latent c_t: N(0, 1) (or Student-t with nu = 5 for the heavy-tailed INT2 workloads) per
    channel, then each token rescaled to unit RMS over its 512 channels (the MLA latent is the
    output of an RMSNorm), rounded to BF16 (round to nearest even);
  - k_R: N(0, 1) per channel, the outlier channels multiplied by a fixed factor (the fixed-
    channel outlier bands of the post-RoPE key), rounded to BF16;
  - q_lat, q_rope: N(0, 1), rounded to BF16;
  - page tables: identity order, or a random permutation of the page pool (ragged serving).
All values are BF16 bit patterns (uint16) and int32 page tables / lengths.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

LATENT, ROPE, ROW = 512, 64, 576


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (sizes follow the DeepSeek-V2-Lite / GLM MLA shapes)."""
    name: str
    batch: int
    heads: int
    seq_len: int                 # cached tokens per sequence (uniform), or the max when ragged
    bits_c: int                  # 4 (C4) or 2 (C2)
    page_size: int
    n_sink: int = 4
    n_recent: int = 128
    clip_q: float = 0.0          # 0.94 for the INT2 latent
    latent_dist: str = "normal"  # "normal" or "student_t5"
    n_outliers: int = 4
    outlier_scale: float = 10.0
    ragged_min: int = 0          # > 0: per-sequence lengths uniform in [ragged_min, seq_len]
    random_pages: bool = False
    steps: int = 1               # decode steps (write one token per sequence, then attend)
    seed: int = 0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(192.0)  # per-head query/key dim of the MLA model: 128 + 64

    def config_kwargs(self) -> dict:
        return dict(bits_c=self.bits_c, page_size=self.page_size, n_sink=self.n_sink,
                    n_recent=self.n_recent, clip_q=self.clip_q)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_c4r4_b1_h16_t1k", 1, 16, 1024, 4, 128),
        Workload("v2lite_c4r4_b32_h16_t8k", 32, 16, 8192, 4, 128),
        Workload("v2lite_c4r4_b32_h16_t32k", 32, 16, 32768, 4, 128),
        Workload("wide_c2r4_b8_h128_t32k", 8, 128, 32768, 2, 64, clip_q=0.94,
                 latent_dist="student_t5", n_outliers=8, outlier_scale=20.0),
        Workload("long_c4r4_b1_h128_t128k", 1, 128, 131072, 4, 128),
        Workload("ragged_c2r4_b64_h16_serve", 64, 16, 16384, 2, 64, clip_q=0.94,
                 latent_dist="student_t5", n_outliers=8, outlier_scale=20.0, ragged_min=512,
                 random_pages=True, steps=256),
    ]
}


def seq_lens_for(w: Workload, rng: np.random.Generator | None = None) -> np.ndarray:
    if w.ragged_min > 0:
        rng = rng or np.random.default_rng(w.seed + 1)
        return rng.integers(w.ragged_min, w.seq_len + 1, size=w.batch).astype(np.int32)
    return np.full(w.batch, w.seq_len, dtype=np.int32)


def draw_tokens(rng: np.random.Generator, n: int, latent_dist: str, outliers: np.ndarray,
                outlier_scale: float):
    """n new tokens: (c bits uint16[n, 512], kr bits uint16[n, 64])."""
    if latent_dist == "student_t5":
        c = rng.standard_t(5, size=(n, LATENT)).astype(np.float32)
    else:
        c = rng.standard_normal((n, LATENT), dtype=np.float32)
    rms = np.sqrt(np.mean(c.astype(np.float64) ** 2, axis=1, keepdims=True)).astype(np.float32)
    c = c / np.maximum(rms, np.float32(1e-30))
    kr = rng.standard_normal((n, ROPE), dtype=np.float32)
    if outliers.size:
        kr[:, outliers] *= np.float32(outlier_scale)
    return bf16_bits(c), bf16_bits(kr)


def draw_queries(rng: np.random.Generator, batch: int, heads: int):
    q_lat = bf16_bits(rng.standard_normal((batch, heads, LATENT), dtype=np.float32))
    q_rope = bf16_bits(rng.standard_normal((batch, heads, ROPE), dtype=np.float32))
    return q_lat, q_rope


def page_table_for(rng: np.random.Generator, batch: int, max_pages: int, random_pages: bool,
                   n_pages: int | None = None):
    """[batch, max_pages] int32 page ids over a pool of n_pages (default batch*max_pages)."""
    n_pages = n_pages or batch * max_pages
    if random_pages:
        perm = rng.permutation(n_pages)[: batch * max_pages]
        return perm.reshape(batch, max_pages).astype(np.int32), n_pages
    return np.arange(batch * max_pages, dtype=np.int32).reshape(batch, max_pages), n_pages


@dataclasses.dataclass
class CacheInputs:
    workload: Workload
    seq_lens: np.ndarray      # [B] int32 tokens to prefill
    c: np.ndarray             # [sum T, 512] BF16 bits, rows grouped by sequence
    kr: np.ndarray            # [sum T, 64] BF16 bits
    cu: np.ndarray            # [B+1] int32 row offsets
    q_lat: np.ndarray         # [B, H, 512] BF16 bits
    q_rope: np.ndarray        # [B, H, 64] BF16 bits
    page_table: np.ndarray    # [B, max_pages] int32
    n_pages: int
    outliers: np.ndarray      # k_R outlier channel indices


def make_inputs(w: Workload, seq_lens: np.ndarray | None = None, extra_pages: int = 0,
                heads: int | None = None) -> CacheInputs:
    """Prefill tokens, queries and page table for a workload (sizes may be overridden)."""
    rng = np.random.default_rng(w.seed)
    outliers = rng.choice(ROPE, w.n_outliers, replace=False) if w.n_outliers else np.zeros(0, int)
    if seq_lens is None:
        seq_lens = seq_lens_for(w)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.shape[0]
    total = int(seq_lens.sum())
    c, kr = draw_tokens(rng, total, w.latent_dist, outliers, w.outlier_scale)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seq_lens)
    q_lat, q_rope = draw_queries(rng, B, heads or w.heads)
    max_pages = int(math.ceil((int(seq_lens.max(initial=0)) + extra_pages * w.page_size + 1) / w.page_size))
    page_table, n_pages = page_table_for(rng, B, max_pages, w.random_pages)
    return CacheInputs(w, seq_lens, c, kr, cu, q_lat, q_rope, page_table, n_pages, outliers)
