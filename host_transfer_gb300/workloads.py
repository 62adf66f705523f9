"""Seeded synthetic workloads for Invariant Bit Packing.

This module only draws numbers: it holds none of the compression arithmetic,
so that the CUDA path and the CPU oracle can be fed the same inputs without
sharing code.  Every generator uses ``numpy.random.Generator(PCG64(seed))``;
floats are drawn in float64 and rounded to float32 (or to bfloat16,
round-to-nearest-even) and returned as 32-bit words.  bfloat16 tensors are
packed two per word, element 2j in bits 0-15 and element 2j+1 in bits 16-31.

The shapes and distributions stand in for the real datasets the paper
measured on (its section « Résultats »: dense and sparse GNN feature sets,
DLRM embedding tables, LLM weights and KV caches), which are not available
here:

==========  ==================================================================
tiny        2048 x 128 fp32, N(0, 0.05) clipped to [-0.25, 0.25]; seed 0;
            sample 256 rows (seed 0), T = 0.99.
dense_gnn   2,000,000 x 128 fp32, N(0,1) rows L2-normalised in float64;
            seed 1; sample 65,536 rows (seed 11), T = 0.99; batches of
            65,536 uniform ids (seed 21 + k).
sparse_gnn  1,000,000 x 512 fp32, 26 non-zeros per row (5 %) at uniform
            positions, values lognormal(-2, 0.5) clipped to <= 1; seed 2;
            sample 65,536 rows (seed 12), T = 0.95; batches of 32,768 ids.
dlrm        8,000,000 x 64 fp32, U(-0.01, 0.01); seed 3; sample 65,536 rows
            (seed 13), T = 0.99; batches of 131,072 ids drawn from a Zipf
            law (s = 1.05) over ranks, ranks mapped to rows by a seeded
            permutation.
llm         32 layers; weights 4096 x 4096 bf16 N(0, 0.02) (rows of 4096
            elements = 2048 words); KV cache [layer, 2, 32 heads, 4096, 128]
            bf16, N(0,1) times a per-(layer, head) scale U(0.5, 4) (rows of
            128 elements = 64 words); seed 4; per-tensor sample of 4,096
            rows, T = 0.99; contiguous decompress of a layer.
==========  ==================================================================
"""

from __future__ import annotations

import numpy as np

CONFIGS = {
    "tiny": dict(n_rows=2048, W=128, T=0.99, seed=0, sample=256, sample_seed=0,
                 batch=2048, batch_seed=20),
    "dense_gnn": dict(n_rows=2_000_000, W=128, T=0.99, seed=1, sample=65_536, sample_seed=11,
                      batch=65_536, batch_seed=21),
    "sparse_gnn": dict(n_rows=1_000_000, W=512, T=0.95, seed=2, sample=65_536, sample_seed=12,
                       batch=32_768, batch_seed=22, nnz=26),
    "dlrm": dict(n_rows=8_000_000, W=64, T=0.99, seed=3, sample=65_536, sample_seed=13,
                 batch=131_072, batch_seed=23, zipf_s=1.05),
    "llm": dict(layers=32, hidden=4096, heads=32, seq=4096, head_dim=128, T=0.99, seed=4,
                sample=4096, sample_seed=14),
}

_CHUNK = 1 << 16  # rows drawn per generator call; fixed so results never depend on it


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _f32_words(x64: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x64.astype(np.float32)).view(np.uint32)


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_pairs_to_words(b16: np.ndarray) -> np.ndarray:
    """View a (..., 2k) uint16 array as (..., k) uint32 words, element 2j low."""
    b16 = np.ascontiguousarray(b16, dtype=np.uint16)
    lo = b16[..., 0::2].astype(np.uint32)
    hi = b16[..., 1::2].astype(np.uint32)
    return lo | (hi << 16)


def _out(n_rows: int, W: int, out):
    if out is None:
        return np.empty((n_rows, W), np.uint32)
    assert out.shape == (n_rows, W) and out.dtype == np.uint32
    return out


def tiny_table(n_rows: int = 2048, W: int = 128, seed: int = 0, out=None) -> np.ndarray:
    out = _out(n_rows, W, out)
    rng = _rng(seed)
    for a in range(0, n_rows, _CHUNK):
        b = min(n_rows, a + _CHUNK)
        x = np.clip(rng.normal(0.0, 0.05, size=(b - a, W)), -0.25, 0.25)
        out[a:b] = _f32_words(x)
    return out


def dense_gnn_table(n_rows: int = 2_000_000, W: int = 128, seed: int = 1, out=None) -> np.ndarray:
    out = _out(n_rows, W, out)
    rng = _rng(seed)
    for a in range(0, n_rows, _CHUNK):
        b = min(n_rows, a + _CHUNK)
        x = rng.standard_normal(size=(b - a, W))
        x /= np.sqrt(np.einsum("ij,ij->i", x, x))[:, None]
        out[a:b] = _f32_words(x)
    return out


def sparse_gnn_table(n_rows: int = 1_000_000, W: int = 512, seed: int = 2, nnz: int = 26,
                     out=None) -> np.ndarray:
    """Exactly ``nnz`` non-zeros per row; positions are a uniform random subset
    (Floyd's subset sampling, vectorised over rows)."""
    out = _out(n_rows, W, out)
    rng = _rng(seed)
    for a in range(0, n_rows, _CHUNK):
        b = min(n_rows, a + _CHUNK)
        n = b - a
        chosen = np.zeros((n, W), dtype=bool)
        rows = np.arange(n)
        for j in range(W - nnz, W):
            t = rng.integers(0, j + 1, size=n)
            taken = chosen[rows, t]
            pick = np.where(taken, j, t)
            chosen[rows, pick] = True
        vals = np.minimum(rng.lognormal(-2.0, 0.5, size=(n, nnz)), 1.0).astype(np.float32)
        blk = np.zeros((n, W), np.float32)
        blk[chosen] = vals.reshape(-1)
        out[a:b] = blk.view(np.uint32)
    return out


def dlrm_table(n_rows: int = 8_000_000, W: int = 64, seed: int = 3, out=None) -> np.ndarray:
    out = _out(n_rows, W, out)
    rng = _rng(seed)
    for a in range(0, n_rows, _CHUNK):
        b = min(n_rows, a + _CHUNK)
        out[a:b] = _f32_words(rng.uniform(-0.01, 0.01, size=(b - a, W)))
    return out


def llm_weight(layer: int, rows: int = 4096, cols: int = 4096, seed: int = 4) -> np.ndarray:
    """One layer's weight matrix as (rows, cols/2) words."""
    rng = _rng(seed * 1_000_003 + 2 * layer)
    x = rng.normal(0.0, 0.02, size=(rows, cols)).astype(np.float32)
    return bf16_pairs_to_words(f32_to_bf16_bits(x))


def llm_kv(layer: int, heads: int = 32, seq: int = 4096, head_dim: int = 128,
           seed: int = 4) -> np.ndarray:
    """One layer's K and V as (2, heads*seq, head_dim/2) words."""
    rng = _rng(seed * 1_000_003 + 2 * layer + 1)
    scale = rng.uniform(0.5, 4.0, size=(2, heads))
    out = np.empty((2, heads, seq, head_dim // 2), np.uint32)
    for kv in range(2):
        for h in range(heads):
            x = (rng.standard_normal(size=(seq, head_dim)) * scale[kv, h]).astype(np.float32)
            out[kv, h] = bf16_pairs_to_words(f32_to_bf16_bits(x))
    return out.reshape(2, heads * seq, head_dim // 2)


def make_table(name: str, n_rows: int | None = None, out=None) -> np.ndarray:
    """Row table of a named configuration, optionally with fewer rows (the
    first ``n_rows`` rows of the full table for chunk-aligned sizes)."""
    c = CONFIGS[name]
    n = c["n_rows"] if n_rows is None else n_rows
    if name == "tiny":
        return tiny_table(n, c["W"], c["seed"], out)
    if name == "dense_gnn":
        return dense_gnn_table(n, c["W"], c["seed"], out)
    if name == "sparse_gnn":
        return sparse_gnn_table(n, c["W"], c["seed"], c["nnz"], out)
    if name == "dlrm":
        return dlrm_table(n, c["W"], c["seed"], out)
    raise KeyError(name)


def sample_ids(n_rows: int, n_sample: int, seed: int) -> np.ndarray:
    """Rows for the preprocess sample: uniform without replacement, sorted."""
    n_sample = min(n_sample, n_rows)
    return np.sort(_rng(seed).choice(n_rows, size=n_sample, replace=False)).astype(np.int64)


def uniform_ids(n_rows: int, batch: int, seed: int) -> np.ndarray:
    return _rng(seed).integers(0, n_rows, size=batch, dtype=np.int64)


class ZipfIds:
    """Truncated Zipf(s) over ranks 1..n (inverse CDF), ranks mapped to rows by
    a seeded permutation."""

    def __init__(self, n_rows: int, s: float = 1.05, seed: int = 3):
        k = np.arange(1, n_rows + 1, dtype=np.float64)
        self.cdf = np.cumsum(k ** (-s))
        self.cdf /= self.cdf[-1]
        self.perm = _rng(seed + 1_000).permutation(n_rows).astype(np.int64)

    def draw(self, batch: int, seed: int) -> np.ndarray:
        u = _rng(seed).random(batch)
        rank = np.minimum(np.searchsorted(self.cdf, u, side="left"), len(self.cdf) - 1)
        return self.perm[rank]


def batch_ids(name: str, k: int, n_rows: int | None = None, batch: int | None = None,
              zipf: ZipfIds | None = None) -> np.ndarray:
    """The k-th id batch of a configuration."""
    c = CONFIGS[name]
    n = c["n_rows"] if n_rows is None else n_rows
    bsz = c["batch"] if batch is None else batch
    seed = c["batch_seed"] * 1000 + k
    if name == "dlrm":
        z = zipf if zipf is not None else ZipfIds(n, c["zipf_s"], c["seed"])
        return z.draw(bsz, seed)
    return uniform_ids(n, bsz, seed)
