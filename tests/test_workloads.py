"""The seeded input generators (host_transfer_gb300/workloads.py) against the
recipe they state: shapes, value ranges and structure of each configuration,
bfloat16 rounding, id distributions, and determinism.  They hold no IBP
arithmetic; these checks pin the inputs both the CUDA path and the oracle
receive."""

import numpy as np

from host_transfer_gb300 import workloads as wl


def _f(words):
    return words.view(np.float32)


def test_tiny_rows_are_clipped_normals():
    t = wl.make_table("tiny")
    assert t.shape == (2048, 128) and t.dtype == np.uint32
    x = _f(t)
    assert np.abs(x).max() <= np.float32(0.25)
    assert 0.04 < x.std() < 0.06
    assert np.array_equal(t, wl.make_table("tiny"))  # same seed, same rows


def test_dense_rows_are_unit_vectors():
    t = wl.make_table("dense_gnn", n_rows=3000)
    x = _f(t).astype(np.float64)
    norms = np.sqrt((x * x).sum(axis=1))
    assert np.allclose(norms, 1.0, atol=1e-6)
    # the first rows of a shorter table are the first rows of the full one
    assert np.array_equal(t[:1000], wl.make_table("dense_gnn", n_rows=1000))


def test_sparse_rows_have_exactly_nnz_non_zeros():
    c = wl.CONFIGS["sparse_gnn"]
    t = wl.make_table("sparse_gnn", n_rows=4000)
    x = _f(t)
    nz = (t != 0).sum(axis=1)
    assert (nz == c["nnz"]).all()
    v = x[t != 0]
    assert (v > 0).all() and (v <= 1.0).all()
    # positions spread over the whole row
    assert (t != 0).any(axis=0).all()
    assert abs(np.log(v).mean() - (-2.0)) < 0.05


def test_dlrm_rows_are_small_uniforms():
    x = _f(wl.make_table("dlrm", n_rows=5000))
    assert np.abs(x).max() <= np.float32(0.01)
    assert abs(x.mean()) < 2e-4 and 0.0055 < x.std() < 0.006


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 0.0], np.float32)
    got = wl.f32_to_bf16_bits(vals)
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even mantissa
    assert list(got) == [0x3F80, 0x3F80, 0x3F82, 0x3F80, 0xC020, 0x0000]
    w = wl.bf16_pairs_to_words(got[:4].reshape(1, 4))
    assert w.shape == (1, 2) and w[0, 0] == (0x3F80 | (0x3F80 << 16)) and w[0, 1] == (0x3F82 | (0x3F80 << 16))


def test_llm_tensors_shapes_and_scales():
    w = wl.llm_weight(0, rows=64, cols=256)
    assert w.shape == (64, 128) and w.dtype == np.uint32
    kv = wl.llm_kv(3, heads=4, seq=256, head_dim=32)
    assert kv.shape == (2, 4 * 256, 16)
    # per-(K/V, head) scales in [0.5, 4]: each head's values have one spread
    lo = (kv & 0xFFFF).astype(np.uint32) << 16
    x = lo.view(np.float32).reshape(2, 4, 256 * 16)
    sd = x.std(axis=2)
    assert (sd > 0.4).all() and (sd < 4.5).all()
    assert np.array_equal(kv, wl.llm_kv(3, heads=4, seq=256, head_dim=32))
    assert not np.array_equal(wl.llm_weight(0, 64, 256), wl.llm_weight(1, 64, 256))


def test_id_batches():
    n = 100_000
    u = wl.batch_ids("dense_gnn", 0, n_rows=n, batch=50_000)
    assert u.dtype == np.int64 and u.min() >= 0 and u.max() < n
    z = wl.ZipfIds(n, 1.05, 3)
    d = z.draw(200_000, 7)
    assert d.min() >= 0 and d.max() < n
    counts = np.bincount(d, minlength=n)
    top = z.perm[0]  # rank 1
    assert counts[top] == counts.max() and counts[top] > 100 * counts.mean()
    assert np.array_equal(d, z.draw(200_000, 7))
    s = wl.sample_ids(1000, 300, 11)
    assert len(np.unique(s)) == 300 and (np.diff(s) > 0).all()
