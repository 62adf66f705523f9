"""The decoder's prefix length (how much of each slot is fetched before the
row's headers are read): its tuning from sampled row lengths, and that no
prefix changes a decoded bit (« Algorithme central », step 3)."""

import ctypes

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp
from oracle import oracle_c as C
from tests.gpu_util import gpu_codec, on_device, place, words_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()
    C.set_threads(8)


def _mixed_rows(rng, n, W):
    """Sparse float rows whose number of non-zero words varies a lot, plus
    some rows of noise (stored raw): stored lengths spread over many chunks."""
    x = np.zeros((n, W), np.float32)
    nnz = rng.integers(0, W // 2 + 1, n)
    for r in range(n):
        cols = rng.choice(W, nnz[r], replace=False)
        x[r, cols] = rng.normal(0, 1, nnz[r])
    rows = x.view(np.uint32).copy()
    rows[::17] = rng.integers(0, 2**32, (len(rows[::17]), W), dtype=np.uint64).astype(np.uint32)
    return rows


def _expected_prefix(lens, n_rows, n_sample, W, lmin_words):
    """The rule ibp_plan_tune_prefix states, applied to the oracle's stored
    lengths of the sampled rows."""
    n_sample = min(n_rows, n_sample)
    sampled = lens[(np.arange(n_sample, dtype=np.uint64) * n_rows) // n_sample]
    c = (sampled.astype(np.int64) + 3) // 4
    best = None
    for P in range((lmin_words + 3) // 4, (W + 3) // 4 + 1):
        cost = int(np.where(c > P, c + 8, P).sum())
        if best is None or cost < best[0]:
            best = (cost, P)
    return min(4 * best[1], W)


@pytest.mark.parametrize("W", [32, 64, 96, 512])
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_tuned_prefix_follows_the_rule_and_keeps_results(W, where):
    rng = np.random.default_rng(W)
    n = 3000
    rows = _mixed_rows(rng, n, W)
    g = gpu_codec(rows, rows[:1000], 0.9, where)
    plan = g["plan"]
    default = plan.info["prefix_words"]
    lens = C.row_words(rows, g["mask"], g["bitval"])
    bm_t = on_device(g["bitmask"])
    for max_sample in (0, 257):
        got = ibp.ibp_plan_tune_prefix(plan, g["slots_t"], bm_t, max_sample=max_sample)
        want = _expected_prefix(lens, n, max_sample or 65536, W, default)
        assert got == want == plan.info["prefix_words"], (max_sample, got, want)
        assert default <= got <= W
    ids = rng.integers(0, n, 4 * n).astype(np.int64)
    ids_t = torch.from_numpy(ids).cuda()
    for words in (0, 5, default + 4, 3 * W // 4, W, 10 * W):
        plan.set_prefix(words)
        out = ibp.ibp_gather_decompress(plan, g["slots_t"], bm_t, ids_t)
        torch.cuda.synchronize()
        assert ibp.ibp_get_status(plan) == ibp.IBP_OK
        assert np.array_equal(words_np(out), rows[ids]), words
        out = ibp.ibp_decompress_contig(plan, g["slots_t"], bm_t, 11, n - 20)
        torch.cuda.synchronize()
        assert np.array_equal(words_np(out), rows[11:n - 9]), words
    plan.set_prefix(0)
    assert plan.info["prefix_words"] == default


def test_prefix_of_unaligned_width():
    """W not a multiple of 4 (word path): any prefix still decodes exactly."""
    rng = np.random.default_rng(3)
    W, n = 45, 800
    rows = _mixed_rows(rng, n, W)
    g = gpu_codec(rows, rows, 0.9, "hbm")
    bm_t = on_device(g["bitmask"])
    got = ibp.ibp_plan_tune_prefix(g["plan"], g["slots_t"], bm_t)
    assert g["plan"].info["segments"] <= got <= W
    ids = torch.from_numpy(rng.integers(0, n, 2 * n).astype(np.int64)).cuda()
    for words in (0, 7, W):
        g["plan"].set_prefix(words)
        out = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm_t, ids)
        torch.cuda.synchronize()
        assert np.array_equal(words_np(out), rows[ids.cpu().numpy()])


def test_packed_layout_ignores_a_long_prefix():
    """A packed row may end before a long prefix; the packed decoder keeps the
    plan's shortest-stream prefix and decodes exactly."""
    rng = np.random.default_rng(5)
    W, n = 128, 2000
    rows = _mixed_rows(rng, n, W)
    g = gpu_codec(rows, rows[:500], 0.9, "hbm")
    plan = g["plan"]
    bm_t = on_device(g["bitmask"])
    plan.set_prefix(W)
    offsets = ibp.ibp_packed_offsets(plan, g["slots_t"], bm_t)
    packed = ibp.ibp_pack(plan, g["slots_t"], offsets)
    ids = rng.integers(0, n, 3 * n).astype(np.int64)
    out = ibp.ibp_gather_decompress_packed(plan, packed, offsets, bm_t, torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows[ids])


@pytest.mark.parametrize("where", ["host", "hbm"])
def test_corrupt_rows_detected_with_full_prefix(where):
    rng = np.random.default_rng(9)
    W = 128
    rows = rng.normal(0, 0.05, (64, W)).astype(np.float32).view(np.uint32)
    g = gpu_codec(rows, rows, 0.9, "host")
    slots = words_np(g["slots_t"]).copy()
    slots[0, :W // 32] = 0  # every word announces 32 bits: stream >= W words
    bad = place(slots, where)
    g["plan"].set_prefix(W)
    ids = np.arange(4, dtype=np.int64)
    out = ibp.ibp_gather_decompress(g["plan"], bad, on_device(g["bitmask"]), torch.from_numpy(ids).cuda())
    assert ibp.ibp_get_status(g["plan"], raise_on_error=False) == ibp.IBP_ECORRUPT
    st, ref = C.decompress(slots, g["bitmask"], ids, g["mask"], g["bitval"])
    assert st == ibp.IBP_ECORRUPT and np.array_equal(words_np(out), ref)


def test_tune_prefix_rejects_bad_arguments():
    rows = np.random.default_rng(1).normal(0, 1, (64, 32)).astype(np.float32).view(np.uint32)
    g = gpu_codec(rows, rows, 0.9, "hbm")
    lib = ibp.load()
    assert lib.ibp_plan_tune_prefix(None, None, 0, None, 0, None, None) == ibp.IBP_EINVAL
    assert lib.ibp_plan_tune_prefix(g["plan"].handle, ctypes.c_void_p(g["slots_t"].data_ptr()), 0,
                                    ctypes.c_void_p(0), 0, None, None) == ibp.IBP_EINVAL
    assert lib.ibp_plan_set_prefix(None, 4) == ibp.IBP_EINVAL
