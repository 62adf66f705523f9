"""Gather-decompress fused with sum / mean pooling against the oracles: the C
oracle decodes the ids' rows, oracle/bag_ref.py pools them; the GPU result
must match bit for bit (« Résultats »: DLRM / GNN consumers of IBP's rows)."""

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp
from oracle import bag_ref as B
from oracle import oracle_c as C
from tests.gpu_util import gpu_codec, on_device, words_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()
    C.set_threads(8)


def _rows(rng, n, W, per_column=False):
    """float32 rows (no NaN or Inf): small values, and every 9th row large
    (those mismatch the Mask and are stored raw)."""
    scale = np.exp(rng.uniform(-6, 1, W)) if per_column else 0.05
    x = (rng.normal(0, 1, (n, W)) * scale).astype(np.float32)
    x[::9] = rng.normal(0, 1e4, (len(x[::9]), W)).astype(np.float32)
    return x.view(np.uint32)


def _bags(rng, n_ids, G):
    sizes = [0, 1, G - 1, G, G + 1, 0, 3 * G + 2, 100, 1, 0]
    while sum(sizes) < n_ids:
        sizes.append(int(rng.integers(0, 4 * G)))
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    offsets = np.minimum(offsets, n_ids)
    offsets[-1] = n_ids
    return offsets


def _expected(g, ids, offsets, mode):
    st, dec = C.decompress(words_np(g["slots_t"]), g["bitmask"], ids, g["mask"], g["bitval"])
    bst, out = B.embedding_bag(dec, offsets, mode)
    return st or bst, out


@pytest.mark.parametrize("W", [32, 64, 128, 256, 512])
@pytest.mark.parametrize("where", ["host", "hbm"])
@pytest.mark.parametrize("mode", [ibp.IBP_BAG_SUM, ibp.IBP_BAG_MEAN])
def test_bag_matches_oracle(W, where, mode):
    rng = np.random.default_rng(W + 7 * mode)
    n = max(64, 120_000 // W)
    rows = _rows(rng, n, W)
    g = gpu_codec(rows, rows[: n // 2], 0.9, where)
    G = max(1, 512 // W)
    n_ids = 3000
    ids = rng.integers(0, n, n_ids).astype(np.int64)
    offsets = _bags(rng, n_ids, G)
    out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                        torch.from_numpy(ids).cuda(), torch.from_numpy(offsets).cuda(), mode)
    code = ibp.ibp_get_status(g["plan"], raise_on_error=False)
    st, want = _expected(g, ids, offsets, mode)
    assert st == 0 and code == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("W", [128, 512])
def test_bag_per_word_plan(W):
    rng = np.random.default_rng(40 + W)
    n = 900
    rows = _rows(rng, n, W, per_column=True)
    g = gpu_codec(rows, rows[:600], 0.95, "hbm")
    assert g["plan"].info["uniform"] == 0
    ids = rng.integers(0, n, 2000).astype(np.int64)
    offsets = _bags(rng, len(ids), max(1, 512 // W))
    for mode in (ibp.IBP_BAG_SUM, ibp.IBP_BAG_MEAN):
        out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                            torch.from_numpy(ids).cuda(), torch.from_numpy(offsets).cuda(), mode)
        assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
        st, want = _expected(g, ids, offsets, mode)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want)


def test_bag_errors_bad_ids_offsets_and_corrupt_slots():
    rng = np.random.default_rng(3)
    W, n = 64, 500
    rows = _rows(rng, n, W)
    g = gpu_codec(rows, np.delete(rows, np.s_[::9], axis=0), 0.9, "hbm")  # Mask from the small rows
    ids = rng.integers(0, n, 200).astype(np.int64)
    ids[[5, 77]] = [n, -3]  # out of range: zero rows, IBP_ERANGE
    offsets = _bags(rng, len(ids), 8)
    out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                        torch.from_numpy(ids).cuda(), torch.from_numpy(offsets).cuda())
    assert ibp.ibp_get_status(g["plan"], raise_on_error=False) == ibp.IBP_ERANGE
    st, want = _expected(g, ids, offsets, B.SUM)
    assert st == ibp.IBP_ERANGE and np.array_equal(out.cpu().numpy().view(np.uint32), want)
    # invalid offsets: a decreasing pair and one past n_ids
    bad_off = np.array([0, 10, 4, 20, 250, 200], np.int64)
    out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                        torch.from_numpy(ids).cuda(), torch.from_numpy(bad_off).cuda())
    assert ibp.ibp_get_status(g["plan"], raise_on_error=False) == ibp.IBP_ERANGE
    st, want = _expected(g, ids, bad_off, B.SUM)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want)
    assert not want[[1, 3, 4]].any()
    # a corrupt slot: zero row, IBP_ECORRUPT
    slots = words_np(g["slots_t"]).copy()
    r = int(np.nonzero([(g["bitmask"][i // 32] >> (i % 32)) & 1 for i in range(n)])[0][0])
    slots[r, :W // 32] = 0
    ids2 = np.array([r, (r + 1) % n, r], np.int64)
    off2 = np.array([0, 2, 3], np.int64)
    out = ibp.ibp_gather_decompress_bag(g["plan"], on_device(slots), on_device(g["bitmask"]),
                                        torch.from_numpy(ids2).cuda(), torch.from_numpy(off2).cuda(), ibp.IBP_BAG_MEAN)
    assert ibp.ibp_get_status(g["plan"], raise_on_error=False) == ibp.IBP_ECORRUPT
    st, dec = C.decompress(slots, g["bitmask"], ids2, g["mask"], g["bitval"])
    _, want = B.embedding_bag(dec, off2, B.MEAN)
    assert st == ibp.IBP_ECORRUPT and np.array_equal(out.cpu().numpy().view(np.uint32), want)


def test_bag_equals_gather_then_sequential_sum():
    """The fused result equals decoding the rows (gather-decompress) and then
    adding them in order in float32 on the GPU."""
    rng = np.random.default_rng(8)
    W, n = 128, 4000
    rows = _rows(rng, n, W)
    g = gpu_codec(rows, rows[:2000], 0.9, "host")
    ids = rng.integers(0, n, 640).astype(np.int64)
    offsets = np.arange(0, 641, 32, dtype=np.int64)  # 20 bags of 32
    ids_t = torch.from_numpy(ids).cuda()
    out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]), ids_t,
                                        torch.from_numpy(offsets).cuda())
    dec = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], on_device(g["bitmask"]), ids_t).view(torch.float32)
    ref = torch.zeros((20, W), dtype=torch.float32, device="cuda")
    for k in range(32):  # one row of every bag per step: sequential order within each bag
        ref += dec.view(20, 32, W)[:, k]
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))


def test_bag_rejects_bad_arguments():
    rng = np.random.default_rng(1)
    rows = _rows(rng, 64, 45)  # W = 45: not a specialised shape
    g = gpu_codec(rows, rows, 0.9, "hbm")
    ids = torch.zeros(4, dtype=torch.int64, device="cuda")
    off = torch.tensor([0, 4], dtype=torch.int64, device="cuda")
    with pytest.raises(ibp.IbpError):
        ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]), ids, off)
    rows = _rows(rng, 64, 64)
    g = gpu_codec(rows, rows, 0.9, "hbm")
    with pytest.raises(ibp.IbpError):
        ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]), ids, off, mode=4)
    empty = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]), ids,
                                          torch.zeros(1, dtype=torch.int64, device="cuda"))
    assert empty.shape == (0, 64)


@pytest.mark.parametrize("W", [32, 64, 128, 512])
def test_bag_row_reuse_hint_from_host(W):
    """Row-reuse copies from host-mapped slots take the small-group kernels;
    results are unchanged."""
    rng = np.random.default_rng(90 + W)
    n = max(64, 60_000 // W)
    rows = _rows(rng, n, W)
    g = gpu_codec(rows, rows[: n // 2], 0.9, "host")
    g["plan"].set_hints(ibp.IBP_HINT_ROW_REUSE)
    hot = rng.integers(0, n, 7)
    ids = np.where(rng.random(2500) < 0.6, hot[rng.integers(0, 7, 2500)], rng.integers(0, n, 2500)).astype(np.int64)
    offsets = _bags(rng, len(ids), max(1, 256 // W))
    for mode in (ibp.IBP_BAG_SUM, ibp.IBP_BAG_MEAN):
        out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                            torch.from_numpy(ids).cuda(), torch.from_numpy(offsets).cuda(), mode)
        assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
        st, want = _expected(g, ids, offsets, mode)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want)


def _bf16_rows(rng, n, W):
    """Rows of 2W bfloat16 values (N(0, 0.5), every 9th row N(0, 1e3)) as W
    words of pairs."""
    from host_transfer_gb300 import workloads

    x = rng.normal(0, 0.5, (n, 2 * W))
    x[::9] = rng.normal(0, 1e3, (len(x[::9]), 2 * W))
    return workloads.bf16_pairs_to_words(workloads.f32_to_bf16_bits(x.astype(np.float32)))


@pytest.mark.parametrize("W", [32, 64, 128, 512])
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_bag_bf16_rows_match_oracle(W, where):
    rng = np.random.default_rng(300 + W)
    n = max(64, 60_000 // W)
    rows = _bf16_rows(rng, n, W)
    g = gpu_codec(rows, np.delete(rows, np.s_[::9], axis=0), 0.9, where)
    ids = rng.integers(0, n, 2500).astype(np.int64)
    offsets = _bags(rng, len(ids), max(1, 512 // W))
    for mode in (ibp.IBP_BAG_SUM, ibp.IBP_BAG_MEAN):
        out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                            torch.from_numpy(ids).cuda(), torch.from_numpy(offsets).cuda(),
                                            mode | ibp.IBP_BAG_BF16)
        assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
        assert out.shape == (len(offsets) - 1, 2 * W)
        st, dec = C.decompress(words_np(g["slots_t"]), g["bitmask"], ids, g["mask"], g["bitval"])
        _, want = B.embedding_bag(dec, offsets, mode, bf16=True)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("W", [128, 256, 512])
@pytest.mark.parametrize("n_bags", [40, 300, 900])
def test_few_large_bags_from_hbm(W, n_bags):
    """Few bags on device slots are pooled by teams of warps that split the
    segments; each column is still added in bag order."""
    rng = np.random.default_rng(500 + W + n_bags)
    n = max(200, 150_000 // W)
    per_column = W == 256
    rows = _rows(rng, n, W, per_column=per_column)
    g = gpu_codec(rows, np.delete(rows, np.s_[::9], axis=0), 0.95 if per_column else 0.9, "hbm")
    sizes = rng.integers(0, 60, n_bags)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    ids = rng.integers(0, n, int(offsets[-1])).astype(np.int64)
    for mode in (ibp.IBP_BAG_SUM, ibp.IBP_BAG_MEAN):
        out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                            torch.from_numpy(ids).cuda(), torch.from_numpy(offsets).cuda(), mode)
        assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
        st, want = _expected(g, ids, offsets, mode)
        assert st == 0 and np.array_equal(out.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("W", [64, 256])
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_bag_bf16_per_word_plan(W, where):
    """bfloat16 rows under per-word Masks (every third element on a scale a
    thousand times smaller): the table decoder's two words per lane pooled as
    four floats, in bag order, against the oracle."""
    from host_transfer_gb300 import workloads

    rng = np.random.default_rng(700 + W)
    n = 900
    scale = np.where(np.arange(2 * W) % 3 == 0, 1e-3, 1.0)
    x = (rng.normal(0, 1, (n, 2 * W)) * scale).astype(np.float32)
    rows = workloads.bf16_pairs_to_words(workloads.f32_to_bf16_bits(x))
    g = gpu_codec(rows, rows[:600], 0.95, where)
    assert g["plan"].info["uniform"] == 0
    ids = rng.integers(0, n, 2500).astype(np.int64)
    offsets = _bags(rng, len(ids), max(1, 512 // W))
    for mode in (ibp.IBP_BAG_SUM, ibp.IBP_BAG_MEAN):
        out = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                            torch.from_numpy(ids).cuda(), torch.from_numpy(offsets).cuda(),
                                            mode | ibp.IBP_BAG_BF16)
        assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
        st, dec = C.decompress(words_np(g["slots_t"]), g["bitmask"], ids, g["mask"], g["bitval"])
        _, want = B.embedding_bag(dec, offsets, mode, bf16=True)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want)


def test_bag_bf16_output_must_be_8_byte_aligned():
    """bfloat16 bags are written as pairs of floats: an output that is only
    4-byte aligned is refused before anything runs."""
    rng = np.random.default_rng(5)
    rows = _rows(rng, 128, 64)
    g = gpu_codec(rows, rows, 0.9, "hbm")
    ids = torch.zeros(4, dtype=torch.int64, device="cuda")
    off = torch.tensor([0, 4], dtype=torch.int64, device="cuda")
    buf = torch.zeros(2 * 128 + 1, dtype=torch.float32, device="cuda")
    with pytest.raises(ibp.IbpError):
        ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]), ids, off,
                                      mode=ibp.IBP_BAG_BF16, out=buf[1:])
    ok = ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], on_device(g["bitmask"]), ids, off,
                                       mode=ibp.IBP_BAG_BF16, out=buf[:-1])
    torch.cuda.synchronize()
    assert ok.data_ptr() == buf.data_ptr()
