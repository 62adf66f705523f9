"""The packed cache layout: offsets, packed words and decode against the
oracle (« Intégration au système », cache compression: only the compressed
part of each row is kept)."""

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp, workloads
from oracle import oracle_c as C
from oracle import packed_ref as P
from tests.gpu_util import gpu_codec, on_device, pinned, words_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()
    C.set_threads(8)


def _expected(rows, mask, bitval):
    """Offsets and packed words of the oracle's slots (oracle/packed_ref.py)."""
    slots, bitmask, _ = C.compress(rows, mask, bitval)
    offsets, packed = P.pack(slots, C.row_words(rows, mask, bitval))
    return offsets, packed, bitmask


def _sparse_rows(rng, n, W, nnz):
    x = np.zeros((n, W), np.float32)
    cols = np.argsort(rng.random((n, W)), axis=1)[:, :nnz]
    x[np.arange(n)[:, None], cols] = rng.lognormal(-2, 0.5, (n, nnz)).clip(max=1.0)
    return x.view(np.uint32)


CASES = {
    "dense_w128": lambda rng: rng.normal(0, 0.05, (3000, 128)).astype(np.float32).view(np.uint32),
    "dlrm_w64": lambda rng: rng.uniform(-0.01, 0.01, (5000, 64)).astype(np.float32).view(np.uint32),
    "sparse_w512": lambda rng: _sparse_rows(rng, 1500, 512, 26),
    "mixed_w32": lambda rng: np.where(rng.random((20000, 1)) < 0.8,
                                      rng.normal(0, 1e-3, (20000, 32)).astype(np.float32).view(np.uint32),
                                      rng.integers(0, 2**32, (20000, 32), dtype=np.uint64).astype(np.uint32)),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_packed_layout_matches_oracle(name, where):
    rng = np.random.default_rng(len(name))
    rows = CASES[name](rng)
    T = 0.95 if name.startswith("sparse") else 0.99
    g = gpu_codec(rows, rows[: min(len(rows), 4096)], T, where)
    bm_t = on_device(g["bitmask"])
    offsets = ibp.ibp_packed_offsets(g["plan"], g["slots_t"], bm_t)
    packed = ibp.ibp_pack(g["plan"], g["slots_t"], offsets)
    torch.cuda.synchronize()
    want_off, want_packed, _ = _expected(rows, g["mask"], g["bitval"])
    assert np.array_equal(offsets.cpu().numpy(), want_off), "offsets differ from the oracle"
    got = words_np(packed)[: want_off[-1]]
    assert np.array_equal(got, want_packed), "packed words differ from the oracle"
    # decode from the packed buffer, in HBM and in pinned host memory
    ids = np.concatenate([rng.permutation(len(rows)), rng.integers(0, len(rows), 999)]).astype(np.int64)
    ids_t = torch.from_numpy(ids).cuda()
    for buf in (packed, pinned(words_np(packed))):
        out = ibp.ibp_gather_decompress_packed(g["plan"], buf, offsets, bm_t, ids_t)
        torch.cuda.synchronize()
        assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
        assert np.array_equal(words_np(out), rows[ids])
    saving = 1 - want_off[-1] / rows.size
    print(f"{name}: packed size saving {100 * saving:.2f} %")


def test_packed_bad_ids_and_corrupt_extents():
    rng = np.random.default_rng(3)
    rows = rng.normal(0, 0.05, (500, 128)).astype(np.float32).view(np.uint32)
    g = gpu_codec(rows, rows, 0.99, "hbm")
    bm_t = on_device(g["bitmask"])
    offsets = ibp.ibp_packed_offsets(g["plan"], g["slots_t"], bm_t)
    packed = ibp.ibp_pack(g["plan"], g["slots_t"], offsets)
    ids = torch.tensor([0, 500, -1, 3, 4], dtype=torch.int64, device="cuda")
    out = ibp.ibp_gather_decompress_packed(g["plan"], packed, offsets, bm_t, ids)
    assert ibp.ibp_get_status(g["plan"], raise_on_error=False) == ibp.IBP_ERANGE
    o = words_np(out)
    assert np.array_equal(o[[0, 3, 4]], rows[[0, 3, 4]]) and not o[[1, 2]].any()
    # row 3 announced shorter than its stream: its extent cuts the stream
    bad = offsets.clone()
    bad[4] = bad[3] + 8  # row 3 now spans 8 words only
    out = ibp.ibp_gather_decompress_packed(g["plan"], packed, bad, bm_t,
                                           torch.tensor([3, 0], dtype=torch.int64, device="cuda"))
    assert ibp.ibp_get_status(g["plan"], raise_on_error=False) == ibp.IBP_ECORRUPT
    o = words_np(out)
    assert not o[0].any() and np.array_equal(o[1], rows[0])


def test_packed_needs_the_specialised_plan_shape():
    rows = np.random.default_rng(4).normal(0, 0.05, (64, 100)).astype(np.float32).view(np.uint32)
    g = gpu_codec(rows, rows, 0.99, "hbm")
    bm_t = on_device(g["bitmask"])
    offsets = ibp.ibp_packed_offsets(g["plan"], g["slots_t"], bm_t)
    packed = ibp.ibp_pack(g["plan"], g["slots_t"], offsets)
    want_off, want_packed, _ = _expected(rows, g["mask"], g["bitval"])
    assert np.array_equal(offsets.cpu().numpy(), want_off)
    assert np.array_equal(words_np(packed)[: want_off[-1]], want_packed)
    with pytest.raises(ibp.IbpError):
        ibp.ibp_gather_decompress_packed(g["plan"], packed, offsets, bm_t,
                                         torch.zeros(4, dtype=torch.int64, device="cuda"))
