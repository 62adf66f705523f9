"""Plan sets: one plan per block of consecutive rows (finer Mask granularity,
e.g. per attention head of a KV cache), decoded in one call and compared with
the oracle block by block (« Algorithme central », steps 1-3, per block)."""

import ctypes

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp
from oracle import oracle_c as C
from tests.gpu_util import empty_like_in, on_device, place, words_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()
    C.set_threads(8)


def _bf16_words(x: np.ndarray) -> np.ndarray:
    """float32 [n, 2W] -> bf16 (round to nearest even) pairs as uint32 [n, W]."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) & 0xFFFF
    return (r[:, 0::2] | (r[:, 1::2] << 16)).astype(np.uint32)


def _kv_blocks(rng, heads, rows, W, scale=None):
    """[head][position] rows of 2W bf16 values, N(0,1) times a per-head scale."""
    scale = rng.uniform(0.5, 4.0, heads) if scale is None else np.asarray(scale, np.float64)
    x = rng.normal(0, 1, (heads, rows, 2 * W)) * scale[:, None, None]
    return _bf16_words(x.reshape(heads * rows, 2 * W))


def _compress_blocks(rows, plans, rows_per_plan, where):
    """Compress block k of rows with plans[k] into one slot table and one
    bitmask (block k at word k * rows_per_plan / 32)."""
    n, W = rows.shape
    rows_t = place(rows, where)
    slots_t = empty_like_in(rows_t, where)
    bitmask = torch.zeros((n + 31) // 32, dtype=torch.int32, device="cuda")
    bpp = rows_per_plan // 32
    stored = 0
    for k, plan in enumerate(plans):
        lo, hi = k * rows_per_plan, (k + 1) * rows_per_plan
        _, _, st = ibp.ibp_compress(plan, rows_t[lo:hi], slots_t[lo:hi], bitmask=bitmask[k * bpp:(k + 1) * bpp])
        stored += int(st.item())
    torch.cuda.synchronize()
    return slots_t, bitmask, stored


@pytest.mark.parametrize("where", ["host", "hbm"])
def test_per_head_plans_match_the_oracle(where):
    rng = np.random.default_rng(11)
    heads, rpp, W = 6, 256, 64
    rows = _kv_blocks(rng, heads, rpp, W)
    plans, masks = [], []
    for k in range(heads):
        blk = rows[k * rpp:(k + 1) * rpp]
        mask, bitval = ibp.ibp_preprocess(on_device(blk), 0.99)
        st, m, b = C.preprocess(blk, 0.99)
        assert st == 0 and np.array_equal(words_np(mask), m) and np.array_equal(words_np(bitval), b)
        plans.append(ibp.ibp_plan_create(mask, bitval))
        masks.append((m, b))
    slots_t, bitmask, stored = _compress_blocks(rows, plans, rpp, where)
    slots, bm = words_np(slots_t), words_np(bitmask)
    for k, (m, b) in enumerate(masks):
        cs, cb, _ = C.compress(rows[k * rpp:(k + 1) * rpp], m, b)
        assert np.array_equal(slots[k * rpp:(k + 1) * rpp], cs), f"slots of block {k}"
        assert np.array_equal(bm[k * rpp // 32:(k + 1) * rpp // 32], cb), f"bitmask of block {k}"
    pset = ibp.ibp_plan_set_create(plans)
    out = ibp.ibp_decompress_contig_set(pset, slots_t, rpp, bitmask)
    assert ibp.ibp_plan_set_get_status(pset) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows)
    # finer masks pay on this data: one Mask for all heads keeps fewer bits
    st, m_all, b_all = C.preprocess(rows, 0.99)
    _, _, stored_all = C.compress(rows, m_all, b_all)
    assert stored < stored_all


def _run_mask(lo, length):
    return ((1 << length) - 1) << lo


def _rows_for(mask, bitval, rng, n, p_match=0.85):
    W = mask.size
    rows = rng.integers(0, 2**32, (n, W), dtype=np.uint64).astype(np.uint32)
    match = rng.random((n, W)) < p_match
    return np.where(match, (rows & ~mask) | (bitval & mask), rows).astype(np.uint32)


@pytest.mark.parametrize("W", [32, 128, 1024])
def test_mixed_plan_shapes_in_one_set(W):
    """Uniform, two-popcount, four-run and no-kept-bit plans in one set: all
    decode through the table path sized for the set."""
    rng = np.random.default_rng(W)
    rpp = 96
    shapes = []
    shapes.append(np.full(W, _run_mask(0, 9), np.uint64))                                   # uniform, 1 run
    shapes.append(np.array([_run_mask(0, 27) | (1 << 31) if w % 3 else _run_mask(26, 4)
                            for w in range(W)], np.uint64))                                  # two popcounts
    shapes.append(np.array([_run_mask(0, 3) | _run_mask(6, 2) | _run_mask(12, 5) | _run_mask(24, 1 + w % 7)
                            for w in range(W)], np.uint64))                                  # 4 runs
    shapes.append(np.array([0 if w % 2 else _run_mask(4, 12) for w in range(W)], np.uint64))  # empty fields
    plans, mb, blocks = [], [], []
    for keep in shapes:
        mask = (~keep & 0xFFFFFFFF).astype(np.uint32)
        bitval = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32) & mask
        plans.append(ibp.ibp_plan_create(torch.from_numpy(mask.view(np.int32)), torch.from_numpy(bitval.view(np.int32))))
        mb.append((mask, bitval))
        blk = _rows_for(mask, bitval, rng, rpp)
        blk[::7] = rng.integers(0, 2**32, (len(blk[::7]), W), dtype=np.uint64).astype(np.uint32)
        blocks.append(blk)
    rows = np.concatenate(blocks)
    # rows_per_plan need not be a multiple of 32 when the bitmask is built by
    # the oracle for the whole table
    slots = np.empty_like(rows)
    bits = np.zeros(len(rows), np.uint8)
    for k, (m, b) in enumerate(mb):
        cs, cb, _ = C.compress(blocks[k], m, b)
        slots[k * rpp:(k + 1) * rpp] = cs
        bits[k * rpp:(k + 1) * rpp] = ((cb[np.arange(rpp) >> 5] >> (np.arange(rpp) & 31).astype(np.uint32)) & 1)
    bitmask = np.zeros((len(rows) + 31) // 32, np.uint32)
    for r in np.nonzero(bits)[0]:
        bitmask[r // 32] |= np.uint32(1 << (r % 32))
    pset = ibp.ibp_plan_set_create(plans)
    for where in ("host", "hbm"):
        out = ibp.ibp_decompress_contig_set(pset, place(slots, where), rpp, on_device(bitmask))
        assert ibp.ibp_plan_set_get_status(pset) == ibp.IBP_OK
        assert np.array_equal(words_np(out), rows), where


def test_corrupt_row_reported_by_the_set():
    rng = np.random.default_rng(5)
    heads, rpp, W = 3, 64, 64
    rows = _kv_blocks(rng, heads, rpp, W, scale=[0.5, 0.25, 0.5])  # small values: invariant exponent bits
    plans = []
    for k in range(heads):
        blk = rows[k * rpp:(k + 1) * rpp]
        mask, bitval = ibp.ibp_preprocess(on_device(blk), 0.9)
        plans.append(ibp.ibp_plan_create(mask, bitval))
    slots_t, bitmask, _ = _compress_blocks(rows, plans, rpp, "hbm")
    bm = words_np(bitmask)
    comp = [r for r in range(rpp, 2 * rpp) if (bm[r // 32] >> (r % 32)) & 1]
    assert comp, "block 1 has compressed rows"
    r = comp[len(comp) // 2]
    slots = words_np(slots_t).copy()
    slots[r, :W // 32] = 0  # every word announces 32 bits: stream >= W words
    pset = ibp.ibp_plan_set_create(plans)
    out = words_np(ibp.ibp_decompress_contig_set(pset, on_device(slots), rpp, bitmask))
    assert ibp.ibp_plan_set_get_status(pset, raise_on_error=False) == ibp.IBP_ECORRUPT
    assert not out[r].any()
    keep = np.ones(len(rows), bool)
    keep[r] = False
    assert np.array_equal(out[keep], rows[keep])
    assert ibp.ibp_plan_set_get_status(pset) == ibp.IBP_OK  # cleared


def test_plan_set_rejects_bad_arguments():
    rng = np.random.default_rng(2)
    a = rng.normal(0, 1, (64, 64)).astype(np.float32).view(np.uint32)
    b = rng.normal(0, 1, (64, 128)).astype(np.float32).view(np.uint32)
    pa = ibp.ibp_plan_create(*ibp.ibp_preprocess(on_device(a), 0.9))
    pb = ibp.ibp_plan_create(*ibp.ibp_preprocess(on_device(b), 0.9))
    with pytest.raises(ibp.IbpError):
        ibp.ibp_plan_set_create([pa, pb])  # different W
    p45 = ibp.ibp_plan_create(*ibp.ibp_preprocess(on_device(a[:, :45].copy()), 0.9))
    with pytest.raises(ibp.IbpError):
        ibp.ibp_plan_set_create([p45])  # W not 32 * 2^k
    lib = ibp.load()
    h = ctypes.c_void_p()
    assert lib.ibp_plan_set_create(None, 1, ctypes.byref(h)) == ibp.IBP_EINVAL
    arr = (ctypes.c_void_p * 1)(pa.handle.value)
    assert lib.ibp_plan_set_create(arr, 0, ctypes.byref(h)) == ibp.IBP_EINVAL
    pset = ibp.ibp_plan_set_create([pa, pa])
    slots = torch.zeros((128, 64), dtype=torch.int32, device="cuda")
    bm = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros((128 * 64 + 1,), dtype=torch.int32, device="cuda")
    # unaligned output
    assert lib.ibp_decompress_contig_set(pset.handle, ctypes.c_void_p(slots.data_ptr()), 64,
                                         ctypes.c_void_p(bm.data_ptr()), ctypes.c_void_p(out.data_ptr() + 4),
                                         None) == ibp.IBP_EINVAL
    # zero rows: a no-op
    assert lib.ibp_decompress_contig_set(pset.handle, ctypes.c_void_p(slots.data_ptr()), 0,
                                         ctypes.c_void_p(bm.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                         None) == ibp.IBP_OK
    assert lib.ibp_decompress_contig_set(None, None, 1, None, None, None) == ibp.IBP_EINVAL
    assert lib.ibp_plan_set_destroy(None) == ibp.IBP_OK
