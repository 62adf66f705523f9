"""Seeded random cases over the decoder instantiations: widths (every
specialised segment count and odd widths for the general kernel), Mask shapes
(uniform, few popcounts, many runs), match rates, raw rows, slots in host
memory or HBM, the row-reuse hint and tuned prefixes.  Slots and bitmask are
compared with the C oracle; gather, contiguous and pooled results must give
back the rows (IBP is lossless) or the pooling oracle's bits."""

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp
from oracle import bag_ref as B
from oracle import oracle_c as C
from tests.gpu_util import on_device, place, words_np

pytestmark = pytest.mark.gpu

WIDTHS = [32, 64, 128, 256, 512, 1024, 2048, 3, 40, 100, 300]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()
    C.set_threads(8)


def _run_mask(lo, length):
    return ((1 << length) - 1) << lo


def _keep(rng, W, shape):
    if shape == "uniform":
        lo = int(rng.integers(0, 8))
        return np.full(W, _run_mask(lo, int(rng.integers(1, 32 - lo))) | _run_mask(30, 2), np.uint64)
    if shape == "two_popcounts":
        a, b = _run_mask(0, 20), _run_mask(0, 9) | _run_mask(28, 4)
        return np.array([a if rng.random() < 0.7 else b for _ in range(W)], np.uint64)
    if shape == "full_and_kept":  # some positions keep nothing (empty fields)
        return np.array([0 if rng.random() < 0.3 else _run_mask(2, 11) for _ in range(W)], np.uint64)
    # up to four runs, random per position
    out = []
    for _ in range(W):
        k, pos = 0, 0
        for _ in range(int(rng.integers(1, 5))):
            pos += int(rng.integers(0, 4))
            ln = int(rng.integers(1, 5))
            if pos + ln > 32:
                break
            k |= _run_mask(pos, ln)
            pos += ln + 1
        out.append(k or 1)
    return np.array(out, np.uint64)


def _case(seed):
    rng = np.random.default_rng(seed)
    W = int(rng.choice(WIDTHS))
    shape = str(rng.choice(["uniform", "two_popcounts", "full_and_kept", "runs"]))
    keep = _keep(rng, W, shape)
    mask = (~keep & 0xFFFFFFFF).astype(np.uint32)
    if shape == "uniform":
        bitval = np.full(W, rng.integers(0, 2**32, dtype=np.uint64), np.uint64).astype(np.uint32) & mask
    else:
        bitval = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32) & mask
    n = int(rng.integers(33, max(34, 200_000 // W)))
    rows = rng.integers(0, 2**32, (n, W), dtype=np.uint64).astype(np.uint32)
    match = rng.random((n, W)) < rng.uniform(0.6, 0.99)
    rows = np.where(match, (rows & ~mask) | (bitval & mask), rows).astype(np.uint32)
    rows[rng.random(n) < 0.05] = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32)  # raw rows
    return rng, W, shape, mask, bitval, rows


@pytest.mark.parametrize("seed", range(48))
def test_fuzz_decoders(seed):
    rng, W, shape, mask, bitval, rows = _case(seed)
    n = rows.shape[0]
    where = "host" if seed % 2 else "hbm"
    plan = ibp.ibp_plan_create(torch.from_numpy(mask.view(np.int32)), torch.from_numpy(bitval.view(np.int32)))
    if seed % 3 == 0:
        plan.set_hints(ibp.IBP_HINT_ROW_REUSE)
    rows_t = place(rows, where)
    slots_t = torch.empty_like(rows_t)
    if where == "host":
        slots_t = slots_t.pin_memory()
    _, bitmask, stored = ibp.ibp_compress(plan, rows_t, slots_t)
    torch.cuda.synchronize()
    cs, cb, cst = C.compress(rows, mask, bitval)
    assert np.array_equal(words_np(slots_t), cs) and np.array_equal(words_np(bitmask), cb)
    assert int(stored.item()) == cst
    if seed % 4 == 1:
        ibp.ibp_plan_tune_prefix(plan, slots_t, bitmask)
    hot = rng.integers(0, n, 5)
    ids = np.where(rng.random(3 * n) < 0.3, hot[rng.integers(0, 5, 3 * n)], rng.integers(0, n, 3 * n)).astype(np.int64)
    ids_t = torch.from_numpy(ids).cuda()
    out = ibp.ibp_gather_decompress(plan, slots_t, bitmask, ids_t)
    first = int(rng.integers(0, n // 2))
    contig = ibp.ibp_decompress_contig(plan, slots_t, bitmask, first, n - first)
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK, (W, shape, where)
    assert np.array_equal(words_np(out), rows[ids]), (W, shape, where)
    assert np.array_equal(words_np(contig), rows[first:]), (W, shape, where)
    # pooled bags where the fused kernel applies (W = 32 * 2^k <= 512, <= 4 runs)
    if W in (32, 64, 128, 256, 512) and plan.info["max_runs"] <= 4 and plan.info["max_runs"] >= 1:
        sizes = rng.integers(0, 40, 60)
        offsets = np.minimum(np.concatenate([[0], np.cumsum(sizes)]), len(ids)).astype(np.int64)
        mode = ibp.IBP_BAG_MEAN if seed % 5 == 0 else ibp.IBP_BAG_SUM
        bf16 = seed % 7 == 0
        pooled = ibp.ibp_gather_decompress_bag(plan, slots_t, bitmask, ids_t, torch.from_numpy(offsets).cuda(),
                                               mode | (ibp.IBP_BAG_BF16 if bf16 else 0))
        assert ibp.ibp_get_status(plan) == ibp.IBP_OK
        _, want = B.embedding_bag(rows[ids], offsets, mode, bf16=bf16)
        got = pooled.cpu().numpy()
        nan = np.isnan(got) | np.isnan(want.view(np.float32))
        assert np.array_equal(np.isnan(got), np.isnan(want.view(np.float32)))
        assert np.array_equal(got.view(np.uint32)[~nan], want[~nan]), (W, shape, where, mode, bf16)
