"""Parity on the five workload configurations at full size.

- Mask/Bitval: the whole preprocess sample goes through both sides;
- slots and bitmask: every slot word and every bitmask word of the whole
  table is compared with the C oracle's compress of the same rows (OpenMP
  over rows; a 2 GB table takes a few seconds on the host cores);
- the oracle decodes the GPU-written slots of a few thousand sampled rows;
- gather-decompress of whole batches (the batch size and id law the
  benchmark uses), from pinned host memory and from HBM, must return the
  original rows exactly - IBP is lossless, so this holds at any size;
- the LLM configuration: every one of the 32 layers (weight, K, V).
"""

import os
import zlib

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp, workloads
from oracle import oracle_c as C
from tests.gpu_util import on_device, words_np

pytestmark = pytest.mark.gpu

N_CHECK = 4096


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()
    C.set_threads(os.cpu_count() or 1)


def _bits_at(bitmask: np.ndarray, ids: np.ndarray) -> np.ndarray:
    return ((bitmask[ids >> 5] >> (ids & 31).astype(np.uint32)) & 1).astype(np.uint8)


def _check_table(name, rows_t, rows, T, sample, batches, contig=None):
    n, W = rows.shape
    mask, bitval = ibp.ibp_preprocess(on_device(sample), T)
    st, m, b = C.preprocess(sample, T)
    torch.cuda.synchronize()
    assert st == 0
    assert np.array_equal(words_np(mask), m), f"{name}: Mask"
    assert np.array_equal(words_np(bitval), b), f"{name}: Bitval"
    plan = ibp.ibp_plan_create(mask, bitval)

    slots_t = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
    _, bitmask_t, stored_t = ibp.ibp_compress(plan, rows_t, slots_t)
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    slots = words_np(slots_t)
    bitmask = words_np(bitmask_t)
    if n % 32:
        assert (int(bitmask[-1]) >> (n % 32)) == 0, f"{name}: bitmask tail bits"

    want_slots, want_bitmask, want_stored = C.compress(rows, m, b)
    assert np.array_equal(bitmask, want_bitmask), f"{name}: bitmask words"
    assert int(stored_t.item()) == want_stored, f"{name}: stored words"
    if not np.array_equal(slots, want_slots):
        bad = np.nonzero((slots != want_slots).any(axis=1))[0]
        raise AssertionError(f"{name}: {len(bad)} slots differ from the oracle, first rows {bad[:8].tolist()}")
    del want_slots
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    chk = np.unique(np.concatenate([rng.choice(n, min(n, N_CHECK), replace=False), [0, n - 1]]))
    st, dec = C.decode_slots(slots[chk], _bits_at(bitmask, chk), m, b)
    assert st == 0 and np.array_equal(dec, rows[chk]), f"{name}: oracle decode of GPU slots"

    saving = 1.0 - int(stored_t.item()) / float(n * W)
    slots_d = slots_t.cuda()
    for ids in batches:
        ids_t = torch.from_numpy(ids).cuda()
        want = rows[ids]
        for src in (slots_t, slots_d):
            out = ibp.ibp_gather_decompress(plan, src, bitmask_t, ids_t)
            torch.cuda.synchronize()
            assert ibp.ibp_get_status(plan) == ibp.IBP_OK
            assert np.array_equal(words_np(out), want), f"{name}: batch round trip"
    if contig is not None:
        first, cnt = contig
        for src in (slots_t, slots_d):
            out = ibp.ibp_decompress_contig(plan, src, bitmask_t, first, cnt)
            torch.cuda.synchronize()
            assert np.array_equal(words_np(out), rows[first:first + cnt]), f"{name}: contig"
    del slots_d
    return saving


@pytest.mark.parametrize("name", ["dense_gnn", "sparse_gnn", "dlrm"])
def test_full_size_table(name):
    c = workloads.CONFIGS[name]
    n, W = c["n_rows"], c["W"]
    rows_t = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
    rows = rows_t.numpy().view(np.uint32)
    workloads.make_table(name, out=rows)
    sample = rows[workloads.sample_ids(n, c["sample"], c["sample_seed"])]
    zipf = workloads.ZipfIds(n, c["zipf_s"], c["seed"]) if name == "dlrm" else None
    batches = [workloads.batch_ids(name, k, zipf=zipf) for k in range(2)]
    saving = _check_table(name, rows_t, rows, c["T"], sample, batches,
                          contig=(n // 3, min(n - n // 3, 100_000)))
    print(f"{name}: space saving {100 * saving:.2f} %")
    assert 0.0 <= saving < 1.0


@pytest.mark.parametrize("layer", range(32))
def test_llm_layer(layer):
    c = workloads.CONFIGS["llm"]
    wt = workloads.llm_weight(layer)
    kv = workloads.llm_kv(layer)
    for name, tab in (("weight", wt), ("K", kv[0]), ("V", kv[1])):
        n, W = tab.shape
        rows_t = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
        rows = rows_t.numpy().view(np.uint32)
        rows[...] = tab
        sample = rows[workloads.sample_ids(n, c["sample"], c["sample_seed"] + layer)]
        saving = _check_table(f"llm[{layer}].{name}", rows_t, rows, c["T"], sample, [],
                              contig=(0, n))
        print(f"llm layer {layer} {name}: space saving {100 * saving:.2f} %")
