"""Stream order with programmatic dependent launch: the decoders may place
their CTAs before the previous kernel of the stream has finished, so a kernel
that writes their inputs (ids, slots, offsets) or reads their output just
before or after them must still see / produce the stream-ordered values."""

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp
from oracle import bag_ref as B
from tests.gpu_util import gpu_codec, on_device, words_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()


def _table(W=128, n=20000, seed=0):
    rng = np.random.default_rng(seed)
    rows = rng.normal(0, 0.05, (n, W)).astype(np.float32).view(np.uint32)
    return rows, gpu_codec(rows, rows[:4000], 0.9, "hbm")


def test_ids_written_by_the_previous_kernel():
    rows, g = _table()
    n = rows.shape[0]
    bm = on_device(g["bitmask"])
    ids = torch.empty(65536, dtype=torch.int64, device="cuda")
    base = torch.arange(65536, dtype=torch.int64, device="cuda")
    outs = []
    for k in range(1, 9):
        torch.remainder(base * (2 * k + 1) + 7 * k, n, out=ids)  # a kernel writes this step's ids
        outs.append(ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm, ids))
    torch.cuda.synchronize()
    b = np.arange(65536, dtype=np.int64)
    for k, out in enumerate(outs, start=1):
        assert np.array_equal(words_np(out), rows[(b * (2 * k + 1) + 7 * k) % n]), k


def test_slots_written_by_the_previous_kernel_and_output_read_by_the_next():
    rows, g = _table(seed=1)
    bm = on_device(g["bitmask"])
    ids = torch.randint(0, rows.shape[0], (30000,), dtype=torch.int64, device="cuda")
    slots = torch.zeros_like(g["slots_t"])
    out = torch.empty((30000, 128), dtype=torch.int32, device="cuda")
    checks = []
    for _ in range(4):
        slots.zero_()
        slots.copy_(g["slots_t"])  # kernels rewrite the slots just before the decode
        ibp.ibp_gather_decompress(g["plan"], slots, bm, ids, out=out)
        checks.append(out.clone())  # a kernel reads the output just after
        out.fill_(-1)
    torch.cuda.synchronize()
    want = rows[ids.cpu().numpy()]
    for c in checks:
        assert np.array_equal(words_np(c), want)


def test_stream_order_inside_a_captured_graph():
    rows, g = _table(W=64, seed=2)
    n = rows.shape[0]
    bm = on_device(g["bitmask"])
    ids = torch.empty(8192, dtype=torch.int64, device="cuda")
    base = torch.arange(8192, dtype=torch.int64, device="cuda")
    offsets = torch.arange(0, 8193, 32, dtype=torch.int64, device="cuda")
    out = torch.empty((8192, 64), dtype=torch.int32, device="cuda")
    pooled = torch.empty((256, 64), dtype=torch.float32, device="cuda")
    keep, keep_bags = [], []
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm, base, out=out)  # warm-up outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
            for k in range(1, 5):
                torch.remainder(base * (4 * k + 1) + k, n, out=ids)
                ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm, ids, out=out)
                ibp.ibp_gather_decompress_bag(g["plan"], g["slots_t"], bm, ids, offsets, out=pooled)
                keep.append(out.clone())
                keep_bags.append(pooled.clone())
        graph.replay()
    torch.cuda.synchronize()
    b = np.arange(8192, dtype=np.int64)
    for k in range(1, 5):
        want = rows[(b * (4 * k + 1) + k) % n]
        assert np.array_equal(words_np(keep[k - 1]), want), k
        st, pw = B.embedding_bag(want, offsets.cpu().numpy(), B.SUM)
        assert st == 0 and np.array_equal(keep_bags[k - 1].cpu().numpy().view(np.uint32), pw), k


@pytest.mark.parametrize("where", ["host", "hbm"])
def test_early_fetch_hint_keeps_results_when_inputs_are_ready(where):
    """IBP_HINT_EARLY_FETCH: the decoder fetches its first ids and prefixes
    while the previous kernel drains.  With inputs that no kernel just before
    writes (here: set up before the loop), the results are those of the plain
    calls, also when a kernel reads each call's output just after it and when
    calls follow one another back to back on one stream."""
    rows, g = _table(seed=3)
    g_in = gpu_codec(rows, rows[:4000], 0.9, where)
    plan, slots = g_in["plan"], g_in["slots_t"]
    bm = on_device(g_in["bitmask"])
    n = rows.shape[0]
    rng = np.random.default_rng(4)
    batches = [torch.from_numpy(rng.integers(0, n, 50000).astype(np.int64)).cuda() for _ in range(6)]
    plan.set_hints(ibp.IBP_HINT_EARLY_FETCH)
    outs, sums = [], []
    for k in range(12):
        out = ibp.ibp_gather_decompress(plan, slots, bm, batches[k % 6])
        outs.append(out)
        sums.append(out.view(torch.float32).sum(dim=1))  # a kernel reads the output just after
    contig = [ibp.ibp_decompress_contig(plan, slots, bm, 17 * k, 4000) for k in range(4)]
    offs = torch.arange(0, 50001, 50, dtype=torch.int64, device="cuda")
    bags = [ibp.ibp_gather_decompress_bag(plan, slots, bm, batches[k], offs) for k in range(3)]
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    for k, out in enumerate(outs):
        want = rows[batches[k % 6].cpu().numpy()]
        assert np.array_equal(words_np(out), want), k
        assert torch.equal(sums[k], torch.from_numpy(want.view(np.float32)).cuda().sum(dim=1))
    for k, out in enumerate(contig):
        assert np.array_equal(words_np(out), rows[17 * k:17 * k + 4000]), k
    for k, out in enumerate(bags):
        st, want = B.embedding_bag(rows[batches[k].cpu().numpy()], offs.cpu().numpy(), B.SUM)
        assert st == 0 and np.array_equal(words_np(out), want), k
    plan.set_hints(0)
    with pytest.raises(ibp.IbpError):
        plan.set_hints(4)


@pytest.mark.parametrize("where", ["host", "hbm"])
def test_status_read_after_each_call_on_the_same_stream(where):
    """ibp_get_status_async between back-to-back decodes on one stream (the
    status kernel launches as a programmatic dependent, the decodes carry the
    early-fetch hint and fill the GPU): every call's status word holds that
    call's error and no other, and the rows are right."""
    rows, g = _table(seed=5)
    g_in = gpu_codec(rows, rows[:4000], 0.9, where)
    plan, slots = g_in["plan"], g_in["slots_t"]
    bm = on_device(g_in["bitmask"])
    n = rows.shape[0]
    rng = np.random.default_rng(6)
    steps, bad_steps = 16, {3, 4, 11}
    batches = []
    for k in range(steps):
        ids = rng.integers(0, n, 50000).astype(np.int64)
        if k in bad_steps:
            ids[-1] = n + k  # the last id of the batch, decoded by the grid's last groups
        batches.append(torch.from_numpy(ids).pin_memory())
    words = torch.full((steps,), -1, dtype=torch.int32, pin_memory=True)
    plan.set_hints(ibp.IBP_HINT_EARLY_FETCH)
    outs = []
    for k in range(steps):
        outs.append(ibp.ibp_gather_decompress(plan, slots, bm, batches[k]))
        ibp.ibp_get_status_async(plan, words[k])
    torch.cuda.synchronize()
    plan.set_hints(0)
    want_words = [ibp.IBP_ERANGE if k in bad_steps else ibp.IBP_OK for k in range(steps)]
    assert words.tolist() == want_words
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    for k, out in enumerate(outs):
        ids = batches[k].numpy()
        o = words_np(out)
        good = ids < n
        assert np.array_equal(o[good], rows[ids[good]]), k
        assert not o[~good].any(), k
