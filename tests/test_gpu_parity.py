"""Bit-exact parity of the CUDA path with the CPU oracle.

Small cases are compared whole (Mask/Bitval, every slot word, the bitmask,
the stored-word count, every decoded word); they span several warps and
groups, ragged segments and ragged row counts.  Edge cases: empty calls,
one-word rows, widths that are not multiples of 4 or 32 (the 4-byte path),
unaligned buffers, masks of 0 and of all ones, random masks (five-step
expand path), per-word masks (table path), special floats, repeated and
out-of-range ids, corrupt slots.
"""

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp, workloads
from oracle import oracle_c as C
from tests.gpu_util import empty_like_in, gpu_codec, on_device, pinned, place, words_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_transfer_gb300 import build

    build.build()
    ibp.load()
    C.set_threads(8)


def _check_codec(rows, sample, T, where, inplace=False):
    """Full comparison of preprocess + compress + decompress with the oracle."""
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    g = gpu_codec(rows, sample, T, where, inplace)
    st, m, b = C.preprocess(sample, T)
    assert st == 0
    assert np.array_equal(g["mask"], m), "Mask differs from the oracle"
    assert np.array_equal(g["bitval"], b), "Bitval differs from the oracle"
    slots, bitmask, stored = C.compress(rows, m, b)
    assert np.array_equal(words_np(g["slots_t"]), slots), "slots differ from the oracle"
    assert np.array_equal(g["bitmask"], bitmask), "bitmask differs from the oracle"
    assert g["stored"] == stored
    # gather every row in a shuffled order with repeats
    n = rows.shape[0]
    rng = np.random.default_rng(n)
    ids = np.concatenate([rng.permutation(n), rng.integers(0, n, n // 3 + 1)]).astype(np.int64)
    ids_t = torch.from_numpy(ids).cuda()
    bm_t = on_device(g["bitmask"])
    out = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm_t, ids_t)
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows[ids])
    return g, ids


@pytest.mark.parametrize("where", ["host", "hbm"])
def test_tiny_config_full_parity(where):
    c = workloads.CONFIGS["tiny"]
    rows = workloads.make_table("tiny")
    sample = rows[workloads.sample_ids(c["n_rows"], c["sample"], c["sample_seed"])]
    g, _ = _check_codec(rows, sample, c["T"], where)
    # contiguous decompress of a ragged middle range
    bm_t = on_device(g["bitmask"])
    out = ibp.ibp_decompress_contig(g["plan"], g["slots_t"], bm_t, 37, 1500)
    torch.cuda.synchronize()
    assert np.array_equal(words_np(out), rows[37:1537])
    info = g["plan"].info
    assert info["W"] == 128 and info["segments"] == 4


def test_tiny_config_in_place_compress():
    c = workloads.CONFIGS["tiny"]
    rows = workloads.make_table("tiny")
    sample = rows[workloads.sample_ids(c["n_rows"], c["sample"], c["sample_seed"])]
    g = gpu_codec(rows, sample, c["T"], "host", inplace=True)
    slots, bitmask, stored = C.compress(rows, g["mask"], g["bitval"])
    assert np.array_equal(words_np(g["slots_t"]), slots)
    assert np.array_equal(g["bitmask"], bitmask)


def _float_rows(rng, n, W, scale=0.05):
    return rng.normal(0, scale, (n, W)).astype(np.float32).view(np.uint32)


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8, 31, 32, 33, 63, 64, 100, 127, 128, 129, 255, 256,
                               257, 512, 1000, 1024, 2048, 4096, 8192])
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_widths_learned_masks(W, where):
    rng = np.random.default_rng(W)
    n = max(33, min(700, 200_000 // W))
    rows = _float_rows(rng, n, W)
    rows[::9] = rng.integers(0, 2**32, (len(rows[::9]), W), dtype=np.uint64).astype(np.uint32)
    _check_codec(rows, rows[: max(1, n // 2)], 0.9, where)


@pytest.mark.parametrize("W", [4, 33, 128, 300])
def test_per_word_masks_table_path(W):
    """Columns with different scales give different Masks per word position."""
    rng = np.random.default_rng(100 + W)
    scale = np.exp(rng.uniform(-8, 3, W))
    x = (rng.normal(0, 1, (400, W)) * scale).astype(np.float32)
    x[:, ::3] = np.abs(x[:, ::3])
    rows = x.view(np.uint32)
    g, _ = _check_codec(rows, rows[:300], 0.97, "hbm")
    assert g["plan"].info["uniform"] == 0


@pytest.mark.parametrize("W", [7, 64, 160])
@pytest.mark.parametrize("runs", ["many", "few"])
def test_random_masks(W, runs):
    """Arbitrary Mask/Bitval (up to 16 runs of kept bits: five-step path)."""
    rng = np.random.default_rng(W)
    n = 300
    if runs == "many":
        base = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32)
    else:
        base = np.full(W, 0x3F800000, np.uint32)
    rows = rng.integers(0, 2**32, (n, W), dtype=np.uint64).astype(np.uint32)
    keepers = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32)
    if runs == "few":
        keepers = np.full(W, 0x807F00FF, np.uint32)
    # most rows agree with base outside `keepers`
    agree = rng.random(n) < 0.8
    rows[agree] = (rows[agree] & keepers) | (base & ~keepers)
    g, _ = _check_codec(rows, rows[:200], 0.75, "hbm")
    if runs == "many":
        assert g["plan"].info["max_runs"] > 4


@pytest.mark.parametrize("W", [32, 64, 512])
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_mask_zero_all_raw(where, W):
    """Sample rows that agree on nothing leave the Mask empty: every row raw
    (whole groups of raw rows are copied in one piece, the last partial group
    row by row)."""
    rows = np.random.default_rng(1).integers(0, 2**32, (101, W), dtype=np.uint64).astype(np.uint32)
    sample = np.stack([np.zeros(W, np.uint32), np.full(W, 0xFFFFFFFF, np.uint32)])
    g, _ = _check_codec(rows, sample, 1.0, where)
    assert not g["bitmask"].any() and g["plan"].info["max_kept_bits"] == 32


@pytest.mark.parametrize("W", [1, 6, 32, 33, 200])
def test_full_mask_headers_only(W):
    bv = (np.arange(W, dtype=np.uint64) * 2654435761 % 2**32).astype(np.uint32)
    rows = np.tile(bv, (70, 1))
    rows[5, 0] ^= 1  # one row breaks one word
    g, _ = _check_codec(rows, np.tile(bv, (3, 1)), 1.0, "hbm")
    S = (W + 31) // 32
    if W > 1:
        assert g["stored"] == 69 * S + min(W, S + 1)


def test_special_floats_round_trip():
    rng = np.random.default_rng(5)
    W = 96
    vals = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 1e-45, -1e-40, 3.4e38, 1.0, -2.5],
                    np.float32).view(np.uint32)
    rows = _float_rows(rng, 500, W)
    rows[::7, ::5] = vals[rng.integers(0, len(vals), rows[::7, ::5].shape)]
    rows[3, :] = vals[rng.integers(0, len(vals), W)]
    _check_codec(rows, rows, 0.95, "host")


def test_bf16_pairs_round_trip():
    rng = np.random.default_rng(6)
    x = rng.normal(0, 0.02, (300, 256)).astype(np.float32)
    rows = workloads.bf16_pairs_to_words(workloads.f32_to_bf16_bits(x))
    _check_codec(rows, rows[:128], 0.99, "host")


def test_unaligned_buffers_take_the_word_path():
    """Slots and outputs offset by one word are not 16-byte aligned."""
    rng = np.random.default_rng(7)
    W, n = 128, 300
    rows = _float_rows(rng, n, W)
    s = on_device(rows[:200])
    mask, bitval = ibp.ibp_preprocess(s, 0.95)
    plan = ibp.ibp_plan_create(mask, bitval)
    buf = torch.empty(n * W + 1, dtype=torch.int32, pin_memory=True)
    buf[1:].numpy()[...] = rows.reshape(-1).view(np.int32)
    rows_t = buf[1:].view(n, W)
    sbuf = torch.empty(n * W + 1, dtype=torch.int32, pin_memory=True)
    slots_t = sbuf[1:].view(n, W)
    _, bitmask, stored = ibp.ibp_compress(plan, rows_t, slots_t)
    obuf = torch.empty(n * W + 1, dtype=torch.int32, device="cuda")
    out = obuf[1:].view(n, W)
    ids = torch.arange(n - 1, -1, -1, dtype=torch.int64, device="cuda")
    ibp.ibp_gather_decompress(plan, slots_t, bitmask, ids, out=out)
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    ms, mb = words_np(mask), words_np(bitval)
    cs, cb, _ = C.compress(rows, ms, mb)
    assert np.array_equal(words_np(slots_t), cs) and np.array_equal(words_np(bitmask), cb)
    assert np.array_equal(words_np(out), rows[::-1])


def test_decoder_on_oracle_slots():
    """The decoder alone, on slots the oracle wrote."""
    rng = np.random.default_rng(8)
    for W in (16, 128, 129, 600):
        rows = _float_rows(rng, 257, W, scale=1e-3)
        _, m, b = C.preprocess(rows[:100], 0.99)
        slots, bitmask, _ = C.compress(rows, m, b)
        plan = ibp.ibp_plan_create(torch.from_numpy(m.view(np.int32)), torch.from_numpy(b.view(np.int32)))
        for where in ("host", "hbm"):
            st = place(slots, where)
            ids = torch.from_numpy(rng.integers(0, 257, 999)).cuda()
            out = ibp.ibp_gather_decompress(plan, st, on_device(bitmask), ids)
            torch.cuda.synchronize()
            assert ibp.ibp_get_status(plan) == ibp.IBP_OK
            assert np.array_equal(words_np(out), rows[ids.cpu().numpy()])


def test_empty_calls_are_no_ops():
    rows = np.zeros((4, 8), np.uint32)
    g = gpu_codec(rows, rows, 0.9, "hbm")
    plan = g["plan"]
    empty_ids = torch.empty(0, dtype=torch.int64, device="cuda")
    out = ibp.ibp_gather_decompress(plan, g["slots_t"], on_device(g["bitmask"]), empty_ids)
    assert out.shape == (0, 8)
    out = ibp.ibp_decompress_contig(plan, g["slots_t"], on_device(g["bitmask"]), 0, 0)
    assert out.shape == (0, 8)
    _, bm, st = ibp.ibp_compress(plan, torch.empty((0, 8), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK


def test_out_of_range_ids_give_zero_rows_and_erange():
    c = workloads.CONFIGS["tiny"]
    rows = workloads.make_table("tiny")
    g = gpu_codec(rows, rows[:256], c["T"], "hbm")
    n = rows.shape[0]
    ids = np.array([0, n, -1, 5, 2**40, n - 1, -(2**62)], np.int64)
    out = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                                    torch.from_numpy(ids).cuda())
    code = ibp.ibp_get_status(g["plan"], raise_on_error=False)
    assert code == ibp.IBP_ERANGE
    o = words_np(out)
    assert np.array_equal(o[[0, 3, 5]], rows[[0, 5, n - 1]])
    assert not o[[1, 2, 4, 6]].any()
    st, ref = C.decompress(words_np(g["slots_t"]), g["bitmask"], ids, g["mask"], g["bitval"])
    assert st == ibp.IBP_ERANGE and np.array_equal(o, ref)
    # the status was cleared by the read
    assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK


@pytest.mark.parametrize("W", [40, 128])
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_corrupt_slots_give_zero_rows_and_ecorrupt(W, where):
    rng = np.random.default_rng(9)
    rows = _float_rows(rng, 64, W)
    g = gpu_codec(rows, rows, 0.9, "host")
    assert g["bitmask"][0] & 0b111 == 0b111
    slots = words_np(g["slots_t"]).copy()
    S = (W + 31) // 32
    slots[0, :S] = 0  # every word announces 32 bits: stream >= W words
    if W % 32:
        slots[1, S - 1] |= 1 << 31  # header bit past the last word
    bad = place(slots, where)
    ids = np.arange(4, dtype=np.int64)
    out = ibp.ibp_gather_decompress(g["plan"], bad, on_device(g["bitmask"]), torch.from_numpy(ids).cuda())
    code = ibp.ibp_get_status(g["plan"], raise_on_error=False)
    assert code == ibp.IBP_ECORRUPT
    o = words_np(out)
    st, ref = C.decompress(slots, g["bitmask"], ids, g["mask"], g["bitval"])
    assert st == ibp.IBP_ECORRUPT and np.array_equal(o, ref)
    assert not o[0].any() and np.array_equal(o[2:], rows[2:4])


def test_preprocess_edge_cases():
    rng = np.random.default_rng(10)
    cases = [
        (rng.integers(0, 2**32, (1, 37), dtype=np.uint64).astype(np.uint32), 1.0),
        (np.array([[0x0F0F0F0F, 1], [0xF0F0F0F0, 1]], np.uint32), 0.5),
        (np.array([[1], [1], [1], [0]], np.uint32), 0.75),
        (np.array([[1], [1], [1], [0]], np.uint32), 0.76),
        (rng.integers(0, 2**32, (4097, 33), dtype=np.uint64).astype(np.uint32), 0.5),
        (_float_rows(rng, 5000, 1000), 0.999),
    ]
    for sample, T in cases:
        for where in ("host", "hbm"):
            s = place(sample, where)
            m, b = ibp.ibp_preprocess(s, T)
            torch.cuda.synchronize()
            st, rm, rb = C.preprocess(sample, T)
            assert np.array_equal(words_np(m), rm) and np.array_equal(words_np(b), rb)


def test_preprocess_rejects_bad_arguments():
    s = torch.zeros((4, 4), dtype=torch.int32, device="cuda")
    for T in (0.0, -1.0, 1.5, float("nan")):
        with pytest.raises(ibp.IbpError):
            ibp.ibp_preprocess(s, T)
    pageable = torch.zeros((4, 4), dtype=torch.int32)
    with pytest.raises(ibp.IbpError):
        ibp.ibp_preprocess(pageable, 0.9)


def test_gather_raw_matches_rows():
    rng = np.random.default_rng(11)
    for W in (3, 64, 128):
        rows = rng.integers(0, 2**32, (1000, W), dtype=np.uint64).astype(np.uint32)
        ids = rng.integers(-5, 1005, 3000).astype(np.int64)
        for where in ("host", "hbm"):
            out = ibp.ibp_gather_raw(place(rows, where), torch.from_numpy(ids).cuda())
            torch.cuda.synchronize()
            want = np.where(((ids >= 0) & (ids < 1000))[:, None], rows[np.clip(ids, 0, 999)], 0)
            assert np.array_equal(words_np(out), want)


def test_streams_and_repeated_calls_agree():
    """Two plans on two streams, calls repeated: identical results."""
    c = workloads.CONFIGS["tiny"]
    rows = workloads.make_table("tiny")
    g = gpu_codec(rows, rows[:256], c["T"], "host")
    bm_t = on_device(g["bitmask"])
    ids = torch.from_numpy(np.random.default_rng(3).integers(0, 2048, 4096)).cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for s in (s1, s2, s1):
        with torch.cuda.stream(s):
            outs.append(ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm_t, ids, stream=s))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, outs[0])
    assert np.array_equal(words_np(outs[0]), rows[ids.cpu().numpy()])


@pytest.mark.parametrize("W", [5, 64, 128, 300])
def test_row_lengths_match_oracle_stored_words(W):
    rng = np.random.default_rng(12 + W)
    rows = _float_rows(rng, 200, W)
    rows[::11] = rng.integers(0, 2**32, (len(rows[::11]), W), dtype=np.uint64).astype(np.uint32)
    g = gpu_codec(rows, rows[:100], 0.9, "host")
    ids = np.concatenate([np.arange(200), [-1, 200, 7]]).astype(np.int64)
    lens = ibp.ibp_row_lengths(g["plan"], g["slots_t"], on_device(g["bitmask"]),
                               torch.from_numpy(ids).cuda())
    code = ibp.ibp_get_status(g["plan"], raise_on_error=False)
    assert code == ibp.IBP_ERANGE
    want = [C.compress(rows[i:i + 1], g["mask"], g["bitval"])[2] for i in range(200)]
    got = lens.cpu().numpy()
    assert got[:200].tolist() == want
    assert got[200] == 0 and got[201] == 0 and got[202] == want[7]


def _explicit_plan_check(mask, bitval, rows, where="hbm", hints=0):
    """Compress + gather with an explicit Mask/Bitval; compare with the oracle."""
    plan = ibp.ibp_plan_create(torch.from_numpy(mask.view(np.int32)), torch.from_numpy(bitval.view(np.int32)))
    plan.set_hints(hints)
    rows_t = place(rows, where)
    slots_t = empty_like_in(rows_t, where)
    _, bitmask, stored = ibp.ibp_compress(plan, rows_t, slots_t)
    n = rows.shape[0]
    ids = np.random.default_rng(n).integers(0, n, 3 * n).astype(np.int64)
    out = ibp.ibp_gather_decompress(plan, slots_t, bitmask, torch.from_numpy(ids).cuda())
    contig = ibp.ibp_decompress_contig(plan, slots_t, bitmask, 3, n - 5)
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    cs, cb, cst = C.compress(rows, mask, bitval)
    assert np.array_equal(words_np(slots_t), cs) and np.array_equal(words_np(bitmask), cb)
    assert int(stored.item()) == cst
    assert np.array_equal(words_np(out), rows[ids])
    assert np.array_equal(words_np(contig), rows[3:n - 2])
    return plan


def _rows_for(mask, bitval, rng, n, p_match=0.85):
    W = mask.size
    rows = rng.integers(0, 2**32, (n, W), dtype=np.uint64).astype(np.uint32)
    match = rng.random((n, W)) < p_match
    rows = np.where(match, (rows & ~mask) | (bitval & mask), rows).astype(np.uint32)
    return rows


def _run_mask(lo, length):
    return ((1 << length) - 1) << lo


@pytest.mark.parametrize("W", [32, 64, 128, 512, 1024])
@pytest.mark.parametrize("kind", ["same_popcount", "two_popcounts", "many_popcounts", "up_to_4_runs"])
def test_per_word_plans_fast_table_modes(W, kind):
    """Per-word Masks of the shapes the table kernel specialises for: the same
    popcount at different positions (no e-plane), two popcounts (one e-plane),
    many popcounts (six e-planes), and up to four runs of kept bits.  W = 32
    decodes one word per lane; wider rows two words per lane (64-word blocks);
    W = 1024 from device slots as two tasks of 16 segments."""
    rng = np.random.default_rng(W + len(kind))
    keep = np.zeros(W, np.uint64)
    for w in range(W):
        if kind == "same_popcount":
            keep[w] = _run_mask(w % 20, 8)  # 8 kept bits, shifting position
        elif kind == "two_popcounts":
            keep[w] = _run_mask(0, 27) | (1 << 31) if w % 3 else _run_mask(26, 4)
        elif kind == "many_popcounts":
            keep[w] = _run_mask(w % 7, 1 + (w * 5) % 30)
        else:
            keep[w] = _run_mask(0, 3) | _run_mask(6, 2) | _run_mask(12, 5) | _run_mask(24, 1 + w % 7)
    mask = (~keep & 0xFFFFFFFF).astype(np.uint32)
    bitval = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32) & mask
    rows = _rows_for(mask, bitval, rng, 700)
    rows[::13] = rng.integers(0, 2**32, (len(rows[::13]), W), dtype=np.uint64).astype(np.uint32)
    plan = _explicit_plan_check(mask, bitval, rows, "hbm")
    _explicit_plan_check(mask, bitval, rows[:200], "host")
    assert plan.info["uniform"] == 0
    if kind == "up_to_4_runs":
        assert plan.info["max_runs"] == 4


@pytest.mark.parametrize("where", ["host", "hbm"])
def test_row_reuse_hint_same_results(where):
    """IBP_HINT_ROW_REUSE changes the cache policy of the row copies only."""
    c = workloads.CONFIGS["tiny"]
    rows = workloads.make_table("tiny")
    g = gpu_codec(rows, rows[:256], c["T"], where)
    rng = np.random.default_rng(21)
    hot = rng.integers(0, len(rows), 5)
    ids = np.where(rng.random(6000) < 0.7, hot[rng.integers(0, 5, 6000)], rng.integers(0, len(rows), 6000))
    ids_t = torch.from_numpy(ids.astype(np.int64)).cuda()
    bm_t = on_device(g["bitmask"])
    plain = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm_t, ids_t)
    g["plan"].set_hints(ibp.IBP_HINT_ROW_REUSE)
    hinted = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm_t, ids_t)
    torch.cuda.synchronize()
    assert torch.equal(plain, hinted)
    assert np.array_equal(words_np(hinted), rows[ids])
    with pytest.raises(ibp.IbpError):
        g["plan"].set_hints(4)  # no such hint


@pytest.mark.parametrize("W", [32, 64, 128, 256, 512, 2048])
@pytest.mark.parametrize("kind", ["uniform", "two_popcounts", "up_to_4_runs"])
def test_row_reuse_hint_from_host_memory(W, kind):
    """Row-reuse copies from host-mapped slots take kernels with smaller
    groups; uniform and per-word plans, every segment count."""
    rng = np.random.default_rng(3 * W + len(kind))
    if kind == "uniform":
        keep = np.full(W, _run_mask(0, 9) | _run_mask(23, 3), np.uint64)
    elif kind == "two_popcounts":
        keep = np.array([_run_mask(0, 27) | (1 << 31) if w % 3 else _run_mask(26, 4) for w in range(W)], np.uint64)
    else:
        keep = np.array([_run_mask(0, 3) | _run_mask(6, 2) | _run_mask(12, 5) | _run_mask(24, 1 + w % 7)
                         for w in range(W)], np.uint64)
    mask = (~keep & 0xFFFFFFFF).astype(np.uint32)
    bitval = rng.integers(0, 2**32, 1 if kind == "uniform" else W, dtype=np.uint64).astype(np.uint32)
    bitval = np.broadcast_to(bitval, (W,)) & mask
    n = max(40, min(900, 300_000 // W))
    rows = _rows_for(mask, bitval, rng, n)
    rows[::11] = rng.integers(0, 2**32, (len(rows[::11]), W), dtype=np.uint64).astype(np.uint32)
    plan = _explicit_plan_check(mask, bitval, rows, "host", hints=ibp.IBP_HINT_ROW_REUSE)
    assert plan.info["uniform"] == (kind == "uniform")


@pytest.mark.parametrize("W", [32, 512])
def test_hbm_long_batches(W):
    """Batches from HBM long enough that every decoding warp cycles through
    its shared-memory stages many times, with a ragged last group."""
    rng = np.random.default_rng(7 * W)
    n = (3 << 21) // W + 13
    rows = _float_rows(rng, n, W)
    rows[::7] = rng.integers(0, 2**32, (len(rows[::7]), W), dtype=np.uint64).astype(np.uint32)
    g, _ = _check_codec(rows, rows[:4096], 0.9, "hbm")
    bm_t = on_device(g["bitmask"])
    ids = rng.integers(0, n, 4 * n + 5).astype(np.int64)
    out = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm_t, torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows[ids])
    out = ibp.ibp_decompress_contig(g["plan"], g["slots_t"], bm_t, 3, n - 4)
    torch.cuda.synchronize()
    assert np.array_equal(words_np(out), rows[3:n - 1])


@pytest.mark.parametrize("W", [1024, 2048])
@pytest.mark.parametrize("shape", ["learned", "per_word"])
def test_wide_rows_in_hbm_split_into_tasks(W, shape):
    """Rows of 32 or 64 segments with slots in HBM are decoded as two tasks per
    row (of 16 or 32 segments), each from its row's headers and its own slice
    of the stream:
    compressed, raw, corrupt rows and bad ids, gathered and contiguous, all
    equal to the oracle's decode of the same slots."""
    rng = np.random.default_rng(W + len(shape))
    n = 300
    rows = _float_rows(rng, n, W)
    if shape == "learned":
        g = gpu_codec(rows, rows[:200], 0.9, "hbm")
    else:  # two Masks alternating by word position (per-word tables), W <= 1024
        if W > 1024:
            pytest.skip("per-word tables take W <= 1024")
        mask = np.where(np.arange(W) % 2 == 0, 0xFF800000, 0xFFF00000).astype(np.uint32)
        bitval = (rows[0] & mask).astype(np.uint32)
        match = rng.random((n, 1)) < 0.8
        rows = np.where(match, (rows & ~mask) | (bitval & mask), rows).astype(np.uint32)
        plan = _explicit_plan_check(mask, bitval, rows, "hbm")
        g = dict(plan=plan, mask=mask, bitval=bitval)
        rows_t = on_device(rows)
        slots_t = torch.empty_like(rows_t)
        _, bm, _ = ibp.ibp_compress(plan, rows_t, slots_t)
        torch.cuda.synchronize()
        g["slots_t"], g["bitmask"] = slots_t, words_np(bm)
    slots = words_np(g["slots_t"]).copy()
    comp = np.nonzero((g["bitmask"][np.arange(n) >> 5] >> (np.arange(n) & 31).astype(np.uint32)) & 1)[0]
    assert len(comp) > 10
    raw_rows = np.setdiff1d(np.arange(n), comp)
    slots[comp[1], :W // 32] = 0  # every word announced raw: stream >= W words
    dev_slots = on_device(slots)
    ids = np.concatenate([rng.integers(0, n, 500), [comp[1], -1, n, n + 7, comp[0]],
                          raw_rows[:3] if len(raw_rows) else []]).astype(np.int64)
    out = ibp.ibp_gather_decompress(g["plan"], dev_slots, on_device(g["bitmask"]), torch.from_numpy(ids).cuda())
    code = ibp.ibp_get_status(g["plan"], raise_on_error=False)
    st, ref = C.decompress(slots, g["bitmask"], ids, g["mask"], g["bitval"])
    # both kinds of error occur: which one a concurrent kernel records first is
    # not fixed, the rows are
    assert code in (ibp.IBP_ERANGE, ibp.IBP_ECORRUPT) and st in (ibp.IBP_ERANGE, ibp.IBP_ECORRUPT)
    assert np.array_equal(words_np(out), ref)
    ok = np.setdiff1d(np.arange(n), [comp[1]])
    out = ibp.ibp_decompress_contig(g["plan"], dev_slots, on_device(g["bitmask"]), int(ok[0]), n - int(ok[0]))
    code = ibp.ibp_get_status(g["plan"], raise_on_error=False)
    st, ref = C.decompress(slots, g["bitmask"], np.arange(int(ok[0]), n), g["mask"], g["bitval"])
    assert code == st and np.array_equal(words_np(out), ref)


@pytest.mark.parametrize("where", ["host", "hbm"])
def test_ids_and_status_word_in_pinned_host_memory(where):
    """Row ids read by the kernel from pinned host memory (zero copy) give the
    same rows as device ids, and ibp_get_status_async moves each call's status
    into a pinned host word without a host wait: OK for a clean call, the data
    error for a call with a bad id, cleared after it is moved."""
    c = workloads.CONFIGS["tiny"]
    rows = workloads.make_table("tiny")
    g = gpu_codec(rows, rows[:256], c["T"], where)
    bm = on_device(g["bitmask"])
    n = rows.shape[0]
    rng = np.random.default_rng(12)
    ids = rng.integers(0, n, 5000).astype(np.int64)
    ids_host = torch.from_numpy(ids).pin_memory()
    words = torch.full((3,), -1, dtype=torch.int32, pin_memory=True)
    out = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm, ids_host)
    ibp.ibp_get_status_async(g["plan"], words[0])
    bad = torch.from_numpy(np.array([1, n + 3, 2], np.int64)).pin_memory()
    out_bad = ibp.ibp_gather_decompress(g["plan"], g["slots_t"], bm, bad)
    ibp.ibp_get_status_async(g["plan"], words[1])
    ibp.ibp_get_status_async(g["plan"], words[2])
    torch.cuda.synchronize()
    assert words.tolist() == [ibp.IBP_OK, ibp.IBP_ERANGE, ibp.IBP_OK]
    assert np.array_equal(words_np(out), rows[ids])
    o = words_np(out_bad)
    assert np.array_equal(o[[0, 2]], rows[[1, 2]]) and not o[1].any()
    assert ibp.ibp_get_status(g["plan"]) == ibp.IBP_OK
    # a device word works too
    dword = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ibp.ibp_get_status_async(g["plan"], dword[0])
    assert int(dword.item()) == ibp.IBP_OK


@pytest.mark.parametrize("W", [64, 128, 512])
@pytest.mark.parametrize("where", ["host", "hbm"])
def test_per_word_plan_groups_with_raw_corrupt_and_bad_rows(W, where):
    """Per-word tables (two Masks alternating by word position; one run of
    kept bits each) on groups that mix compressed, raw and corrupt rows and
    bad ids: from device slots the rows are rebuilt two words per lane, with
    straight-line code for groups whose rows are all compressed and a per-row
    path for the others.  Rows and status against the oracle's decode of the
    same slots."""
    rng = np.random.default_rng(40 + W)
    n = 600
    rows = _float_rows(rng, n, W)
    mask = np.where(np.arange(W) % 2 == 0, 0xFF800000, 0xFFF00000).astype(np.uint32)
    bitval = (rows[0] & mask).astype(np.uint32)
    match = rng.random((n, 1)) < 0.8
    rows = np.where(match, (rows & ~mask) | (bitval & mask), rows).astype(np.uint32)
    plan = _explicit_plan_check(mask, bitval, rows, where)
    assert plan.info["uniform"] == 0 and plan.info["max_runs"] == 1
    rows_t = place(rows, where)
    slots_t = empty_like_in(rows_t, where)
    _, bm, _ = ibp.ibp_compress(plan, rows_t, slots_t)
    torch.cuda.synchronize()
    bitmask = words_np(bm)
    slots = words_np(slots_t).copy()
    comp = np.nonzero((bitmask[np.arange(n) >> 5] >> (np.arange(n) & 31).astype(np.uint32)) & 1)[0]
    raw_rows = np.setdiff1d(np.arange(n), comp)
    assert len(comp) > 50 and len(raw_rows) > 5
    bad_rows = comp[3:9]
    slots[bad_rows, :W // 32] = 0  # every word announced raw: stream >= W words
    dev = place(slots, where)
    ids = rng.integers(0, n, 3000).astype(np.int64)
    ids[::37] = bad_rows[np.arange(len(ids[::37])) % len(bad_rows)]
    ids[5::101] = n + 3
    out = ibp.ibp_gather_decompress(plan, dev, bm, torch.from_numpy(ids).cuda())
    code = ibp.ibp_get_status(plan, raise_on_error=False)
    st, ref = C.decompress(slots, bitmask, ids, mask, bitval)
    assert code in (ibp.IBP_ERANGE, ibp.IBP_ECORRUPT) and st in (ibp.IBP_ERANGE, ibp.IBP_ECORRUPT)
    assert np.array_equal(words_np(out), ref)
    # all-compressed groups only: the straight-line path, status clean
    good = np.setdiff1d(comp, bad_rows)
    ids = good[rng.integers(0, len(good), 2000)].astype(np.int64)
    out = ibp.ibp_gather_decompress(plan, dev, bm, torch.from_numpy(ids).cuda())
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows[ids])


@pytest.mark.parametrize("W", [256, 512])
def test_short_stage_rows_from_device_slots(W):
    """Sparse rows (5 % non-zeros) under a per-word plan, slots in HBM: once
    the prefix is tuned the plan records short rows and device decodes stage
    W / 4 words per row.  A few denser rows (stored longer than W / 4 words,
    decoded from their slots), raw rows (copied from their slots), corrupt
    rows and bad ids mixed in; rows and status against the oracle's decode of
    the same slots."""
    rng = np.random.default_rng(70 + W)
    n = 6000
    rows = workloads.sparse_gnn_table(n_rows=n, W=W, seed=W, nnz=max(1, W // 20))
    dense = rng.choice(n, 20, replace=False)  # 0.33 %: long compressed rows
    raw = rng.choice(np.setdiff1d(np.arange(n), dense), 12, replace=False)  # 0.2 %: raw rows
    rows[dense, : 2 * W // 5] = rng.lognormal(-2, 0.5, (len(dense), 2 * W // 5)).astype(np.float32).view(np.uint32)
    rows[raw] = rng.integers(0, 2**32, (len(raw), W), dtype=np.uint64).astype(np.uint32)
    g = gpu_codec(rows, rows[:3000], 0.95, "hbm")
    plan = g["plan"]
    assert plan.info["uniform"] == 0 and plan.info["max_runs"] <= 2
    bm = on_device(g["bitmask"])
    words = ibp.ibp_plan_tune_prefix(plan, g["slots_t"], bm)
    info = plan.info
    assert info["short_rows"] == 1 and words <= W // 4
    slots = words_np(g["slots_t"]).copy()
    comp = np.nonzero((g["bitmask"][np.arange(n) >> 5] >> (np.arange(n) & 31).astype(np.uint32)) & 1)[0]
    assert np.isin(dense, comp).all() and not np.isin(raw, comp).any()
    bad = np.setdiff1d(comp, dense)[:4]
    slots[bad, : W // 32] = 0  # every word announced raw: stream >= W words
    dev = on_device(slots)
    ids = rng.integers(0, n, 20000).astype(np.int64)
    ids[::50] = dense[np.arange(len(ids[::50])) % len(dense)]
    ids[7::80] = raw[np.arange(len(ids[7::80])) % len(raw)]
    ids[11::997] = bad[np.arange(len(ids[11::997])) % len(bad)]
    ids[13::1999] = -5
    out = ibp.ibp_gather_decompress(plan, dev, bm, torch.from_numpy(ids).cuda())
    code = ibp.ibp_get_status(plan, raise_on_error=False)
    st, ref = C.decompress(slots, g["bitmask"], ids, g["mask"], g["bitval"])
    assert code in (ibp.IBP_ERANGE, ibp.IBP_ECORRUPT) and st in (ibp.IBP_ERANGE, ibp.IBP_ECORRUPT)
    assert np.array_equal(words_np(out), ref)
    # clean ids only: every row exact, status clean; contiguous too
    ok = np.setdiff1d(np.arange(n), bad)
    ids = ok[rng.integers(0, len(ok), 20000)].astype(np.int64)
    out = ibp.ibp_gather_decompress(plan, dev, bm, torch.from_numpy(ids).cuda())
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows[ids])
    first = int(bad.max()) + 1
    out = ibp.ibp_decompress_contig(plan, dev, bm, first, n - first)
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows[first:])


@pytest.mark.parametrize("W", [256, 512])
def test_short_stage_rows_at_the_stage_boundary(W):
    """Short stage rows hold W / 4 words: rows whose streams are W / 4 - 1,
    W / 4 (staged) and W / 4 + 1, W / 4 + 2 words (decoded from their slots),
    among rows that all fit, under an explicit per-word plan (one and two
    kept bits, alternating).  Stored lengths come from the oracle."""
    rng = np.random.default_rng(500 + W)
    RW = W // 4
    mask = np.where(np.arange(W) % 2 == 0, 0xFFFFFFFE, 0xFFFFFFFC).astype(np.uint32)
    bitval = np.zeros(W, np.uint32)
    base = rng.integers(0, 2, (1, W)).astype(np.uint32)  # every word matches

    def with_unmatched(k):
        r = base.copy()
        pos = rng.choice(W, k, replace=False)
        r[0, pos] = rng.integers(1 << 20, 1 << 31, k).astype(np.uint32)
        return r

    # candidates around the boundary: the oracle's stored length picks them
    cands = np.concatenate([with_unmatched(k) for k in range(1, W // 2) for _ in range(3)])
    lw = C.row_words(cands, mask, bitval)
    picks = [cands[lw == L][:3] for L in (RW - 1, RW, RW + 1, RW + 2)]
    assert all(len(p) for p in picks), [int((lw == L).sum()) for L in (RW - 1, RW, RW + 1, RW + 2)]
    n = 4000
    rows = np.repeat(base, n, axis=0)
    rows ^= (rng.random((n, W)) < 0.5).astype(np.uint32)  # kept bits only: still matching
    special = np.concatenate(picks)
    at = rng.choice(n, len(special), replace=False)
    rows[at] = special
    plan = ibp.ibp_plan_create(torch.from_numpy(mask.view(np.int32)), torch.from_numpy(bitval.view(np.int32)))
    rows_t = on_device(rows)
    slots_t = torch.empty_like(rows_t)
    _, bm, _ = ibp.ibp_compress(plan, rows_t, slots_t)
    ibp.ibp_plan_tune_prefix(plan, slots_t, bm)
    assert plan.info["short_rows"] == 1 and plan.info["prefix_words"] <= RW
    slots = words_np(slots_t)
    cs, cb, _ = C.compress(rows, mask, bitval)
    assert np.array_equal(slots, cs) and np.array_equal(words_np(bm), cb)
    ids = np.concatenate([np.repeat(at, 5), rng.integers(0, n, 6000)]).astype(np.int64)
    rng.shuffle(ids)
    out = ibp.ibp_gather_decompress(plan, slots_t, bm, torch.from_numpy(ids).cuda())
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    assert np.array_equal(words_np(out), rows[ids])
