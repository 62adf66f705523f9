"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle (Python ``oracle.ibp_ref`` and C ``oracle.oracle_c``)
against something fixed independently of it: hand-derived rows, a second
formulation of pext/pdep, exhaustive enumeration of 8-bit toy words, the size
identity, the round trip, closed forms of the preprocess, and special cases.
"""

import math
import os

import numpy as np
import pytest

from oracle import ibp_ref as R
from oracle import oracle_c as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_rows.txt")


def _load_golden():
    examples = []
    cur = None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "example":
            cur = {"name": vals[0]}
            examples.append(cur)
            continue
        nums = [int(v, 16) for v in vals]
        cur[key] = nums
    for e in examples:
        W = e["W"][0]
        for k in ("mask", "bitval"):
            if len(e[k]) == 1:
                e[k] = e[k] * W
        assert len(e["row"]) == W and len(e["slot"]) == W
    return examples


EXAMPLES = _load_golden()


# ---------------------------------------------------------------------------
# hand-derived rows


@pytest.mark.parametrize("ex", EXAMPLES, ids=[e["name"] for e in EXAMPLES])
def test_hand_rows_python(ex):
    slot, comp, used = R.compress_row(ex["row"], ex["mask"], ex["bitval"])
    assert slot == ex["slot"]
    assert comp == bool(ex["compressed"][0])
    assert used == ex["stored"][0]
    st, row = R.decode_row(slot, comp, ex["mask"], ex["bitval"])
    assert st == R.OK and row == ex["row"]


@pytest.mark.parametrize("ex", EXAMPLES, ids=[e["name"] for e in EXAMPLES])
def test_hand_rows_c(ex):
    rows = np.array([ex["row"]], np.uint32)
    slots, bitmask, stored = C.compress(rows, np.array(ex["mask"], np.uint32),
                                        np.array(ex["bitval"], np.uint32))
    assert slots[0].tolist() == ex["slot"]
    assert int(bitmask[0]) == ex["compressed"][0]
    assert stored == ex["stored"][0]
    st, out = C.decompress(slots, bitmask, np.array([0]), np.array(ex["mask"], np.uint32),
                           np.array(ex["bitval"], np.uint32))
    assert st == 0 and out[0].tolist() == ex["row"]


# ---------------------------------------------------------------------------
# pext / pdep: exhaustive on 8-bit words against a second formulation


def _positions(keep, B):
    return [p for p in range(B) if (keep >> p) & 1]


def test_pext_pdep_exhaustive_8bit():
    B = 8
    for keep in range(256):
        pos = _positions(keep, B)
        for x in range(256):
            # pext: read bit pos[j] of x into bit j
            want = sum(((x >> p) & 1) << j for j, p in enumerate(pos))
            assert R.pext(x, keep, B) == want
            # pdep: bit j of x lands at pos[j]
            want = sum(((x >> j) & 1) << p for j, p in enumerate(pos))
            assert R.pdep(x, keep, B) == want
            # the two are inverse on their ranges
            assert R.pdep(R.pext(x, keep, B), keep, B) == x & keep
            assert R.pext(R.pdep(x, keep, B), keep, B) == x & ((1 << len(pos)) - 1)


# ---------------------------------------------------------------------------
# word level: every (mask, x) of 8-bit words, Bitval inside and outside


def _bitval_choices(m, x, rng):
    sub = rng.integers(0, 256) & m
    return {x & m, (x ^ m) & m, sub, 0}


def test_word_level_exhaustive_8bit():
    B = 8
    rng = np.random.default_rng(0)
    for m in range(256):
        keep = ~m & 0xFF
        p = bin(m).count("1")
        for x in range(256):
            for b in _bitval_choices(m, x, rng):
                stream, nbits, flags = R.encode_row([x], [m], [b], B)
                match = ((x ^ b) & m) == 0
                assert flags == [1 if match else 0]
                # size identity on one word: header (B) + field
                assert nbits == B + ((B - p) if match else B)
                # the stream starts with the header, then the field
                field = (stream[1] if len(stream) > 1 else 0)
                if match:
                    assert stream[0] == 1
                    if p < B:
                        assert field & ((1 << (B - p)) - 1) == R.pext(x, keep, B)
                else:
                    assert stream[0] == 0 and field == x
                assert R.decode_stream(stream + [0], 1, [m], [b], B) == [x]


def test_bitval_outside_mask_is_ignored():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        W = int(rng.integers(1, 70))
        m = [int(v) for v in rng.integers(0, 2**32, W, dtype=np.uint64)]
        b = [int(v) for v in rng.integers(0, 2**32, W, dtype=np.uint64)]
        x = [bm & mm if rng.random() < 0.7 else int(rng.integers(0, 2**32)) for bm, mm in zip(b, m)]
        bin_ = [bb & mm for bb, mm in zip(b, m)]
        slot, comp, used = R.compress_row(x, m, b)
        assert (slot, comp, used) == R.compress_row(x, m, bin_)
        # Bitval bits outside the Mask never reach a decoded word either
        assert R.decode_row(slot, comp, m, b) == (R.OK, x)
    rows = np.random.default_rng(2).integers(0, 2**32, (64, 40), dtype=np.uint64).astype(np.uint32)
    m = rows[0] & rows[1]
    b = rows[2]
    rows[::2] = (rows[::2] & ~m) | (b & m)
    slots, bitmask, _ = C.compress(rows, m, b)
    st, back = C.decompress(slots, bitmask, np.arange(64), m, b)
    assert st == 0 and np.array_equal(back, rows)


# ---------------------------------------------------------------------------
# rows of toy words: exhaustive for W = 2, B = 8


@pytest.mark.parametrize("m,b", [(0xF0, 0x30), (0x81, 0x01), (0xFF, 0x5A), (0x00, 0x00), (0x7E, 0x00)])
def test_rows_exhaustive_8bit_w2(m, b):
    B, W = 8, 2
    p = bin(m).count("1")
    for x0 in range(256):
        for x1 in range(256):
            x = [x0, x1]
            stream, nbits, flags = R.encode_row(x, [m] * W, [b] * W, B)
            # size identity: S*B header bits + per word (B - p) or B
            assert nbits == B + sum((B - p) if f else B for f in flags)
            slot, comp, used = R.compress_row(x, [m] * W, [b] * W, B)
            assert comp == (math.ceil(nbits / B) < W)
            st, back = R.decode_row(slot, comp, [m] * W, [b] * W, B)
            assert st == R.OK and back == x


# ---------------------------------------------------------------------------
# 32-bit rows: size identity and round trip


def _float_rows(rng, n, W):
    x = rng.normal(0, 0.05, size=(n, W)).astype(np.float32).view(np.uint32)
    return x


def test_size_identity_32bit_w_multiple_of_32():
    """For W % 32 == 0 the stream has sum over words of 1 + 32 - popcount(mask)
    bits when the word matches and 33 bits otherwise."""
    rng = np.random.default_rng(2)
    W = 64
    rows = _float_rows(rng, 40, W)
    st, mask, bitval = R.preprocess(rows[:20].tolist(), 0.9)
    assert st == R.OK
    for x in rows.tolist():
        _, nbits, flags = R.encode_row(x, mask, bitval)
        want = sum((1 + 32 - bin(mask[w]).count("1")) if flags[w] else 33 for w in range(W))
        assert nbits == want


def test_size_identity_partial_segment():
    rng = np.random.default_rng(3)
    W = 45  # two segments, 19 header bits unused
    rows = _float_rows(rng, 30, W)
    _, mask, bitval = R.preprocess(rows.tolist(), 0.8)
    for x in rows.tolist():
        _, nbits, flags = R.encode_row(x, mask, bitval)
        want = 64 + sum((32 - bin(mask[w]).count("1")) if flags[w] else 32 for w in range(W))
        assert nbits == want


def test_round_trip_python_random_garbage():
    rng = np.random.default_rng(4)
    for W in (1, 3, 31, 32, 33, 64, 97):
        rows = [[int(v) for v in rng.integers(0, 2**32, W, dtype=np.uint64)] for _ in range(8)]
        mask = [int(v) for v in rng.integers(0, 2**32, W, dtype=np.uint64)]
        bitval = [int(v) & mm for v, mm in zip(rng.integers(0, 2**32, W, dtype=np.uint64), mask)]
        # half of the rows are made to match
        for r in rows[:4]:
            for w in range(W):
                r[w] = (r[w] & ~mask[w] & 0xFFFFFFFF) | bitval[w]
        slots, bm, _ = R.compress(rows, mask, bitval)
        st, back = R.gather_decompress(slots, bm, list(range(len(rows))), mask, bitval)
        assert st == R.OK and back == rows


def test_round_trip_c_special_floats():
    rng = np.random.default_rng(5)
    W = 96
    vals = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 1e-45, -1e-40, 3.4e38, 1.0, -2.5],
                    np.float32).view(np.uint32)
    rows = _float_rows(rng, 500, W)
    rows[::7, ::5] = vals[rng.integers(0, len(vals), rows[::7, ::5].shape)]
    rows[3, :] = vals[rng.integers(0, len(vals), W)]
    _, mask, bitval = C.preprocess(rows, 0.95)
    slots, bitmask, _ = C.compress(rows, mask, bitval)
    st, back = C.decompress(slots, bitmask, np.arange(len(rows)), mask, bitval)
    assert st == 0 and np.array_equal(back, rows)


def test_round_trip_c_random_masks():
    rng = np.random.default_rng(6)
    for W in (1, 2, 5, 32, 40, 129):
        rows = rng.integers(0, 2**32, (300, W), dtype=np.uint64).astype(np.uint32)
        mask = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32)
        bitval = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32) & mask
        rows[::2] = (rows[::2] & ~mask) | bitval
        slots, bitmask, _ = C.compress(rows, mask, bitval)
        st, back = C.decompress(slots, bitmask, np.arange(len(rows)), mask, bitval)
        assert st == 0 and np.array_equal(back, rows)


# ---------------------------------------------------------------------------
# preprocess closed forms


def _rand_sample(rng, s, W):
    base = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32)
    flips = rng.integers(0, 2**32, (s, W), dtype=np.uint64).astype(np.uint32)
    keep = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32)
    return base ^ (flips & keep & rng.integers(0, 2**32, (s, W), dtype=np.uint64).astype(np.uint32))


@pytest.mark.parametrize("s", [1, 2, 7, 64])
def test_preprocess_T1_closed_form(s):
    """T = 1: a bit is invariant iff all rows agree, i.e. mask = ~(OR ^ AND)
    and Bitval = AND on those positions."""
    rng = np.random.default_rng(s)
    x = _rand_sample(rng, s, 37)
    orv = np.bitwise_or.reduce(x, axis=0)
    andv = np.bitwise_and.reduce(x, axis=0)
    want_m = ~(orv ^ andv)
    want_b = andv & want_m
    st, m, b = C.preprocess(x, 1.0)
    assert st == 0 and np.array_equal(m, want_m) and np.array_equal(b, want_b)
    st, m2, b2 = R.preprocess(x.tolist(), 1.0)
    assert st == R.OK and m2 == want_m.tolist() and b2 == want_b.tolist()


@pytest.mark.parametrize("s,T", [(5, 0.5), (9, 0.3), (33, 0.01)])
def test_preprocess_majority_closed_form(s, T):
    """T <= 0.5 with an odd sample: every position is invariant and Bitval is
    the bitwise majority."""
    rng = np.random.default_rng(10 + s)
    x = rng.integers(0, 2**32, (s, 21), dtype=np.uint64).astype(np.uint32)
    bits = np.unpackbits(x.view(np.uint8).reshape(s, 21, 4), axis=2, bitorder="little")
    maj = (bits.sum(axis=0) * 2 > s).astype(np.uint8)
    want_b = np.packbits(maj, axis=1, bitorder="little").view(np.uint32).reshape(21)
    st, m, b = C.preprocess(x, T)
    assert st == 0 and np.all(m == 0xFFFFFFFF) and np.array_equal(b, want_b)
    st, m2, b2 = R.preprocess(x.tolist(), T)
    assert m2 == [0xFFFFFFFF] * 21 and b2 == want_b.tolist()


def test_preprocess_tie_and_threshold_edges():
    # two rows disagreeing on every bit: ones = zeros = 1.
    x = np.array([[0x0F0F0F0F], [0xF0F0F0F0]], np.uint32)
    # T = 0.5: t = ceil(1.0) = 1, max(1, 1) >= 1 -> invariant; tie -> Bitval 0
    st, m, b = C.preprocess(x, 0.5)
    assert m[0] == 0xFFFFFFFF and b[0] == 0
    # T = 0.51: t = ceil(1.02) = 2 -> nothing invariant
    st, m, b = C.preprocess(x, 0.51)
    assert m[0] == 0 and b[0] == 0
    # four rows, bit 0 set in exactly three: T = 0.75 -> t = 3 -> invariant, value 1
    y = np.array([[1], [1], [1], [0]], np.uint32)
    st, m, b = C.preprocess(y, 0.75)
    assert m[0] & 1 and b[0] & 1
    st, m, b = C.preprocess(y, 0.76)  # t = ceil(3.04) = 4
    assert not (m[0] & 1)
    assert R.preprocess(y.tolist(), 0.75)[1][0] & 1 == 1
    assert R.preprocess(y.tolist(), 0.76)[1][0] & 1 == 0


def test_preprocess_rejects_bad_arguments():
    x = np.zeros((4, 3), np.uint32)
    for T in (0.0, -0.1, 1.0000001, float("nan")):
        assert C.preprocess(x, T)[0] == 1
        assert R.preprocess(x.tolist(), T)[0] == R.EINVAL
    assert C.preprocess(np.zeros((0, 3), np.uint32), 0.9)[0] == 1
    assert R.preprocess([], 0.9)[0] == R.EINVAL


# ---------------------------------------------------------------------------
# special cases


def test_mask_zero_stores_every_row_raw():
    rng = np.random.default_rng(20)
    for W in (1, 4, 32, 100):
        rows = rng.integers(0, 2**32, (50, W), dtype=np.uint64).astype(np.uint32)
        z = np.zeros(W, np.uint32)
        slots, bitmask, stored = C.compress(rows, z, z)
        assert np.array_equal(slots, rows) and not bitmask.any() and stored == 50 * W


def test_full_mask_rows_equal_bitval_give_headers_only():
    for W in (2, 31, 32, 33, 64, 200):
        S = (W + 31) // 32
        bv = np.arange(W, dtype=np.uint32) * 2654435761
        rows = np.tile(bv, (33, 1))
        slots, bitmask, stored = C.compress(rows, np.full(W, 0xFFFFFFFF, np.uint32), bv)
        assert stored == 33 * S
        assert bitmask[0] == 0xFFFFFFFF and bitmask[1] == 1
        for s in range(S):
            nbits = min(32, W - 32 * s)
            want = 0xFFFFFFFF if nbits == 32 else (1 << nbits) - 1
            assert np.all(slots[:, s] == want)
        assert not slots[:, S:].any()


def test_sparse_zero_rows_header_only():
    """A mask learned on mostly-zero rows makes an all-zero row a stream of
    header words and zero-length fields."""
    W = 512
    rng = np.random.default_rng(21)
    x = np.zeros((200, W), np.float32)
    nz = rng.integers(0, W, (200, 3))
    x[np.arange(200)[:, None], nz] = rng.uniform(0.1, 0.9, (200, 3))
    words = x.view(np.uint32)
    st, m, b = C.preprocess(words, 0.95)
    zero_row = np.zeros((1, W), np.uint32)
    slots, bitmask, stored = C.compress(zero_row, m, b)
    kept = 32 * 16 + sum(32 - bin(int(v)).count("1") for v in m)
    assert stored == (kept + 31) // 32
    assert np.all(slots[0, :16] == 0xFFFFFFFF)


# ---------------------------------------------------------------------------
# the two oracles agree (written independently)


@pytest.mark.parametrize("W,T", [(4, 0.9), (37, 0.99), (64, 0.75), (128, 0.99)])
def test_c_and_python_oracles_agree(W, T):
    rng = np.random.default_rng(W)
    rows = _float_rows(rng, 60, W)
    rows[5] = rng.integers(0, 2**32, W, dtype=np.uint64).astype(np.uint32)
    st, mc, bc = C.preprocess(rows[:40], T)
    st2, mp, bp = R.preprocess(rows[:40].tolist(), T)
    assert mc.tolist() == mp and bc.tolist() == bp
    sc, bmc, stc = C.compress(rows, mc, bc)
    sp, bmp, stp = R.compress(rows.tolist(), mp, bp)
    assert sc.tolist() == sp and bmc.tolist() == bmp and stc == stp
    ids = rng.integers(-3, len(rows) + 3, 80)
    stc, outc = C.decompress(sc, bmc, ids, mc, bc)
    stp, outp = R.gather_decompress(sp, bmp, ids.tolist(), mp, bp)
    assert stc == stp and outc.tolist() == outp


def test_out_of_range_and_corrupt_slots():
    W = 64
    rng = np.random.default_rng(30)
    rows = _float_rows(rng, 40, W)
    _, m, b = C.preprocess(rows, 0.9)
    slots, bitmask, _ = C.compress(rows, m, b)
    assert bitmask[0] & 1
    st, out = C.decompress(slots, bitmask, np.array([0, 40, -1]), m, b)
    assert st == R.ERANGE and not out[1:].any() and np.array_equal(out[0], rows[0])
    bad = slots.copy()
    bad[0, :2] = 0  # every word now announces 32 bits: the stream exceeds W words
    st, out = C.decompress(bad, bitmask, np.array([1, 0]), m, b)
    assert st == R.ECORRUPT and not out[1].any() and np.array_equal(out[0], rows[1])
    # W = 40: the second header has 24 bits past the last word
    W2 = 40
    r2 = _float_rows(rng, 8, W2)
    _, m2, b2 = C.preprocess(r2, 0.9)
    s2, bm2, _ = C.compress(r2, m2, b2)
    assert bm2[0] & 1
    s2[0, 1] |= 1 << 20  # header bit of word 52 >= W
    st, out = C.decompress(s2, bm2, np.array([0]), m2, b2)
    assert st == R.ECORRUPT and not out.any()
    assert R.decode_row(s2[0].tolist(), True, m2.tolist(), b2.tolist())[0] == R.ECORRUPT


def test_row_words_sum_to_stored_words():
    """Per-row stored words add up to the total the compress reports, and equal
    W exactly for the rows stored raw."""
    rng = np.random.default_rng(40)
    rows = _float_rows(rng, 300, 96)
    rows[::5] = rng.integers(0, 2**32, (60, 96), dtype=np.uint64).astype(np.uint32)
    _, m, b = C.preprocess(rows, 0.9)
    slots, bitmask, stored = C.compress(rows, m, b)
    words = C.row_words(rows, m, b)
    assert int(words.sum()) == stored
    bits = (bitmask[np.arange(300) >> 5] >> (np.arange(300) & 31).astype(np.uint32)) & 1
    assert np.all(words[bits == 0] == 96) and np.all(words[bits == 1] < 96)
    for r in (0, 1, 7):
        assert words[r] == R.compress_row(rows[r].tolist(), m.tolist(), b.tolist())[2]
