"""Pins of the packed-layout oracle (oracle/packed_ref.py) and of the two C
oracle entry points that the full-size GPU parity tests lean on
(compress_some, decode_slots), each against something other than itself:
a hand-built example, and the whole-table oracle functions that the hand rows
and the brute-force tests already pin."""

import os

import numpy as np
import pytest

from oracle import ibp_ref as R
from oracle import oracle_c as C
from oracle import packed_ref as P

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "packed_rows.txt")


def _load():
    ex = {"row": [], "packed": []}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key in ("W", "stored", "offsets"):
            ex[key] = [int(v) for v in vals]
        elif key in ("row", "packed"):
            ex[key].append([int(v, 16) for v in vals])
        else:
            ex[key] = [int(v, 16) for v in vals]
    return ex


EX = _load()


def _mask_bitval(ex):
    W = ex["W"][0]
    return [ex["mask"][0]] * W, [ex["bitval"][0]] * W


def test_hand_example_python_oracle():
    m, b = _mask_bitval(EX)
    slots, bitmask, stored = R.compress(EX["row"], m, b)
    lens = [R.compress_row(x, m, b)[2] for x in EX["row"]]
    assert lens == EX["stored"]
    assert bitmask == EX["bitmask"]
    assert stored == sum(EX["stored"])
    offsets, packed = P.pack(slots, lens)
    assert offsets.tolist() == EX["offsets"]
    assert packed.tolist() == [w for row in EX["packed"] for w in row]


def test_hand_example_c_oracle():
    m, b = (np.array(v, np.uint32) for v in _mask_bitval(EX))
    rows = np.array(EX["row"], np.uint32)
    slots, bitmask, _ = C.compress(rows, m, b)
    words = C.row_words(rows, m, b)
    assert words.tolist() == EX["stored"]
    offsets, packed = P.pack(slots, words)
    assert offsets.tolist() == EX["offsets"]
    assert packed.tolist() == [w for row in EX["packed"] for w in row]


def test_offsets_closed_form():
    """offsets[r] = sum over earlier rows of 4 * ceil(s / 4); the total is the
    last entry; every row starts on a multiple of 4 words."""
    rng = np.random.default_rng(7)
    s = rng.integers(1, 129, 1000)
    off = P.packed_offsets(s)
    want = np.concatenate([[0], np.cumsum(-(-s // 4) * 4)])
    assert np.array_equal(off, want)
    assert np.all(off % 4 == 0)
    assert P.packed_offsets([]).tolist() == [0]


def test_packed_rows_round_trip_through_the_decoder():
    """Each packed row, padded back to W with zeros, is the row's slot, and the
    oracle decoder gives the row back."""
    rng = np.random.default_rng(8)
    rows = rng.normal(0, 0.05, (200, 64)).astype(np.float32).view(np.uint32)
    rows[::7] = rng.integers(0, 2**32, (29, 64), dtype=np.uint64).astype(np.uint32)
    _, m, b = C.preprocess(rows, 0.99)
    slots, bitmask, _ = C.compress(rows, m, b)
    offsets, packed = P.pack(slots, C.row_words(rows, m, b))
    for r in range(len(rows)):
        seg = packed[offsets[r]:offsets[r + 1]]
        slot = np.zeros(64, np.uint32)
        slot[: len(seg)] = seg
        assert np.array_equal(slot, slots[r])
    st, out = C.decompress(slots, bitmask, np.arange(len(rows)), m, b)
    assert st == 0 and np.array_equal(out, rows)


def _mixed_rows(rng, n, W):
    """Float rows, a fifth of them replaced by random words (stored raw), and
    the Mask/Bitval of the float rows."""
    rows = rng.normal(0, 0.05, (n, W)).astype(np.float32).view(np.uint32)
    _, m, b = C.preprocess(rows[:256], 0.99)
    raw = rng.random(n) < 0.2
    rows[raw] = rng.integers(0, 2**32, (int(raw.sum()), W), dtype=np.uint64).astype(np.uint32)
    return rows, m, b


@pytest.mark.parametrize("W", [64, 100, 512])
def test_compress_some_is_compress_at_the_ids(W):
    """Slot i and bit i of compress_some(rows, ids) are slot ids[i] and bit
    ids[i] of the whole-table compress, for ids in any order, with repeats."""
    rng = np.random.default_rng(W)
    rows, m, b = _mixed_rows(rng, 700, W)
    slots, bitmask, _ = C.compress(rows, m, b)
    ids = np.concatenate([rng.permutation(700)[:300], [0, 699, 5, 5, 5]]).astype(np.int64)
    got, bits = C.compress_some(rows, ids, m, b)
    want_bits = (bitmask[ids >> 5] >> (ids & 31).astype(np.uint32)) & 1
    assert np.array_equal(got, slots[ids])
    assert np.array_equal(bits.astype(np.uint32), want_bits)
    assert 0 < bits.sum() < len(ids)  # both kinds of row are exercised


@pytest.mark.parametrize("W", [64, 100])
def test_decode_slots_is_decompress_of_the_same_slots(W):
    """decode_slots on rows taken out of a table gives what decompress gives
    on the table at those ids, corrupt slots included."""
    rng = np.random.default_rng(W + 1)
    rows, m, b = _mixed_rows(rng, 400, W)
    slots, bitmask, _ = C.compress(rows, m, b)
    bits = ((bitmask[np.arange(400) >> 5] >> (np.arange(400) & 31).astype(np.uint32)) & 1).astype(np.uint8)
    comp = np.nonzero(bits)[0]
    bad = slots.copy()
    # all-ones words: with W = 100 the last header sets bits past the last
    # word, so the slot is corrupt; with W = 64 it decodes to some row
    bad[comp[3]] = 0xFFFFFFFF
    ids = rng.permutation(400)[:250]
    ids = np.concatenate([ids, [comp[3]]]).astype(np.int64)
    st_a, out_a = C.decode_slots(bad[ids], bits[ids], m, b)
    st_b, out_b = C.decompress(bad, bitmask, ids, m, b)
    assert np.array_equal(out_a, out_b)
    assert st_a == st_b
    if W == 100:
        assert st_a == R.ECORRUPT
    ok = ids != comp[3]
    assert np.array_equal(out_a[ok], rows[ids[ok]])
