"""Pins of the pooling oracle (oracle/bag_ref.py) to facts that do not come
from the oracle itself: exact integer arithmetic, the IEEE single precision
results of fixed addition orders, and the reading's special cases."""

import numpy as np

from oracle import bag_ref as B


def _f(rows):
    return np.asarray(rows, np.float32).view(np.uint32)


def _vals(out):
    return out.view(np.float32)


def test_sums_of_small_integers_are_exact():
    rng = np.random.default_rng(0)
    n, W = 500, 24
    x = rng.integers(-1000, 1000, (n, W)).astype(np.float32)  # sums stay far below 2^24
    offsets = np.concatenate([[0], np.sort(rng.integers(0, n, 40)), [n]]).astype(np.int64)
    st, out = B.embedding_bag(_f(x), offsets, B.SUM)
    assert st == B.OK
    want = np.stack([x[offsets[b]:offsets[b + 1]].astype(np.float64).sum(axis=0) for b in range(len(offsets) - 1)])
    assert np.array_equal(_vals(out).astype(np.float64), want)


def test_mean_with_power_of_two_bag_sizes_is_exact():
    rng = np.random.default_rng(1)
    x = rng.integers(-500, 500, (64, 8)).astype(np.float32)
    offsets = np.array([0, 1, 3, 7, 15, 31, 63, 64], np.int64)  # sizes 1, 2, 4, 8, 16, 32, 1
    st, out = B.embedding_bag(_f(x), offsets, B.MEAN)
    assert st == B.OK
    for b in range(len(offsets) - 1):
        seg = x[offsets[b]:offsets[b + 1]].astype(np.float64)
        assert np.array_equal(_vals(out)[b].astype(np.float64), seg.sum(axis=0) / len(seg))


def test_rows_are_added_in_increasing_position_order():
    # 1e8 is exact in single precision and its neighbours are 8 apart, so
    # 1 + 1e8 rounds back to 1e8: the result depends on the order.
    x = np.array([[1e8], [-1e8], [1.0], [1.0], [1e8], [-1e8]], np.float32)
    st, out = B.embedding_bag(_f(x), np.array([0, 3, 6], np.int64), B.SUM)
    assert st == B.OK
    assert _vals(out)[0, 0] == 1.0   # (1e8 - 1e8) + 1
    assert _vals(out)[1, 0] == 0.0   # (1 + 1e8) - 1e8 = 1e8 - 1e8


def test_special_cases_of_the_reading():
    x = np.array([[-0.0, 3.5], [2.0, -1.0], [5.0, 7.0]], np.float32)
    # empty bags, a one-row bag, a bag of -0.0 (the sum starts from +0.0)
    offsets = np.array([0, 0, 1, 1, 3], np.int64)
    st, s = B.embedding_bag(_f(x), offsets, B.SUM)
    _, m = B.embedding_bag(_f(x), offsets, B.MEAN)
    assert st == B.OK
    assert not s[0].any() and not m[0].any() and not s[2].any() and not m[2].any()
    assert s[1, 0] == 0 and _vals(s)[1, 1] == 3.5  # +0.0 + -0.0 = +0.0
    assert np.array_equal(_vals(s)[3], [7.0, 6.0]) and np.array_equal(_vals(m)[3], [3.5, 3.0])


def test_invalid_offsets_give_zero_bags_and_erange():
    x = np.ones((4, 3), np.float32)
    for offsets in ([0, 3, 2, 4], [0, 5], [-1, 2], [0, 2, 2]):
        st, out = B.embedding_bag(_f(x), np.array(offsets, np.int64), B.SUM)
        bad = [b for b in range(len(offsets) - 1)
               if not (0 <= offsets[b] <= offsets[b + 1] <= 4)]
        assert st == (B.ERANGE if bad else B.OK)
        for b in bad:
            assert not out[b].any()


def test_a_planted_order_mistake_is_caught():
    """The order pin fails for an oracle that sums in reverse."""
    x = np.array([[1.0], [1e8], [-1e8]], np.float32)
    fwd = B.embedding_bag(_f(x), np.array([0, 3], np.int64), B.SUM)[1]
    rev = B.embedding_bag(_f(x[::-1].copy()), np.array([0, 3], np.int64), B.SUM)[1]
    assert _vals(fwd)[0, 0] == 0.0 and _vals(rev)[0, 0] == 1.0


def test_bf16_rows_widen_exactly_and_pool_per_element():
    # bf16 1.5 = 0x3FC0, -2.0 = 0xC000, 0.375 = 0x3EC0: exact in both formats
    w = np.array([[0xC0003FC0], [0x3EC03FC0]], np.uint32)  # rows (1.5, -2.0) and (1.5, 0.375)
    st, out = B.embedding_bag(w, np.array([0, 2], np.int64), B.SUM, bf16=True)
    assert st == B.OK and out.shape == (1, 2)
    assert np.array_equal(out.view(np.float32)[0], [3.0, -1.625])
    st, m = B.embedding_bag(w, np.array([0, 2], np.int64), B.MEAN, bf16=True)
    assert np.array_equal(m.view(np.float32)[0], [1.5, -0.8125])


def test_bf16_widening_matches_torch_for_every_pattern():
    """Every bf16 pattern (both halves of a word) widens as torch's own
    bfloat16 -> float32 conversion does (NaNs compared as NaNs)."""
    import torch

    h = np.arange(0, 1 << 16, dtype=np.uint32)
    words = (h | (h[::-1] << 16)).reshape(-1, 1)
    f = B.bf16_words_to_f32(words)
    ref = torch.from_numpy(h.astype(np.int32).astype(np.int16)).view(torch.bfloat16).float().numpy()
    for col, src in ((0, ref), (1, ref[::-1])):
        nan = np.isnan(src)
        assert np.array_equal(np.isnan(f[:, col]), nan)
        assert np.array_equal(f[~nan, col].view(np.uint32), src[~nan].view(np.uint32))
