"""Oracle of the packed cache layout.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only the tests use it.  It shares no code with the CUDA library under
``host_transfer_gb300/``.

Source: the page "Résumé Technique : Réduire le goulot d'étranglement de la
mémoire GPU par la compression sans perte pour le ML", section « Intégration
au système », first use: compressing the tensors held in a GPU software cache
raises the cache's effective capacity.  Fixed-size slots save no room, so a
cache has to keep only the words of each row that a reader needs.  The page
gives no layout; the reading taken here:

* row r keeps the first ``s_r`` words of its slot rounded up to a multiple of
  4 (so every row starts on a 16-byte boundary), where ``s_r`` is the row's
  stored length: Lw (its stream) when it is stored compressed, W when raw;
* the rows follow one another in row order, with nothing between them;
* ``offsets[r]`` is the word where row r starts, ``offsets[n]`` the total.

The words past Lw in a compressed slot are the slot's zero tail, so the
rounding pads with zeros.  A raw row is W words, a multiple of 4 (the layout
requires W % 4 == 0).

Parity status: pinned by tests/test_packed_oracle_pins.py (a hand-built
three-row example, tests/golden/packed_rows.txt).
"""

from __future__ import annotations

import numpy as np


def round4(n):
    """Words a packed row occupies for a stored length of ``n`` words."""
    return (np.asarray(n, dtype=np.int64) + 3) // 4 * 4


def packed_offsets(stored_words) -> np.ndarray:
    """offsets[0..n]: exclusive running sum of the rows' rounded lengths."""
    lens = round4(stored_words)
    out = np.zeros(len(lens) + 1, np.int64)
    running = 0
    for r, n in enumerate(lens):
        out[r] = running
        running += int(n)
    out[len(lens)] = running
    return out


def pack(slots, stored_words) -> tuple[np.ndarray, np.ndarray]:
    """(offsets, packed words) of the slots (n x W words) of rows whose stored
    lengths are ``stored_words``."""
    slots = np.asarray(slots, dtype=np.uint32)
    offsets = packed_offsets(stored_words)
    packed = np.zeros(int(offsets[-1]), np.uint32)
    for r in range(slots.shape[0]):
        a, b = int(offsets[r]), int(offsets[r + 1])
        packed[a:b] = slots[r, : b - a]
    return offsets, packed
