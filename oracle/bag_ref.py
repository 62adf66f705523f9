"""Plain oracle of the pooled consumer of decoded rows (an "embedding bag").

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library under
``host_transfer_gb300/``.

Source: the page "Résumé Technique : Réduire le goulot d'étranglement de la
mémoire GPU par la compression sans perte pour le ML", section « Résultats »:
the rows IBP moves feed DLRM embedding tables and GNN feature aggregation, and
« Algorithme central », step 3 (last point): the decoder overlaps fetching
with the logic that consumes the data.  The consumer of a DLRM or GNN lookup
pools the rows of each bag (the ids of one sample's sparse feature, or one
node's neighbours).  The pages do not define the pooling; the reading taken
is the usual one, stated here in full:

* rows are W float32 values (the decoded 32-bit words read as IEEE single),
  or, with bf16=True, 2W bfloat16 values (word j holds element 2j in bits
  0-15 and element 2j+1 in bits 16-31), each widened exactly to float32
  (its 16 bits become the high half of a float32);
* bag b holds the id positions k in [offsets[b], offsets[b+1]);
* sum:  out[b] = row(ids[k0]) + row(ids[k0+1]) + ..., added in IEEE single
  precision one row after another in increasing k, starting from +0.0 (no
  reassociation, no fused operations);
* mean: the sum divided by the bag size, one correctly rounded single
  precision division; an empty bag gives zeros in both modes;
* a bag whose offsets are not 0 <= offsets[b] <= offsets[b+1] <= n_ids is
  invalid: its output is zeros and the status is ERANGE;
* a row whose id is out of range decodes to zeros (status ERANGE) and still
  counts in its bag's size, as in gather-decompress followed by pooling.

Parity status: pinned (tests/test_bag_oracle_pins.py).
"""

from __future__ import annotations

import numpy as np

OK = 0
ERANGE = 5
SUM = 0
MEAN = 1


def bf16_words_to_f32(words: np.ndarray) -> np.ndarray:
    """uint32 [n, W] of bf16 pairs -> float32 [n, 2W] (exact widening)."""
    w = np.ascontiguousarray(words, dtype=np.uint32)
    out = np.empty((w.shape[0], 2 * w.shape[1]), np.uint32)
    out[:, 0::2] = (w & 0xFFFF) << 16
    out[:, 1::2] = w & 0xFFFF0000
    return out.view(np.float32)


def embedding_bag(decoded: np.ndarray, offsets: np.ndarray, mode: int, bf16: bool = False):
    """Pool decoded rows.

    decoded: uint32 [n_ids, W], row k = the decoded row of id position k.
    offsets: int64 [n_bags + 1].
    Returns (status, out) with out uint32 [n_bags, W] (or [n_bags, 2W] for
    bf16 rows) of float32 bits.
    """
    decoded = np.ascontiguousarray(decoded, dtype=np.uint32)
    n_ids = decoded.shape[0]
    vals = bf16_words_to_f32(decoded) if bf16 else decoded.view(np.float32)
    W = vals.shape[1]
    offsets = np.asarray(offsets, dtype=np.int64)
    n_bags = offsets.size - 1
    out = np.zeros((n_bags, W), np.float32)
    status = OK
    for b in range(n_bags):
        lo, hi = int(offsets[b]), int(offsets[b + 1])
        if not (0 <= lo <= hi <= n_ids):
            status = status or ERANGE
            continue
        acc = np.zeros(W, np.float32)  # +0.0
        with np.errstate(over="ignore", invalid="ignore"):  # IEEE overflow / NaN are results, not errors
            for k in range(lo, hi):
                acc = acc + vals[k]  # elementwise IEEE single additions, in order of k
            if mode == MEAN and hi > lo:
                acc = acc / np.float32(hi - lo)
        out[b] = acc
    return status, out.view(np.uint32)
