"""Plain, bit-by-bit Python oracle of Invariant Bit Packing (IBP).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code, table or helper with the CUDA
library under ``host_transfer_gb300/``.

Source: the page "Résumé Technique : Réduire le goulot d'étranglement de la
mémoire GPU par la compression sans perte pour le ML" (gist.science, French
summary of the paper "Reducing the GPU Memory Bottleneck with Lossless
Compression for ML"), section « Algorithme central », steps 1 (preprocess),
2 (compression) and 3 (decompression), and section « Intégration au système »
(fixed-size in-place slots, GPU-resident per-tensor bitmask).  The Korean page
of the same paper ("... -- Extended", sections 핵심 알고리즘 and 시스템 통합)
says the same thing.

The pages describe the method in prose only.  Every bit-level choice below
that they leave open is a reading, stated where it is made:

* chunk = one word; the word width is the parameter ``B`` (32 for the real
  format, 8 for the exhaustive toy tests);
* one Mask/Bitval word per word position of the row;
* invariance: with ``t = ceil(T * S_rows)`` computed in IEEE double, a bit
  position is invariant when max(#ones, #zeros) >= t; its Bitval bit is 1
  exactly when #ones > #zeros (a tie gives 0);
* participation bits of B consecutive words form one B-bit header word; all
  header words of a row come first, then the payload fields back to back,
  least significant bit first, with no padding;
* a row is stored compressed only when its stream is strictly shorter than
  the row in words; the slot's tail after the stream is zero;
* a word with an all-zero mask still "matches" and keeps all B bits.

Parity status: pinned (see tests/test_oracle_pins.py).
"""

from __future__ import annotations

import math

# Status codes shared by name (not by code) with the library's C ABI.
OK = 0
EINVAL = 1
ECORRUPT = 4
ERANGE = 5


def _full(B: int) -> int:
    return (1 << B) - 1


def popcount(x: int) -> int:
    n = 0
    while x:
        n += x & 1
        x >>= 1
    return n


def pext(x: int, keep: int, B: int = 32) -> int:
    """Gather the bits of ``x`` at the set positions of ``keep`` (ascending)
    into the low bits of the result.  This is the "invariant bits are removed
    and the remaining bits are shifted to fill the gap" of step 2."""
    out = 0
    k = 0
    for pos in range(B):
        if (keep >> pos) & 1:
            out |= ((x >> pos) & 1) << k
            k += 1
    return out


def pdep(v: int, keep: int, B: int = 32) -> int:
    """Scatter the low bits of ``v`` to the set positions of ``keep``
    (ascending): the inverse placement used by step 3."""
    out = 0
    k = 0
    for pos in range(B):
        if (keep >> pos) & 1:
            out |= ((v >> k) & 1) << pos
            k += 1
    return out


def threshold(T: float, s_rows: int) -> int:
    """Number of sampled rows that must agree on a bit: ceil(T * S_rows), in
    IEEE double (Python floats are IEEE doubles)."""
    return int(math.ceil(T * float(s_rows)))


def preprocess(sample, T: float, B: int = 32):
    """Step 1 (« Prétraitement »): from a sample of rows (a list of rows, each
    a list of W words), find for each word position w and bit b whether at
    least a fraction T of the rows share that bit, and with which value.

    Returns (status, mask, bitval) with mask/bitval lists of W words.
    """
    s_rows = len(sample)
    if s_rows == 0 or not (T > 0.0 and T <= 1.0):
        return EINVAL, None, None
    W = len(sample[0])
    t = threshold(T, s_rows)
    mask = [0] * W
    bitval = [0] * W
    for w in range(W):
        for b in range(B):
            ones = 0
            for r in range(s_rows):
                ones += (sample[r][w] >> b) & 1
            zeros = s_rows - ones
            if max(ones, zeros) >= t:
                mask[w] |= 1 << b
                if ones > zeros:
                    bitval[w] |= 1 << b
    return OK, mask, bitval


class _BitWriter:
    """A stream of bits; bit k of the stream is bit (k mod B) of word k // B."""

    def __init__(self, B: int):
        self.B = B
        self.bits: list[int] = []

    def put(self, value: int, nbits: int):
        for i in range(nbits):
            self.bits.append((value >> i) & 1)

    def words(self) -> list[int]:
        B = self.B
        n = (len(self.bits) + B - 1) // B
        out = [0] * n
        for k, bit in enumerate(self.bits):
            out[k // B] |= bit << (k % B)
        return out


class _BitReader:
    def __init__(self, words, B: int):
        self.words = words
        self.B = B
        self.pos = 0

    def get(self, nbits: int) -> int:
        v = 0
        for i in range(nbits):
            k = self.pos + i
            v |= ((self.words[k // self.B] >> (k % self.B)) & 1) << i
        self.pos += nbits
        return v


def segments(W: int, B: int = 32) -> int:
    return (W + B - 1) // B


def encode_row(x, mask, bitval, B: int = 32):
    """Step 2 (« Compression ») for one row.

    Returns (stream_words, stream_bits, flags): the full participation-header
    plus payload stream, its length in bits and the per-word match flags.
    """
    W = len(x)
    full = _full(B)
    flags = []
    fields = []
    for w in range(W):
        m = mask[w]
        keep = ~m & full
        match = ((x[w] ^ bitval[w]) & m) == 0
        flags.append(1 if match else 0)
        if match:
            fields.append((pext(x[w], keep, B), B - popcount(m)))
        else:
            fields.append((x[w], B))
    bw = _BitWriter(B)
    S = segments(W, B)
    for s in range(S):
        h = 0
        for i in range(B):
            w = s * B + i
            if w < W and flags[w]:
                h |= 1 << i
        bw.put(h, B)
    for value, nbits in fields:
        bw.put(value, nbits)
    return bw.words(), len(bw.bits), flags


def compress_row(x, mask, bitval, B: int = 32):
    """Row rule (« Intégration au système »: fixed-size in-place buffers):
    returns (slot, compressed, stored_words)."""
    W = len(x)
    stream, nbits, _ = encode_row(x, mask, bitval, B)
    Lw = (nbits + B - 1) // B
    if Lw < W:
        return stream + [0] * (W - Lw), True, Lw
    return list(x), False, W


def compress(rows, mask, bitval, B: int = 32):
    """All rows.  Returns (slots, bitmask words, total stored words)."""
    n = len(rows)
    slots = []
    bitmask = [0] * ((n + 31) // 32)
    stored = 0
    for r, x in enumerate(rows):
        slot, comp, used = compress_row(x, mask, bitval, B)
        slots.append(slot)
        stored += used
        if comp:
            bitmask[r // 32] |= 1 << (r % 32)
    return slots, bitmask, stored


def stream_bits(headers, W: int, mask, B: int = 32) -> int:
    """Length in bits of a row's stream as announced by its header words."""
    nbits = B * len(headers)
    for w in range(W):
        if (headers[w // B] >> (w % B)) & 1:
            nbits += B - popcount(mask[w])
        else:
            nbits += B
    return nbits


def decode_stream(words, W: int, mask, bitval, B: int = 32):
    """Step 3 (« Décompression ») proper: read the S header words, then for
    each word take its field (B - popcount(mask) bits if its participation bit
    is set, else B bits) and put the invariant bits of Bitval back at the Mask
    positions."""
    full = _full(B)
    S = segments(W, B)
    rd = _BitReader(words, B)
    headers = [rd.get(B) for _ in range(S)]
    out = []
    for w in range(W):
        m = mask[w]
        keep = ~m & full
        if (headers[w // B] >> (w % B)) & 1:
            v = rd.get(B - popcount(m))
            out.append(pdep(v, keep, B) | (bitval[w] & m))
        else:
            out.append(rd.get(B))
    return out


def decode_row(slot, compressed: bool, mask, bitval, B: int = 32):
    """One slot: returns (status, row).  A raw slot is the row itself.  A
    compressed slot is corrupt when a header bit past the last word is set or
    when its headers announce a stream of W words or more (such a row would
    have been stored raw); a corrupt slot decodes to zeros."""
    W = len(slot)
    if not compressed:
        return OK, list(slot)
    S = segments(W, B)
    headers = slot[:S]
    for s in range(S):
        for i in range(B):
            if s * B + i >= W and (headers[s] >> i) & 1:
                return ECORRUPT, [0] * W
    if (stream_bits(headers, W, mask, B) + B - 1) // B >= W:
        return ECORRUPT, [0] * W
    return OK, decode_stream(slot, W, mask, bitval, B)


def gather_decompress(slots, bitmask, ids, mask, bitval, B: int = 32):
    """Decode the rows named by ``ids`` (in order).  Returns (status, rows):
    the first error met, and zero rows where an id is out of range or a slot
    is corrupt."""
    n_rows = len(slots)
    W = len(mask)
    status = OK
    out = []
    for r in ids:
        if r < 0 or r >= n_rows:
            if status == OK:
                status = ERANGE
            out.append([0] * W)
            continue
        comp = (bitmask[r // 32] >> (r % 32)) & 1
        st, row = decode_row(slots[r], bool(comp), mask, bitval, B)
        if st != OK and status == OK:
            status = st
        out.append(row)
    return status, out
