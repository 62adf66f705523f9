"""ctypes wrapper of the C oracle (oracle/ibp_oracle.c).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline of the benchmark, never by the library.  Builds
``oracle/libibp_oracle.so`` with gcc on first use (or from ``build()``).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ibp_oracle.c")
_LIB = os.path.join(_HERE, "libibp_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", _LIB + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    u32p = ctypes.POINTER(ctypes.c_uint32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    u64 = ctypes.c_uint64
    lib.ibp_ref_set_threads.argtypes = [ctypes.c_int]
    lib.ibp_ref_threads.restype = ctypes.c_int
    lib.ibp_ref_preprocess.argtypes = [u32p, u64, ctypes.c_uint32, ctypes.c_double, u32p, u32p]
    lib.ibp_ref_compress.argtypes = [u32p, u64, ctypes.c_uint32, u32p, u32p, u32p, u32p,
                                     ctypes.POINTER(ctypes.c_uint64)]
    lib.ibp_ref_compress_some.argtypes = [u32p, u64, ctypes.c_uint32, u32p, u32p, i64p, u64,
                                          u32p, ctypes.POINTER(ctypes.c_uint8)]
    lib.ibp_ref_decompress.argtypes = [u32p, u64, ctypes.c_uint32, u32p, u32p, u32p, i64p, u64,
                                       u32p, ctypes.POINTER(ctypes.c_int)]
    lib.ibp_ref_row_words.argtypes = [u32p, u64, ctypes.c_uint32, u32p, u32p, u32p]
    lib.ibp_ref_decode_slots.argtypes = [u32p, ctypes.POINTER(ctypes.c_uint8), u64,
                                         ctypes.c_uint32, u32p, u32p, u32p,
                                         ctypes.POINTER(ctypes.c_int)]
    _lib = lib
    return lib


def _p(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _u32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint32:
        a = a.view(np.uint32) if a.dtype.itemsize == 4 else a.astype(np.uint32)
    return a


def set_threads(n: int) -> None:
    _load().ibp_ref_set_threads(int(n))


def threads() -> int:
    return int(_load().ibp_ref_threads())


def preprocess(sample: np.ndarray, T: float):
    """sample: (S_rows, W) 32-bit words.  Returns (status, mask, bitval)."""
    lib = _load()
    sample = _u32(sample)
    s_rows, W = sample.shape
    mask = np.zeros(W, np.uint32)
    bitval = np.zeros(W, np.uint32)
    st = lib.ibp_ref_preprocess(_p(sample, ctypes.c_uint32), s_rows, W, float(T),
                                _p(mask, ctypes.c_uint32), _p(bitval, ctypes.c_uint32))
    return st, mask, bitval


def compress(rows: np.ndarray, mask: np.ndarray, bitval: np.ndarray):
    """rows: (N, W) words.  Returns (slots, bitmask, stored_words)."""
    lib = _load()
    rows = _u32(rows)
    n, W = rows.shape
    slots = np.empty_like(rows)
    bitmask = np.zeros((n + 31) // 32, np.uint32)
    stored = ctypes.c_uint64(0)
    st = lib.ibp_ref_compress(_p(rows, ctypes.c_uint32), n, W, _p(_u32(mask), ctypes.c_uint32),
                              _p(_u32(bitval), ctypes.c_uint32), _p(slots, ctypes.c_uint32),
                              _p(bitmask, ctypes.c_uint32), ctypes.byref(stored))
    assert st == 0, st
    return slots, bitmask, int(stored.value)


def row_words(rows: np.ndarray, mask: np.ndarray, bitval: np.ndarray) -> np.ndarray:
    """Per row: Lw if stored compressed, else W."""
    lib = _load()
    rows = _u32(rows)
    n, W = rows.shape
    out = np.empty(n, np.uint32)
    st = lib.ibp_ref_row_words(_p(rows, ctypes.c_uint32), n, W, _p(_u32(mask), ctypes.c_uint32),
                               _p(_u32(bitval), ctypes.c_uint32), _p(out, ctypes.c_uint32))
    assert st == 0, st
    return out


def compress_some(rows: np.ndarray, ids: np.ndarray, mask: np.ndarray, bitval: np.ndarray):
    """Compress only rows[ids].  Returns (slots (len(ids), W), compressed bits (uint8))."""
    lib = _load()
    rows = _u32(rows)
    n, W = rows.shape
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    slots = np.empty((len(ids), W), np.uint32)
    bits = np.empty(len(ids), np.uint8)
    st = lib.ibp_ref_compress_some(_p(rows, ctypes.c_uint32), n, W, _p(_u32(mask), ctypes.c_uint32),
                                   _p(_u32(bitval), ctypes.c_uint32), _p(ids, ctypes.c_int64),
                                   len(ids), _p(slots, ctypes.c_uint32), _p(bits, ctypes.c_uint8))
    assert st == 0, st
    return slots, bits


def decompress(slots: np.ndarray, bitmask: np.ndarray, ids: np.ndarray, mask: np.ndarray,
               bitval: np.ndarray):
    """Returns (status, rows (len(ids), W))."""
    lib = _load()
    slots = _u32(slots)
    n, W = slots.shape
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    out = np.empty((len(ids), W), np.uint32)
    status = ctypes.c_int(0)
    st = lib.ibp_ref_decompress(_p(slots, ctypes.c_uint32), n, W, _p(_u32(bitmask), ctypes.c_uint32),
                                _p(_u32(mask), ctypes.c_uint32), _p(_u32(bitval), ctypes.c_uint32),
                                _p(ids, ctypes.c_int64), len(ids), _p(out, ctypes.c_uint32),
                                ctypes.byref(status))
    assert st == 0, st
    return int(status.value), out


def decode_slots(slots: np.ndarray, comp: np.ndarray, mask: np.ndarray, bitval: np.ndarray):
    """Decode standalone slots (n, W) with per-slot compressed flags."""
    lib = _load()
    slots = _u32(slots)
    n, W = slots.shape
    comp = np.ascontiguousarray(comp, dtype=np.uint8)
    out = np.empty((n, W), np.uint32)
    status = ctypes.c_int(0)
    st = lib.ibp_ref_decode_slots(_p(slots, ctypes.c_uint32), _p(comp, ctypes.c_uint8), n, W,
                                  _p(_u32(mask), ctypes.c_uint32), _p(_u32(bitval), ctypes.c_uint32),
                                  _p(out, ctypes.c_uint32), ctypes.byref(status))
    assert st == 0, st
    return int(status.value), out
