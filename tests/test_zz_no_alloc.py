"""ibp_preprocess_noalloc - the preprocess entry point that allocates nothing -
checked through the C ABI against ibp_preprocess and against the oracle.

Some callers cannot let a library allocate device memory: a process whose
device memory is all owned by its own allocator, or a device without
stream-ordered memory pools.  For them the counters of the preprocess live
in a fixed per-GPU array that every call shares, so each call must clear
what it uses: the second and third calls below would see the first call's
counts otherwise.  This file is collected last so that a run stopping at the
first failure has run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from host_transfer_gb300 import ibp
from oracle import oracle_c as C

pytestmark = pytest.mark.gpu

IBP_NOALLOC_MAX_W = 4096
# CUmemPool_attribute values (cuda.h): the used-memory high watermark of a pool
CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8


def _call(lib, name, sample, T, mask, bitval):
    stream = torch.cuda.current_stream().cuda_stream
    return getattr(lib, name)(ctypes.c_void_p(sample.data_ptr()), sample.shape[0], sample.shape[1],
                              ctypes.c_double(T), ctypes.c_void_p(mask.data_ptr()),
                              ctypes.c_void_p(bitval.data_ptr()), ctypes.c_void_p(stream))


def _sample(seed, n, W):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 0.05, (n, W)).astype(np.float32).view(np.int32)
    return torch.from_numpy(x).cuda()


class _DefaultPool:
    """The high watermark of the current device's default stream-ordered memory
    pool (where cudaMallocAsync takes its memory), read through the driver."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def reset_high(self):
        zero = ctypes.c_uint64(0)  # setting 0 resets the watermark to the current use
        assert self.cu.cuMemPoolSetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(zero)) == 0

    def high(self) -> int:
        v = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolGetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(v)) == 0
        return v.value


def test_noalloc_matches_preprocess_and_oracle_on_calls_in_a_row():
    from host_transfer_gb300 import build

    build.build()
    lib = ibp.load()
    cases = [(_sample(1, 5000, 128), 0.99), (_sample(2, 3000, IBP_NOALLOC_MAX_W), 0.9),
             (_sample(3, 777, 128), 0.75)]
    for sample, T in cases:
        W = sample.shape[1]
        m0 = torch.empty(W, dtype=torch.int32, device="cuda")
        b0 = torch.empty_like(m0)
        m1 = torch.full_like(m0, -1)
        b1 = torch.full_like(m0, -1)
        assert _call(lib, "ibp_preprocess", sample, T, m0, b0) == ibp.IBP_OK
        assert _call(lib, "ibp_preprocess_noalloc", sample, T, m1, b1) == ibp.IBP_OK
        torch.cuda.synchronize()
        # integer results: bit-exact, the same bar as every other parity test
        assert torch.equal(m0, m1) and torch.equal(b0, b1)
        st, m, b = C.preprocess(sample.cpu().numpy().view(np.uint32), T)
        assert st == 0
        assert np.array_equal(m1.cpu().numpy().view(np.uint32), m), "Mask differs from the oracle"
        assert np.array_equal(b1.cpu().numpy().view(np.uint32), b), "Bitval differs from the oracle"


def test_noalloc_takes_no_memory_from_the_pool():
    """ibp_preprocess takes its scratch from the default memory pool (its call
    raises the pool's high watermark); ibp_preprocess_noalloc must not."""
    lib = ibp.load()
    pool = _DefaultPool()
    sample = _sample(5, 2048, 1024)
    m = torch.empty(1024, dtype=torch.int32, device="cuda")
    b = torch.empty_like(m)
    torch.cuda.synchronize()
    pool.reset_high()
    before = pool.high()
    assert _call(lib, "ibp_preprocess", sample, 0.99, m, b) == ibp.IBP_OK
    torch.cuda.synchronize()
    assert pool.high() >= before + 128 * 1024, "the pool check does not see a stream-ordered allocation"
    torch.cuda.synchronize()
    pool.reset_high()
    before = pool.high()
    alloc_before = torch.cuda.memory_allocated()
    for _ in range(2):
        assert _call(lib, "ibp_preprocess_noalloc", sample, 0.99, m, b) == ibp.IBP_OK
    torch.cuda.synchronize()
    assert pool.high() == before
    assert torch.cuda.memory_allocated() == alloc_before


def test_noalloc_rejects_rows_above_its_limit():
    lib = ibp.load()
    sample = _sample(4, 4, IBP_NOALLOC_MAX_W + 1)
    m = torch.empty(IBP_NOALLOC_MAX_W + 1, dtype=torch.int32, device="cuda")
    assert _call(lib, "ibp_preprocess_noalloc", sample, 0.9, m, m.clone()) == ibp.IBP_EINVAL
    assert b"IBP_NOALLOC_MAX_W" in lib.ibp_last_error_detail()


def test_noalloc_call_captured_in_a_graph():
    """After a first call outside any capture, a call is captured in a CUDA
    graph; replays on new samples written into the same buffer give the
    oracle's Mask and Bitval each time (each replay clears its counters)."""
    lib = ibp.load()
    W, n, T = 256, 1500, 0.9
    sample = _sample(6, n, W)
    m = torch.empty(W, dtype=torch.int32, device="cuda")
    b = torch.empty_like(m)
    assert _call(lib, "ibp_preprocess_noalloc", sample, T, m, b) == ibp.IBP_OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rc = _call(lib, "ibp_preprocess_noalloc", sample, T, m, b)
    assert rc == ibp.IBP_OK
    for seed in (7, 8):
        sample.copy_(_sample(seed, n, W))
        m.fill_(-1)
        b.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        st, mo, bo = C.preprocess(sample.cpu().numpy().view(np.uint32), T)
        assert st == 0
        assert np.array_equal(m.cpu().numpy().view(np.uint32), mo), seed
        assert np.array_equal(b.cpu().numpy().view(np.uint32), bo), seed
