"""ibp_preprocess_noalloc - the preprocess entry point that allocates nothing -
checked through the C ABI against ibp_preprocess.

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

pytestmark = pytest.mark.gpu

IBP_NOALLOC_MAX_W = 4096


def _call(lib, name, sample, T, mask, bitval):
    stream = torch.cuda.current_stream().cuda_stream
    return getattr(lib, name)(ctypes.c_void_p(sample.data_ptr()), sample.shape[0], sample.shape[1],
                              ctypes.c_double(T), ctypes.c_void_p(mask.data_ptr()),
                              ctypes.c_void_p(bitval.data_ptr()), ctypes.c_void_p(stream))


def _sample(seed, n, W):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 0.05, (n, W)).astype(np.float32).view(np.int32)
    return torch.from_numpy(x).cuda()


def test_noalloc_matches_preprocess_on_calls_in_a_row():
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


def test_noalloc_rejects_rows_above_its_limit():
    lib = ibp.load()
    sample = _sample(4, 4, IBP_NOALLOC_MAX_W + 1)
    m = torch.empty(IBP_NOALLOC_MAX_W + 1, dtype=torch.int32, device="cuda")
    assert _call(lib, "ibp_preprocess_noalloc", sample, 0.9, m, m.clone()) == ibp.IBP_EINVAL
    assert b"IBP_NOALLOC_MAX_W" in lib.ibp_last_error_detail()
