"""Helpers shared by the GPU tests: pinned/device tensors from numpy words and
one call of the CUDA path (preprocess -> plan -> compress)."""

import numpy as np
import torch

from host_transfer_gb300 import ibp


def pinned(a: np.ndarray) -> torch.Tensor:
    t = torch.empty(a.shape, dtype=torch.int32, pin_memory=True)
    t.numpy()[...] = np.ascontiguousarray(a).view(np.int32)
    return t


def on_device(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def place(a: np.ndarray, where: str) -> torch.Tensor:
    return pinned(a) if where == "host" else on_device(a)


def empty_like_in(t: torch.Tensor, where: str) -> torch.Tensor:
    if where == "host":
        return torch.empty(t.shape, dtype=torch.int32, pin_memory=True)
    return torch.empty(t.shape, dtype=torch.int32, device="cuda")


def words_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def gpu_codec(rows: np.ndarray, sample: np.ndarray, T: float, where: str = "host",
              inplace: bool = False):
    """Runs the CUDA path on rows: preprocess on `sample`, plan, compress.
    Returns dict(plan, mask, bitval, rows_t, slots_t, bitmask, stored)."""
    s = on_device(sample)
    mask, bitval = ibp.ibp_preprocess(s, T)
    plan = ibp.ibp_plan_create(mask, bitval)
    rows_t = place(rows, where)
    slots_t = rows_t if inplace else empty_like_in(rows_t, where)
    _, bitmask, stored = ibp.ibp_compress(plan, rows_t, slots_t)
    torch.cuda.synchronize()
    assert ibp.ibp_get_status(plan) == ibp.IBP_OK
    return dict(plan=plan, mask=words_np(mask), bitval=words_np(bitval), rows_t=rows_t,
                slots_t=slots_t, bitmask=words_np(bitmask), stored=int(stored.item()))
