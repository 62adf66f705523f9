"""Python binding of libibp (ctypes).  Argument marshalling only: every step
runs in the library's CUDA kernels.  PyTorch supplies device memory, pinned
host memory and streams.

Names follow the C ABI in include/ibp.h:

    mask, bitval = ibp_preprocess(sample, T)
    plan = ibp_plan_create(mask, bitval)
    bitmask, stored = ibp_compress(plan, rows)                 # in place
    out = ibp_gather_decompress(plan, slots, bitmask, row_ids)
    out = ibp_decompress_contig(plan, slots, bitmask, first_row, n)
    ibp_get_status(plan)                                         # raises on a data error

Word tensors: any contiguous tensor whose last dimension is a whole number of
32-bit words (int32/uint32/float32, or bfloat16/float16 with an even last
dimension) is viewed as rows of 32-bit words.  Tables passed as host tensors
must be pinned (``pin_memory=True``): kernels read them in place (zero copy).
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libibp.so")

IBP_OK = 0
IBP_EINVAL = 1
IBP_ECUDA = 2
IBP_ENOMEM = 3
IBP_ECORRUPT = 4
IBP_ERANGE = 5
IBP_ETIMEOUT = 6

IBP_HINT_ROW_REUSE = 1
IBP_HINT_EARLY_FETCH = 2

_lib = None


class IbpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if _lib is not None:
            detail = _lib.ibp_last_error_detail().decode(errors="replace")
            msg = _lib.ibp_strerror(code).decode()
        else:
            msg = f"status {code}"
        super().__init__(f"{where}: {msg}" + (f" ({detail})" if detail else ""))


class PlanInfo(ctypes.Structure):
    _fields_ = [("W", ctypes.c_uint32), ("segments", ctypes.c_uint32), ("uniform", ctypes.c_uint32),
                ("max_runs", ctypes.c_uint32), ("min_kept_bits", ctypes.c_uint32),
                ("max_kept_bits", ctypes.c_uint32), ("metadata_bytes", ctypes.c_uint64),
                ("device", ctypes.c_int), ("prefix_words", ctypes.c_uint32),
                ("short_rows", ctypes.c_uint32)]


def load():
    """Load libibp.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing; build it with `python -m host_transfer_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, u64, u32, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
    sigs = {
        "ibp_strerror": ([i32], ctypes.c_char_p),
        "ibp_version": ([], i32),
        "ibp_last_error_detail": ([], ctypes.c_char_p),
        "ibp_preprocess": ([vp, u64, u32, ctypes.c_double, vp, vp, vp], i32),
        "ibp_preprocess_noalloc": ([vp, u64, u32, ctypes.c_double, vp, vp, vp], i32),
        "ibp_plan_create": ([vp, vp, u32, i32, ctypes.POINTER(vp)], i32),
        "ibp_plan_destroy": ([vp], i32),
        "ibp_plan_get_info": ([vp, ctypes.POINTER(PlanInfo)], i32),
        "ibp_plan_get_mask": ([vp, vp, vp], i32),
        "ibp_plan_set_hints": ([vp, u32], i32),
        "ibp_plan_tune_prefix": ([vp, vp, u64, vp, u64, ctypes.POINTER(u32), vp], i32),
        "ibp_plan_set_prefix": ([vp, u32], i32),
        "ibp_gather_decompress_bag": ([vp, vp, u64, vp, vp, u64, vp, u64, u32, vp, vp], i32),
        "ibp_plan_set_create": ([ctypes.POINTER(vp), u32, ctypes.POINTER(vp)], i32),
        "ibp_plan_set_destroy": ([vp], i32),
        "ibp_decompress_contig_set": ([vp, vp, u64, vp, vp, vp], i32),
        "ibp_plan_set_get_status": ([vp, vp], i32),
        "ibp_compress": ([vp, vp, vp, u64, vp, vp, vp], i32),
        "ibp_gather_decompress": ([vp, vp, u64, vp, vp, u64, vp, vp], i32),
        "ibp_decompress_contig": ([vp, vp, u64, vp, u64, u64, vp, vp], i32),
        "ibp_get_status": ([vp, vp], i32),
        "ibp_get_status_async": ([vp, vp, vp], i32),
        "ibp_gather_raw": ([vp, u64, u32, vp, u64, vp, vp], i32),
        "ibp_row_lengths": ([vp, vp, u64, vp, vp, u64, vp, vp], i32),
        "ibp_packed_offsets": ([vp, vp, u64, vp, vp, vp], i32),
        "ibp_pack": ([vp, vp, u64, vp, vp, vp], i32),
        "ibp_gather_decompress_packed": ([vp, vp, vp, u64, vp, vp, u64, vp, vp], i32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != IBP_OK:
        raise IbpError(code, where)


def words(t: torch.Tensor) -> torch.Tensor:
    """View a contiguous tensor as 32-bit words (int32), keeping its rows."""
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    if t.element_size() == 4:
        return t.view(torch.int32)
    if t.element_size() == 2:
        if t.shape[-1] % 2:
            raise ValueError("16-bit rows need an even number of elements")
        return t.view(torch.int32)
    if t.element_size() == 8 and t.dtype == torch.int64:
        raise ValueError("int64 tensors are not word tensors")
    raise ValueError(f"unsupported dtype {t.dtype}")


def _rows(t: torch.Tensor):
    w = words(t)
    if w.dim() == 1:
        w = w.view(1, -1)
    w = w.reshape(-1, w.shape[-1])
    return w, w.shape[0], w.shape[1]


def _word_rows(t: torch.Tensor):
    """(data pointer, rows, words per row) of a contiguous word tensor, without
    building views (the per-call path of the gather entry points)."""
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    es = t.element_size()
    last = t.shape[-1] if t.dim() else 1
    if es == 4:
        W = last
    elif es == 2 and last % 2 == 0:
        W = last // 2
    else:
        raise ValueError(f"unsupported dtype {t.dtype} / row length")
    n = (t.numel() * es) // (4 * W) if W else 0
    return t.data_ptr(), n, W


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device) -> int:
    """The cudaStream_t to launch on, as a plain int: `stream`, else torch's
    current stream of `device` (read as a raw handle: no Stream object per
    call)."""
    if stream is None:
        if _raw_stream is not None:
            idx = device if isinstance(device, int) else torch.device(device).index
            return _raw_stream(torch.cuda.current_device() if idx is None else idx)
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    """A tensor's data pointer as a plain int (ctypes passes it as void*)."""
    return t.data_ptr() if t is not None else None


def _device_of(*ts) -> torch.device:
    for t in ts:
        if t is not None and t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def ibp_preprocess(sample: torch.Tensor, T: float, mask: torch.Tensor | None = None,
                   bitval: torch.Tensor | None = None, stream=None):
    """Mask and Bitval (int32 device tensors of W words) from sampled rows."""
    lib = load()
    s, n, W = _rows(sample)
    dev = _device_of(sample, mask, bitval)
    if mask is None:
        mask = torch.empty(W, dtype=torch.int32, device=dev)
    if bitval is None:
        bitval = torch.empty(W, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.ibp_preprocess(_ptr(s), n, W, float(T), _ptr(mask), _ptr(bitval),
                                  _stream(stream, dev)), "ibp_preprocess")
    return mask, bitval


def ibp_preprocess_noalloc(sample: torch.Tensor, T: float, mask: torch.Tensor, bitval: torch.Tensor,
                           stream=None):
    """ibp_preprocess for callers that cannot let the library allocate device
    memory: its scratch is a fixed per-GPU array (W <= IBP_NOALLOC_MAX_W), and
    the caller passes the outputs.  Calls that overlap on the GPU race."""
    lib = load()
    s, n, W = _rows(sample)
    dev = _device_of(sample, mask, bitval)
    with torch.cuda.device(dev):
        _check(lib.ibp_preprocess_noalloc(_ptr(s), n, W, float(T), _ptr(mask), _ptr(bitval),
                                          _stream(stream, dev)), "ibp_preprocess_noalloc")
    return mask, bitval


class Plan:
    """A device plan (Mask, Bitval and derived tables).  Frees itself."""

    def __init__(self, handle: int, W: int, device: int):
        self.handle = ctypes.c_void_p(handle)
        self.W = W
        self.device = device

    @property
    def info(self) -> dict:
        lib = load()
        inf = PlanInfo()
        _check(lib.ibp_plan_get_info(self.handle, ctypes.byref(inf)), "ibp_plan_get_info")
        return {k: getattr(inf, k) for k, _ in PlanInfo._fields_}

    def set_hints(self, hints: int):
        """IBP_HINT_* access hints for later decompress calls (0 = default)."""
        _check(load().ibp_plan_set_hints(self.handle, int(hints)), "ibp_plan_set_hints")

    def set_prefix(self, words: int):
        """Words fetched from every slot before its headers are read (0 = default)."""
        _check(load().ibp_plan_set_prefix(self.handle, int(words)), "ibp_plan_set_prefix")

    def mask_bitval(self):
        lib = load()
        m = torch.empty(self.W, dtype=torch.int32)
        b = torch.empty(self.W, dtype=torch.int32)
        _check(lib.ibp_plan_get_mask(self.handle, _ptr(m), _ptr(b)), "ibp_plan_get_mask")
        return m, b

    def destroy(self):
        if self.handle is not None and self.handle.value:
            load().ibp_plan_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def ibp_plan_create(mask: torch.Tensor, bitval: torch.Tensor, device: int | None = None) -> Plan:
    lib = load()
    m = words(mask.contiguous()).reshape(-1)
    b = words(bitval.contiguous()).reshape(-1)
    if m.numel() != b.numel():
        raise ValueError("mask and bitval differ in length")
    if device is None:
        device = m.device.index if m.is_cuda else torch.cuda.current_device()
    h = ctypes.c_void_p()
    _check(lib.ibp_plan_create(_ptr(m), _ptr(b), m.numel(), int(device), ctypes.byref(h)),
           "ibp_plan_create")
    return Plan(h.value, m.numel(), int(device))


def bitmask_words(n_rows: int) -> int:
    return (n_rows + 31) // 32


def ibp_compress(plan: Plan, rows: torch.Tensor, slots: torch.Tensor | None = None,
                 bitmask: torch.Tensor | None = None, stored: torch.Tensor | None = None,
                 stream=None):
    """Compress rows into slots (in place when slots is None).  Returns
    (slots, bitmask, stored) where stored is a device int64 tensor with the
    words a reader fetches (added to `stored` when given)."""
    lib = load()
    r, n, W = _rows(rows)
    if W != plan.W:
        raise ValueError(f"rows have {W} words, plan has {plan.W}")
    dev = torch.device("cuda", plan.device)
    s = r if slots is None else _rows(slots)[0]
    if bitmask is None:
        bitmask = torch.empty(bitmask_words(n), dtype=torch.int32, device=dev)
    if stored is None:
        stored = torch.zeros(1, dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        _check(lib.ibp_compress(plan.handle, _ptr(r), _ptr(s), n, _ptr(bitmask), _ptr(stored),
                                _stream(stream, dev)), "ibp_compress")
    return (rows if slots is None else slots), bitmask, stored


def ibp_gather_decompress(plan: Plan, slots: torch.Tensor, bitmask: torch.Tensor,
                          row_ids: torch.Tensor, out: torch.Tensor | None = None, stream=None,
                          n_rows: int | None = None) -> torch.Tensor:
    lib = load()
    sp, n, W = _word_rows(slots)
    if W != plan.W:
        raise ValueError(f"slots have {W} words, plan has {plan.W}")
    if row_ids.dtype != torch.int64 or not row_ids.is_contiguous():
        raise ValueError("row_ids must be a contiguous int64 tensor")
    k = row_ids.numel()
    if out is None:
        out = torch.empty((k, W), dtype=torch.int32, device=torch.device("cuda", plan.device))
    _check(lib.ibp_gather_decompress(plan.handle, sp, n if n_rows is None else n_rows,
                                     _ptr(bitmask), _ptr(row_ids), k, _ptr(out),
                                     _stream(stream, plan.device)), "ibp_gather_decompress")
    return out


def ibp_decompress_contig(plan: Plan, slots: torch.Tensor, bitmask: torch.Tensor, first_row: int,
                          n: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    lib = load()
    sp, n_rows, W = _word_rows(slots)
    if W != plan.W:
        raise ValueError(f"slots have {W} words, plan has {plan.W}")
    if out is None:
        out = torch.empty((n, W), dtype=torch.int32, device=torch.device("cuda", plan.device))
    _check(lib.ibp_decompress_contig(plan.handle, sp, n_rows, _ptr(bitmask), int(first_row), int(n),
                                     _ptr(out), _stream(stream, plan.device)),
           "ibp_decompress_contig")
    return out


def ibp_get_status(plan: Plan, stream=None, raise_on_error: bool = True) -> int:
    lib = load()
    dev = torch.device("cuda", plan.device)
    code = lib.ibp_get_status(plan.handle, _stream(stream, dev))
    if raise_on_error and code != IBP_OK:
        raise IbpError(code, "ibp_get_status")
    return code


def ibp_get_status_async(plan: Plan, status_out: torch.Tensor, stream=None) -> torch.Tensor:
    """Enqueue the move of the plan's status word into `status_out` (one int32
    word of pinned host or device memory; a view of a larger tensor is fine)
    and return without waiting: read it after synchronising with the stream."""
    lib = load()
    if status_out.element_size() != 4 or not status_out.is_contiguous():
        raise ValueError("status_out must be a contiguous 32-bit word")
    _check(lib.ibp_get_status_async(plan.handle, _ptr(status_out), _stream(stream, plan.device)),
           "ibp_get_status_async")
    return status_out


def ibp_row_lengths(plan: Plan, slots: torch.Tensor, bitmask: torch.Tensor, row_ids: torch.Tensor,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Words a reader fetches per requested row (int32 device tensor)."""
    lib = load()
    s, n, W = _rows(slots)
    dev = torch.device("cuda", plan.device)
    k = row_ids.numel()
    if out is None:
        out = torch.empty(k, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.ibp_row_lengths(plan.handle, _ptr(s), n, _ptr(bitmask), _ptr(row_ids), k,
                                   _ptr(out), _stream(stream, dev)), "ibp_row_lengths")
    return out


IBP_BAG_SUM = 0
IBP_BAG_MEAN = 1
IBP_BAG_BF16 = 2


def ibp_gather_decompress_bag(plan: Plan, slots: torch.Tensor, bitmask: torch.Tensor, row_ids: torch.Tensor,
                              bag_offsets: torch.Tensor, mode: int = IBP_BAG_SUM,
                              out: torch.Tensor | None = None, stream=None,
                              n_rows: int | None = None) -> torch.Tensor:
    """Pooled rows per bag (float32 device tensor [n_bags, W], or [n_bags, 2W]
    with IBP_BAG_BF16 in mode) of the rows row_ids[bag_offsets[b] ..
    bag_offsets[b+1])."""
    lib = load()
    sp, n, W = _word_rows(slots)
    if W != plan.W:
        raise ValueError(f"slots have {W} words, plan has {plan.W}")
    for name, t in (("row_ids", row_ids), ("bag_offsets", bag_offsets)):
        if t.dtype != torch.int64 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int64 tensor")
    n_bags = bag_offsets.numel() - 1
    dev = torch.device("cuda", plan.device)
    if out is None:
        width = 2 * W if int(mode) & IBP_BAG_BF16 else W
        out = torch.empty((max(n_bags, 0), width), dtype=torch.float32, device=dev)
    if n_bags <= 0:
        return out
    with torch.cuda.device(dev):
        _check(lib.ibp_gather_decompress_bag(plan.handle, sp, n if n_rows is None else n_rows, _ptr(bitmask),
                                             _ptr(row_ids) if row_ids.numel() else None, row_ids.numel(),
                                             _ptr(bag_offsets), n_bags, int(mode), _ptr(out),
                                             _stream(stream, dev)), "ibp_gather_decompress_bag")
    return out


class PlanSet:
    """Plans for consecutive row blocks of one table (finer Mask granularity).
    Keeps its plans alive; frees itself."""

    def __init__(self, plans):
        lib = load()
        self.plans = list(plans)
        if not self.plans:
            raise ValueError("a plan set needs at least one plan")
        arr = (ctypes.c_void_p * len(self.plans))(*[p.handle.value for p in self.plans])
        h = ctypes.c_void_p()
        _check(lib.ibp_plan_set_create(arr, len(self.plans), ctypes.byref(h)), "ibp_plan_set_create")
        self.handle = h
        self.W = self.plans[0].W
        self.device = self.plans[0].device

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.ibp_plan_set_destroy(self.handle)
            self.handle = None


def ibp_plan_set_create(plans) -> PlanSet:
    return PlanSet(plans)


def ibp_decompress_contig_set(pset: PlanSet, slots: torch.Tensor, rows_per_plan: int, bitmask: torch.Tensor,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode n_plans * rows_per_plan rows; row block k with plan k."""
    lib = load()
    sp, n, W = _word_rows(slots)
    dev = torch.device("cuda", pset.device)
    total = rows_per_plan * len(pset.plans)
    if n < total:
        raise ValueError(f"slots hold {n} rows, the set decodes {total}")
    if out is None:
        out = torch.empty((total, W), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.ibp_decompress_contig_set(pset.handle, sp, int(rows_per_plan), _ptr(bitmask), _ptr(out),
                                             _stream(stream, dev)), "ibp_decompress_contig_set")
    return out


def ibp_plan_set_get_status(pset: PlanSet, stream=None, raise_on_error: bool = True) -> int:
    lib = load()
    dev = torch.device("cuda", pset.device)
    code = lib.ibp_plan_set_get_status(pset.handle, _stream(stream, dev))
    if raise_on_error and code != IBP_OK:
        raise IbpError(code, "ibp_plan_set_get_status")
    return code


def ibp_plan_tune_prefix(plan: Plan, slots: torch.Tensor, bitmask: torch.Tensor, max_sample: int = 0,
                         stream=None) -> int:
    """Set the plan's prefix from the stored lengths of sampled rows of a
    compressed table; returns the prefix in words.  Synchronises the stream."""
    lib = load()
    sp, n, W = _word_rows(slots)
    got = ctypes.c_uint32(0)
    dev = torch.device("cuda", plan.device)
    with torch.cuda.device(dev):
        _check(lib.ibp_plan_tune_prefix(plan.handle, sp, n, _ptr(bitmask), int(max_sample), ctypes.byref(got),
                                        _stream(stream, dev)), "ibp_plan_tune_prefix")
    return int(got.value)


def ibp_packed_offsets(plan: Plan, slots: torch.Tensor, bitmask: torch.Tensor,
                       offsets: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Row offsets (int64 device tensor of n_rows + 1 words) of the packed cache
    layout of these slots; offsets[-1] is the packed size in words."""
    lib = load()
    sp, n, W = _word_rows(slots)
    if offsets is None:
        offsets = torch.empty(n + 1, dtype=torch.int64, device=torch.device("cuda", plan.device))
    _check(lib.ibp_packed_offsets(plan.handle, sp, n, _ptr(bitmask), _ptr(offsets),
                                  _stream(stream, plan.device)), "ibp_packed_offsets")
    return offsets


def ibp_pack(plan: Plan, slots: torch.Tensor, offsets: torch.Tensor, packed: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """Packed copy of the slots (int32 device tensor of offsets[-1] words).
    Allocating it reads offsets[-1] back to the host (a synchronisation)."""
    lib = load()
    sp, n, W = _word_rows(slots)
    if packed is None:
        total = int(offsets[-1].item())
        packed = torch.empty(max(total, 4), dtype=torch.int32, device=torch.device("cuda", plan.device))
    _check(lib.ibp_pack(plan.handle, sp, n, _ptr(offsets), _ptr(packed), _stream(stream, plan.device)),
           "ibp_pack")
    return packed


def ibp_gather_decompress_packed(plan: Plan, packed: torch.Tensor, offsets: torch.Tensor,
                                 bitmask: torch.Tensor, row_ids: torch.Tensor,
                                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    lib = load()
    if row_ids.dtype != torch.int64 or not row_ids.is_contiguous():
        raise ValueError("row_ids must be a contiguous int64 tensor")
    n_rows = offsets.numel() - 1
    k = row_ids.numel()
    if out is None:
        out = torch.empty((k, plan.W), dtype=torch.int32, device=torch.device("cuda", plan.device))
    _check(lib.ibp_gather_decompress_packed(plan.handle, _ptr(packed), _ptr(offsets), n_rows,
                                            _ptr(bitmask), _ptr(row_ids), k, _ptr(out),
                                            _stream(stream, plan.device)), "ibp_gather_decompress_packed")
    return out


def ibp_gather_raw(rows: torch.Tensor, row_ids: torch.Tensor, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    lib = load()
    rp, n, W = _word_rows(rows)
    dev = _device_of(row_ids, out)
    k = row_ids.numel()
    if out is None:
        out = torch.empty((k, W), dtype=torch.int32, device=dev)
    _check(lib.ibp_gather_raw(rp, n, W, _ptr(row_ids), k, _ptr(out), _stream(stream, dev)),
           "ibp_gather_raw")
    return out
