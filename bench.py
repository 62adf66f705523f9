#!/usr/bin/env python
"""Benchmark of IBP gather-decompress on one GB300 (or N replicas).

Workload (default): the dense GNN feature table - 2,000,000 rows x 128 fp32
(1.02 GB), N(0,1) rows L2-normalised, in pinned host memory, compressed in
place on the GPU with Mask/Bitval learned from 65,536 sampled rows at
T = 0.99.  A step is one gather-decompress of a batch of 65,536 uniform row
ids into HBM: the kernel reads the compressed slots straight from host memory
(zero copy), rebuilds the rows and writes them to HBM.

One JSON line on stdout.  `value` is decompressed output GB/s (uncompressed
bytes) over all ranks, timed with CUDA events over K steps after W warm-up
steps; slots are in pinned host memory, ids already on the device.  Also
reported: the H2D copy ceiling measured in the same run, the space saving,
the same kernel on HBM-resident slots against the HBM roofline, the
uncompressed zero-copy gather of the same rows, an end-to-end leg through the
public API (ids copied from pinned host memory, status read back each step)
and the CPU oracle timed on the host cores.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]
    torchrun --nproc-per-node N bench.py --gpus N     (independent replicas)
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decompressed GB/s (uncompressed bytes) vs PCIe/compress-ratio and HBM roofline; space saving %"
HBM_FALLBACK_GBS = 6800.0
POOL = 64  # distinct id batches; step k uses batch k % POOL (64 x 30 MB of slots > L2)
SOAK_S = 0.5  # untimed decode loop under the clock sampler before the warm-up


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", choices=["dense_gnn", "sparse_gnn", "dlrm", "llm"], default="dense_gnn")
    p.add_argument("--layers", type=int, default=8, help="llm: layers generated (steps cycle over them)")
    p.add_argument("--rows", type=int, default=None, help="fewer table rows (quick runs only)")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle sample budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed helpers (independent replicas: no data-path collective)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def batch_seed_offset(rank: int) -> int:
    """Replica r draws its own id batches: batch k of rank r uses index
    k + 100000 * r of the configuration's batch sequence."""
    return 100_000 * rank


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            if self.uuid and f[1] != self.uuid:
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


KERNEL_SOURCES = ["ibp_decompress_fast.cuh", "ibp_decompress_fast_u.cu", "ibp_decompress_fast_t.cu",
                  "ibp_decompress_fast_up.cu", "ibp_decompress_fast_tp.cu", "ibp_decompress_fast_ur.cu",
                  "ibp_decompress_fast_tr.cu", "ibp_decompress_fast_td.cu", "ibp_decompress_fast_ud.cu",
                  "ibp_decompress_fast_set.cu",
                  "ibp_decompress.cu", "ibp_internal.cuh", "ibp_api.cu"]


def kernel_sources_sha() -> str:
    """sha256 over the sources of the decompress kernels."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "host_transfer_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def kernel_traffic(kind: str, config: str) -> dict:
    """Measured traffic per launch of one bench leg from the committed ncu
    summary, when it was taken on this workload and the current kernel sources
    (else {}): dram = DRAM bytes read + written; link = bytes over the host
    link (sysmem sectors x 32)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        rec = json.load(open(path))
        sha = kernel_sources_sha()
    except (OSError, ValueError):
        return {}
    ent = rec.get(config, {}).get(kind)
    if not ent or ent.get("kernel_source_sha256") != sha:
        return {}
    return {"dram": ent.get("dram_bytes_read", 0) + ent.get("dram_bytes_write", 0),
            "link": ent.get("link_bytes")}


def workload_desc(name: str, n_rows: int) -> str:
    from host_transfer_gb300 import workloads

    c = workloads.CONFIGS[name]
    return {
        "dense_gnn": f"dense GNN features: {n_rows:,} rows x 128 fp32, N(0,1) rows L2-normalised, "
                     f"pinned host, T=0.99, gather batches of {c['batch']:,} uniform ids into HBM",
        "sparse_gnn": f"sparse GNN features: {n_rows:,} rows x 512 fp32, 95% zeros, lognormal "
                      f"non-zeros, pinned host, T=0.95, gather batches of {c['batch']:,} uniform ids",
        "dlrm": f"DLRM embedding table: {n_rows:,} rows x 64 fp32 U(-0.01,0.01), pinned host, "
                f"T=0.99, gather batches of {c['batch']:,} Zipf(1.05) ids",
    }[name]


def graph_of(torch, fn, count, first, pool):
    """Capture fn(k) for k = first .. first + count - 1 (batch k mod pool) as
    one CUDA graph, so the timed steps run back to back on the GPU with no
    host enqueue time between them."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for k in range(count):
            fn((first + k) % pool)
    return g


def make_batches(name, n_rows, count, offset):
    from host_transfer_gb300 import workloads

    zipf = None
    if name == "dlrm":
        c = workloads.CONFIGS[name]
        zipf = workloads.ZipfIds(n_rows, c["zipf_s"], c["seed"])
    return np.stack([workloads.batch_ids(name, offset + k, n_rows=n_rows, zipf=zipf) for k in range(count)])


def cpu_oracle_decode(slots, bitmask, mask, bitval, batches, seconds, threads):
    """Time the C oracle decoding rows of the same batches for about
    `seconds`; returns (GB/s of uncompressed output, rows decoded, seconds)."""
    from oracle import oracle_c

    oracle_c.set_threads(threads)
    W = slots.shape[1]
    chunk = 8192
    rows_done, t_used, k = 0, 0.0, 0
    flat = batches.reshape(-1)
    nchunks = max(1, flat.size // chunk)
    while t_used < seconds:
        ids = flat[(k % nchunks) * chunk:(k % nchunks + 1) * chunk]
        t0 = time.perf_counter()
        st, _ = oracle_c.decompress(slots, bitmask, ids, mask, bitval)
        t_used += time.perf_counter() - t0
        assert st == 0
        rows_done += len(ids)
        k += 1
    return rows_done * 4 * W / t_used / 1e9, rows_done, t_used


def cpu_oracle_compress(rows, mask, bitval, seconds, threads):
    """Time the C oracle compressing `rows` (repeated for about `seconds`);
    returns (GB/s of uncompressed input, rows compressed, seconds)."""
    from oracle import oracle_c

    oracle_c.set_threads(threads)
    rows_done, t_used = 0, 0.0
    while t_used < seconds:
        t0 = time.perf_counter()
        oracle_c.compress(rows, mask, bitval)
        t_used += time.perf_counter() - t0
        rows_done += rows.shape[0]
    return rows_done * 4 * rows.shape[1] / t_used / 1e9, rows_done, t_used


# ---------------------------------------------------------------------------


def run_reference(args):
    """The CPU oracle as the reference arm: each step decodes a bounded
    sample of a batch of the same workload on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.config == "llm":
        raise SystemExit("--impl reference covers the row-table configurations")
    from host_transfer_gb300 import workloads
    from oracle import oracle_c

    name = args.config
    c = workloads.CONFIGS[name]
    n = args.rows or c["n_rows"]
    W = c["W"]
    rows = workloads.make_table(name, n_rows=n)
    sample = rows[workloads.sample_ids(n, c["sample"], c["sample_seed"])]
    threads = os.cpu_count() or 1
    oracle_c.set_threads(threads)
    st, m, b = oracle_c.preprocess(sample, c["T"])
    per_step = 16384  # rows of each batch the oracle decodes per step
    batches = make_batches(name, n, args.warmup + args.steps, 0)[:, :per_step]
    # compress only the rows the steps touch, into a small table
    need = np.unique(batches)
    small_slots, bits = oracle_c.compress_some(rows, need, m, b)
    small_bm = np.zeros((len(need) + 31) // 32, np.uint32)
    for i in np.nonzero(bits)[0]:
        small_bm[i // 32] |= np.uint32(1 << (i % 32))
    remap = np.searchsorted(need, batches)
    for k in range(args.warmup):
        oracle_c.decompress(small_slots, small_bm, remap[k], m, b)
    t0 = time.perf_counter()
    for k in range(args.warmup, args.warmup + args.steps):
        st, _ = oracle_c.decompress(small_slots, small_bm, remap[k], m, b)
        assert st == 0
    dt = time.perf_counter() - t0
    gbs = args.steps * per_step * 4 * W / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": workload_desc(name, n), "rows_per_step": per_step},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} ids of each batch decoded by the bit-by-bit C oracle "
                                   f"(OpenMP over rows, {threads} threads)"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from host_transfer_gb300 import build, ibp, workloads

    build.build()
    ibp.load()
    name = args.config
    c = workloads.CONFIGS[name]
    n = args.rows or c["n_rows"]
    W = c["W"]
    B = c["batch"]
    K, WU = args.steps, args.warmup
    stream = torch.cuda.current_stream(dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # table in pinned host memory
    t0 = time.perf_counter()
    table = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
    rows_np = table.numpy().view(np.uint32)
    workloads.make_table(name, n_rows=n, out=rows_np)
    gen_s = time.perf_counter() - t0
    pool = min(POOL, WU + K)
    batches = make_batches(name, n, pool, batch_seed_offset(rank))
    last = (WU + K - 1) % pool
    expect_last = rows_np[batches[last]].copy()  # originals of the last timed batch
    ids_d = torch.from_numpy(batches).to(dev)
    out = torch.empty((B, W), dtype=torch.int32, device=dev)

    # preprocess (step 1) on the GPU
    sample_d = torch.from_numpy(rows_np[workloads.sample_ids(n, c["sample"], c["sample_seed"])].view(np.int32)).to(dev)
    e0, e1 = ev(), ev()
    e0.record(stream)
    mask, bitval = ibp.ibp_preprocess(sample_d, c["T"])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    preprocess_ms = e0.elapsed_time(e1)
    plan = ibp.ibp_plan_create(mask, bitval, device=local)
    hints = ibp.IBP_HINT_ROW_REUSE if name == "dlrm" else 0  # Zipf ids repeat hot rows
    plan.set_hints(hints)
    info = plan.info

    # H2D ceiling: cudaMemcpyAsync of the pinned table (1 GB) to HBM, median of 10
    table_d = torch.empty((n, W), dtype=torch.int32, device=dev)
    h2d = []
    for _ in range(10):
        a, b = ev(), ev()
        a.record(stream)
        table_d.copy_(table, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        h2d.append(table.numel() * 4 / (a.elapsed_time(b) * 1e-3) / 1e9)
    h2d_gbs = statistics.median(h2d)

    def time_steps(fn, count, first, label):
        """Warm up eagerly, then time `count` steps replayed as a CUDA graph
        (inside the NVTX range `label`)."""
        for k in range(WU):
            fn(k % pool)
        g = graph_of(torch, fn, count, first, pool)
        g.replay()  # untimed first replay
        torch.cuda.synchronize(dev)
        a, b = ev(), ev()
        torch.cuda.nvtx.range_push(label)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b)

    # uncompressed gathers of the same rows: zero copy from host, and from HBM
    raw_host_ms = time_steps(lambda k: ibp.ibp_gather_raw(table, ids_d[k], out=out), K, WU, "raw_host_timed")
    raw_hbm_ms = time_steps(lambda k: ibp.ibp_gather_raw(table_d, ids_d[k], out=out), K, WU, "raw_hbm_timed")

    # compress in place on the pinned table (step 2, zero copy)
    e0, e1 = ev(), ev()
    e0.record(stream)
    _, bitmask, stored = ibp.ibp_compress(plan, table)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ibp.ibp_get_status(plan)
    compress_ms = e0.elapsed_time(e1)
    # prefix fetched before the headers, from the stored lengths of sampled rows
    prefix_words = ibp.ibp_plan_tune_prefix(plan, table, bitmask)
    stored_words = int(stored.item())
    saving = 1.0 - stored_words / float(n * W)

    # words each batch reads
    lens = torch.stack([ibp.ibp_row_lengths(plan, table, bitmask, ids_d[k]) for k in range(pool)])
    per_batch = lens.to(torch.int64).sum(dim=1).cpu().numpy()
    link_words = int(sum(per_batch[(WU + k) % pool] for k in range(K)))
    f_batch = link_words / float(K * B * W)
    table_d.copy_(table)  # compressed slots in HBM for the cache-resident leg
    torch.cuda.synchronize(dev)

    # ---- timed region: host-resident gather-decompress -------------------
    # K steps captured once as a CUDA graph (launch-bound loops belong in
    # graphs); the replay is the timed region.
    def dec_host(k):
        ibp.ibp_gather_decompress(plan, table, bitmask, ids_d[k], out=out)

    def dec_hbm(k):
        ibp.ibp_gather_decompress(plan, table_d, bitmask, ids_d[k], out=out)

    for k in range(WU):
        dec_host(k % pool)
    ibp.ibp_get_status(plan)
    g_host = graph_of(torch, dec_host, K, WU, pool)
    g_hbm = graph_of(torch, dec_hbm, K, WU, pool)
    # untimed first replays: a graph's first launch also uploads it
    g_host.replay()
    g_hbm.replay()
    torch.cuda.synchronize(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    t_soak = time.perf_counter()
    k = 0
    while time.perf_counter() - t_soak < SOAK_S:  # untimed: clocks settle under this load
        dec_host(k % pool)
        k += 1
        if k % 64 == 0:
            torch.cuda.synchronize(dev)
    for k in range(WU):
        dec_host(k % pool)
    torch.cuda.synchronize(dev)
    g0, g1 = ev(), ev()
    torch.cuda.nvtx.range_push("host_timed")  # ncu --nvtx --nvtx-include host_timed/
    g0.record(stream)
    g_host.replay()
    g1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    total_ms = g0.elapsed_time(g1)
    launch_ms = total_ms / K
    ibp.ibp_get_status(plan)
    parity = bool(np.array_equal(out.cpu().numpy().view(np.uint32), expect_last))

    # ---- HBM-resident gather-decompress -----------------------------------
    for k in range(WU):
        dec_hbm(k % pool)
    torch.cuda.synchronize(dev)
    a, b = ev(), ev()
    torch.cuda.nvtx.range_push("hbm_timed")  # ncu --nvtx --nvtx-include hbm_timed/
    a.record(stream)
    g_hbm.replay()
    b.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    hbm_total_ms = a.elapsed_time(b)
    hbm_launch_ms = hbm_total_ms / K
    ibp.ibp_get_status(plan)
    parity = parity and bool(np.array_equal(out.cpu().numpy().view(np.uint32), expect_last))
    del g_host, g_hbm

    # ---- fused consumer: gather-decompress + sum pooling (embedding bag) ----
    # Bags of POOLING consecutive ids of each batch; the fused call writes one
    # pooled row per bag.  Unfused reference: gather-decompress, then torch's
    # sum over each bag.
    POOLING = 32
    n_bags = B // POOLING
    bag_off = torch.arange(0, n_bags * POOLING + 1, POOLING, dtype=torch.int64, device=dev)
    bag_out = torch.empty((n_bags, W), dtype=torch.float32, device=dev)
    bag_ref = torch.empty((n_bags, W), dtype=torch.float32, device=dev)
    bag_res = {}
    for where, src in (("host", table), ("hbm", table_d)):
        fused_ms = time_steps(lambda k: ibp.ibp_gather_decompress_bag(plan, src, bitmask, ids_d[k], bag_off, out=bag_out),
                              K, WU, f"bag_{where}_timed") / K
        ibp.ibp_get_status(plan)
        # the last timed batch's bags against its decoded rows added in order
        ibp.ibp_gather_decompress(plan, src, bitmask, ids_d[last], out=out)
        rows_f = out[:n_bags * POOLING].view(torch.float32).view(n_bags, POOLING, W)
        bag_ref.zero_()
        for j in range(POOLING):
            bag_ref += rows_f[:, j]
        bag_ok = bool(torch.equal(bag_out.view(torch.int32), bag_ref.view(torch.int32)))

        def unfused(k):
            ibp.ibp_gather_decompress(plan, src, bitmask, ids_d[k], out=out)
            torch.sum(out[:n_bags * POOLING].view(torch.float32).view(n_bags, POOLING, W), dim=1, out=bag_ref)

        unfused_ms = time_steps(unfused, K, WU, f"bag_unfused_{where}_timed") / K
        bag_res[where] = {"value": round(n_bags * POOLING * 4 * W / (fused_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                          "ms_per_step": round(fused_ms, 4), "unfused_ms_per_step": round(unfused_ms, 4),
                          "speedup_vs_unfused": round(unfused_ms / fused_ms, 3),
                          "parity": "bit-exact" if bag_ok else "MISMATCH"}
        parity = parity and bag_ok

    # ---- packed HBM cache: only the stored words of each row ---------------
    offsets = ibp.ibp_packed_offsets(plan, table, bitmask)
    packed_words = int(offsets[-1].item())
    del table_d  # the packed cache replaces the slot copy in HBM
    packed = torch.empty(max(packed_words, 4), dtype=torch.int32, device=dev)
    ibp.ibp_pack(plan, table, offsets, packed)  # fill from pinned host memory

    def dec_packed(k):
        ibp.ibp_gather_decompress_packed(plan, packed, offsets, bitmask, ids_d[k], out=out)

    for k in range(WU):
        dec_packed(k % pool)
    g_pk = graph_of(torch, dec_packed, K, WU, pool)
    g_pk.replay()
    torch.cuda.synchronize(dev)
    a, b = ev(), ev()
    torch.cuda.nvtx.range_push("packed_timed")
    a.record(stream)
    g_pk.replay()
    b.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    pk_ms = a.elapsed_time(b) / K
    ibp.ibp_get_status(plan)
    parity = parity and bool(np.array_equal(out.cpu().numpy().view(np.uint32), expect_last))
    del g_pk
    # stored words rounded to 16 bytes per row, as the packed rows hold them
    pk_words = int(sum(((lens[(WU + k) % pool].to(torch.int64) + 3) // 4 * 4).sum().item() for k in range(K)))
    pk_alg_bytes = (pk_words * 4 + K * B * (4 * W + 8 + 16) + K * B / 8) / K
    pk_achieved = pk_alg_bytes / (pk_ms * 1e-3) / 1e9

    # ---- end to end through the public API ----------------------------------
    ids_host = torch.from_numpy(batches).pin_memory()
    ids_step = torch.empty(B, dtype=torch.int64, device=dev)
    for k in range(WU):
        ids_step.copy_(ids_host[k % pool], non_blocking=True)
        ibp.ibp_gather_decompress(plan, table, bitmask, ids_step, out=out)
        ibp.ibp_get_status(plan)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for k in range(WU, WU + K):
        ids_step.copy_(ids_host[k % pool], non_blocking=True)   # H2D: this step's ids
        ibp.ibp_gather_decompress(plan, table, bitmask, ids_step, out=out)
        ibp.ibp_get_status(plan)                                 # D2H: the call's status word
    e2e_s = time.perf_counter() - t0

    out_bytes = K * B * 4 * W
    ms_step = max_over_ranks(total_ms / K, world)
    value = world * B * 4 * W / (ms_step * 1e-3) / 1e9
    e2e_gbs = world * out_bytes / max_over_ranks(e2e_s, world) / 1e9

    # rooflines
    peaks = measured_peaks()
    hbm_peak = peaks.get("hbm_gbs") or HBM_FALLBACK_GBS
    link_bytes_launch = link_words * 4 / K
    host_achieved = link_bytes_launch / (launch_ms * 1e-3) / 1e9
    hbm_alg_bytes = (link_words * 4 + K * B * (4 * W + 8) + K * B / 8) / K
    hbm_achieved = hbm_alg_bytes / (hbm_launch_ms * 1e-3) / 1e9
    traffic_host = kernel_traffic("host_resident", name)
    traffic_hbm = kernel_traffic("hbm_resident", name)
    traffic_pk = kernel_traffic("packed_hbm_cache", name)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": WU, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": workload_desc(name, n), "batch": B, "W": W, "T": c["T"],
                   "prefix_words": prefix_words,
                   "slots": "pinned host memory, read zero-copy by the kernel",
                   "l2": f"inputs larger than L2: {n * W * 4 / 1e9:.2f} GB table, random ids",
                   "parallelism": f"replicas x{world}"},
        "space_saving_pct": round(100 * saving, 3),
        "compressed_fraction_batch": round(f_batch, 5),
        "unique_ids_per_batch": round(float(np.mean([np.unique(b).size for b in batches])), 1),
        "h2d_gbs": round(h2d_gbs, 2),
        "host_ceiling_gbs": round(h2d_gbs / f_batch, 2),
        "frac_of_host_ceiling": round((B * 4 * W / (launch_ms * 1e-3) / 1e9) / (h2d_gbs / f_batch), 4),
        "roofline": {"bound": "host_link", "achieved": round(host_achieved, 2), "peak": round(h2d_gbs, 2),
                     "unit": "GB/s", "frac": round(host_achieved / h2d_gbs, 4),
                     "traffic": traffic_host.get("link"), "dram_traffic": traffic_host.get("dram"),
                     "traffic_source": "ncu: host-link bytes (sysmem sectors x 32) and DRAM bytes per launch",
                     "peak_source": "cudaMemcpyAsync pinned->HBM of the 1 GB table, median of 10, same run",
                     "kernel": "k_decompress (host-resident slots)",
                     "bytes_per_launch": round(link_bytes_launch)},
        "hbm_resident": {
            "value": round(B * 4 * W / (hbm_total_ms / K * 1e-3) / 1e9, 3), "unit": "GB/s",
            "ms_per_step": round(hbm_total_ms / K, 4),
            "roofline": {"bound": "hbm", "achieved": round(hbm_achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(hbm_achieved / hbm_peak, 4), "traffic": traffic_hbm.get("dram"),
                         "peak_source": "MEASURED_PEAKS.json hbm_gbs" if peaks.get("hbm_gbs") else "fallback",
                         "kernel": "k_decompress (HBM-resident slots)",
                         "bytes_per_launch": round(hbm_alg_bytes)}},
        "packed_hbm_cache": {
            "value": round(B * 4 * W / (pk_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
            "ms_per_step": round(pk_ms, 4),
            "capacity_saving_pct": round(100 * (1 - packed_words / float(n * W)), 3),
            "roofline": {"bound": "hbm", "achieved": round(pk_achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(pk_achieved / hbm_peak, 4), "traffic": traffic_pk.get("dram"),
                         "kernel": "k_decompress_fast (packed layout)", "bytes_per_launch": round(pk_alg_bytes)}},
        "bag_fused": {"what": f"gather-decompress fused with sum pooling, bags of {POOLING} ids "
                              f"({n_bags} per step); value = decoded bytes / s; unfused = gather-decompress "
                              f"then torch.sum per bag",
                      "slots_host": bag_res["host"], "slots_hbm": bag_res["hbm"]},
        "uncompressed_gather": {
            "zero_copy_host_gbs": round(K * B * 4 * W / (raw_host_ms * 1e-3) / 1e9, 3),
            "hbm_gbs": round(K * B * 4 * W / (raw_hbm_ms * 1e-3) / 1e9, 3)},
        "speedup_vs_uncompressed_host": round((raw_host_ms / K) / (total_ms / K), 4),
        "preprocess_ms": round(preprocess_ms, 3),
        "compress_gbs": round(n * W * 4 / (compress_ms * 1e-3) / 1e9, 3),
        "metadata_bytes": info["metadata_bytes"],
        "plan": {k: info[k] for k in ("uniform", "max_runs", "min_kept_bits", "max_kept_bits")},
        "hints": "IBP_HINT_ROW_REUSE" if hints else "none",
        "parity": "bit-exact" if parity else "MISMATCH",
        "e2e": {"value": round(e2e_gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": B * 8,
                "d2h_bytes_per_step": 4},
        "gpu_launches": K,
        "clocks": clocks,
        "table_gen_s": round(gen_s, 2),
        "id_batches": f"{pool} distinct batches, step k uses batch k mod {pool}",
        "timing": "K steps captured as one CUDA graph, replay timed with CUDA events; e2e: eager API calls",
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        gbs, nrows, secs = cpu_oracle_decode(rows_np, bitmask.cpu().numpy().view(np.uint32),
                                             mask.cpu().numpy().view(np.uint32),
                                             bitval.cpu().numpy().view(np.uint32),
                                             batches, args.cpu_seconds, threads)
        m_np, b_np = mask.cpu().numpy().view(np.uint32), bitval.cpu().numpy().view(np.uint32)
        gbs1, nrows1, secs1 = cpu_oracle_decode(rows_np, bitmask.cpu().numpy().view(np.uint32), m_np, b_np,
                                                batches, args.cpu_seconds / 4, 1)
        sub = workloads.make_table(name, n_rows=min(n, 65536))  # the table's first rows, uncompressed
        cgbs, crows, csecs = cpu_oracle_compress(sub, m_np, b_np, args.cpu_seconds / 4, threads)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": f"{nrows} ids of the timed batches decoded by the bit-by-bit C "
                                          f"oracle in {secs:.1f} s (OpenMP over rows)",
                                "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                                                  "sample": f"{nrows1} ids decoded in {secs1:.1f} s"},
                                "compress": {"value": round(cgbs, 4), "unit": "GB/s (input)", "cores": threads,
                                             "sample": f"the table's first {sub.shape[0]} rows compressed "
                                                       f"{crows // sub.shape[0]} times in {csecs:.1f} s"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_llm(args):
    """LLM offload: per layer a 4096 x 4096 bf16 weight and the layer's K and V
    cache [32 heads x 4096 positions, 128] bf16, each compressed in place in
    pinned host memory with its own Mask/Bitval (4,096 sampled rows, T =
    0.99).  A step is the contiguous decompress of one layer (weight, K, V:
    96 MiB of output) into HBM; steps cycle over the layers."""
    import torch

    from host_transfer_gb300 import build, ibp, workloads

    build.build()
    ibp.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    c = workloads.CONFIGS["llm"]
    L, K, WU = args.layers, args.steps, args.warmup

    def ev():
        return torch.cuda.Event(enable_timing=True)

    t0 = time.perf_counter()
    layers = []  # per layer: [(plan, slots, bitmask, n_rows, out, stored_words)] for weight, K, V
    stored = {"weight": 0, "K": 0, "V": 0}
    total = {"weight": 0, "K": 0, "V": 0}
    for li in range(L):
        kv = workloads.llm_kv(li, c["heads"], c["seq"], c["head_dim"], c["seed"])
        tensors = [("weight", workloads.llm_weight(li, c["hidden"], c["hidden"], c["seed"])),
                   ("K", kv[0]), ("V", kv[1])]
        entry = []
        for name, tab in tensors:
            n, W = tab.shape
            host = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
            host.numpy()[...] = tab.view(np.int32)
            sample = torch.from_numpy(tab[workloads.sample_ids(n, c["sample"], c["sample_seed"] + li)]
                                      .view(np.int32)).to(dev)
            mask, bitval = ibp.ibp_preprocess(sample, c["T"])
            plan = ibp.ibp_plan_create(mask, bitval, device=0)
            _, bitmask, st = ibp.ibp_compress(plan, host)
            ibp.ibp_plan_tune_prefix(plan, host, bitmask)
            out = torch.empty((n, W), dtype=torch.int32, device=dev)
            entry.append((plan, host, bitmask, n, out))
            stored[name] += int(st.item())
            total[name] += n * W
        layers.append(entry)
    torch.cuda.synchronize(dev)
    gen_s = time.perf_counter() - t0
    step_bytes = sum(e[3] * e[1].shape[1] * 4 for e in layers[0])
    f = sum(stored.values()) / float(sum(total.values()))

    def step(k):
        for plan, host, bitmask, n, out in layers[k % L]:
            ibp.ibp_decompress_contig(plan, host, bitmask, 0, n, out=out)

    # H2D ceiling on one layer's pinned buffers (the uncompressed transfer)
    h2d = []
    for _ in range(5):
        a, b = ev(), ev()
        a.record(stream)
        for plan, host, bitmask, n, out in layers[0]:
            out.copy_(host, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        h2d.append(step_bytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    h2d_gbs = statistics.median(h2d)

    for k in range(WU):
        step(k)
    torch.cuda.synchronize(dev)
    g = graph_of(torch, step, K, WU, L)
    g.replay()
    torch.cuda.synchronize(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < SOAK_S:
        g.replay()
        torch.cuda.synchronize(dev)
    a, b = ev(), ev()
    torch.cuda.nvtx.range_push("llm_timed")
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = a.elapsed_time(b) / K
    last = (WU + K - 1) % L
    for plan, host, bitmask, n, out in layers[last]:
        ibp.ibp_get_status(plan)
    # parity of the last decoded layer against freshly generated tensors
    kv = workloads.llm_kv(last, c["heads"], c["seq"], c["head_dim"], c["seed"])
    want = [workloads.llm_weight(last, c["hidden"], c["hidden"], c["seed"]), kv[0], kv[1]]
    parity = all(np.array_equal(e[4].cpu().numpy().view(np.uint32), w) for e, w in zip(layers[last], want))
    value = step_bytes / (ms * 1e-3) / 1e9
    link = value * f

    # ---- KV with one Mask/Bitval per attention head (plan sets) -----------
    # Same layers; K and V are compressed again, block of 4096 positions per
    # head with that head's plan, into their own pinned buffers; a step
    # decodes the layer's weight (per-tensor plan, as above) and its K and V
    # with one plan-set call each.
    heads, seq = c["heads"], c["seq"]
    ph_layers = []
    st_ph = {"K": 0, "V": 0}
    for li in range(L):
        kv = workloads.llm_kv(li, heads, seq, c["head_dim"], c["seed"])
        entry = []
        for name, tab in (("K", kv[0]), ("V", kv[1])):
            n, W = tab.shape
            host = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
            host.numpy()[...] = tab.view(np.int32)
            bitmask = torch.zeros((n + 31) // 32, dtype=torch.int32, device=dev)
            stw = torch.zeros(1, dtype=torch.int64, device=dev)
            plans = []
            for h in range(heads):
                blk = tab[h * seq:(h + 1) * seq]
                sample = torch.from_numpy(blk[workloads.sample_ids(seq, c["sample"], c["sample_seed"] + li)]
                                          .view(np.int32)).to(dev)
                plan = ibp.ibp_plan_create(*ibp.ibp_preprocess(sample, c["T"]), device=0)
                ibp.ibp_compress(plan, host[h * seq:(h + 1) * seq], bitmask=bitmask[h * seq // 32:(h + 1) * seq // 32],
                                 stored=stw)
                plans.append(plan)
            torch.cuda.synchronize(dev)
            for h, plan in enumerate(plans):
                ibp.ibp_plan_tune_prefix(plan, host[h * seq:(h + 1) * seq], bitmask[h * seq // 32:(h + 1) * seq // 32])
            entry.append((ibp.ibp_plan_set_create(plans), host, bitmask, seq, layers[li][1 if name == "K" else 2][4]))
            st_ph[name] += int(stw.item())
        ph_layers.append(entry)
    f_ph = (stored["weight"] + st_ph["K"] + st_ph["V"]) / float(sum(total.values()))

    def step_ph(k):
        plan, host, bitmask, n, out = layers[k % L][0]
        ibp.ibp_decompress_contig(plan, host, bitmask, 0, n, out=out)
        for pset, host, bitmask, rpp, out in ph_layers[k % L]:
            ibp.ibp_decompress_contig_set(pset, host, rpp, bitmask, out=out)

    for k in range(WU):
        step_ph(k)
    torch.cuda.synchronize(dev)
    g_ph = graph_of(torch, step_ph, K, WU, L)
    g_ph.replay()
    torch.cuda.synchronize(dev)
    a, b = ev(), ev()
    torch.cuda.nvtx.range_push("llm_ph_timed")
    a.record(stream)
    g_ph.replay()
    b.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    ms_ph = a.elapsed_time(b) / K
    for pset, *_ in ph_layers[last]:
        ibp.ibp_plan_set_get_status(pset)
    parity_ph = all(np.array_equal(e[4].cpu().numpy().view(np.uint32), w)
                    for e, w in zip([layers[last][0]] + ph_layers[last], want))
    value_ph = step_bytes / (ms_ph * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": WU,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32", "data": "synthetic",
        "config": {"workload": f"LLM offload bf16: {L} of 32 layers (4096 x 4096 weight + K and V "
                               f"[32 heads, 4096, 128]) in pinned host memory, per-tensor Mask/Bitval, "
                               f"T=0.99; a step = contiguous decompress of one layer (96 MiB) into HBM",
                   "layers": L, "l2": f"inputs larger than L2: {L} x 96 MiB"},
        "space_saving_pct": {k: round(100 * (1 - stored[k] / total[k]), 3) for k in total},
        "compressed_fraction": round(f, 5),
        "h2d_gbs": round(h2d_gbs, 2),
        "host_ceiling_gbs": round(h2d_gbs / f, 2),
        "frac_of_host_ceiling": round(value / (h2d_gbs / f), 4),
        "roofline": {"bound": "host_link", "achieved": round(link, 2), "peak": round(h2d_gbs, 2),
                     "unit": "GB/s", "frac": round(link / h2d_gbs, 4), "traffic": None,
                     "peak_source": "cudaMemcpyAsync pinned->HBM of one layer, median of 5, same run",
                     "kernel": "k_decompress_fast (contiguous, host-resident slots)"},
        "parity": "bit-exact" if parity else "MISMATCH",
        "kv_per_head": {
            "what": "K and V with one Mask/Bitval per attention head (32 plans per tensor, plan-set decode); "
                    "weight per tensor as above",
            "value": round(value_ph, 3), "unit": "GB/s", "ms_per_step": round(ms_ph, 4),
            "space_saving_pct": {"K": round(100 * (1 - st_ph["K"] / total["K"]), 3),
                                 "V": round(100 * (1 - st_ph["V"] / total["V"]), 3)},
            "compressed_fraction": round(f_ph, 5),
            "frac_of_host_ceiling": round(value_ph / (h2d_gbs / f_ph), 4),
            "parity": "bit-exact" if parity_ph else "MISMATCH"},
        "gpu_launches": 3 * K, "clocks": clocks, "table_gen_s": round(gen_s, 2),
        "timing": "K steps captured as one CUDA graph, replay timed with CUDA events",
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.config == "llm":
        run_llm(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
