#!/usr/bin/env python
"""Benchmark of IBP gather-decompress on one GB300 (or N replicas).

Headline workload (default, `--config all`): LLM offload in bf16, all 32
layers.  Each layer holds a 4096 x 4096 weight and its K and V caches [32
heads, 4096 positions, 128]; bf16 pairs are packed into 32-bit words, and the
layer sits in pinned host memory.  Each tensor is compressed in place on the
GPU with its own Mask/Bitval (4,096 sampled rows, T = 0.99).  A step is the
contiguous decompress of one layer (weight, K, V: 96 MiB of output) into HBM;
the kernels read the compressed slots straight from host memory (zero copy).
Steps cycle over the layers.

The line nests the three row tables under "configs", each measured the same
way (gather-decompress of id batches):
- sparse GNN (1M x 512 fp32, 95 % zeros);
- DLRM (8M x 64 fp32, Zipf ids);
- dense GNN (2M x 128 fp32).

One JSON line on stdout.  Every config reports:
- `value`: decompressed output GB/s (uncompressed bytes), timed with CUDA
  events over K steps replayed as one CUDA graph after W warm-up steps; slots
  are in pinned host memory and ids are already on the device;
- the H2D copy ceiling measured in the same run, and the space saving;
- the same decode with the slots in HBM, against the HBM roofline; decoded
  rows go to a ring of output buffers larger than L2, so their writes reach
  DRAM;
- an end-to-end leg through the public API: eager calls, each step's inputs
  coming from host memory, each step's status word read back to host memory;
- the CPU oracle, timed on the host cores.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]
                    [--config all|llm|dense_gnn|sparse_gnn|dlrm]
    torchrun --nproc-per-node N bench.py --gpus N     (independent replicas)
"""

from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decompressed GB/s (uncompressed bytes) vs PCIe/compress-ratio and HBM roofline; space saving %"
HBM_FALLBACK_GBS = 6800.0
L2_FALLBACK_BYTES = 129 * 2**20
POOL = 64  # distinct id batches; step s uses batch s % POOL
SOAK_S = 0.5  # untimed decode loop under the clock sampler before each timed region
TABLES = ["sparse_gnn", "dlrm", "dense_gnn"]  # nested under the LLM headline, in this order
POOLING = 32  # ids per bag in the fused pooling legs


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", choices=["all", "llm", "dense_gnn", "sparse_gnn", "dlrm"], default="all")
    p.add_argument("--layers", type=int, default=32, help="llm: layers generated (steps cycle over them)")
    p.add_argument("--rows", type=int, default=None, help="fewer table rows (quick runs only)")
    p.add_argument("--cpu-seconds", type=float, default=6.0, help="CPU oracle sample of the headline")
    p.add_argument("--nested-cpu-seconds", type=float, default=2.0, help="CPU oracle sample of a nested config")
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
# measured peaks and committed ncu traffic figures


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


KERNEL_SOURCES = ["ibp_decompress_fast.cuh", "ibp_decode_pipe.cuh", "ibp_decompress_fast_u.cu",
                  "ibp_decompress_fast_t.cu", "ibp_decompress_fast_up.cu", "ibp_decompress_fast_tp.cu",
                  "ibp_decompress_fast_ur.cu", "ibp_decompress_fast_tr.cu", "ibp_decompress_fast_td.cu",
                  "ibp_decompress_fast_ud.cu", "ibp_decompress_fast_set.cu",
                  "ibp_decompress.cu", "ibp_internal.cuh", "ibp_api.cu"]


def kernel_sources_sha() -> str:
    """sha256 over the sources of the decompress kernels."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        path = os.path.join(ROOT, "host_transfer_gb300", "csrc", f)
        if os.path.exists(path):
            h.update(open(path, "rb").read())
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


# ---------------------------------------------------------------------------
# workloads and the config objects both arms print


def table_workload(name: str, n_rows: int) -> str:
    from host_transfer_gb300 import workloads

    c = workloads.CONFIGS[name]
    return {
        "dense_gnn": f"dense GNN features: {n_rows:,} rows x 128 fp32, N(0,1) rows L2-normalised, "
                     f"pinned host, T=0.99, gather batches of {c['batch']:,} uniform ids into HBM",
        "sparse_gnn": f"sparse GNN features: {n_rows:,} rows x 512 fp32, 95% zeros, lognormal "
                      f"non-zeros, pinned host, T=0.95, gather batches of {c['batch']:,} uniform ids into HBM",
        "dlrm": f"DLRM embedding table: {n_rows:,} rows x 64 fp32 U(-0.01,0.01), pinned host, "
                f"T=0.99, gather batches of {c['batch']:,} Zipf(1.05) ids into HBM",
    }[name]


def llm_workload(layers: int) -> str:
    return (f"LLM offload bf16: {layers} layers x (4096 x 4096 weight + K and V [32 heads, 4096, 128]), "
            f"bf16 pairs in 32-bit words, pinned host, per-tensor Mask/Bitval at T=0.99; a step = "
            f"contiguous decompress of one layer (96 MiB) into HBM")


def config_of(name: str, args, world: int) -> dict:
    """The `config` object of a workload; the same for both arms."""
    from host_transfer_gb300 import workloads

    par = f"replicas x{world}"
    if name == "llm":
        return {"workload": llm_workload(args.layers), "layers": args.layers,
                "l2": f"inputs larger than L2: {args.layers} x 96 MiB, one layer per step",
                "parallelism": par}
    c = workloads.CONFIGS[name]
    n = args.rows or c["n_rows"]
    return {"workload": table_workload(name, n), "batch": c["batch"], "W": c["W"], "T": c["T"],
            "l2": f"inputs larger than L2: {n * c['W'] * 4 / 1e9:.2f} GB table, random ids",
            "parallelism": par}


def make_batches(name, n_rows, count, offset):
    from host_transfer_gb300 import workloads

    zipf = None
    if name == "dlrm":
        c = workloads.CONFIGS[name]
        zipf = workloads.ZipfIds(n_rows, c["zipf_s"], c["seed"])
    return np.stack([workloads.batch_ids(name, offset + k, n_rows=n_rows, zipf=zipf) for k in range(count)])


def llm_layer(li: int):
    """[(name, words)] of one layer: the weight, K and V."""
    from host_transfer_gb300 import workloads

    c = workloads.CONFIGS["llm"]
    kv = workloads.llm_kv(li, c["heads"], c["seq"], c["head_dim"], c["seed"])
    return [("weight", workloads.llm_weight(li, c["hidden"], c["hidden"], c["seed"])), ("K", kv[0]), ("V", kv[1])]


def llm_layers(count: int):
    """Layers 0 .. count-1, drawn in parallel (numpy's generators release the
    GIL; every layer has its own seed, so the result does not depend on the
    thread count)."""
    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        return list(ex.map(llm_layer, range(count)))


def llm_sample(li: int, tab: np.ndarray) -> np.ndarray:
    from host_transfer_gb300 import workloads

    c = workloads.CONFIGS["llm"]
    return tab[workloads.sample_ids(tab.shape[0], c["sample"], c["sample_seed"] + li)]


# ---------------------------------------------------------------------------
# CPU oracle timings (test infrastructure: the oracle never runs on the GPU
# path; here it is the reported baseline)


def oracle_compress_rows(rows, sample, T, timing=None):
    """The oracle's own Mask/Bitval from `sample` and its slots of `rows`;
    `timing` (a list) collects (bytes of rows, seconds) of the compress."""
    from oracle import oracle_c

    st, m, b = oracle_c.preprocess(sample, T)
    assert st == 0
    t0 = time.perf_counter()
    slots, bitmask, _ = oracle_c.compress(rows, m, b)
    if timing is not None:
        timing.append((rows.size * 4, time.perf_counter() - t0))
    return slots, bitmask, m, b


def _decode_for(slots, bitmask, m, b, ids_of, seconds):
    """The C oracle decoding id chunks ids_of(k), k = 0, 1, ..., until about
    `seconds` have been spent; returns (ids decoded, seconds)."""
    from oracle import oracle_c

    done, used, k = 0, 0.0, 0
    while used < seconds:
        ids = ids_of(k)
        t0 = time.perf_counter()
        st, _ = oracle_c.decompress(slots, bitmask, ids, m, b)
        used += time.perf_counter() - t0
        assert st == 0
        done += len(ids)
        k += 1
    return done, used


def cpu_extras(gbs1, secs1, comp, threads):
    """The single-thread decode rate and the compress rate of the oracle."""
    nbytes = sum(n for n, _ in comp)
    csecs = sum(t for _, t in comp)
    return {"single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"the same decode on one thread for {secs1:.1f} s"},
            "compress": {"value": round(nbytes / csecs / 1e9, 4), "unit": "GB/s of input rows", "cores": threads,
                         "sample": f"{nbytes / 1e6:.0f} MB of rows compressed once by the C oracle in "
                                   f"{csecs:.2f} s (OpenMP over rows)"}}


def cpu_table_baseline(rows, sample, T, id_batches, seconds, threads):
    """The C oracle decoding `id_batches` (ids into `rows`) for about
    `seconds` on all `threads`, and for a quarter of that on one thread, on
    slots it compressed itself.  Returns (GB/s of uncompressed output, ids
    decoded, seconds, extras: the single-thread and compress rates)."""
    from oracle import oracle_c

    oracle_c.set_threads(threads)
    remap = id_batches.reshape(-1)
    comp = []
    slots, bitmask, m, b = oracle_compress_rows(rows, sample, T, comp)
    W = rows.shape[1]
    chunk = 8192
    nchunks = max(1, remap.size // chunk)
    ids_of = lambda k: remap[(k % nchunks) * chunk:(k % nchunks + 1) * chunk]  # noqa: E731
    done, used = _decode_for(slots, bitmask, m, b, ids_of, seconds)
    oracle_c.set_threads(1)
    one = lambda k: remap[(k * 512) % max(1, remap.size - 512):][:512]  # noqa: E731
    done1, used1 = _decode_for(slots, bitmask, m, b, one, seconds / 4)
    oracle_c.set_threads(threads)
    extras = cpu_extras(done1 * 4 * W / used1 / 1e9, used1, comp, threads)
    return done * 4 * W / used / 1e9, done, used, extras


def cpu_llm_baseline(layer, seconds, threads):
    """The C oracle decoding one whole layer (weight, K, V) again and again for
    about `seconds`.  Returns (GB/s of uncompressed output, layers, seconds)."""
    from oracle import oracle_c

    oracle_c.set_threads(threads)
    comp, timing = [], []
    for name, tab in layer:
        slots, bitmask, m, b = oracle_compress_rows(tab, llm_sample(0, tab), 0.99, timing)
        comp.append((slots, bitmask, m, b, np.arange(tab.shape[0], dtype=np.int64)))
    step_bytes = sum(t.size * 4 for _, t in layer)
    done, used = 0, 0.0
    while used < seconds:
        t0 = time.perf_counter()
        for slots, bitmask, m, b, ids in comp:
            st, _ = oracle_c.decompress(slots, bitmask, ids, m, b)
            assert st == 0
        used += time.perf_counter() - t0
        done += 1
    # one thread: the weight rows, 64 at a time
    oracle_c.set_threads(1)
    slots, bitmask, m, b, ids = comp[0]
    W = layer[0][1].shape[1]
    done1, used1 = _decode_for(slots, bitmask, m, b, lambda k: ids[(64 * k) % (len(ids) - 64):][:64], seconds / 4)
    oracle_c.set_threads(threads)
    extras = cpu_extras(done1 * 4 * W / used1 / 1e9, used1, timing, threads)
    return done * step_bytes / used / 1e9, done, used, extras


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the same workload and the same steps


def reference_line(args, name, world, value, ms, threads, sample_desc):
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32", "data": "synthetic", "config": config_of(name, args, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample_desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args):
    """The CPU oracle as the reference arm: each step decodes exactly what a
    step of the GPU arm decodes (the same layer, or the same id batch), on
    the host cores, with slots the oracle compressed itself."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from host_transfer_gb300 import workloads
    from oracle import oracle_c

    threads = os.cpu_count() or 1
    oracle_c.set_threads(threads)
    K, WU = args.steps, args.warmup
    name = "llm" if args.config in ("all", "llm") else args.config
    if name == "llm":
        L = args.layers
        T = workloads.CONFIGS["llm"]["T"]
        used = sorted({s % L for s in range(WU + K)})
        pool_threads = max(1, min(16, os.cpu_count() or 1))
        with ThreadPoolExecutor(pool_threads) as ex:  # generators and the C preprocess release the GIL
            layers = dict(zip(used, ex.map(llm_layer, used)))
            masks = {li: list(ex.map(lambda t: oracle_c.preprocess(llm_sample(li, t[1]), T), layers[li]))
                     for li in used}
        comp = {}
        for li in used:
            comp[li] = []
            for (tname, tab), (st, m, b) in zip(layers[li], masks[li]):
                assert st == 0
                slots, bitmask, _ = oracle_c.compress(tab, m, b)
                comp[li].append((slots, bitmask, m, b, np.arange(tab.shape[0], dtype=np.int64)))
        step_bytes = sum(t.size * 4 for _, t in layers[used[0]])
        del layers

        def step(s):
            for slots, bitmask, m, b, ids in comp[s % L]:
                st, _ = oracle_c.decompress(slots, bitmask, ids, m, b)
                assert st == 0

        for s in range(WU):
            step(s)
        t0 = time.perf_counter()
        for s in range(WU, WU + K):
            step(s)
        dt = time.perf_counter() - t0
        value = K * step_bytes / dt / 1e9
        desc = (f"every step decodes one whole layer (weight, K, V: 96 MiB), as a GPU step does, with the "
                f"bit-by-bit C oracle (OpenMP over rows, {threads} threads)")
    else:
        c = workloads.CONFIGS[name]
        n = args.rows or c["n_rows"]
        W, B = c["W"], c["batch"]
        rows = workloads.make_table(name, n_rows=n)
        sample = rows[workloads.sample_ids(n, c["sample"], c["sample_seed"])]
        pool = min(POOL, WU + K)
        batches = make_batches(name, n, pool, 0)
        need, remap = np.unique(batches, return_inverse=True)
        remap = remap.reshape(batches.shape)
        slots, bitmask, m, b = oracle_compress_rows(rows[need], sample, c["T"])
        del rows
        for s in range(WU):
            oracle_c.decompress(slots, bitmask, remap[s % pool], m, b)
        t0 = time.perf_counter()
        for s in range(WU, WU + K):
            st, _ = oracle_c.decompress(slots, bitmask, remap[s % pool], m, b)
            assert st == 0
        dt = time.perf_counter() - t0
        value = K * B * 4 * W / dt / 1e9
        desc = (f"every step decodes the same {B:,} ids as a GPU step, with the bit-by-bit C oracle "
                f"(OpenMP over rows, {threads} threads)")
    print(json.dumps(reference_line(args, name, world, value, 1e3 * dt / K, threads, desc)), flush=True)


# ---------------------------------------------------------------------------
# GPU arm


class Ctx:
    """Device, stream, step counts and the ceilings shared by every leg."""

    def __init__(self, args):
        import torch

        self.torch = torch
        self.args = args
        self.rank, self.world, self.local = dist_env()
        torch.cuda.set_device(self.local)
        self.dev = torch.device("cuda", self.local)
        self.stream = torch.cuda.current_stream(self.dev)
        self.K, self.WU = args.steps, args.warmup
        props = torch.cuda.get_device_properties(self.dev)
        self.l2 = int(getattr(props, "L2_cache_size", 0) or L2_FALLBACK_BYTES)
        try:
            self.uuid = "GPU-" + str(props.uuid)
        except Exception:
            self.uuid = None
        peaks = measured_peaks()
        self.hbm_peak = peaks.get("hbm_gbs") or HBM_FALLBACK_GBS
        self.hbm_peak_src = "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks.get("hbm_gbs") else "fallback"
        self.cpu_ok = self.rank == 0 and self.world == 1 and not args.no_cpu_baseline
        self.h2d_gbs = self.measure_h2d()

    def ev(self):
        return self.torch.cuda.Event(enable_timing=True)

    def sync(self):
        self.torch.cuda.synchronize(self.dev)

    def measure_h2d(self) -> float:
        """cudaMemcpyAsync of a 1 GiB pinned buffer into HBM, median of 10: the
        ceiling of the host link for every host-resident leg of the run."""
        torch = self.torch
        src = torch.empty(2**28, dtype=torch.int32, pin_memory=True)
        src.fill_(1)
        dst = torch.empty(2**28, dtype=torch.int32, device=self.dev)
        rates = []
        for _ in range(10):
            a, b = self.ev(), self.ev()
            a.record(self.stream)
            dst.copy_(src, non_blocking=True)
            b.record(self.stream)
            self.sync()
            rates.append(src.numel() * 4 / (a.elapsed_time(b) * 1e-3) / 1e9)
        del src, dst
        return statistics.median(rates)

    def graph(self, fn, first, count):
        """fn(s) for steps s = first .. first + count - 1 captured as one CUDA
        graph (launch-bound loops belong in graphs)."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for k in range(count):
                fn(first + k)
        return g

    def time_graph(self, g, label) -> float:
        """One timed replay of g (CUDA events on the launching stream, NVTX
        range `label`); returns milliseconds."""
        torch = self.torch
        self.sync()
        a, b = self.ev(), self.ev()
        torch.cuda.nvtx.range_push(label)
        a.record(self.stream)
        g.replay()
        b.record(self.stream)
        torch.cuda.nvtx.range_pop()
        self.sync()
        return a.elapsed_time(b)

    def time_steps(self, fn, label) -> float:
        """W eager warm-up steps, then the K timed steps as one graph (after
        an untimed first replay, which also uploads the graph); ms total."""
        for s in range(self.WU):
            fn(s)
        g = self.graph(fn, self.WU, self.K)
        g.replay()
        ms = self.time_graph(g, label)
        del g
        return ms

    def timed_with_clocks(self, fn, label):
        """As time_steps, with nvidia-smi sampling the clocks through an untimed
        soak of the same steps and the timed replay; returns (ms, clocks)."""
        for s in range(self.WU):
            fn(s)
        g = self.graph(fn, self.WU, self.K)
        g.replay()
        self.sync()
        sampler = ClockSampler(self.uuid)
        barrier(self.world)
        self.sync()
        sampler.start()
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < SOAK_S:  # untimed: clocks settle under this load
            g.replay()
            self.sync()
        ms = self.time_graph(g, label)
        barrier(self.world)
        clocks = sampler.stop()
        del g
        return ms, clocks

    def time_eager(self, step):
        """Wall time of the K timed steps s = W .. W+K-1 issued eagerly, with one
        synchronisation at the end; returns (seconds, seconds until the last
        step was enqueued).  Garbage is collected first, so that no object
        whose release synchronises the device (a plan's memory) is freed
        inside the timed loop."""
        gc.collect()
        self.sync()
        barrier(self.world)
        t0 = time.perf_counter()
        for s in range(self.WU, self.WU + self.K):
            step(s)
        t1 = time.perf_counter()
        self.sync()
        return time.perf_counter() - t0, t1 - t0

    def ring_count(self, out_bytes: int) -> int:
        """Output buffers in a ring whose total is at least twice L2, so that
        every step's writes reach DRAM rather than staying in L2."""
        return max(2, math.ceil(2 * self.l2 / out_bytes))


def roofline(bound, achieved, peak, peak_source, kernel, bytes_per_launch, traffic, **extra):
    d = {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": "GB/s",
         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_source,
         "kernel": kernel, "bytes_per_launch": round(bytes_per_launch)}
    d.update(extra)
    return d


def run_table(ctx: Ctx, name: str, cpu_seconds: float) -> dict:
    """One row table: gather-decompress legs, fused pooling, packed cache,
    end to end and the CPU oracle."""
    torch = ctx.torch
    from host_transfer_gb300 import ibp, workloads

    c = workloads.CONFIGS[name]
    n = ctx.args.rows or c["n_rows"]
    W, B = c["W"], c["batch"]
    K, WU, dev, stream = ctx.K, ctx.WU, ctx.dev, ctx.stream
    last = WU + K - 1  # step index of the last timed step

    t0 = time.perf_counter()
    table = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
    rows_np = table.numpy().view(np.uint32)
    workloads.make_table(name, n_rows=n, out=rows_np)
    gen_s = time.perf_counter() - t0
    pool = min(POOL, WU + K)
    batches = make_batches(name, n, pool, batch_seed_offset(ctx.rank))
    expect_last = rows_np[batches[last % pool]].copy()  # originals of the last timed batch
    sample_np = rows_np[workloads.sample_ids(n, c["sample"], c["sample_seed"])]
    cpu_keep = cpu_rows = cpu_sample = None
    if ctx.cpu_ok:  # rows the CPU baseline decodes, copied before the in-place compress
        cpu_keep = np.unique(batches[:2])
        cpu_rows = rows_np[cpu_keep].copy()
        cpu_sample = sample_np.copy()
    ids_d = torch.from_numpy(batches).to(dev)
    ring_n = ctx.ring_count(B * W * 4)
    ring = torch.empty((ring_n, B, W), dtype=torch.int32, device=dev)

    def out_of(s):
        return ring[s % ring_n]

    # preprocess (step 1) on the GPU
    sample_d = torch.from_numpy(sample_np.view(np.int32)).to(dev)
    e0, e1 = ctx.ev(), ctx.ev()
    e0.record(stream)
    mask, bitval = ibp.ibp_preprocess(sample_d, c["T"])
    e1.record(stream)
    ctx.sync()
    preprocess_ms = e0.elapsed_time(e1)
    plan = ibp.ibp_plan_create(mask, bitval, device=ctx.local)
    # the ids, bitmask and slots of a step are written before the loop, never by
    # the kernel just before a decode; Zipf ids repeat hot rows
    hints = ibp.IBP_HINT_EARLY_FETCH | (ibp.IBP_HINT_ROW_REUSE if name == "dlrm" else 0)
    plan.set_hints(hints)
    info = plan.info

    # uncompressed gathers of the same rows: zero copy from host, and from HBM
    table_d = torch.empty((n, W), dtype=torch.int32, device=dev)
    table_d.copy_(table)
    raw_host_ms = ctx.time_steps(lambda s: ibp.ibp_gather_raw(table, ids_d[s % pool], out=out_of(s)),
                                 f"{name}_raw_host_timed")
    raw_hbm_ms = ctx.time_steps(lambda s: ibp.ibp_gather_raw(table_d, ids_d[s % pool], out=out_of(s)),
                                f"{name}_raw_hbm_timed")

    # compress in place on the pinned table (step 2, zero copy)
    e0, e1 = ctx.ev(), ctx.ev()
    e0.record(stream)
    _, bitmask, stored = ibp.ibp_compress(plan, table)
    e1.record(stream)
    ctx.sync()
    ibp.ibp_get_status(plan)
    compress_ms = e0.elapsed_time(e1)
    prefix_words = ibp.ibp_plan_tune_prefix(plan, table, bitmask)
    stored_words = int(stored.item())
    saving = 1.0 - stored_words / float(n * W)

    # words each batch reads, all ids and unique ids
    lens = torch.stack([ibp.ibp_row_lengths(plan, table, bitmask, ids_d[k]) for k in range(pool)])
    lens_np = lens.to(torch.int64).cpu().numpy()
    per_batch = lens_np.sum(axis=1)
    per_batch_unique = np.array([lens_np[k][np.unique(batches[k], return_index=True)[1]].sum()
                                 for k in range(pool)])
    steps = range(WU, WU + K)
    link_words = int(sum(per_batch[s % pool] for s in steps))
    link_words_unique = int(sum(per_batch_unique[s % pool] for s in steps))
    f_batch = link_words / float(K * B * W)
    table_d.copy_(table)  # compressed slots in HBM for the cache-resident leg
    ctx.sync()

    def dec_host(s):
        ibp.ibp_gather_decompress(plan, table, bitmask, ids_d[s % pool], out=out_of(s))

    def dec_hbm(s):
        ibp.ibp_gather_decompress(plan, table_d, bitmask, ids_d[s % pool], out=out_of(s))

    # ---- timed region: host-resident gather-decompress ------------------
    # ncu --clock-control none --nvtx --nvtx-include "<name>_host_timed/" selects it
    total_ms, clocks = ctx.timed_with_clocks(dec_host, f"{name}_host_timed")
    ibp.ibp_get_status(plan)
    parity = bool(np.array_equal(out_of(last).cpu().numpy().view(np.uint32), expect_last))
    launch_ms = total_ms / K

    # ---- end to end through the public API ----------------------------------
    # Eager calls as a user makes them: every step's ids sit in pinned host
    # memory and the decode kernel reads them there (zero copy, like the
    # compressed rows), and the step's status word is moved into pinned host
    # memory by a status read enqueued right after the decode on the same
    # stream; the host checks every step's word after the last step.  Two
    # calls per step; the status read launches as a programmatic dependent, so
    # consecutive decodes still overlap.  Run right after the
    # graph-timed leg, over the same steps, so that both see the host table in
    # the same state (the GPU's translations of its pages warm).
    ids_host = torch.from_numpy(batches).pin_memory()
    status_host = torch.full((WU + K,), -1, dtype=torch.int32, pin_memory=True)
    # set-up, untimed: the GPU's first access to newly pinned pages is slow, so
    # every batch's ids are read once by the kernel before any step
    for k in range(pool):
        ibp.ibp_gather_decompress(plan, table, bitmask, ids_host[k], out=out_of(k))
    ctx.sync()

    # The per-step tensors (views of the pinned id and status buffers and of
    # the output ring) are made once, as a pipeline that reuses its buffers
    # holds them: building a view per call costs the host more than the call.
    ids_v = [ids_host[k] for k in range(pool)]
    out_v = [out_of(k) for k in range(ring_n)]
    status_v = [status_host[k] for k in range(WU + K)]

    def e2e_step(s):
        # H2D: step s's ids and compressed rows, read by the kernel
        ibp.ibp_gather_decompress(plan, table, bitmask, ids_v[s % pool], out=out_v[s % ring_n], stream=stream)
        ibp.ibp_get_status_async(plan, status_v[s], stream=stream)  # D2H: step s's status

    for s in range(WU):
        e2e_step(s)
    e2e_s, enqueue_s = ctx.time_eager(e2e_step)
    e2e_ok = bool((status_host == 0).all().item())
    parity = parity and e2e_ok and bool(np.array_equal(out_of(last).cpu().numpy().view(np.uint32), expect_last))

    # ---- HBM-resident gather-decompress ------------------------------------
    hbm_ms = ctx.time_steps(dec_hbm, f"{name}_hbm_timed") / K
    ibp.ibp_get_status(plan)
    parity = parity and bool(np.array_equal(out_of(last).cpu().numpy().view(np.uint32), expect_last))

    # ---- fused consumer: gather-decompress + sum pooling (embedding bag) ----
    n_bags = B // POOLING
    bag_off = torch.arange(0, n_bags * POOLING + 1, POOLING, dtype=torch.int64, device=dev)
    bag_out = torch.empty((n_bags, W), dtype=torch.float32, device=dev)
    bag_ref = torch.empty((n_bags, W), dtype=torch.float32, device=dev)
    bag_res = {}
    for where, src in (("host", table), ("hbm", table_d)):
        fused_ms = ctx.time_steps(
            lambda s: ibp.ibp_gather_decompress_bag(plan, src, bitmask, ids_d[s % pool], bag_off, out=bag_out),
            f"{name}_bag_{where}_timed") / K
        ibp.ibp_get_status(plan)
        # the last timed batch's bags against its decoded rows added in order
        rows_f = out_of(last)[:n_bags * POOLING].view(torch.float32).view(n_bags, POOLING, W)
        bag_ref.zero_()
        for j in range(POOLING):
            bag_ref += rows_f[:, j]
        bag_ok = bool(torch.equal(bag_out.view(torch.int32), bag_ref.view(torch.int32)))

        def unfused(s, src=src):
            o = out_of(s)
            ibp.ibp_gather_decompress(plan, src, bitmask, ids_d[s % pool], out=o)
            torch.sum(o[:n_bags * POOLING].view(torch.float32).view(n_bags, POOLING, W), dim=1, out=bag_ref)

        unfused_ms = ctx.time_steps(unfused, f"{name}_bag_unfused_{where}_timed") / K
        bag_res[where] = {"value": round(n_bags * POOLING * 4 * W / (fused_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                          "ms_per_step": round(fused_ms, 4), "unfused_ms_per_step": round(unfused_ms, 4),
                          "speedup_vs_unfused": round(unfused_ms / fused_ms, 3),
                          "parity": "bit-exact" if bag_ok else "MISMATCH"}
        parity = parity and bag_ok
        # the unfused leg rewrote the ring: restore the last step's rows
        dec_hbm(last)

    # ---- packed HBM cache: only the stored words of each row ---------------
    offsets = ibp.ibp_packed_offsets(plan, table, bitmask)
    packed_words = int(offsets[-1].item())
    del table_d  # the packed cache replaces the slot copy in HBM
    packed = torch.empty(max(packed_words, 4), dtype=torch.int32, device=dev)
    ibp.ibp_pack(plan, table, offsets, packed)  # fill from pinned host memory
    pk_ms = ctx.time_steps(
        lambda s: ibp.ibp_gather_decompress_packed(plan, packed, offsets, bitmask, ids_d[s % pool], out=out_of(s)),
        f"{name}_packed_timed") / K
    ibp.ibp_get_status(plan)
    parity = parity and bool(np.array_equal(out_of(last).cpu().numpy().view(np.uint32), expect_last))
    pk_words = int(sum(((lens[s % pool].to(torch.int64) + 3) // 4 * 4).sum().item() for s in steps))
    pk_alg_bytes = (pk_words * 4 + K * B * (4 * W + 8 + 16) + K * B / 8) / K
    del packed, offsets

    # ---- numbers -------------------------------------------------------------
    world = ctx.world
    ms_step = max_over_ranks(launch_ms, world)
    value = world * B * 4 * W / (ms_step * 1e-3) / 1e9
    e2e_gbs = world * K * B * 4 * W / max_over_ranks(e2e_s, world) / 1e9
    link_bytes_launch = link_words * 4 / K
    host_achieved = link_bytes_launch / (launch_ms * 1e-3) / 1e9
    hbm_alg_bytes = (link_words * 4 + K * B * (4 * W + 8) + K * B / 8) / K
    hbm_achieved = hbm_alg_bytes / (hbm_ms * 1e-3) / 1e9
    pk_achieved = pk_alg_bytes / (pk_ms * 1e-3) / 1e9
    ceiling = ctx.h2d_gbs / f_batch
    traffic_host = kernel_traffic("host_resident", name)
    traffic_hbm = kernel_traffic("hbm_resident", name)
    traffic_pk = kernel_traffic("packed_hbm_cache", name)
    h2d_src = "cudaMemcpyAsync of a 1 GiB pinned buffer into HBM, median of 10, same run"

    res = {
        "value": round(value, 3), "unit": "GB/s", "ms_per_step": round(ms_step, 4),
        "config": config_of(name, ctx.args, world),
        "slots": "pinned host memory, read zero-copy by the kernel",
        "prefix_words": prefix_words,
        "space_saving_pct": round(100 * saving, 3),
        "compressed_fraction_batch": round(f_batch, 5),
        "unique_ids_per_batch": round(float(np.mean([np.unique(b).size for b in batches])), 1),
        "h2d_gbs": round(ctx.h2d_gbs, 2),
        "host_ceiling_gbs": round(ceiling, 2),
        "frac_of_host_ceiling": round((B * 4 * W / (launch_ms * 1e-3) / 1e9) / ceiling, 4),
        "roofline": roofline("host_link", host_achieved, ctx.h2d_gbs, h2d_src,
                             "k_decompress_fast (slots in pinned host memory)", link_bytes_launch,
                             traffic_host.get("link"), dram_traffic=traffic_host.get("dram"),
                             traffic_source="ncu: host-link bytes (sysmem sectors x 32) per launch"),
        "hbm_resident": {
            "value": round(B * 4 * W / (hbm_ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(hbm_ms, 4),
            "roofline": roofline("hbm", hbm_achieved, ctx.hbm_peak, ctx.hbm_peak_src,
                                 "k_decompress_fast (slots in HBM)", hbm_alg_bytes, traffic_hbm.get("dram"),
                                 output_ring=f"{ring_n} x {B * W * 4 / 2**20:.1f} MiB output buffers "
                                             f"(> 2 x L2): decoded rows are written to DRAM")},
        "packed_hbm_cache": {
            "value": round(B * 4 * W / (pk_ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(pk_ms, 4),
            "capacity_saving_pct": round(100 * (1 - packed_words / float(n * W)), 3),
            "roofline": roofline("hbm", pk_achieved, ctx.hbm_peak, ctx.hbm_peak_src,
                                 "k_decompress_fast (packed layout in HBM)", pk_alg_bytes, traffic_pk.get("dram"))},
        "bag_fused": {"what": f"gather-decompress fused with sum pooling, bags of {POOLING} ids "
                              f"({n_bags} per step); value = decoded bytes / s; unfused = gather-decompress "
                              f"then torch.sum per bag",
                      "slots_host": bag_res["host"], "slots_hbm": bag_res["hbm"]},
        "uncompressed_gather": {
            "zero_copy_host_gbs": round(K * B * 4 * W / (raw_host_ms * 1e-3) / 1e9, 3),
            "hbm_gbs": round(K * B * 4 * W / (raw_hbm_ms * 1e-3) / 1e9, 3)},
        "speedup_vs_uncompressed_host": round((raw_host_ms / K) / launch_ms, 4),
        "preprocess_ms": round(preprocess_ms, 3),
        "compress_gbs": round(n * W * 4 / (compress_ms * 1e-3) / 1e9, 3),
        "metadata_bytes": info["metadata_bytes"],
        "plan": {k: info[k] for k in ("uniform", "max_runs", "min_kept_bits", "max_kept_bits")},
        "hints": " | ".join(h for h, bit in (("IBP_HINT_EARLY_FETCH", ibp.IBP_HINT_EARLY_FETCH),
                                              ("IBP_HINT_ROW_REUSE", ibp.IBP_HINT_ROW_REUSE)) if hints & bit),
        "parity": "bit-exact" if parity else "MISMATCH",
        "e2e": {"value": round(e2e_gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": B * 8 + link_words * 4 // K,
                "d2h_bytes_per_step": 4, "enqueue_ms_per_step": round(1e3 * enqueue_s / K, 4),
                "what": "eager API calls; per step the ids and the compressed rows read from pinned host memory "
                        "by the kernel (the step's host-to-device bytes) and the status word moved into pinned host "
                        "memory by a status read on the same stream; wall clock, one synchronisation at the end"},
        "gpu_launches": K,
        "clocks": clocks,
        "table_gen_s": round(gen_s, 2),
        "id_batches": f"{pool} distinct batches, step s uses batch s mod {pool}",
        "timing": "K steps captured as one CUDA graph, replay timed with CUDA events",
    }
    if name == "dlrm":
        # Zipf ids repeat rows within a batch; a repeat served from L1 never
        # crosses the link, so the link rate is also given on unique rows.
        uniq_bytes = link_words_unique * 4 / K
        res["link_unique_rows"] = {
            "bytes_per_launch": round(uniq_bytes),
            "achieved_gbs": round(uniq_bytes / (launch_ms * 1e-3) / 1e9, 2),
            "frac_of_h2d": round(uniq_bytes / (launch_ms * 1e-3) / 1e9 / ctx.h2d_gbs, 4),
            "what": "the compressed bytes of the batch's unique rows (each must cross the link at least "
                    "once) per launch time, against the H2D copy rate",
        }
        if traffic_host.get("link"):
            res["link_unique_rows"]["measured_link_bytes_per_row"] = round(traffic_host["link"] / B, 1)
    if ctx.cpu_ok:
        threads = os.cpu_count() or 1
        remap = np.searchsorted(cpu_keep, batches[:2])  # the two batches' ids into the kept rows
        gbs, nids, secs, extras = cpu_table_baseline(cpu_rows, cpu_sample, c["T"], remap, cpu_seconds, threads)
        res["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                               "sample": f"{nids} ids of two of the bench's batches decoded by the bit-by-bit "
                                         f"C oracle in {secs:.1f} s (OpenMP over rows), on slots it compressed "
                                         f"itself", **extras}
    del table, ring
    return res


def run_llm(ctx: Ctx, cpu_seconds: float) -> dict:
    """LLM offload: contiguous decompress of one layer per step."""
    torch = ctx.torch
    from host_transfer_gb300 import ibp, workloads

    c = workloads.CONFIGS["llm"]
    L, K, WU, dev, stream = ctx.args.layers, ctx.K, ctx.WU, ctx.dev, ctx.stream
    last = WU + K - 1
    t0 = time.perf_counter()
    originals = llm_layers(L)
    gen_s = time.perf_counter() - t0

    # per tensor: pinned host slots (compressed in place), plan, bitmask, HBM output
    layers = []
    stored = {"weight": 0, "K": 0, "V": 0}
    total = {"weight": 0, "K": 0, "V": 0}
    t0 = time.perf_counter()
    for li in range(L):
        entry = []
        for name, tab in originals[li]:
            n, W = tab.shape
            host = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
            host.numpy()[...] = tab.view(np.int32)
            sample = torch.from_numpy(llm_sample(li, tab).view(np.int32)).to(dev)
            mask, bitval = ibp.ibp_preprocess(sample, c["T"])
            plan = ibp.ibp_plan_create(mask, bitval, device=ctx.local)
            plan.set_hints(ibp.IBP_HINT_EARLY_FETCH)  # the layers are written once, before the steps
            _, bitmask, st = ibp.ibp_compress(plan, host)
            ibp.ibp_plan_tune_prefix(plan, host, bitmask)
            out = torch.empty((n, W), dtype=torch.int32, device=dev)
            entry.append({"name": name, "plan": plan, "host": host, "bitmask": bitmask, "n": n, "W": W,
                          "out": out, "stored": int(st.item())})
            stored[name] += entry[-1]["stored"]
            total[name] += n * W
        layers.append(entry)
    ctx.sync()
    setup_s = time.perf_counter() - t0
    step_bytes = sum(e["n"] * e["W"] * 4 for e in layers[0])
    f = sum(stored.values()) / float(sum(total.values()))
    steps = range(WU, WU + K)
    link_bytes = {k: sum(e["stored"] * 4 for s in steps for e in layers[s % L] if e["name"] == k)
                  for k in ("weight", "K", "V")}

    def dec(s, which=("weight", "K", "V"), src="host"):
        for e in layers[s % L]:
            if e["name"] in which:
                ibp.ibp_decompress_contig(e["plan"], e[src], e["bitmask"], 0, e["n"], out=e["out"])

    def check(layer_ids) -> bool:
        ok = True
        for li in layer_ids:
            for e, (_, want) in zip(layers[li], originals[li]):
                ok = ok and bool(np.array_equal(e["out"].cpu().numpy().view(np.uint32), want))
        return ok

    timed_layers = sorted({s % L for s in steps})

    # ---- timed region: host-resident contiguous decompress ------------------
    # ncu --clock-control none --nvtx --nvtx-include "llm_host_timed/" selects it
    total_ms, clocks = ctx.timed_with_clocks(dec, "llm_host_timed")
    for e in layers[last % L]:
        ibp.ibp_get_status(e["plan"])
    parity = check(timed_layers)
    ms = total_ms / K
    # ---- end to end through the public API ----------------------------------
    # Eager calls: every step decodes one layer from its pinned host slots (the
    # kernels read the compressed bytes over the host link) and moves each
    # tensor's status word into pinned host memory, where the host checks them
    # after the last step.  Each status read is enqueued right after its decode
    # on the same stream; it launches as a programmatic dependent, so the
    # decodes still overlap one another's start and drain.  Run right after the graph-timed leg, over the same layers,
    # so that both see the host slots in the same state (the GPU's translations
    # of their pages warm).
    status_host = torch.full((WU + K, 3), -1, dtype=torch.int32, pin_memory=True)

    status_v = [[status_host[k, j] for j in range(3)] for k in range(WU + K)]  # views made once

    def e2e_step(s):
        for e, word in zip(layers[s % L], status_v[s]):
            ibp.ibp_decompress_contig(e["plan"], e["host"], e["bitmask"], 0, e["n"], out=e["out"], stream=stream)
            ibp.ibp_get_status_async(e["plan"], word, stream=stream)  # D2H: this tensor's status

    for s in range(WU):
        e2e_step(s)
    e2e_s, enqueue_s = ctx.time_eager(e2e_step)
    e2e_ok = bool((status_host == 0).all().item())
    parity = parity and e2e_ok and check([last % L])
    del status_host

    # the launches of each kernel on their own (weight rows; K and V rows)
    w_ms = ctx.time_steps(lambda s: dec(s, ("weight",)), "llm_weight_host_timed") / K
    kv_ms = ctx.time_steps(lambda s: dec(s, ("K", "V")), "llm_kv_host_timed") / K

    # ---- HBM-resident: the compressed layers copied into HBM ----------------
    for entry in layers:
        for e in entry:
            e["dev"] = e["host"].to(dev)
    ctx.sync()
    for entry in layers:  # outputs are rewritten below: clear them first
        for e in entry:
            e["out"].zero_()
    hbm_ms = ctx.time_steps(lambda s: dec(s, src="dev"), "llm_hbm_timed") / K
    parity = parity and check(timed_layers)
    hbm_w_ms = ctx.time_steps(lambda s: dec(s, ("weight",), "dev"), "llm_weight_hbm_timed") / K
    hbm_kv_ms = ctx.time_steps(lambda s: dec(s, ("K", "V"), "dev"), "llm_kv_hbm_timed") / K
    for entry in layers:
        for e in entry:
            del e["dev"]

    # ---- KV with one Mask/Bitval per attention head (plan sets) -----------
    # The same layers; K and V compressed again, one block of 4096 positions
    # per head with that head's plan, into their own pinned buffers; a step
    # decodes the layer's weight (per-tensor plan, as above) and its K and V
    # with one plan-set call each.
    heads, seq = c["heads"], c["seq"]
    ph_layers = []
    st_ph = {"K": 0, "V": 0}
    for li in range(L):
        entry = []
        for name, tab in originals[li][1:]:
            n, W = tab.shape
            host = torch.empty((n, W), dtype=torch.int32, pin_memory=True)
            host.numpy()[...] = tab.view(np.int32)
            bitmask = torch.zeros((n + 31) // 32, dtype=torch.int32, device=dev)
            stw = torch.zeros(1, dtype=torch.int64, device=dev)
            plans = []
            for h in range(heads):
                blk = tab[h * seq:(h + 1) * seq]
                sample = torch.from_numpy(llm_sample(li, blk).view(np.int32)).to(dev)
                plan = ibp.ibp_plan_create(*ibp.ibp_preprocess(sample, c["T"]), device=ctx.local)
                plan.set_hints(ibp.IBP_HINT_EARLY_FETCH)  # copied into the set below
                ibp.ibp_compress(plan, host[h * seq:(h + 1) * seq],
                                 bitmask=bitmask[h * seq // 32:(h + 1) * seq // 32], stored=stw)
                plans.append(plan)
            ctx.sync()
            for h, plan in enumerate(plans):
                ibp.ibp_plan_tune_prefix(plan, host[h * seq:(h + 1) * seq], bitmask[h * seq // 32:(h + 1) * seq // 32])
            out = layers[li][1 if name == "K" else 2]["out"]
            entry.append((ibp.ibp_plan_set_create(plans), host, bitmask, seq, out))
            st_ph[name] += int(stw.item())
        ph_layers.append(entry)
    f_ph = (stored["weight"] + st_ph["K"] + st_ph["V"]) / float(sum(total.values()))

    def dec_ph(s):
        dec(s, ("weight",))
        for pset, host, bitmask, rpp, out in ph_layers[s % L]:
            ibp.ibp_decompress_contig_set(pset, host, rpp, bitmask, out=out)

    for entry in layers:
        for e in entry:
            e["out"].zero_()
    ph_ms = ctx.time_steps(dec_ph, "llm_ph_host_timed") / K
    for pset, *_ in ph_layers[last % L]:
        ibp.ibp_plan_set_get_status(pset)
    parity_ph = check(timed_layers)
    del ph_layers

    # ---- numbers -------------------------------------------------------------
    world = ctx.world
    ms_step = max_over_ranks(ms, world)
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    e2e_gbs = world * K * step_bytes / max_over_ranks(e2e_s, world) / 1e9
    link_step = sum(link_bytes.values()) / K
    h2d_src = "cudaMemcpyAsync of a 1 GiB pinned buffer into HBM, median of 10, same run"
    per_kernel = {}
    for kind, kms, khbm, names in (("weight", w_ms, hbm_w_ms, ("weight",)), ("kv", kv_ms, hbm_kv_ms, ("K", "V"))):
        lb = sum(link_bytes[k] for k in names) / K / len(names)  # per launch
        out_b = step_bytes / 3  # per launch: one 32 MiB tensor
        n_l = len(names)
        hbm_b = lb + out_b
        per_kernel[kind] = {
            "launches_per_step": n_l, "host_ms_per_launch": round(kms / n_l, 4),
            "hbm_ms_per_launch": round(khbm / n_l, 4),
            "link_bytes_per_launch": round(lb),
            "host_link_frac": round(lb / (kms / n_l * 1e-3) / 1e9 / ctx.h2d_gbs, 4),
            "hbm_frac": round(hbm_b / (khbm / n_l * 1e-3) / 1e9 / ctx.hbm_peak, 4)}
    hbm_step_bytes = link_step + step_bytes
    res = {
        "value": round(value, 3), "unit": "GB/s", "ms_per_step": round(ms_step, 4),
        "config": config_of("llm", ctx.args, world),
        "slots": "pinned host memory, read zero-copy by the kernel",
        "space_saving_pct": {k: round(100 * (1 - stored[k] / total[k]), 3) for k in total},
        "compressed_fraction": round(f, 5),
        "h2d_gbs": round(ctx.h2d_gbs, 2),
        "host_ceiling_gbs": round(ctx.h2d_gbs / f, 2),
        "frac_of_host_ceiling": round(value / world / (ctx.h2d_gbs / f), 4),
        # every launch of the step is k_decompress_fast (the weight's, K's and
        # V's instantiation): bytes per launch and launch time are the step's
        # over its three launches; "kernels" splits them, each timed alone
        "roofline": roofline("host_link", link_step / (ms * 1e-3) / 1e9, ctx.h2d_gbs, h2d_src,
                             "k_decompress_fast (weight, K, V of one layer: 3 launches per step, host slots)",
                             link_step / 3, kernel_traffic("host_resident", "llm").get("link"),
                             traffic_source="ncu: host-link bytes (sysmem sectors x 32) per launch",
                             bytes_per_step=round(link_step)),
        "kernels": per_kernel,
        "hbm_resident": {
            "value": round(step_bytes / (hbm_ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(hbm_ms, 4),
            "roofline": roofline("hbm", hbm_step_bytes / (hbm_ms * 1e-3) / 1e9, ctx.hbm_peak, ctx.hbm_peak_src,
                                 "k_decompress_fast (weight, K, V of one layer: 3 launches per step, slots in HBM)",
                                 hbm_step_bytes / 3, kernel_traffic("hbm_resident", "llm").get("dram"),
                                 output="each layer has its own 96 MiB of outputs (32 layers: 3 GiB > L2)")},
        "kv_per_head": {
            "what": "K and V with one Mask/Bitval per attention head (32 plans per tensor, plan-set decode); "
                    "weight per tensor as above",
            "value": round(step_bytes / (ph_ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ph_ms, 4),
            "space_saving_pct": {"K": round(100 * (1 - st_ph["K"] / total["K"]), 3),
                                 "V": round(100 * (1 - st_ph["V"] / total["V"]), 3)},
            "compressed_fraction": round(f_ph, 5),
            "frac_of_host_ceiling": round(step_bytes / (ph_ms * 1e-3) / 1e9 / (ctx.h2d_gbs / f_ph), 4),
            "parity": "bit-exact" if parity_ph else "MISMATCH"},
        "parity": "bit-exact" if parity else "MISMATCH",
        "e2e": {"value": round(e2e_gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": round(link_step),
                "d2h_bytes_per_step": 12, "enqueue_ms_per_step": round(1e3 * enqueue_s / K, 4),
                "what": "eager API calls; per step one layer's compressed slots read from pinned host memory by "
                        "the kernels (the step's host-to-device bytes) and three status words moved into pinned "
                        "host memory by status reads on the same stream; wall clock, one synchronisation at the end"},
        "gpu_launches": 3 * K,
        "clocks": clocks,
        "table_gen_s": round(gen_s, 2),
        "setup_s": round(setup_s, 2),
        "timing": "K steps captured as one CUDA graph, replay timed with CUDA events",
    }
    if ctx.cpu_ok:
        threads = os.cpu_count() or 1
        gbs, nl, secs, extras = cpu_llm_baseline(originals[0], cpu_seconds, threads)
        res["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                               "sample": f"layer 0 (weight, K, V) compressed by the oracle itself and decoded "
                                         f"{nl} times by the bit-by-bit C oracle in {secs:.1f} s "
                                         f"(OpenMP over rows)", **extras}
    return res


def headline_line(ctx: Ctx, res: dict) -> dict:
    """The driver's JSON line around one config's result."""
    line = {"metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": ctx.world, "steps": ctx.K,
            "warmup": ctx.WU, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u32", "data": "synthetic"}
    for k, v in res.items():
        if k not in ("value", "unit", "ms_per_step"):
            line[k] = v
    return line


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    from host_transfer_gb300 import build, ibp

    build.build()
    ibp.load()
    ctx = Ctx(args)
    if args.config in ("all", "llm"):
        line = headline_line(ctx, run_llm(ctx, args.cpu_seconds))
        if args.config == "all":
            nested = {}
            for name in TABLES:
                nested[name] = run_table(ctx, name, args.nested_cpu_seconds)
                torch.cuda.empty_cache()
            line["configs"] = nested
            line["parity_all_configs"] = "bit-exact" if all(
                r["parity"] == "bit-exact" for r in [line] + list(nested.values())) else "MISMATCH"
    else:
        line = headline_line(ctx, run_table(ctx, args.config, args.cpu_seconds))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
