// ibp_api.cu - the C ABI of libibp: argument checks, pointer resolution,
// plan lifetime, status word.  Kernels live in the other .cu files.
#include <cuda_runtime.h>

#include <vector>
#include <stdio.h>
#include <string.h>

#include <cmath>
#include <new>

#include "ibp_internal.cuh"

namespace ibp {

static thread_local char g_detail[256] = "";

void set_cuda_error(cudaError_t e, const char* where) {
  snprintf(g_detail, sizeof(g_detail), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
}

void set_detail(const char* text) { snprintf(g_detail, sizeof(g_detail), "%s", text); }

void clear_error_detail() { g_detail[0] = 0; }

int check_launch(const char* where) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(e, where);
    return IBP_ECUDA;
  }
  return IBP_OK;
}

int resolve_ptr(const void* p, int device, const void** dev, int* on_device) {
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return IBP_EINVAL;
  }
  *on_device = 1;
  switch (attr.type) {
    case cudaMemoryTypeDevice:
      if (attr.device != device) return IBP_EINVAL;
      *dev = p;
      return IBP_OK;
    case cudaMemoryTypeManaged:
      *dev = p;
      return IBP_OK;
    case cudaMemoryTypeHost:
      if (attr.devicePointer == nullptr) return IBP_EINVAL;
      *dev = attr.devicePointer;
      *on_device = 0;
      return IBP_OK;
    default:
      return IBP_EINVAL;  // pageable host memory
  }
}

int resolve_ptr(const void* p, int device, const void** dev) {
  int on_device;
  return resolve_ptr(p, device, dev, &on_device);
}

int sm_count(int device) {
  // per device; set once, read by any host thread
  static std::atomic<int> cached[64];
  if (device >= 0 && device < 64) {
    const int c = cached[device].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 1;
  }
  if (device >= 0 && device < 64) cached[device].store(n, std::memory_order_relaxed);
  return n;
}

// Makes `device` current for the lifetime of the guard (and restores the
// previous device only when it had to change it).
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  bool changed = false;
  explicit DeviceGuard(int device) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      set_cuda_error(cudaGetLastError(), "cudaGetDevice");
      return;
    }
    if (prev != device) {
      cudaError_t e = cudaSetDevice(device);
      if (e != cudaSuccess) {
        ok = false;
        set_cuda_error(e, "cudaSetDevice");
        cudaGetLastError();
      } else {
        changed = true;
      }
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace ibp

using namespace ibp;

extern "C" {

const char* ibp_strerror(int status) {
  switch (status) {
    case IBP_OK: return "IBP_OK: success";
    case IBP_EINVAL: return "IBP_EINVAL: invalid argument";
    case IBP_ECUDA: return "IBP_ECUDA: CUDA runtime error";
    case IBP_ENOMEM: return "IBP_ENOMEM: device allocation failed";
    case IBP_ECORRUPT: return "IBP_ECORRUPT: corrupt compressed slot";
    case IBP_ERANGE: return "IBP_ERANGE: row id out of range";
    case IBP_ETIMEOUT: return "IBP_ETIMEOUT: bounded wait expired";
    default: return "IBP_?: unknown status";
  }
}

int ibp_version(void) { return IBP_VERSION; }

const char* ibp_last_error_detail(void) { return g_detail; }

int ibp_preprocess(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T, uint32_t* mask,
                   uint32_t* bitval, void* stream) {
  g_detail[0] = 0;
  if (W == 0 || W > IBP_MAX_W || s_rows == 0 || s_rows >= (1ull << 32)) return IBP_EINVAL;
  if (!(T > 0.0 && T <= 1.0)) return IBP_EINVAL;
  if (!sample || !mask || !bitval) return IBP_EINVAL;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) {
    set_cuda_error(cudaGetLastError(), "cudaGetDevice");
    return IBP_ECUDA;
  }
  const void *ds, *dm, *db;
  if (resolve_ptr(sample, device, &ds) || resolve_ptr(mask, device, &dm) ||
      resolve_ptr(bitval, device, &db))
    return IBP_EINVAL;
  return launch_preprocess(static_cast<const uint32_t*>(ds), s_rows, W, T,
                           const_cast<uint32_t*>(static_cast<const uint32_t*>(dm)),
                           const_cast<uint32_t*>(static_cast<const uint32_t*>(db)),
                           static_cast<cudaStream_t>(stream));
}

int ibp_plan_create(const uint32_t* mask, const uint32_t* bitval, uint32_t W, int device,
                    ibp_plan** out) {
  g_detail[0] = 0;
  if (!out || !mask || !bitval || W == 0 || W > IBP_MAX_W) return IBP_EINVAL;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    set_cuda_error(cudaGetLastError(), "cudaGetDeviceCount");
    return IBP_ECUDA;
  }
  if (device < 0 || device >= ndev) return IBP_EINVAL;
  DeviceGuard g(device);
  if (!g.ok) return IBP_ECUDA;

  ibp_plan* p = new (std::nothrow) ibp_plan();
  if (!p) return IBP_ENOMEM;
  p->device = device;
  p->W = W;
  p->S = (W + 31) / 32;
  // Layout (words): mask, bm, pcnt, rmask[4], rshift, mv[5] = 13 W; planes 6 S;
  // eplanes 6 S; status 1 (padded to 4).
  const size_t words = 13ull * W + 12ull * p->S + 4;
  p->d_bytes = words * 4;
  cudaError_t e = cudaMalloc(&p->d_block, p->d_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return IBP_ENOMEM;
  }
  e = cudaHostAlloc(reinterpret_cast<void**>(&p->h_status), 4, cudaHostAllocDefault);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(p->d_block);
    delete p;
    return IBP_ENOMEM;
  }
  uint32_t* base = static_cast<uint32_t*>(p->d_block);
  PlanView& v = p->view;
  v.W = W;
  v.S = p->S;
  v.mask = base;
  v.bm = base + 1ull * W;
  v.pcnt = base + 2ull * W;
  v.rmask = base + 3ull * W;
  v.rshift = base + 7ull * W;
  v.mv = base + 8ull * W;
  v.planes = base + 13ull * W;
  v.eplanes = base + 13ull * W + 6ull * p->S;
  v.status = base + 13ull * W + 12ull * p->S;
  // Mask and Bitval go to the mask and bm slots; the table kernel cleans bm.
  e = cudaMemcpy(const_cast<uint32_t*>(v.mask), mask, 4ull * W, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(const_cast<uint32_t*>(v.bm), bitval, 4ull * W, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemset(v.status, 0, 4);
  if (e != cudaSuccess) {
    set_cuda_error(e, "ibp_plan_create copy");
    cudaGetLastError();
    cudaFree(p->d_block);
    cudaFreeHost(p->h_status);
    delete p;
    return IBP_ECUDA;
  }
  int rc = build_plan_tables(p);
  if (rc != IBP_OK) {
    cudaFree(p->d_block);
    cudaFreeHost(p->h_status);
    delete p;
    return rc;
  }
  *out = p;
  return IBP_OK;
}

int ibp_plan_destroy(ibp_plan* plan) {
  if (!plan) return IBP_OK;
  DeviceGuard g(plan->device);
  cudaError_t e = cudaFree(plan->d_block);
  const cudaError_t e2 = cudaFreeHost(plan->h_status);
  if (e == cudaSuccess) e = e2;
  delete plan;
  if (e != cudaSuccess) {
    set_cuda_error(e, "cudaFree");
    return IBP_ECUDA;
  }
  return IBP_OK;
}

// Words a decompress call fetches from every row before it reads the row's
// headers: the shortest stream the plan allows (in whole 16-byte chunks on the
// vector path), or the longer prefix set by ibp_plan_tune_prefix /
// ibp_plan_set_prefix (slot layout only), never more than W.
static uint32_t prefix_words(const ibp_plan* plan, bool vec, bool packed = false) {
  const uint32_t W = plan->W;
  uint32_t pre = vec ? ((plan->lmin + 3u) / 4u) * 4u : plan->lmin;
  if (!packed && plan->prefix > pre) pre = vec ? ((plan->prefix + 3u) / 4u) * 4u : plan->prefix;
  return pre < W ? pre : W;
}

int ibp_plan_get_info(const ibp_plan* plan, ibp_plan_info* out) {
  if (!plan || !out) return IBP_EINVAL;
  out->W = plan->W;
  out->segments = plan->S;
  out->uniform = plan->uniform;
  out->max_runs = plan->max_runs;
  out->min_kept_bits = plan->min_kept;
  out->max_kept_bits = plan->max_kept;
  out->metadata_bytes = plan->d_bytes;
  out->device = plan->device;
  out->prefix_words = prefix_words(plan, true);
  out->short_rows = plan->short_rows;
  return IBP_OK;
}

int ibp_plan_set_hints(ibp_plan* plan, uint32_t hints) {
  if (!plan || (hints & ~(IBP_HINT_ROW_REUSE | IBP_HINT_EARLY_FETCH))) return IBP_EINVAL;
  plan->view.hints = hints;
  return IBP_OK;
}

int ibp_plan_set_prefix(ibp_plan* plan, uint32_t words) {
  if (!plan) return IBP_EINVAL;
  plan->prefix = words < plan->W ? words : plan->W;
  return IBP_OK;
}

int ibp_plan_tune_prefix(ibp_plan* plan, const uint32_t* slots, uint64_t n_rows, const uint32_t* bitmask,
                         uint64_t max_sample, uint32_t* prefix_words_out, void* stream) {
  g_detail[0] = 0;
  if (!plan || !slots || !bitmask || n_rows == 0) return IBP_EINVAL;
  const uint64_t W = plan->W;
  if (n_rows > (~0ull) / (4 * W)) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void *dsl, *dbm;
  if (resolve_ptr(slots, plan->device, &dsl) || resolve_ptr(bitmask, plan->device, &dbm)) return IBP_EINVAL;
  const uint64_t n_sample = n_rows < (max_sample ? max_sample : 65536ull) ? n_rows : (max_sample ? max_sample : 65536ull);
  const uint32_t nb = static_cast<uint32_t>((W + 3) / 4 + 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* d_hist = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&d_hist), 4ull * nb, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return IBP_ENOMEM;
  }
  std::vector<uint32_t> hist(nb, 0);
  e = cudaMemsetAsync(d_hist, 0, 4ull * nb, st);
  int rc = e == cudaSuccess ? IBP_OK : IBP_ECUDA;
  if (rc == IBP_OK)
    rc = launch_length_hist(plan, static_cast<const uint32_t*>(dsl), n_rows, static_cast<const uint32_t*>(dbm),
                            n_sample, d_hist, st);
  if (rc == IBP_OK) {
    e = cudaMemcpyAsync(hist.data(), d_hist, 4ull * nb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
      set_cuda_error(e, "ibp_plan_tune_prefix");
      rc = IBP_ECUDA;
    }
  }
  cudaFreeAsync(d_hist, st);
  if (rc != IBP_OK) {
    cudaGetLastError();
    return rc;
  }
  // Chunks fetched per row with a prefix of P chunks: max(P, c) for a row of
  // c chunks, plus kRefetch for each row that needs a second, dependent fetch
  // (c > P).  Take the P with the smallest total, the shortest on ties.
  constexpr uint64_t kRefetch = 8;
  const uint32_t pmin = (plan->lmin + 3u) / 4u;
  uint32_t best_p = pmin;
  uint64_t best = ~0ull;
  for (uint32_t P = pmin; P < nb; ++P) {
    uint64_t cost = 0;
    for (uint32_t c = 0; c < nb; ++c) cost += hist[c] * (c > P ? c + kRefetch : P);
    if (cost < best) {
      best = cost;
      best_p = P;
    }
  }
  plan->prefix = static_cast<uint32_t>(4ull * best_p < W ? 4ull * best_p : W);
  // Short rows: at least 99 % of the sampled rows store at most W / 4 words
  // (raw rows store W).  Decodes from device memory then stage W / 4 words
  // per row and read the few longer rows from their slots.
  uint64_t total = 0, short_n = 0;
  for (uint32_t c = 0; c < nb; ++c) {
    total += hist[c];
    if (4ull * c <= W / 4) short_n += hist[c];
  }
  plan->short_rows = (total > 0 && 100ull * short_n >= 99ull * total) ? 1u : 0u;
  if (prefix_words_out) *prefix_words_out = prefix_words(plan, W % 4 == 0);
  return IBP_OK;
}

int ibp_plan_get_mask(const ibp_plan* plan, uint32_t* mask, uint32_t* bitval) {
  if (!plan) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  cudaError_t e = cudaSuccess;
  if (mask) e = cudaMemcpy(mask, plan->view.mask, 4ull * plan->W, cudaMemcpyDefault);
  if (e == cudaSuccess && bitval)
    e = cudaMemcpy(bitval, plan->view.bm, 4ull * plan->W, cudaMemcpyDefault);
  if (e != cudaSuccess) {
    set_cuda_error(e, "ibp_plan_get_mask");
    cudaGetLastError();
    return IBP_ECUDA;
  }
  return IBP_OK;
}

int ibp_compress(const ibp_plan* plan, const uint32_t* rows, uint32_t* slots, uint64_t n_rows,
                 uint32_t* bitmask, uint64_t* stored_words, void* stream) {
  g_detail[0] = 0;
  if (!plan) return IBP_EINVAL;
  if (n_rows == 0) return IBP_OK;
  if (!rows || !slots || !bitmask) return IBP_EINVAL;
  const uint64_t W = plan->W;
  if (n_rows > (~0ull) / (4 * W)) return IBP_EINVAL;
  // in place, or no overlap at all
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(rows), s0 = reinterpret_cast<uintptr_t>(slots);
  const uintptr_t len = n_rows * W * 4;
  if (r0 != s0 && r0 < s0 + len && s0 < r0 + len) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void *dr, *ds, *db, *dst = nullptr;
  if (resolve_ptr(rows, plan->device, &dr) || resolve_ptr(slots, plan->device, &ds) ||
      resolve_ptr(bitmask, plan->device, &db))
    return IBP_EINVAL;
  if (stored_words && resolve_ptr(stored_words, plan->device, &dst)) return IBP_EINVAL;
  CompressArgs a;
  a.pv = plan->view;
  a.rows = static_cast<const uint32_t*>(dr);
  a.slots = const_cast<uint32_t*>(static_cast<const uint32_t*>(ds));
  a.n_rows = n_rows;
  a.bitmask = const_cast<uint32_t*>(static_cast<const uint32_t*>(db));
  a.stored = const_cast<unsigned long long*>(static_cast<const unsigned long long*>(dst));
  a.vec = (W % 4 == 0) && aligned16(a.rows) && aligned16(a.slots);
  a.rowcap = static_cast<uint32_t>(((W + 31) / 32) * 32);
  return launch_compress(plan, a, static_cast<cudaStream_t>(stream));
}

static int decompress_common(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                             const uint32_t* bitmask, const int64_t* ids, uint64_t first,
                             uint64_t n_out, uint32_t* out, void* stream,
                             const uint64_t* offsets = nullptr) {
  const uint64_t W = plan->W;
  if (n_rows > (~0ull) / (4 * W) || n_out > (~0ull) / (4 * W)) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void *dsl, *dbm, *dout, *dids = nullptr;
  int slots_on_device = 1;
  if (resolve_ptr(slots, plan->device, &dsl, &slots_on_device) || resolve_ptr(bitmask, plan->device, &dbm) ||
      resolve_ptr(out, plan->device, &dout))
    return IBP_EINVAL;
  if (ids && resolve_ptr(ids, plan->device, &dids)) return IBP_EINVAL;
  const void* doff = nullptr;
  if (offsets && resolve_ptr(offsets, plan->device, &doff)) return IBP_EINVAL;
  DecodeArgs a{};
  a.offsets = static_cast<const uint64_t*>(doff);
  a.dev_slots = static_cast<uint32_t>(slots_on_device);
  a.pv = plan->view;
  a.slots = static_cast<const uint32_t*>(dsl);
  a.bitmask = static_cast<const uint32_t*>(dbm);
  a.ids = static_cast<const int64_t*>(dids);
  a.first = first;
  a.n_rows = n_rows;
  a.n_out = n_out;
  a.out = const_cast<uint32_t*>(static_cast<const uint32_t*>(dout));
  a.vec = (W % 4 == 0) && aligned16(a.slots) && aligned16(a.out);
  a.rowcap = static_cast<uint32_t>(((W + 31) / 32) * 32);
  // prefix fetched before the headers (never past the row: W % 4 == 0 on the
  // vector path)
  a.pre = prefix_words(plan, a.vec != 0, offsets != nullptr);
  uint32_t G = 1152u / static_cast<uint32_t>(W + 4);
  a.G = G < 1 ? 1 : (G > 32 ? 32 : G);
  if (a.offsets) {  // the packed layout is decoded by the specialised kernel only
    if (!fast_decompress_applies(plan, a)) return IBP_EINVAL;
    return launch_decompress_fast(plan, a, static_cast<cudaStream_t>(stream));
  }
  return launch_decompress(plan, a, static_cast<cudaStream_t>(stream));
}

int ibp_gather_decompress(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                          const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                          uint32_t* out, void* stream) {
  g_detail[0] = 0;
  if (!plan) return IBP_EINVAL;
  if (n_ids == 0) return IBP_OK;
  if (!slots || !bitmask || !row_ids || !out || n_rows == 0) return IBP_EINVAL;
  return decompress_common(plan, slots, n_rows, bitmask, row_ids, 0, n_ids, out, stream);
}

int ibp_decompress_contig(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                          const uint32_t* bitmask, uint64_t first_row, uint64_t n, uint32_t* out,
                          void* stream) {
  g_detail[0] = 0;
  if (!plan) return IBP_EINVAL;
  if (n == 0) return IBP_OK;
  if (!slots || !bitmask || !out) return IBP_EINVAL;
  if (first_row >= n_rows || n > n_rows - first_row) return IBP_EINVAL;
  return decompress_common(plan, slots, n_rows, bitmask, nullptr, first_row, n, out, stream);
}

int ibp_packed_offsets(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                       const uint32_t* bitmask, uint64_t* offsets, void* stream) {
  g_detail[0] = 0;
  if (!plan || !offsets || plan->W % 4u) return IBP_EINVAL;
  if (n_rows == 0) {
    DeviceGuard g(plan->device);
    if (!g.ok) return IBP_ECUDA;
    cudaError_t e = cudaMemsetAsync(offsets, 0, sizeof(uint64_t), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      set_cuda_error(e, "cudaMemsetAsync");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    return IBP_OK;
  }
  if (!slots || !bitmask || n_rows > (~0ull) / (4ull * plan->W)) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void *ds, *db, *dof;
  if (resolve_ptr(slots, plan->device, &ds) || resolve_ptr(bitmask, plan->device, &db) ||
      resolve_ptr(offsets, plan->device, &dof))
    return IBP_EINVAL;
  return launch_packed_offsets(plan, static_cast<const uint32_t*>(ds), n_rows,
                               static_cast<const uint32_t*>(db),
                               const_cast<uint64_t*>(static_cast<const uint64_t*>(dof)),
                               static_cast<cudaStream_t>(stream));
}

int ibp_pack(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows, const uint64_t* offsets,
             uint32_t* packed, void* stream) {
  g_detail[0] = 0;
  if (!plan || plan->W % 4u) return IBP_EINVAL;
  if (n_rows == 0) return IBP_OK;
  if (!slots || !offsets || !packed || n_rows > (~0ull) / (4ull * plan->W)) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void *ds, *dof, *dp;
  if (resolve_ptr(slots, plan->device, &ds) || resolve_ptr(offsets, plan->device, &dof) ||
      resolve_ptr(packed, plan->device, &dp))
    return IBP_EINVAL;
  if (!aligned16(ds) || !aligned16(dp)) return IBP_EINVAL;
  return launch_pack(static_cast<const uint32_t*>(ds), n_rows, plan->W,
                     static_cast<const uint64_t*>(dof),
                     const_cast<uint32_t*>(static_cast<const uint32_t*>(dp)), plan->device,
                     static_cast<cudaStream_t>(stream));
}

int ibp_gather_decompress_packed(const ibp_plan* plan, const uint32_t* packed,
                                 const uint64_t* offsets, uint64_t n_rows,
                                 const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                                 uint32_t* out, void* stream) {
  g_detail[0] = 0;
  if (!plan) return IBP_EINVAL;
  if (n_ids == 0) return IBP_OK;
  if (!packed || !offsets || !bitmask || !row_ids || !out || n_rows == 0) return IBP_EINVAL;
  return decompress_common(plan, packed, n_rows, bitmask, row_ids, 0, n_ids, out, stream, offsets);
}

int ibp_get_status(const ibp_plan* plan, void* stream) {
  g_detail[0] = 0;
  if (!plan) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  // h_status is the plan's one pinned word: one caller at a time
  std::lock_guard<std::mutex> lock(const_cast<ibp_plan*>(plan)->status_mu);
  // one copy into the plan's pinned word, ordered on the stream, then one wait
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(plan->h_status, plan->view.status, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  const uint32_t st = e == cudaSuccess ? *plan->h_status : 0u;
  if (e == cudaSuccess && st != 0) {
    e = cudaMemsetAsync(plan->view.status, 0, 4, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) {
    set_cuda_error(e, "ibp_get_status");
    cudaGetLastError();
    return IBP_ECUDA;
  }
  return static_cast<int>(st);
}

}  // extern "C"

// Moves the status word to *dst and clears it, in one atomic exchange (so an
// error recorded concurrently by another stream's kernel is either moved or
// kept, never lost).  Launched as a programmatic dependent: it lets the next
// kernel of the stream launch at once and then waits, before the exchange,
// for the previous grid to complete with its memory visible.  A decode that
// follows it on the same stream therefore still fetches its first ids and
// prefixes while the previous decode drains; its own status writes come after
// its wait, which ends only once this grid (and so the previous decode) has
// completed.
__global__ void k_take_status(uint32_t* status, uint32_t* dst) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) *dst = atomicExch(status, 0u);
}

extern "C" {

int ibp_get_status_async(const ibp_plan* plan, uint32_t* status_out, void* stream) {
  g_detail[0] = 0;
  if (!plan || !status_out) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void* dst;
  if (resolve_ptr(status_out, plan->device, &dst)) return IBP_EINVAL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_take_status, plan->view.status,
                                           const_cast<uint32_t*>(static_cast<const uint32_t*>(dst)));
  if (e != cudaSuccess) {
    set_cuda_error(e, "k_take_status");
    cudaGetLastError();
    return IBP_ECUDA;
  }
  return check_launch("k_take_status");
}

int ibp_row_lengths(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                    const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                    uint32_t* lengths, void* stream) {
  g_detail[0] = 0;
  if (!plan) return IBP_EINVAL;
  if (n_ids == 0) return IBP_OK;
  if (!slots || !bitmask || !row_ids || !lengths || n_rows == 0) return IBP_EINVAL;
  if (n_rows > (~0ull) / (4ull * plan->W) || n_ids > (1ull << 40)) return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void *ds, *db, *di, *dl;
  if (resolve_ptr(slots, plan->device, &ds) || resolve_ptr(bitmask, plan->device, &db) ||
      resolve_ptr(row_ids, plan->device, &di) || resolve_ptr(lengths, plan->device, &dl))
    return IBP_EINVAL;
  return launch_row_lengths(plan, static_cast<const uint32_t*>(ds), n_rows,
                            static_cast<const uint32_t*>(db), static_cast<const int64_t*>(di), n_ids,
                            const_cast<uint32_t*>(static_cast<const uint32_t*>(dl)),
                            static_cast<cudaStream_t>(stream));
}

int ibp_gather_raw(const uint32_t* rows, uint64_t n_rows, uint32_t W, const int64_t* row_ids,
                   uint64_t n_ids, uint32_t* out, void* stream) {
  g_detail[0] = 0;
  if (W == 0 || W > IBP_MAX_W) return IBP_EINVAL;
  if (n_ids == 0) return IBP_OK;
  if (!rows || !row_ids || !out || n_rows == 0) return IBP_EINVAL;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) {
    set_cuda_error(cudaGetLastError(), "cudaGetDevice");
    return IBP_ECUDA;
  }
  const void *dr, *di, *dout;
  if (resolve_ptr(rows, device, &dr) || resolve_ptr(row_ids, device, &di) ||
      resolve_ptr(out, device, &dout))
    return IBP_EINVAL;
  const bool vec = (W % 4 == 0) && aligned16(dr) && aligned16(dout);
  return launch_gather_raw(static_cast<const uint32_t*>(dr), n_rows, W,
                           static_cast<const int64_t*>(di), n_ids,
                           const_cast<uint32_t*>(static_cast<const uint32_t*>(dout)), vec, device,
                           static_cast<cudaStream_t>(stream));
}

}  // extern "C"

int ibp_gather_decompress_bag(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                              const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                              const int64_t* bag_offsets, uint64_t n_bags, uint32_t mode, float* out,
                              void* stream) {
  g_detail[0] = 0;
  if (!plan) return IBP_EINVAL;
  if (n_bags == 0) return IBP_OK;
  if (!slots || !bitmask || !bag_offsets || !out || n_rows == 0 || (mode & ~(IBP_BAG_MEAN | IBP_BAG_BF16)))
    return IBP_EINVAL;
  if ((n_ids > 0 && !row_ids) || n_rows >= (1ull << 31) || n_ids > (1ull << 40) || n_bags > (1ull << 40))
    return IBP_EINVAL;
  DeviceGuard g(plan->device);
  if (!g.ok) return IBP_ECUDA;
  const void *dsl, *dbm, *doff, *dout, *dids = nullptr;
  int slots_on_device = 1;
  if (resolve_ptr(slots, plan->device, &dsl, &slots_on_device) || resolve_ptr(bitmask, plan->device, &dbm) ||
      resolve_ptr(bag_offsets, plan->device, &doff) || resolve_ptr(out, plan->device, &dout))
    return IBP_EINVAL;
  if (row_ids && resolve_ptr(row_ids, plan->device, &dids)) return IBP_EINVAL;
  // bfloat16 rows: the pooled pairs of floats are written with 8-byte stores
  if ((mode & IBP_BAG_BF16) && (reinterpret_cast<uintptr_t>(dout) & 7u)) return IBP_EINVAL;
  BagArgs a{};
  DecodeArgs& d = a.d;
  d.pv = plan->view;
  d.slots = static_cast<const uint32_t*>(dsl);
  d.bitmask = static_cast<const uint32_t*>(dbm);
  d.ids = static_cast<const int64_t*>(dids);
  d.n_rows = n_rows;
  d.n_out = n_ids;
  d.vec = (plan->W % 4 == 0) && aligned16(d.slots);
  d.dev_slots = static_cast<uint32_t>(slots_on_device);
  d.rowcap = ((plan->W + 31) / 32) * 32;
  d.pre = prefix_words(plan, d.vec != 0);
  d.G = 1;
  a.offsets = static_cast<const int64_t*>(doff);
  a.n_ids = n_ids;
  a.n_bags = n_bags;
  a.out = static_cast<float*>(const_cast<void*>(dout));
  a.mean = (mode & IBP_BAG_MEAN) ? 1u : 0u;
  a.bf16 = (mode & IBP_BAG_BF16) ? 1u : 0u;
  return launch_bag(plan, a, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Plan sets: one plan per block of consecutive rows (finer Mask granularity)

struct ibp_plan_set {
  int device;
  uint32_t W, S, n, max_runs, npl;
  std::vector<const ibp_plan*> plans;
  ibp::PlanView* d_views;  // n views in device memory
};

int ibp_plan_set_create(const ibp_plan* const* plans, uint32_t n_plans, ibp_plan_set** out) {
  g_detail[0] = 0;
  if (!out) return IBP_EINVAL;
  *out = nullptr;
  if (!plans || n_plans == 0 || n_plans > 65535u || !plans[0]) return IBP_EINVAL;
  const ibp_plan* p0 = plans[0];
  const uint32_t S = p0->S, W = p0->W;
  const bool pow2 = S == 1 || S == 2 || S == 4 || S == 8 || S == 16 || S == 32;
  if (W != 32u * S || !pow2) return IBP_EINVAL;
  std::vector<PlanView> views(n_plans);
  uint32_t max_runs = 0, npl = 0;
  for (uint32_t i = 0; i < n_plans; ++i) {
    const ibp_plan* p = plans[i];
    if (!p || p->device != p0->device || p->W != W || p->max_runs > static_cast<uint32_t>(kMaxRuns))
      return IBP_EINVAL;
    max_runs = p->max_runs > max_runs ? p->max_runs : max_runs;
    npl = p->view.npl > npl ? p->view.npl : npl;
    views[i] = p->view;
    views[i].pre = prefix_words(p, true);  // the plan's own prefix, as of now
  }
  DeviceGuard g(p0->device);
  if (!g.ok) return IBP_ECUDA;
  ibp_plan_set* set = new (std::nothrow) ibp_plan_set();
  if (!set) return IBP_ENOMEM;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&set->d_views), sizeof(PlanView) * n_plans);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete set;
    return IBP_ENOMEM;
  }
  e = cudaMemcpy(set->d_views, views.data(), sizeof(PlanView) * n_plans, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    set_cuda_error(e, "ibp_plan_set_create");
    cudaGetLastError();
    cudaFree(set->d_views);
    delete set;
    return IBP_ECUDA;
  }
  set->device = p0->device;
  set->W = W;
  set->S = S;
  set->n = n_plans;
  set->max_runs = max_runs;
  set->npl = npl;
  set->plans.assign(plans, plans + n_plans);
  *out = set;
  return IBP_OK;
}

int ibp_plan_set_destroy(ibp_plan_set* set) {
  if (!set) return IBP_OK;
  DeviceGuard g(set->device);
  cudaError_t e = cudaFree(set->d_views);
  delete set;
  if (e != cudaSuccess) {
    set_cuda_error(e, "cudaFree");
    return IBP_ECUDA;
  }
  return IBP_OK;
}

int ibp_decompress_contig_set(const ibp_plan_set* set, const uint32_t* slots, uint64_t rows_per_plan,
                              const uint32_t* bitmask, uint32_t* out, void* stream) {
  g_detail[0] = 0;
  if (!set) return IBP_EINVAL;
  if (rows_per_plan == 0) return IBP_OK;
  if (!slots || !bitmask || !out) return IBP_EINVAL;
  if (rows_per_plan >= (1ull << 31) / set->n) return IBP_EINVAL;  // every row id fits in 31 bits
  const uint64_t n_rows = rows_per_plan * set->n;
  DeviceGuard g(set->device);
  if (!g.ok) return IBP_ECUDA;
  const void *dsl, *dbm, *dout;
  int slots_on_device = 1;
  if (resolve_ptr(slots, set->device, &dsl, &slots_on_device) || resolve_ptr(bitmask, set->device, &dbm) ||
      resolve_ptr(out, set->device, &dout))
    return IBP_EINVAL;
  DecodeArgs a{};
  a.pv = set->plans[0]->view;
  a.slots = static_cast<const uint32_t*>(dsl);
  a.bitmask = static_cast<const uint32_t*>(dbm);
  a.n_rows = n_rows;
  a.n_out = n_rows;
  a.out = const_cast<uint32_t*>(static_cast<const uint32_t*>(dout));
  a.vec = aligned16(a.slots) && aligned16(a.out);
  if (!a.vec) return IBP_EINVAL;  // the set decoder is the 16-byte vector path
  a.dev_slots = static_cast<uint32_t>(slots_on_device);
  a.rowcap = set->W;
  a.pre = set->W;  // each CTA takes its plan's prefix from the device views
  a.G = 1;
  a.plans = set->d_views;
  a.rows_per_plan = rows_per_plan;
  a.n_plans = set->n;
  return launch_fast_set(set->plans[0], set->max_runs, set->npl, a, static_cast<cudaStream_t>(stream));
}

int ibp_plan_set_get_status(const ibp_plan_set* set, void* stream) {
  g_detail[0] = 0;
  if (!set) return IBP_EINVAL;
  int first = IBP_OK;
  for (const ibp_plan* p : set->plans) {
    const int st = ibp_get_status(p, stream);
    if (st == IBP_ECUDA) return st;
    if (first == IBP_OK) first = st;
  }
  return first;
}
