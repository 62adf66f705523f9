// ibp_noalloc.cu - ibp_preprocess without any device allocation.
//
// ibp_preprocess needs 128 * W bytes of scratch for its per-bit counters and
// gets them from cudaMallocAsync.  Some callers cannot allocate device memory
// from inside this library: processes whose device memory is wholly owned by
// their own allocator (a framework's caching allocator, a fixed arena sized at
// start-up), and devices or drivers without stream-ordered memory pools
// (cudaDevAttrMemoryPoolsSupported = 0).  ibp_preprocess_noalloc serves them:
// its counters live in the file-scope array below, a fixed
// IBP_NOALLOC_MAX_W * 32 words (512 KiB) that every GPU which loads the library
// keeps until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ibp_internal.cuh"

namespace ibp {

// Per-bit counters for one preprocess call: ones[w * 32 + b].  Shared by every
// call on a device; each call clears the part it uses before counting.
static __device__ __align__(256) uint32_t g_noalloc_ones[IBP_NOALLOC_MAX_W * 32];

// Device address of g_noalloc_ones per device, with the id of the context it
// was looked up in.  In host code the name g_noalloc_ones is only a host-side
// stand-in for the symbol, never a device address, so kernels always get the
// looked-up pointer.  The module (and so the array) is loaded anew in a new
// context, e.g. after cudaDeviceReset, and may then sit at another address:
// the context id tells a stale entry from a valid one.
static std::mutex g_noalloc_mu;
struct NoallocEntry {
  unsigned long long ctx_id;
  uint32_t* ptr;
};
static NoallocEntry g_noalloc[64] = {};

// cuCtxGetId of the current context, through the runtime's driver entry
// point (the library does not link the driver library itself).
static int current_ctx_id(unsigned long long* id) {
  using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);
  static std::atomic<CtxGetId> fn_cache{nullptr};  // looked up once, any host thread
  CtxGetId fn = fn_cache.load(std::memory_order_acquire);
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) {
      set_cuda_error(e != cudaSuccess ? e : cudaErrorSymbolNotFound, "cudaGetDriverEntryPointByVersion(cuCtxGetId)");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    fn = reinterpret_cast<CtxGetId>(f);
    fn_cache.store(fn, std::memory_order_release);
  }
  if (fn(nullptr, id) != CUDA_SUCCESS) {
    set_detail("cuCtxGetId: no current context");
    return IBP_ECUDA;
  }
  return IBP_OK;
}

// `device` is the current device.  Looks the array up the first time it is
// used in the device's current context.
static int noalloc_scratch(int device, uint32_t** out) {
  if (device < 0 || device >= 64) return IBP_EINVAL;
  unsigned long long ctx = 0;
  int rc = current_ctx_id(&ctx);
  if (rc != IBP_OK) return rc;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocEntry& ent = g_noalloc[device];
  if (!ent.ptr || ent.ctx_id != ctx) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_ones);
    if (e != cudaSuccess || p == nullptr) {
      set_cuda_error(e, "cudaGetSymbolAddress(g_noalloc_ones)");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    ent.ptr = static_cast<uint32_t*>(p);
    ent.ctx_id = ctx;
  }
  *out = ent.ptr;
  return IBP_OK;
}

}  // namespace ibp

using namespace ibp;

extern "C" int ibp_preprocess_noalloc(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T,
                                      uint32_t* mask, uint32_t* bitval, void* stream) {
  clear_error_detail();
  if (W > IBP_NOALLOC_MAX_W) {
    set_detail("ibp_preprocess_noalloc: W is above IBP_NOALLOC_MAX_W (4096)");
    return IBP_EINVAL;
  }
  if (W == 0 || s_rows == 0 || s_rows >= (1ull << 32)) return IBP_EINVAL;
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
  uint32_t* ones = nullptr;
  int rc = noalloc_scratch(device, &ones);
  if (rc != IBP_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The counters keep the previous call's values: clear the W * 32 in use.
  cudaError_t e = cudaMemsetAsync(ones, 0, 32ull * W * sizeof(uint32_t), st);
  if (e != cudaSuccess) {
    set_cuda_error(e, "cudaMemsetAsync");
    cudaGetLastError();
    return IBP_ECUDA;
  }
  return launch_count_and_threshold(static_cast<const uint32_t*>(ds), s_rows, W, T, ones,
                                    const_cast<uint32_t*>(static_cast<const uint32_t*>(dm)),
                                    const_cast<uint32_t*>(static_cast<const uint32_t*>(db)), st);
}
