// ibp_internal.cuh - shared internals of libibp (not part of the ABI).
//
// Plan tables, device bit helpers and the launchers each kernel file
// provides.  Everything here is written for sm_103a; the library is built
// only for that target.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "ibp.h"

namespace ibp {

constexpr int kMaxRuns = 4;     // runs of kept bits handled by the run tables
constexpr int kPlanes = 6;      // bit planes of a kept-bit count (0..32)
constexpr int kWarp = 32;

// Row kinds decided before a row's payload is fetched (kCompSlot: a
// compressed row decoded from its slot instead of a shared-memory stage).
enum RowKind : uint32_t { kNone = 0, kRaw = 1, kComp = 2, kBadRange = 3, kCorrupt = 4, kCompSlot = 5 };

// Device view of a plan, passed to kernels by value.
//
// Per word position w (arrays of W words):
//   mask[w]     invariant bits
//   bm[w]       Bitval[w] & Mask[w]
//   pcnt[w]     popcount(Mask[w]) (bits a matching word drops)
//   rmask[k*W+w], k < kMaxRuns: k-th run of kept bits (~Mask[w]) at its
//               position in the word; 0 for missing runs
//   rshift[w]   byte k = left shift that moves run k from its packed position
//               (kept bits before it) to its place in the word
//   mv[i*W+w], i < 5: move masks of the five-step parallel-suffix
//               compress/expand (Hacker's Delight, sections 7-4 and 7-5) for
//               ~Mask[w]; used when some word has more than kMaxRuns runs
// Per segment s (S = ceil(W/32) segments):
//   planes[s*6+k] bit i = bit k of pcnt[32s+i]; lets one lane sum
//               popcount(Mask) over the matching words of a segment with six
//               popcounts.
//   eplanes[s*6+k] bit i = bit k of e_w, w = 32s+i, where
//               pcnt[w] = p_min + p_scale * e_w (p_min the smallest popcount,
//               p_scale the gcd of the differences); e_w < 2^npl.  With two
//               distinct popcounts npl = 1, so a prefix sum of pcnt over the
//               matching lanes is p_min * popc(H & lt) + p_scale *
//               popc(H & E_0 & lt).
struct PlanView {
  uint32_t W, S;
  const uint32_t* mask;
  const uint32_t* bm;
  const uint32_t* pcnt;
  const uint32_t* rmask;
  const uint32_t* rshift;
  const uint32_t* mv;
  const uint32_t* planes;
  const uint32_t* eplanes;
  uint32_t* status;
  uint32_t p_min, p_scale, npl;
  uint32_t hints;  // IBP_HINT_* bits set by ibp_plan_set_hints
  uint32_t pre;    // words fetched before the headers (read from device views of plan sets)
  // Uniform plans (every word position has the same Mask/Bitval): scalars.
  uint32_t u_mask, u_bm, u_p, u_keep;
  uint32_t u_rmask[kMaxRuns];
  uint32_t u_rsh[kMaxRuns];
  uint32_t u_mv[5];
};

}  // namespace ibp

struct ibp_plan {
  int device;
  uint32_t W, S;
  uint32_t uniform, max_runs, min_kept, max_kept;
  uint32_t lmin;  // min(W, words of the shortest possible compressed stream)
  uint32_t prefix;  // words fetched before the headers (slot layout); 0 = from lmin
  uint32_t short_rows;  // the tuner found 99 % of the sampled rows at most W / 4 words long
  void* d_block;  // single device allocation holding every table + status
  uint32_t* h_status;  // pinned host word the status is read back into
  std::mutex status_mu;  // serialises ibp_get_status calls on this plan (h_status)
  size_t d_bytes;
  ibp::PlanView view;
};

namespace ibp {

// ---------------------------------------------------------------------------
// Host-side helpers (ibp_api.cu)

void set_cuda_error(cudaError_t e, const char* where);
// Plain text for ibp_last_error_detail (argument errors, not CUDA errors).
void set_detail(const char* text);
void clear_error_detail();
int check_launch(const char* where);
// Resolves a pointer to an address a kernel on `device` can dereference.
// Accepts device memory of `device`, managed memory, and mapped pinned host
// memory.  Returns IBP_OK or IBP_EINVAL.
int resolve_ptr(const void* p, int device, const void** dev);
// As resolve_ptr; also sets *on_device to 1 for device or managed memory and
// to 0 for mapped host memory.
int resolve_ptr(const void* p, int device, const void** dev, int* on_device);
int sm_count(int device);

// ---------------------------------------------------------------------------
// Launchers (one per kernel file)

struct DecodeArgs {
  PlanView pv;
  const uint32_t* slots;   // row 0 of the table
  const uint32_t* bitmask;
  const int64_t* ids;      // nullptr: rows first, first + 1, ...
  const uint64_t* offsets; // packed layout: row r at slots[offsets[r] .. offsets[r+1]); else nullptr
  uint64_t first;
  uint64_t n_rows;         // rows in the table
  uint64_t n_out;          // rows to produce
  uint32_t* out;
  uint32_t G;              // rows per group
  uint32_t rowcap;         // stage words per row: W rounded up to a multiple of 32
  uint32_t pre;            // words fetched for every row before its headers are read
  uint32_t vec;            // 16-byte copies allowed
  uint32_t dev_slots;      // slots in device (or managed) memory, not host-mapped
  // plan sets: row block y of rows_per_plan rows is decoded with plans[y]
  const PlanView* plans;   // device array of n_plans views, or nullptr
  uint64_t rows_per_plan;
  uint32_t n_plans;
};

int launch_decompress(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
// Specialised decompress for uniform plans with W = 32 * 2^k <= 2048 words,
// at most kMaxRuns runs of kept bits, 16-byte aligned buffers and fewer than
// 2^31 rows (ibp_decompress_fast.cu).
bool fast_decompress_applies(const ibp_plan* plan, const DecodeArgs& a);
int launch_decompress_fast(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
// Gather-decompress fused with sum / mean pooling (ibp_bag.cu).
struct BagArgs {
  DecodeArgs d;            // plan, slots, bitmask, ids, n_rows, pre, vec (n_out unused)
  const int64_t* offsets;  // n_bags + 1 bag boundaries into ids
  uint64_t n_ids;
  uint64_t n_bags;
  float* out;              // n_bags x W
  uint32_t mean;           // 0: sum, 1: mean
  uint32_t bf16;           // rows of bfloat16 pairs: out has 2W floats per bag
};
// Specialised shapes only (as fast_decompress_applies, S <= 16); else IBP_EINVAL.
int launch_bag(const ibp_plan* plan, BagArgs& a, cudaStream_t stream);

// Plan sets (ibp_decompress_fast_set.cu): contiguous decode through the
// specialised kernel's table path with the set's most runs (2 or 4) and
// e-planes (0, 1 or 6); W = 32 * S, S <= 32, 16-byte aligned buffers.
int launch_fast_set(const ibp_plan* plan0, uint32_t max_runs, uint32_t npl, DecodeArgs& a, cudaStream_t stream);

// Packed cache layout (ibp_packed.cu): per-row stored lengths rounded up to
// 4 words and their exclusive scan; the copy of slots into packed rows.
int launch_packed_offsets(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                          const uint32_t* bitmask, uint64_t* offsets, cudaStream_t stream);
int launch_pack(const uint32_t* slots, uint64_t n_rows, uint32_t W, const uint64_t* offsets,
                uint32_t* packed, int device, cudaStream_t stream);

struct CompressArgs {
  PlanView pv;
  const uint32_t* rows;
  uint32_t* slots;
  uint64_t n_rows;
  uint32_t* bitmask;
  unsigned long long* stored;  // may be null
  uint32_t rowcap;  // words per row buffer: W rounded up to a multiple of 32
  uint32_t vec;
};

int launch_compress(const ibp_plan* plan, CompressArgs& a, cudaStream_t stream);

int launch_preprocess(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T,
                      uint32_t* mask, uint32_t* bitval, cudaStream_t stream);

// The two preprocess launches (bit counts, then Mask/Bitval) on a caller-
// provided zeroed counter array of 32 * W words.
int launch_count_and_threshold(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T,
                               uint32_t* ones, uint32_t* mask, uint32_t* bitval,
                               cudaStream_t stream);

// Builds the tables of a plan whose d_block is allocated and whose mask and
// bitval arrays already hold the caller's Mask/Bitval.  Fills the summary
// fields and the uniform scalars.  Synchronous.
int build_plan_tables(ibp_plan* plan);

int launch_row_lengths(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                       const uint32_t* bitmask, const int64_t* ids, uint64_t n_ids,
                       uint32_t* lengths, cudaStream_t stream);
// Histogram of the stored lengths (16-byte chunks) of n_sample evenly spaced
// rows into hist[0 .. ceil(W/4)] (zeroed by the caller).
int launch_length_hist(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                       const uint32_t* bitmask, uint64_t n_sample, uint32_t* hist, cudaStream_t stream);

int launch_gather_raw(const uint32_t* rows, uint64_t n_rows, uint32_t W, const int64_t* ids,
                      uint64_t n_ids, uint32_t* out, bool vec, int device, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Device helpers

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 16-byte asynchronous global -> shared copy, cached in L2 only (streaming
// rows: each is read once per call).
__device__ __forceinline__ void cp_async16(uint32_t* smem_dst, const void* gsrc) {
  uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gsrc) : "memory");
}

// The same copy, also allocating in L1: a row requested again by the same SM
// (repeated ids, e.g. Zipf-distributed lookups) is then served from L1
// instead of crossing the host link again.  Mapped host memory is not kept
// in L2, so L1 is the only on-chip place a repeat can hit.
__device__ __forceinline__ void cp_async16_l1(uint32_t* smem_dst, const void* gsrc) {
  uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gsrc) : "memory");
}

// Row copy of the decoders: L1-allocating when the plan carries
// IBP_HINT_ROW_REUSE (warp-uniform branch).
__device__ __forceinline__ void cp_row16(bool l1, uint32_t* smem_dst, const void* gsrc) {
  if (l1)
    cp_async16_l1(smem_dst, gsrc);
  else
    cp_async16(smem_dst, gsrc);
}

__device__ __forceinline__ void cp_async4(uint32_t* smem_dst, const void* gsrc) {
  uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Plain (coherent) 32-bit load; works on device and mapped host memory.
__device__ __forceinline__ uint32_t ld_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void record_status(uint32_t* status, uint32_t code) {
  atomicCAS(status, 0u, code);
}

// Place the low kept bits of v at the kept positions of a word, using up to
// R runs: run k of the kept mask, starting at bit position lo_k with s_k kept
// bits before it, receives (v << (lo_k - s_k)) & run_k.
template <int R>
__device__ __forceinline__ uint32_t deposit_runs(uint32_t v, const uint32_t* rm, const uint32_t* rs) {
  uint32_t y = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) y |= (v << rs[k]) & rm[k];
  return y;
}

// deposit_runs with the shifts packed one per byte (byte k = shift of run
// k).  A 32-bit rotate uses only the low 5 bits of its count, so no byte
// needs masking out; under the run's mask the rotate equals the shift: bits
// that wrap around land below the run (its shift is at most its position),
// and the field's garbage above its kept bits lands outside the run.
template <int R>
__device__ __forceinline__ uint32_t deposit_runs_packed(uint32_t v, const uint32_t* rm, uint32_t shifts) {
  uint32_t y = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) y |= __funnelshift_l(v, v, shifts >> (8 * k)) & rm[k];
  return y;
}

// Inverse of deposit_runs: gather the kept bits of x to the low bits.
template <int R>
__device__ __forceinline__ uint32_t extract_runs(uint32_t x, const uint32_t* rm, const uint32_t* rs) {
  uint32_t v = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) v |= (x & rm[k]) >> rs[k];
  return v;
}

// Five-step parallel-suffix expand (Hacker's Delight, 2nd ed., section 7-5)
// with precomputed move masks mv[0..4] of the kept mask `keep`.
__device__ __forceinline__ uint32_t expand5(uint32_t v, const uint32_t* mv, uint32_t keep) {
#pragma unroll
  for (int i = 4; i >= 0; --i) {
    const uint32_t t = v << (1u << i);
    v = (v & ~mv[i]) | (t & mv[i]);
  }
  return v & keep;
}

// Five-step parallel-suffix compress (Hacker's Delight, section 7-4).
__device__ __forceinline__ uint32_t compress5(uint32_t x, const uint32_t* mv, uint32_t keep) {
  x &= keep;
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const uint32_t t = x & mv[i];
    x = (x ^ t) | (t >> (1u << i));
  }
  return x;
}

}  // namespace ibp
