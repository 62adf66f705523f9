/*
 * ibp.h - C ABI of libibp, a GB300 (sm_103a) implementation of Invariant Bit
 * Packing (IBP): lossless compression of fixed-width tensor rows by dropping
 * the bits that a Mask marks invariant, and warp-parallel decompression of
 * those rows from zero-copy pinned host memory or from HBM.
 *
 * The method is the one of "Reducing the GPU Memory Bottleneck with Lossless
 * Compression for ML", as summarised on the page "Résumé Technique : Réduire
 * le goulot d'étranglement de la mémoire GPU par la compression sans perte
 * pour le ML" (sections « Algorithme central » and « Intégration au
 * système »).  Each entry point below cites the passage it implements.
 *
 * ---------------------------------------------------------------------------
 * Data format (the readings this library takes where the pages are silent)
 * ---------------------------------------------------------------------------
 * A row is W 32-bit words (fp32 values, or bf16/fp16 pairs with element 2j in
 * bits 0-15).  Mask[w] marks the invariant bits of word position w and
 * Bitval[w] their values.  Word w of a row "matches" when
 * ((x ^ Bitval[w]) & Mask[w]) == 0; a matching word keeps its 32 - popcount(
 * Mask[w]) non-invariant bits (in ascending order), any other word keeps all
 * 32.  Per 32-word segment s, header word H_s has bit i set when word 32s+i
 * matched (bits past the last word are 0).  The stream of a row is H_0 ..
 * H_{S-1} (S = ceil(W/32)) followed by the kept fields back to back, least
 * significant bit first (stream bit k is bit k%32 of stream word k/32).  If
 * the stream is Lw < W words, the row's slot holds the stream and zeros after
 * it, and the row's bit in the bitmask is 1; otherwise the slot holds the row
 * unchanged and the bit is 0.  Bit r of the bitmask is bit r%32 of word r/32.
 *
 * ---------------------------------------------------------------------------
 * Conventions
 * ---------------------------------------------------------------------------
 * - Return value: an ibp_status code.  Argument errors are returned before
 *   anything is launched.  Data errors found by a kernel (bad row id,
 *   corrupt slot) are recorded in the plan's device status word and read by
 *   ibp_get_status().
 * - Memory: "device-accessible" means device memory of the plan's GPU, or
 *   page-locked host memory mapped into the device address space (memory from
 *   cudaHostAlloc / cudaMallocHost, or torch pin_memory=True, or memory
 *   registered with cudaHostRegister and cudaHostRegisterMapped).  Pageable
 *   host memory is rejected with IBP_EINVAL.  Kernels read and write mapped
 *   host memory directly (zero copy).
 * - Ownership: the caller owns every buffer passed in.  A plan owns its device
 *   tables and one status word.  No call allocates on the decompress path.
 * - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   Calls other than ibp_plan_create / ibp_plan_destroy / ibp_get_status are
 *   asynchronous with respect to the host and ordered on `stream`.  The
 *   decompress kernels are launched as programmatic dependents: their blocks
 *   may be placed on the GPU while the previous kernel of the stream drains,
 *   but they read and write no per-call data (ids, slots, bitmask, outputs,
 *   status) before that kernel has completed, so stream order holds.  (With
 *   IBP_HINT_EARLY_FETCH set on the plan, the caller states that the previous
 *   kernel wrote none of the inputs, and the reads may start earlier; see
 *   ibp_plan_set_hints.)
 * - Alignment: slots, rows and outputs whose base is 16-byte aligned and whose
 *   W is a multiple of 4 take the 16-byte vector path; anything else takes a
 *   4-byte path with identical results.
 * - Limits: 1 <= W <= IBP_MAX_W words.
 */
#ifndef IBP_H_
#define IBP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 3: ibp_plan_info.short_rows, ibp_get_status_async, IBP_HINT_EARLY_FETCH */
#define IBP_VERSION 3
#define IBP_MAX_W 8192u
#define IBP_NOALLOC_MAX_W 4096u

/* Hints for ibp_plan_set_hints (bit flags). */
#define IBP_HINT_ROW_REUSE 1u   /* calls request the same rows repeatedly (skewed ids) */
#define IBP_HINT_EARLY_FETCH 2u /* a call's inputs are not written by the kernel just before it */

typedef enum ibp_status {
  IBP_OK = 0,       /* success */
  IBP_EINVAL = 1,   /* invalid argument (size, pointer kind, T, ...) */
  IBP_ECUDA = 2,    /* a CUDA runtime call failed; see ibp_last_error_detail() */
  IBP_ENOMEM = 3,   /* a device allocation failed */
  IBP_ECORRUPT = 4, /* a compressed slot announced an impossible stream */
  IBP_ERANGE = 5,   /* a row id was outside [0, n_rows) */
  IBP_ETIMEOUT = 6  /* a bounded wait expired */
} ibp_status;

/* Opaque per-device plan: Mask, Bitval and the derived decode tables. */
typedef struct ibp_plan ibp_plan;
typedef struct ibp_plan_set ibp_plan_set;

typedef struct ibp_plan_info {
  uint32_t W;              /* words per row */
  uint32_t segments;       /* ceil(W / 32): header words per compressed row */
  uint32_t uniform;        /* 1 when every word position has the same Mask and Bitval */
  uint32_t max_runs;       /* most runs of kept (non-invariant) bits in one word */
  uint32_t min_kept_bits;  /* fewest kept bits of any word position */
  uint32_t max_kept_bits;  /* most kept bits of any word position */
  uint64_t metadata_bytes; /* device bytes of the plan's tables (Mask + Bitval + derived) */
  int device;              /* CUDA device of the plan */
  uint32_t prefix_words;   /* words a decompress call fetches from every slot before
                              reading the row's headers (slot layout, aligned buffers) */
  uint32_t short_rows;     /* 1 when ibp_plan_tune_prefix found at least 99 % of the
                              sampled rows storing at most W / 4 words: decodes of
                              per-word-table plans from device memory then stage W / 4
                              words per row and read longer rows from their slots */
} ibp_plan_info;

/* Human-readable name of a status code.  Never NULL. */
const char* ibp_strerror(int status);

/* IBP_VERSION of the loaded library. */
int ibp_version(void);

/* Text of the last CUDA error seen by a library call on this thread ("" if
 * none).  Valid until the next library call on this thread. */
const char* ibp_last_error_detail(void);

/*
 * Preprocess - « Algorithme central », step 1 (Prétraitement): analyse a batch
 * of rows and find the bit positions that hold the same value in at least a
 * fraction T of them; emit a fixed-size Mask (which positions) and Bitval
 * (their values).
 *
 * sample  device-accessible, s_rows x W words, row-major.
 * s_rows  number of sampled rows, 1 <= s_rows < 2^32.
 * W       words per row, 1 <= W <= IBP_MAX_W.
 * T       fraction in (0, 1].  With t = ceil(T * s_rows) evaluated in IEEE
 *         double, bit b of word w is invariant when max(#ones, #zeros) >= t
 *         over the sample; its Bitval bit is 1 when #ones > #zeros (a tie
 *         gives 0).  Bitval is 0 outside the Mask.
 * mask, bitval  device-accessible outputs of W words each.
 * stream  CUDA stream; the results are ready when the stream reaches them.
 *
 * Uses 128 * W bytes of device scratch, allocated and freed in stream order
 * (cudaMallocAsync / cudaFreeAsync).  Errors: IBP_EINVAL (sizes, T, pointer
 * kinds), IBP_ENOMEM, IBP_ECUDA.
 */
int ibp_preprocess(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T,
                   uint32_t* mask, uint32_t* bitval, void* stream);

/*
 * Preprocess that allocates nothing.  The paper has no counterpart: this
 * entry point exists for callers that cannot let a library allocate device
 * memory - a process whose device memory is wholly owned by its own allocator
 * (a framework's caching allocator, an arena reserved at start-up), or a
 * device or driver without stream-ordered memory pools
 * (cudaDevAttrMemoryPoolsSupported = 0), where the cudaMallocAsync scratch of
 * ibp_preprocess is not an option.
 *
 * Same arguments, results and errors as ibp_preprocess, on the current
 * device.  The per-bit counters live instead in a fixed array of
 * IBP_NOALLOC_MAX_W * 32 words (512 KiB) that the library places in the
 * memory of every GPU it is loaded on, held until the process exits.  No
 * cudaMalloc, cudaFree or other allocating call is made.
 *
 * - W must be at most IBP_NOALLOC_MAX_W; a larger W returns IBP_EINVAL before
 *   anything runs, and ibp_last_error_detail() then names the limit.
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.  The address is kept with the id of the device's context: after
 *   cudaDeviceReset, or any other new context on the device, the module is
 *   loaded again and the next call looks the address up again (that call,
 *   too, belongs before any capture).
 * - Every call on a device shares the one array, and each call clears the part
 *   it uses on `stream` before counting: calls that overlap on the GPU (on
 *   different streams, without ordering between them) race and give wrong
 *   Masks.  Order such calls on one stream or with events.
 */
int ibp_preprocess_noalloc(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T,
                           uint32_t* mask, uint32_t* bitval, void* stream);

/*
 * Plan - « Algorithme central », step 1, last point: the Mask/Bitval metadata
 * is kept in GPU memory (a few kilobytes) and reused for the whole dataset.
 * Copies Mask and Bitval to `device` and derives the per-word decode tables
 * there (kept-bit counts, runs of kept bits, shift tables).
 *
 * mask, bitval  W words each, in any memory (pageable host, pinned host or
 *               device); read once during the call.  Bitval bits outside the
 *               Mask are ignored.
 * device        CUDA device ordinal that will run the plan's kernels.
 * out           receives the new plan; unchanged on error.
 *
 * Synchronous.  Errors: IBP_EINVAL, IBP_ENOMEM, IBP_ECUDA.
 */
int ibp_plan_create(const uint32_t* mask, const uint32_t* bitval, uint32_t W, int device,
                    ibp_plan** out);

/* Frees the plan's device memory (synchronises its device).  NULL is ignored. */
int ibp_plan_destroy(ibp_plan* plan);

/* Fills *out with the plan's shape and table statistics. */
int ibp_plan_get_info(const ibp_plan* plan, ibp_plan_info* out);

/*
 * Access hints for the decompress calls made with this plan (a bit set of
 * IBP_HINT_*; 0 restores the default).  IBP_HINT_ROW_REUSE changes speed,
 * never results; IBP_HINT_EARLY_FETCH states a property of the caller's
 * stream, and results are unchanged whenever that property holds.
 *
 * IBP_HINT_ROW_REUSE: the row ids of a call repeat a lot (skewed lookups such
 * as Zipf-distributed embedding ids).  Row copies then also allocate in the
 * SM's L1, so a repeat is served on chip instead of being fetched again over
 * the host link (mapped host memory is not kept in L2).  For ids without
 * repeats it costs a few percent, so it is off by default.
 *
 * IBP_HINT_EARLY_FETCH: the ids (and packed or bag offsets), bitmask and slots
 * that a decompress call reads are not written by the kernel
 * launched just before it on the same stream (they were written by the host,
 * by a copy, or by an earlier kernel).  The decoder is launched as a
 * programmatic dependent of that kernel, so its blocks can be placed on the
 * GPU while that kernel drains; with this hint they already fetch their first
 * ids and row prefixes there, instead of waiting for the kernel to complete,
 * which hides a launch's start-up latency behind the previous launch's tail.
 * Every write (output rows, status word) still waits for that kernel to
 * complete, so a kernel that reads the previous call's output is unaffected.
 * This library's decompress and status-read kernels let the kernel after them
 * start early in the same way, so when the kernel just before is one of them,
 * the inputs must not be written by the kernels before it either, back to
 * the first kernel that is not one of them (e.g. decompress, status read,
 * decompress: the second decompress must not read what the first one
 * writes).  If those kernels do write the call's inputs, the call may read
 * stale values: leave the hint off then (a copy or an event between them is
 * not a kernel and keeps full ordering).  Used by ibp_gather_decompress,
 * ibp_decompress_contig, ibp_gather_decompress_packed,
 * ibp_gather_decompress_bag and ibp_decompress_contig_set (each plan's hints
 * as the set copied them).
 *
 * Takes effect for calls issued after it returns; not synchronised with
 * calls in flight.  Errors: IBP_EINVAL (NULL plan, unknown bits).
 */
int ibp_plan_set_hints(ibp_plan* plan, uint32_t hints);

/*
 * Prefix length.  A decompress call first fetches the leading words of every
 * requested slot, reads the row's participation headers there (« Algorithme
 * central », step 3: the headers say how long the row's stream is), and then
 * fetches whatever of the stream is left.  By default the prefix is the
 * shortest stream the plan allows (Mask popcounts over every word position),
 * so nothing is ever over-read; when the table's rows are longer than that -
 * a Mask with few invariant bits in some positions, rows of mixed length - most
 * rows need the second, dependent fetch, which over the host link costs a
 * round trip and a partly re-read sector.
 *
 * ibp_plan_tune_prefix reads the headers of min(n_rows, max_sample) evenly
 * spaced rows of a compressed table (row i * n_rows / n_sample; max_sample 0 =
 * 65536), takes their stored lengths in 16-byte chunks (W for raw rows) and
 * sets the prefix P (in chunks, from the default up to W) that minimises
 * sum over sampled rows of (c > P ? c + 8 : P), c the row's chunks: words
 * fetched plus a penalty of 8 chunks for each second fetch.  The prefix in
 * words is written to *prefix_words when that is not NULL.  From the same
 * sample it records whether at least 99 % of the rows store at most W / 4
 * words (ibp_plan_info.short_rows): then decodes of per-word-table plans with
 * rows of 256 or 512 words (at most two runs of kept bits per word and two
 * kept-bit counts) from device memory stage W / 4 words per row, so
 * more warps fit on an SM, and read the few longer rows from their slots
 * (when the prefix is at most W / 4 words).  slots and bitmask
 * are as for ibp_gather_decompress (host-mapped or device memory).
 * Synchronises `stream`.  Errors: IBP_EINVAL, IBP_ENOMEM, IBP_ECUDA.
 *
 * ibp_plan_set_prefix sets it directly in words (0 restores the default; a
 * value below the default counts as the default; capped at W).
 *
 * Both change speed, never results, and take effect for calls issued after
 * they return.  They apply to the slot layout; the packed layout always uses
 * the default, since a packed row may end before a longer prefix.  Neither
 * has a counterpart in the paper: its decoder (« Algorithme central », step 3)
 * has a warp read a row's contiguous compressed segment, without saying how
 * the warp learns the segment's length before reading it.
 */
int ibp_plan_tune_prefix(ibp_plan* plan, const uint32_t* slots, uint64_t n_rows, const uint32_t* bitmask,
                         uint64_t max_sample, uint32_t* prefix_words, void* stream);
int ibp_plan_set_prefix(ibp_plan* plan, uint32_t words);

/* The plan's Mask and Bitval (W words each) copied to host memory `mask` and
 * `bitval` (either may be NULL).  Synchronous. */
int ibp_plan_get_mask(const ibp_plan* plan, uint32_t* mask, uint32_t* bitval);

/*
 * Compress - « Algorithme central », step 2 (Compression), run on the GPU over
 * zero-copy memory, and « Intégration au système » (fixed-size in-place
 * buffers, a GPU-resident bitmask of the compressed tensors).  One warp per
 * row: match test per word, removal of the invariant bits, participation
 * headers by warp ballot, bit offsets by warp scan, row kept raw when the
 * stream would not be shorter than the row.
 *
 * rows          device-accessible input, n_rows x W words.
 * slots         device-accessible output, n_rows x W words.  May be the same
 *               pointer as rows (in-place); must not overlap it otherwise.
 * n_rows        rows to compress (0 is a no-op).
 * bitmask       device-accessible output of ceil(n_rows / 32) words, fully
 *               written (bits past n_rows are 0).
 * stored_words  optional device-accessible uint64: the number of words a
 *               reader fetches for these rows (Lw per compressed row, W per raw
 *               row) is ADDED to it.  NULL to skip.
 *
 * Asynchronous on `stream`.  Errors: IBP_EINVAL, IBP_ECUDA.
 */
int ibp_compress(const ibp_plan* plan, const uint32_t* rows, uint32_t* slots, uint64_t n_rows,
                 uint32_t* bitmask, uint64_t* stored_words, void* stream);

/*
 * Gather-decompress - « Algorithme central », step 3 (Décompression): a warp
 * reads a row's compressed segment from CPU (or GPU) memory into a shared-
 * memory workspace, computes each lane's starting bit offset with warp
 * primitives, rebuilds its words by reinserting the Bitval bits at the Mask
 * positions, and overlaps the fetch of the next rows with the decoding of the
 * current ones.  Only the compressed prefix of a slot is read.
 *
 * slots    device-accessible, the whole table: n_rows x W words (the output
 *          of ibp_compress, or the same format from any writer).
 * n_rows   rows in the table; ids must lie in [0, n_rows).
 * bitmask  device-accessible, ceil(n_rows / 32) words.
 * row_ids  device-accessible, n_ids int64 row ids (repeats allowed).
 * out      device-accessible, n_ids x W words: out row i = row row_ids[i].
 *
 * An id outside [0, n_rows) records IBP_ERANGE and gives a zero row; a
 * compressed slot whose headers announce a stream of W words or more, or set
 * a header bit past the last word, records IBP_ECORRUPT and gives a zero row.
 * Asynchronous on `stream`; no allocation.  Errors: IBP_EINVAL, IBP_ECUDA.
 */
int ibp_gather_decompress(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                          const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                          uint32_t* out, void* stream);

/*
 * Contiguous decompress - step 3 for the rows first_row .. first_row + n - 1
 * of the table (e.g. one offloaded weight matrix or KV block), written to a
 * dense n x W output.  Arguments as for ibp_gather_decompress; first_row + n
 * must not exceed n_rows (IBP_EINVAL).
 */
int ibp_decompress_contig(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                          const uint32_t* bitmask, uint64_t first_row, uint64_t n,
                          uint32_t* out, void* stream);

/*
 * Packed cache layout - « Intégration au système », cache compression:
 * compressing the tensors held in a GPU software cache raises the cache's
 * effective capacity.  Fixed-size slots save no space, so a cache keeps each
 * row's stored words only (Lw for a compressed row, W for a raw one), rounded
 * up to 4 words so that rows start on 16-byte boundaries, back to back.
 * offsets[r] is the word where row r starts and offsets[n_rows] the total
 * number of words.  Requires W % 4 == 0.
 *
 * ibp_packed_offsets: fills offsets (device-accessible, n_rows + 1 uint64)
 *   from the rows' headers in `slots` (as for ibp_gather_decompress).  Uses
 *   8 bytes per 4096 rows of scratch from cudaMallocAsync, freed in stream
 *   order.  Errors: IBP_EINVAL, IBP_ENOMEM, IBP_ECUDA.
 * ibp_pack: copies each row's stored words from `slots` (device-accessible,
 *   e.g. pinned host memory: filling an HBM cache) to `packed`
 *   (device-accessible, offsets[n_rows] words, 16-byte aligned) at
 *   offsets[r].  `offsets` must come from ibp_packed_offsets for these slots.
 * ibp_gather_decompress_packed: ibp_gather_decompress reading the packed
 *   layout.  A row whose headers announce more words than its packed extent,
 *   or a raw row whose extent is not W, records IBP_ECORRUPT and gives a zero
 *   row.  Needs the specialised decoder's plan shape (W = 32 * 2^k <= 2048,
 *   at most four runs of kept bits per word, W <= 1024 for per-word Masks,
 *   16-byte aligned packed buffer and output, fewer than 2^31 rows);
 *   IBP_EINVAL otherwise.
 * All three are asynchronous on `stream`.
 */
int ibp_packed_offsets(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                       const uint32_t* bitmask, uint64_t* offsets, void* stream);
int ibp_pack(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows, const uint64_t* offsets,
             uint32_t* packed, void* stream);
int ibp_gather_decompress_packed(const ibp_plan* plan, const uint32_t* packed,
                                 const uint64_t* offsets, uint64_t n_rows,
                                 const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                                 uint32_t* out, void* stream);

/*
 * Gather-decompress fused with pooling (an "embedding bag").  « Résultats »:
 * IBP's rows feed DLRM embedding tables and GNN feature aggregation, whose
 * consumer pools the rows of each bag; « Algorithme central », step 3: the
 * fetch overlaps the logic that consumes the data.  Here the decoded rows are
 * added in registers and never written out: only one pooled row per bag is.
 *
 * Rows are W float32 values (the decoded words read as IEEE single).  Bag b
 * holds the id positions k in [bag_offsets[b], bag_offsets[b+1]).
 * IBP_BAG_SUM: out[b] = row(row_ids[k0]) + row(row_ids[k0+1]) + ..., added in
 * IEEE single precision in increasing k from +0.0 (no reassociation, no fused
 * multiply-add): bit-identical to gather-decompress followed by that loop.
 * IBP_BAG_MEAN: that sum divided by the bag size (one correctly rounded
 * division); an empty bag gives zeros in both modes.
 * IBP_BAG_BF16 (or-ed into mode): the rows hold 2W bfloat16 values, word j
 * holding element 2j in bits 0-15 and 2j+1 in bits 16-31; each is widened
 * exactly to float and pooled as above, and out holds 2W floats per bag.
 *
 * slots, bitmask, n_rows  as for ibp_gather_decompress; W = 32 * 2^k <= 512,
 *                 at most 4 runs of kept bits per word, slots 16-byte aligned,
 *                 n_rows < 2^31 (IBP_EINVAL otherwise).
 * row_ids     device-accessible int64[n_ids] (may be NULL when n_ids == 0).
 * bag_offsets device-accessible int64[n_bags + 1].  A bag whose offsets are
 *             not 0 <= bag_offsets[b] <= bag_offsets[b+1] <= n_ids gives zeros
 *             and records IBP_ERANGE.
 * out         device-accessible float[n_bags * W] (n_bags * 2W with IBP_BAG_BF16;
 *             8-byte aligned then).
 * Data errors as in ibp_gather_decompress: a bad id or a corrupt slot adds a
 * zero row (it still counts in the bag's size) and records IBP_ERANGE /
 * IBP_ECORRUPT.  Asynchronous on `stream`.  Errors: IBP_EINVAL, IBP_ECUDA.
 */
#define IBP_BAG_SUM 0u
#define IBP_BAG_MEAN 1u
#define IBP_BAG_BF16 2u
int ibp_gather_decompress_bag(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                              const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                              const int64_t* bag_offsets, uint64_t n_bags, uint32_t mode, float* out,
                              void* stream);

/*
 * Plan sets - finer Mask granularity.  « Résultats » reports its savings per
 * tensor (one Mask/Bitval per tensor); an attention KV cache mixes heads whose
 * values have different scales, so one Mask for the whole tensor finds almost
 * no invariant bits.  A plan set gives each block of consecutive rows its own
 * plan (for a KV cache laid out [head][position][dim]: one plan per head) and
 * decodes all the blocks in one launch.
 *
 * ibp_plan_set_create: plans[0 .. n_plans) (1 <= n_plans <= 65535), all on
 * one device with the same W, W = 32 * S with S in {1, 2, 4, 8, 16, 32}, each
 * with at most 4 runs of kept bits per word.  The set copies the plans' device
 * views (table addresses, status word, hints) once: the plans must outlive
 * the set, and hints or prefixes set later are not seen by it.  Synchronous.  Errors:
 * IBP_EINVAL, IBP_ENOMEM, IBP_ECUDA.  ibp_plan_set_destroy frees it (NULL is
 * ignored).
 *
 * ibp_decompress_contig_set: the table is n_plans * rows_per_plan slots of W
 * words; row k * rows_per_plan + i was compressed with plans[k] and is decoded
 * with it into out row k * rows_per_plan + i.  bitmask covers all the rows
 * (bit r of word r / 32): when rows_per_plan is a multiple of 32, compressing
 * block k with plans[k] into bitmask + k * rows_per_plan / 32 builds it.
 * slots (host-mapped or device memory) and out (n_plans * rows_per_plan * W
 * words, device-accessible) must be 16-byte aligned; n_plans * rows_per_plan
 * < 2^31.  Each row is fetched with its plan's prefix as it was when the set
 * was created (tune the plans' prefixes first).
 * Data errors are recorded in the status word of the row's plan.
 * Asynchronous on `stream`.  Errors: IBP_EINVAL, IBP_ECUDA.
 *
 * ibp_plan_set_get_status: ibp_get_status of every plan of the set (each is
 * cleared); returns the first error found (IBP_OK if none).
 */
int ibp_plan_set_create(const ibp_plan* const* plans, uint32_t n_plans, ibp_plan_set** out);
int ibp_plan_set_destroy(ibp_plan_set* set);
int ibp_decompress_contig_set(const ibp_plan_set* set, const uint32_t* slots, uint64_t rows_per_plan,
                              const uint32_t* bitmask, uint32_t* out, void* stream);
int ibp_plan_set_get_status(const ibp_plan_set* set, void* stream);

/*
 * Synchronises `stream`, returns the first data error recorded by the plan's
 * kernels since the last call (IBP_OK if none) and clears it.  The status
 * word is shared by every call made with this plan, on any stream.  Calls on
 * one plan from several host threads are serialised inside the library.
 */
int ibp_get_status(const ibp_plan* plan, void* stream);

/*
 * Status read that does not wait: enqueues on `stream` one small kernel that
 * moves the plan's status word into *status_out and clears it (one atomic
 * exchange), and returns at once.  Once the stream has passed that kernel,
 * *status_out holds the first data error recorded by the plan's kernels
 * ordered before it (IBP_OK if none); read it after synchronising with the
 * stream (an event, cudaStreamSynchronize).  A caller can so check the result
 * of every decompress call without stopping the GPU between calls, e.g. one
 * word of a pinned ring per call, checked a few calls later.  The kernel is
 * launched as a programmatic dependent of the previous kernel of `stream` and
 * lets the next one launch at once, so a status read between two decompress
 * calls on one stream keeps their overlap (IBP_HINT_EARLY_FETCH): no event or
 * side stream is needed to keep the decodes back to back.
 *
 * status_out  device-accessible uint32 (mapped pinned host memory, or device
 *             memory), owned by the caller; written by the kernel.
 * Errors: IBP_EINVAL (NULL plan or word, word not device-accessible),
 * IBP_ECUDA.
 */
int ibp_get_status_async(const ibp_plan* plan, uint32_t* status_out, void* stream);

/*
 * Fetched length per row - « Intégration au système »: a fixed-size buffer of
 * which only the compressed part is read.  lengths[i] = words a reader
 * fetches for row row_ids[i]: Lw (the stream length announced by the row's
 * headers) for a compressed row, W for a raw row, 0 for an id outside
 * [0, n_rows) (which also records IBP_ERANGE).  A compressed row whose headers
 * announce W words or more reports W.
 *
 * slots, bitmask, row_ids  as for ibp_gather_decompress.
 * lengths  device-accessible output, n_ids uint32.
 * Asynchronous on `stream`.  Errors: IBP_EINVAL, IBP_ECUDA.
 */
int ibp_row_lengths(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                    const uint32_t* bitmask, const int64_t* row_ids, uint64_t n_ids,
                    uint32_t* lengths, void* stream);

/*
 * Uncompressed gather (measurement baseline): out row i = rows row
 * row_ids[i], the ideal uncompressed transfer of the same rows that
 * ibp_gather_decompress rebuilds (« Résultats », overhead against the ideal
 * uncompressed transfer rate).  Ids outside [0, n_rows) give zero rows.
 * Arguments as for ibp_gather_decompress.  Asynchronous on `stream`.
 */
int ibp_gather_raw(const uint32_t* rows, uint64_t n_rows, uint32_t W, const int64_t* row_ids,
                   uint64_t n_ids, uint32_t* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* IBP_H_ */
