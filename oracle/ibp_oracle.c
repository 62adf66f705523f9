/*
 * ibp_oracle.c - plain bit-by-bit C oracle of Invariant Bit Packing (IBP).
 *
 * TEST INFRASTRUCTURE ONLY.  The CUDA library never links, includes or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load it (through oracle/oracle_c.py).  It shares no code, header
 * or table with host_transfer_gb300/csrc.
 *
 * Source: the page "Résumé Technique : Réduire le goulot d'étranglement de la
 * mémoire GPU par la compression sans perte pour le ML" (French summary of
 * "Reducing the GPU Memory Bottleneck with Lossless Compression for ML"),
 * section « Algorithme central » steps 1-3, and section « Intégration au
 * système » (fixed-size in-place buffers, GPU-resident bitmask).
 *
 * Readings of what the pages leave open (the same as oracle/ibp_ref.py):
 *   - one chunk = one 32-bit word, one Mask/Bitval word per word position;
 *   - invariant iff max(#ones, #zeros) >= ceil(T * S_rows) (IEEE double),
 *     Bitval bit = (#ones > #zeros);
 *   - per 32-word segment one 32-bit participation header; all headers first,
 *     then the payload fields, LSB first, no padding;
 *   - a row is stored compressed iff its stream is < W words; tail zeroed;
 *   - a word whose mask is 0 "matches" and keeps its 32 bits.
 *
 * Everything is done one bit at a time on purpose: this is the slow, obvious
 * version.  The only concession to size is an OpenMP loop over independent
 * rows (each row is computed exactly as in the serial code).
 *
 * Parity status: pinned by tests/test_oracle_pins.py (hand rows, brute force
 * against the Python oracle, size identity, round trip, closed forms).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_OK 0
#define REF_EINVAL 1
#define REF_ECORRUPT 4
#define REF_ERANGE 5

static int g_threads = 1;

void ibp_ref_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

int ibp_ref_threads(void) { return g_threads; }

static uint32_t bit_of(uint32_t x, unsigned b) { return (x >> b) & 1u; }

static unsigned count_ones(uint32_t x) {
  unsigned n = 0;
  for (unsigned b = 0; b < 32; ++b) n += bit_of(x, b);
  return n;
}

/* --- step 1: preprocess ---------------------------------------------------- */

int ibp_ref_preprocess(const uint32_t* sample, uint64_t s_rows, uint32_t W,
                       double T, uint32_t* mask, uint32_t* bitval) {
  if (s_rows == 0 || W == 0 || !(T > 0.0 && T <= 1.0)) return REF_EINVAL;
  uint64_t t = (uint64_t)ceil(T * (double)s_rows);
  /* ones[w*32 + b] = number of sampled rows with bit b of word w set; the
   * rows are read once, in order */
  uint64_t* ones = (uint64_t*)calloc((size_t)W * 32, sizeof(uint64_t));
  for (uint64_t r = 0; r < s_rows; ++r)
    for (uint32_t w = 0; w < W; ++w)
      for (unsigned b = 0; b < 32; ++b) ones[w * 32 + b] += bit_of(sample[r * W + w], b);
  for (uint32_t w = 0; w < W; ++w) {
    uint32_t m = 0, v = 0;
    for (unsigned b = 0; b < 32; ++b) {
      uint64_t n1 = ones[w * 32 + b];
      uint64_t n0 = s_rows - n1;
      uint64_t most = n1 > n0 ? n1 : n0;
      if (most >= t) {
        m |= 1u << b;
        if (n1 > n0) v |= 1u << b;
      }
    }
    mask[w] = m;
    bitval[w] = v;
  }
  free(ones);
  return REF_OK;
}

/* --- bit cursor over a word array ----------------------------------------- */

static void put_bit(uint32_t* words, uint64_t k, uint32_t bit) {
  if (bit) words[k / 32] |= 1u << (k % 32);
}

static uint32_t get_bit(const uint32_t* words, uint64_t k) {
  return (words[k / 32] >> (k % 32)) & 1u;
}

/* --- step 2: compress one row ---------------------------------------------- */

/* Writes the stream for row x into `stream` (zeroed, capacity cap_words) and
 * returns its length in bits.  Bits beyond cap_words*32 are counted but not
 * written. */
static uint64_t encode_row(const uint32_t* x, uint32_t W, const uint32_t* mask,
                           const uint32_t* bitval, uint32_t* stream,
                           uint64_t cap_words) {
  uint32_t S = (W + 31) / 32;
  uint64_t cap_bits = cap_words * 32;
  uint64_t pos = (uint64_t)S * 32; /* payload starts after the headers */
  for (uint32_t w = 0; w < W; ++w) {
    uint32_t m = mask[w];
    int match = ((x[w] ^ bitval[w]) & m) == 0;
    if (match) {
      /* participation bit w of the header area */
      if ((uint64_t)w < cap_bits) put_bit(stream, w, 1);
      /* keep only the non-invariant bits, in ascending position */
      for (unsigned b = 0; b < 32; ++b) {
        if (bit_of(m, b)) continue;
        if (pos < cap_bits) put_bit(stream, pos, bit_of(x[w], b));
        pos++;
      }
    } else {
      for (unsigned b = 0; b < 32; ++b) {
        if (pos < cap_bits) put_bit(stream, pos, bit_of(x[w], b));
        pos++;
      }
    }
  }
  return pos;
}

/* Returns 1 if the row is stored compressed; writes the W-word slot. */
static int compress_one(const uint32_t* x, uint32_t W, const uint32_t* mask,
                        const uint32_t* bitval, uint32_t* slot,
                        uint64_t* used_words) {
  uint32_t* tmp = (uint32_t*)calloc(W, sizeof(uint32_t));
  uint64_t bits = encode_row(x, W, mask, bitval, tmp, W);
  uint64_t Lw = (bits + 31) / 32;
  int comp = Lw < W;
  if (comp) {
    for (uint32_t k = 0; k < W; ++k) slot[k] = k < Lw ? tmp[k] : 0u;
    *used_words = Lw;
  } else {
    for (uint32_t k = 0; k < W; ++k) slot[k] = x[k];
    *used_words = W;
  }
  free(tmp);
  return comp;
}

/* Compress n_rows rows (row-major, W words each) into slots (may equal rows).
 * bitmask gets ceil(n_rows/32) words; stored_words (optional) the total
 * number of words a reader has to fetch. */
int ibp_ref_compress(const uint32_t* rows, uint64_t n_rows, uint32_t W,
                     const uint32_t* mask, const uint32_t* bitval,
                     uint32_t* slots, uint32_t* bitmask,
                     uint64_t* stored_words) {
  if (W == 0) return REF_EINVAL;
  uint64_t nbm = (n_rows + 31) / 32;
  for (uint64_t i = 0; i < nbm; ++i) bitmask[i] = 0;
  uint64_t total = 0;
  int64_t n = (int64_t)n_rows;
#pragma omp parallel for num_threads(g_threads) schedule(static) reduction(+ : total)
  for (int64_t r = 0; r < n; ++r) {
    uint32_t* tmp = (uint32_t*)malloc((size_t)W * sizeof(uint32_t));
    uint64_t used = 0;
    int comp = compress_one(rows + (uint64_t)r * W, W, mask, bitval, tmp, &used);
    memcpy(slots + (uint64_t)r * W, tmp, (size_t)W * sizeof(uint32_t));
    free(tmp);
    total += used;
    if (comp) {
#pragma omp atomic
      bitmask[r / 32] |= 1u << (r % 32);
    }
  }
  if (stored_words) *stored_words = total;
  return REF_OK;
}

/* Words a reader fetches for each row (Lw when the row is stored compressed,
 * W when it is stored raw): the per-row sizes of a packed layout. */
int ibp_ref_row_words(const uint32_t* rows, uint64_t n_rows, uint32_t W,
                      const uint32_t* mask, const uint32_t* bitval, uint32_t* words) {
  if (W == 0) return REF_EINVAL;
  int64_t n = (int64_t)n_rows;
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    uint32_t* tmp = (uint32_t*)malloc((size_t)W * sizeof(uint32_t));
    uint64_t used = 0;
    compress_one(rows + (uint64_t)r * W, W, mask, bitval, tmp, &used);
    free(tmp);
    words[r] = (uint32_t)used;
  }
  return REF_OK;
}

/* Compress only the rows listed in ids (each a row of `rows`); slot i and bit
 * i of out_bits describe row ids[i].  Used to check sampled rows of a table
 * too large to run through the bit-by-bit code whole. */
int ibp_ref_compress_some(const uint32_t* rows, uint64_t n_rows, uint32_t W,
                          const uint32_t* mask, const uint32_t* bitval,
                          const int64_t* ids, uint64_t n_ids, uint32_t* slots,
                          uint8_t* out_bits) {
  if (W == 0) return REF_EINVAL;
  for (uint64_t i = 0; i < n_ids; ++i)
    if (ids[i] < 0 || (uint64_t)ids[i] >= n_rows) return REF_ERANGE;
  int64_t n = (int64_t)n_ids;
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t used;
    out_bits[i] = (uint8_t)compress_one(rows + (uint64_t)ids[i] * W, W, mask,
                                        bitval, slots + (uint64_t)i * W, &used);
  }
  return REF_OK;
}

/* --- step 3: decompress ---------------------------------------------------- */

static int decode_one(const uint32_t* slot, int comp, uint32_t W,
                      const uint32_t* mask, const uint32_t* bitval,
                      uint32_t* out) {
  if (!comp) {
    for (uint32_t k = 0; k < W; ++k) out[k] = slot[k];
    return REF_OK;
  }
  uint32_t S = (W + 31) / 32;
  /* header bits past the last word must be clear */
  for (uint64_t k = W; k < (uint64_t)S * 32; ++k) {
    if (get_bit(slot, k)) {
      for (uint32_t j = 0; j < W; ++j) out[j] = 0;
      return REF_ECORRUPT;
    }
  }
  /* length of the stream from the headers */
  uint64_t bits = (uint64_t)S * 32;
  for (uint32_t w = 0; w < W; ++w)
    bits += get_bit(slot, w) ? 32 - count_ones(mask[w]) : 32;
  if ((bits + 31) / 32 >= W) {
    for (uint32_t j = 0; j < W; ++j) out[j] = 0;
    return REF_ECORRUPT;
  }
  uint64_t pos = (uint64_t)S * 32;
  for (uint32_t w = 0; w < W; ++w) {
    uint32_t m = mask[w];
    uint32_t y = 0;
    if (get_bit(slot, w)) {
      for (unsigned b = 0; b < 32; ++b) {
        if (bit_of(m, b)) {
          y |= bit_of(bitval[w], b) << b; /* reinsert the invariant bit */
        } else {
          y |= get_bit(slot, pos) << b;
          pos++;
        }
      }
    } else {
      for (unsigned b = 0; b < 32; ++b) {
        y |= get_bit(slot, pos) << b;
        pos++;
      }
    }
    out[w] = y;
  }
  return REF_OK;
}

/* Decode the rows named by ids into out (n_ids rows of W words).  *status
 * gets the first error met in id order; out-of-range ids and corrupt slots
 * give zero rows. */
int ibp_ref_decompress(const uint32_t* slots, uint64_t n_rows, uint32_t W,
                       const uint32_t* bitmask, const uint32_t* mask,
                       const uint32_t* bitval, const int64_t* ids,
                       uint64_t n_ids, uint32_t* out, int* status) {
  if (W == 0) return REF_EINVAL;
  int64_t n = (int64_t)n_ids;
  int* st = (int*)calloc(n_ids ? n_ids : 1, sizeof(int));
#pragma omp parallel for num_threads(g_threads) schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t r = ids[i];
    uint32_t* o = out + (uint64_t)i * W;
    if (r < 0 || (uint64_t)r >= n_rows) {
      for (uint32_t k = 0; k < W; ++k) o[k] = 0;
      st[i] = REF_ERANGE;
      continue;
    }
    int comp = (bitmask[r / 32] >> (r % 32)) & 1u;
    st[i] = decode_one(slots + (uint64_t)r * W, comp, W, mask, bitval, o);
  }
  int first = REF_OK;
  for (uint64_t i = 0; i < n_ids; ++i)
    if (st[i] != REF_OK) {
      first = st[i];
      break;
    }
  free(st);
  if (status) *status = first;
  return REF_OK;
}

/* Decode slots given one by one (slot i with compressed flag comp[i]), the
 * decoder alone, for checking GPU-written slots of sampled rows. */
int ibp_ref_decode_slots(const uint32_t* slots, const uint8_t* comp,
                         uint64_t n, uint32_t W, const uint32_t* mask,
                         const uint32_t* bitval, uint32_t* out, int* status) {
  if (W == 0) return REF_EINVAL;
  int first = REF_OK;
  for (uint64_t i = 0; i < n; ++i) {
    int s = decode_one(slots + i * W, comp[i], W, mask, bitval, out + i * W);
    if (s != REF_OK && first == REF_OK) first = s;
  }
  if (status) *status = first;
  return REF_OK;
}
