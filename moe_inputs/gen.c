/*
 * Counter-based synthetic input generator (bf16 bit patterns).
 *
 * Holds none of the mixture-of-experts arithmetic: it only turns a stream key
 * and an element counter into a bf16 value drawn from a caller-supplied
 * 65536-entry quantile table.  The same definition is restated in numpy in
 * moe_inputs/__init__.py (used when this library cannot be built) and both are
 * checked against each other by the CPU test suite.
 *
 * Element value at counter c (64-bit) of the stream with key k:
 *     h = mix32(mix32(lo32(c) ^ k) ^ (hi32(c) + 0x632be5ab))
 *     v = table[h >> 16]
 * where mix32 is the 32-bit integer finaliser x ^= x>>16; x *= 0x7feb352d;
 * x ^= x>>15; x *= 0x846ca68b; x ^= x>>16 (a bijection on 32-bit words).
 */
#include <stddef.h>
#include <stdint.h>

static inline uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352dU;
  x ^= x >> 15;
  x *= 0x846ca68bU;
  x ^= x >> 16;
  return x;
}

uint32_t moegen_mix32(uint32_t x) { return mix32(x); }

/* Stream key for (seed, tensor id, a, b); a and b are free sub-stream indices
 * (layer, expert, redraw attempt ...). */
uint32_t moegen_key(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b) {
  uint32_t k = mix32(seed ^ 0x9e3779b9U);
  k = mix32(k ^ tensor);
  k = mix32(k ^ a);
  k = mix32(k ^ b);
  return k;
}

/* out[i] = table[hash(key, start + i) >> 16] for i in [0, count). */
void moegen_fill(uint16_t* out, uint64_t count, uint64_t start, uint32_t key,
                 const uint16_t* table) {
  int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t c = start + (uint64_t)i;
    uint32_t h = mix32(mix32((uint32_t)c ^ key) ^ ((uint32_t)(c >> 32) + 0x632be5abU));
    out[i] = table[h >> 16];
  }
}

/* Fill rows of a [rows, cols] matrix where row r draws from counters
 * [row_index[r] * cols, row_index[r] * cols + cols) of the stream: used to
 * regenerate selected rows (a sample of tokens) without the whole tensor. */
void moegen_fill_rows(uint16_t* out, const int64_t* row_index, int64_t rows,
                      int64_t cols, uint32_t key, const uint16_t* table) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    uint64_t base = (uint64_t)row_index[r] * (uint64_t)cols;
    for (int64_t j = 0; j < cols; ++j) {
      uint64_t c = base + (uint64_t)j;
      uint32_t h = mix32(mix32((uint32_t)c ^ key) ^ ((uint32_t)(c >> 32) + 0x632be5abU));
      out[r * cols + j] = table[h >> 16];
    }
  }
}
