/*
 * Host filler of the seeded input generator (definition in synth_hash.h).
 * Test and benchmark inputs only; no fused GEMM + epilogue arithmetic here.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "synth_hash.h"

/* sigma -> the fp32 multiplier that turns the centred Irwin-Hall integer into
 * a draw of standard deviation sigma. */
float synth_scale(double sigma) {
  return (float)(sigma / sqrt((8.0 / 3.0) * (65536.0 * 65536.0 - 1.0)));
}

static void store_value(void* out, int dtype, size_t pos, float v) {
  if (dtype == SYNTH_F16)
    ((uint16_t*)out)[pos] = synth_f32_to_f16_bits(v);
  else if (dtype == SYNTH_BF16)
    ((uint16_t*)out)[pos] = synth_f32_to_bf16_bits(v);
  else
    ((float*)out)[pos] = v;
}

/*
 * Fill nrows rows of a logical [*, cols] row-major tensor with N(0, sigma)
 * draws. Row r of the output holds logical row row_ids[r] (or r when row_ids
 * is NULL). dtype: SYNTH_F16 / SYNTH_BF16 (uint16 bits) or SYNTH_F32.
 */
void synth_fill_normal(void* out, int dtype, int64_t cols, const int64_t* row_ids,
                       int64_t nrows, uint64_t seed, uint32_t tensor_id, double sigma) {
  uint64_t key = synth_key(seed, tensor_id);
  float scale = synth_scale(sigma);
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t lr = row_ids ? row_ids[r] : r;
    for (int64_t c = 0; c < cols; ++c) {
      uint64_t e = (uint64_t)lr * (uint64_t)cols + (uint64_t)c;
      float v = (float)synth_irwin_hall8(key, e) * scale;
      store_value(out, dtype, (size_t)r * (size_t)cols + (size_t)c, v);
    }
  }
}

/*
 * Bernoulli(1/2) bit matrix of logical shape [M, N], stored as column words:
 * word (w, j) holds rows 32w..32w+31 of column j, row 32w+b in bit b; bits of
 * rows >= M are 0. Fills nw word-rows (word_rows[i], or i when NULL).
 */
void synth_fill_mask_words(uint32_t* out, int64_t M, int64_t N, const int64_t* word_rows,
                           int64_t nw, uint64_t seed, uint32_t tensor_id) {
  uint64_t key = synth_key(seed, tensor_id);
  for (int64_t r = 0; r < nw; ++r) {
    int64_t w = word_rows ? word_rows[r] : r;
    int64_t valid = M - 32 * w;
    uint32_t keep = valid >= 32 ? 0xFFFFFFFFu : (valid <= 0 ? 0u : ((1u << valid) - 1u));
    for (int64_t j = 0; j < N; ++j) {
      uint64_t h = synth_at(key, (uint64_t)w * (uint64_t)N + (uint64_t)j);
      out[(size_t)r * (size_t)N + (size_t)j] = (uint32_t)h & keep;
    }
  }
}

/* count distinct sample rows in [0, M): t-th draw is h(t) mod M (duplicates kept) */
void synth_sample_rows(int64_t* out, int64_t count, int64_t M, uint64_t seed,
                       uint32_t tensor_id) {
  uint64_t key = synth_key(seed, tensor_id);
  for (int64_t t = 0; t < count; ++t) out[t] = (int64_t)(synth_at(key, (uint64_t)t) % (uint64_t)M);
}

/* raw hash access, for the generator's own tests */
uint64_t synth_hash(uint64_t seed, uint32_t tensor_id, uint64_t index) {
  return synth_at(synth_key(seed, tensor_id), index);
}

int32_t synth_irwin_hall(uint64_t seed, uint32_t tensor_id, uint64_t element) {
  return synth_irwin_hall8(synth_key(seed, tensor_id), element);
}

/* SplitMix64's output mix alone, for the generator's own tests */
uint64_t synth_mix(uint64_t z) { return synth_mix64(z); }
