/*
 * Seeded, counter-based normal generator for synthetic MoE layer inputs.
 *
 * This file holds no arithmetic of the MoE method itself. It only draws
 * numbers. Both the CPU oracle tests and the CUDA path tests feed from it, so
 * that the two sides see bit-identical inputs.
 *
 * Definition (own construction from two published building blocks):
 *   fmix(z)   : the SplitMix64 output function (Steele, Lea and Flood,
 *               "Fast splittable pseudorandom number generators", OOPSLA 2014):
 *               z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31.
 *   h(v)      = fmix(v + GAMMA), GAMMA = 0x9E3779B97F4A7C15.
 *   stream    = h(h(h(h(seed) ^ tensor_id) ^ row) ^ attempt)
 *   draw(n)   = h(stream + (n + 1) * GAMMA)            (n = 0, 1, 2, ...)
 *   uniform   = ((draw >> 11) + 0.5) * 2^-53           (open interval (0,1))
 *   pair p of a row uses u1 = uniform(draw(2p)), u2 = uniform(draw(2p+1))
 *   Box-Muller (1958): r = sqrt(-2 ln u1), a = 2 pi u2,
 *               column 2p   -> r cos a,   column 2p+1 -> r sin a.
 *   value     = std * z, evaluated in double, rounded to float (round to
 *               nearest even); for bf16 the float is then rounded to nearest
 *               even on its upper 16 bits.
 *
 * Rows are independent streams, so any row range can be drawn alone (an
 * expert's slice of a weight tensor, or one redrawn token row).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t fmix(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t h64(uint64_t v) { return fmix(v + GAMMA); }

static inline double unif(uint64_t r) {
  return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline uint64_t row_stream(uint64_t seed, uint64_t tensor_id,
                                  uint64_t row, uint64_t attempt) {
  return h64(h64(h64(h64(seed) ^ tensor_id) ^ row) ^ attempt);
}

static inline uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static void draw_row(uint64_t stream, int64_t ncols, double stdv, int as_bf16,
                     float* out_f32, uint16_t* out_bf16) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t p = 0; 2 * p < ncols; ++p) {
    /* draw(2p) and draw(2p+1) */
    double u1 = unif(h64(stream + (uint64_t)(2 * p + 1) * GAMMA));
    double u2 = unif(h64(stream + (uint64_t)(2 * p + 2) * GAMMA));
    double r = sqrt(-2.0 * log(u1));
    double a = two_pi * u2;
    double z[2];
    z[0] = r * cos(a);
    z[1] = r * sin(a);
    for (int q = 0; q < 2; ++q) {
      int64_t c = 2 * p + q;
      if (c >= ncols) break;
      float f = (float)(stdv * z[q]);
      if (as_bf16) {
        uint16_t b = f32_to_bf16_bits(f);
        if (out_bf16) out_bf16[c] = b;
        if (out_f32) out_f32[c] = bf16_bits_to_f32(b);
      } else {
        if (out_f32) out_f32[c] = f;
      }
    }
  }
}

/* Rows [row0, row0+nrows) of a tensor with ncols columns.
 * attempts: optional per-row redraw counter (indexed from row0), NULL = 0.
 * out_f32 (nrows*ncols floats) and/or out_bf16 (nrows*ncols uint16) may be
 * NULL; at least one must be given. Returns 0, or -1 on bad arguments. */
int synth_normal_rows(uint64_t seed, uint64_t tensor_id, int64_t row0,
                      int64_t nrows, int64_t ncols, const int32_t* attempts,
                      double stdv, int as_bf16, float* out_f32,
                      uint16_t* out_bf16) {
  if (nrows < 0 || ncols < 0 || row0 < 0) return -1;
  if (!out_f32 && !out_bf16) return -1;
  if (out_bf16 && !as_bf16) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    uint64_t att = attempts ? (uint64_t)(uint32_t)attempts[r] : 0u;
    uint64_t s = row_stream(seed, tensor_id, (uint64_t)(row0 + r), att);
    draw_row(s, ncols, stdv, as_bf16, out_f32 ? out_f32 + r * ncols : 0,
             out_bf16 ? out_bf16 + r * ncols : 0);
  }
  return 0;
}

/* Exact widening of bf16 bit patterns to float (for building host copies). */
void synth_bf16_to_f32(const uint16_t* in, float* out, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits_to_f32(in[i]);
}

int synth_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
