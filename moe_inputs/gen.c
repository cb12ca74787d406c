/*
 * Seeded synthetic-input generator for the sparse MoE FFN layer workloads.
 *
 * This file holds no arithmetic of the MoE method itself: it only turns
 * (seed, stream, tensor slot, element index) into bytes.  Both the fp64
 * oracle tests and the CUDA parity tests draw their inputs from here.
 *
 * Definition (stateless, counter based):
 *   draw(key, i)   = i-th output of splitmix64 seeded with `key`
 *                  = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 *                    with mix64 the splitmix64 finaliser (Steele, Lea, Flood,
 *                    "Fast splittable pseudorandom number generators", 2014).
 *   Tensor slot j of a stream uses draw indices j * 2^40 + i.
 *   uniform(i)     = ((draw >> 11) + 0.5) * 2^-53            in (0, 1)
 *   normal(i)      = Box-Muller on the pair m = i / 2:
 *                    r = sqrt(-2 ln u(2m)), t = 2*pi*u(2m+1),
 *                    even i -> r cos t, odd i -> r sin t  (then * std)
 *   bf16(v)        = round-to-nearest-even of (float)v to 16 bits.
 *   byte(i)        = byte (i % 8) of draw(i / 8), little-endian order.
 *   int_range(i)   = lo + draw(i) % (hi - lo + 1).
 *
 * Compiled with -ffp-contract=off so that x86-64 and aarch64 hosts give the
 * same bytes (libm differences can still move a value across a bf16 rounding
 * boundary in rare cases; every consumer regenerates on the machine it runs).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL
#define SLOT_SHIFT 40

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * GOLDEN_GAMMA);
}

static inline double uniform01(uint64_t key, uint64_t i) {
  return ((double)(draw(key, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* NaN stays NaN */
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline double normal_at(uint64_t key, uint64_t base, uint64_t i) {
  uint64_t m = i >> 1;
  double u1 = uniform01(key, base + 2 * m);
  double u2 = uniform01(key, base + 2 * m + 1);
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(t) : r * cos(t);
}

/* bf16 tensor of n elements ~ N(0, std^2); element i of slot `slot`. */
void gen_normal_bf16(uint64_t key, uint32_t slot, uint64_t first, uint64_t n,
                     double std, uint16_t* out) {
  uint64_t base = (uint64_t)slot << SLOT_SHIFT;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = f32_to_bf16_rne((float)(std * normal_at(key, base, first + (uint64_t)i)));
}

/* fp64 normal draws (no rounding), for tests that need raw values. */
void gen_normal_f64(uint64_t key, uint32_t slot, uint64_t first, uint64_t n, double* out) {
  uint64_t base = (uint64_t)slot << SLOT_SHIFT;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = normal_at(key, base, first + (uint64_t)i);
}

void gen_uniform_f64(uint64_t key, uint32_t slot, uint64_t first, uint64_t n, double* out) {
  uint64_t base = (uint64_t)slot << SLOT_SHIFT;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = uniform01(key, base + first + (uint64_t)i);
}

/* n uniformly random bytes. */
void gen_bytes(uint64_t key, uint32_t slot, uint64_t n, uint8_t* out) {
  uint64_t base = (uint64_t)slot << SLOT_SHIFT;
  int64_t nw = (int64_t)(n / 8);
#pragma omp parallel for schedule(static)
  for (int64_t w = 0; w < nw; ++w) {
    uint64_t v = draw(key, base + (uint64_t)w);
    for (int b = 0; b < 8; ++b) out[w * 8 + b] = (uint8_t)(v >> (8 * b));
  }
  for (uint64_t i = (uint64_t)nw * 8; i < n; ++i)
    out[i] = (uint8_t)(draw(key, base + i / 8) >> (8 * (i % 8)));
}

/* n integers uniform in [lo, hi], stored as bytes (lo, hi within 0..255). */
void gen_int_range_u8(uint64_t key, uint32_t slot, uint64_t n, uint32_t lo, uint32_t hi,
                      uint8_t* out) {
  uint64_t base = (uint64_t)slot << SLOT_SHIFT;
  uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = (uint8_t)(lo + draw(key, base + (uint64_t)i) % span);
}

uint64_t gen_draw(uint64_t key, uint32_t slot, uint64_t i) {
  return draw(key, ((uint64_t)slot << SLOT_SHIFT) + i);
}
