/*
 * Seeded synthetic input generator for the sparse-decode KV offload workloads.
 *
 * This file holds NO arithmetic of the offload method (no scoring, selection,
 * residency or copying rule).  It only turns (seed, kind, request, layer, sub,
 * index) into bf16 numbers, so that the CPU oracle and the CUDA path can be
 * fed bit-identical inputs.  Both sides consume its output; neither shares
 * any other code with the other.
 *
 * Definition (stated so that it can be re-implemented independently):
 *   mix(z)      = SplitMix64 finaliser:
 *                   z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *                   z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   key         = mix(mix(mix(mix(seed ^ (kind << 56)) + r) + l) + sub)
 *   x_j         = mix(key + (j + 1) * 0x9E3779B97F4A7C15)      (counter based)
 *   U(j)        = ((x_j >> 11) + 0.5) * 2^-53                   in (0, 1)
 *   normal pair i (stream values 2i and 2i+1), Box-Muller in fp64:
 *                 rad = sqrt(-2 ln U(2i)),  th = 2*pi*U(2i+1)
 *                 v(2i) = rad cos th,  v(2i+1) = rad sin th
 *   bf16(v)     = fp64 -> fp32 (C cast, round to nearest even), then fp32 ->
 *                 bf16 round to nearest even on the upper 16 bits.
 *
 *   Query walk (one state per (request, layer, sub)), fp64 state:
 *       q_0     = normal stream (QINIT), values 0..D-1
 *       q_{s+1} = a * q_s + sqrt(1 - a^2) * eps_s,
 *                 eps_s = normal stream (QNOISE), values s*D .. s*D+D-1
 *   The query used at step s is bf16(q_s).
 *
 * Deterministic for a given platform and libm; tests always run both sides
 * on the same machine.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t gen_mix(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

uint64_t gen_stream_key(uint64_t seed, int32_t kind, int64_t r, int64_t l, int64_t sub) {
  uint64_t h = gen_mix(seed ^ ((uint64_t)(uint32_t)kind << 56));
  h = gen_mix(h + (uint64_t)r);
  h = gen_mix(h + (uint64_t)l);
  h = gen_mix(h + (uint64_t)sub);
  return h;
}

static inline double gen_uniform(uint64_t key, int64_t j) {
  uint64_t x = gen_mix(key + (uint64_t)(j + 1) * GEN_GAMMA);
  return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Normal value j of a stream, fp64. */
static inline double gen_normal_at(uint64_t key, int64_t j) {
  int64_t i = j >> 1;
  double u1 = gen_uniform(key, 2 * i);
  double u2 = gen_uniform(key, 2 * i + 1);
  double rad = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (j & 1) ? rad * sin(th) : rad * cos(th);
}

uint16_t gen_f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

/* Fill out[0..n) with bf16 values j0..j0+n-1 of stream (seed, kind, r, l, sub). */
void gen_normal_bf16(uint64_t seed, int32_t kind, int64_t r, int64_t l, int64_t sub,
                     int64_t j0, int64_t n, uint16_t* out) {
  uint64_t key = gen_stream_key(seed, kind, r, l, sub);
#pragma omp parallel for schedule(static) if (n > 65536)
  for (int64_t i = 0; i < n; ++i) out[i] = gen_f32_to_bf16((float)gen_normal_at(key, j0 + i));
}

/* Fill out[0..n) with fp64 values j0..j0+n-1 (for distribution tests). */
void gen_normal_f64(uint64_t seed, int32_t kind, int64_t r, int64_t l, int64_t sub,
                    int64_t j0, int64_t n, double* out) {
  uint64_t key = gen_stream_key(seed, kind, r, l, sub);
  for (int64_t i = 0; i < n; ++i) out[i] = gen_normal_at(key, j0 + i);
}

/*
 * Token rows for a block of units: for unit index i in [0, n_units) with
 * (r, l) = (rs[i], ls[i]) and tokens t in [t0, t0 + n_tok), element e in
 * [0, width): value index t*width + e of stream (seed, kind, r, l, 0).
 * out layout: [n_units][n_tok][width], rows of one unit contiguous, unit
 * stride unit_stride elements (>= n_tok*width).
 */
void gen_token_rows_bf16(uint64_t seed, int32_t kind, int32_t n_units, const int64_t* rs,
                         const int64_t* ls, int64_t t0, int64_t n_tok, int32_t width,
                         int64_t unit_stride, uint16_t* out) {
  int64_t total = (int64_t)n_units * n_tok;
#pragma omp parallel for schedule(static) if (total > 64)
  for (int64_t w = 0; w < total; ++w) {
    int64_t i = w / n_tok, t = t0 + w % n_tok;
    uint64_t key = gen_stream_key(seed, kind, rs[i], ls[i], 0);
    uint16_t* dst = out + i * unit_stride + (t - t0) * width;
    for (int32_t e = 0; e < width; ++e)
      dst[e] = gen_f32_to_bf16((float)gen_normal_at(key, t * (int64_t)width + e));
  }
}

/*
 * Random-walk queries for one (request, layer, sub) stream triple.
 * out: [n_steps][dim] bf16, step s holds bf16(q_s).
 */
void gen_query_walk(uint64_t seed, int32_t kind_init, int32_t kind_noise, int64_t r, int64_t l,
                    int64_t sub, double a, int32_t n_steps, int32_t dim, uint16_t* out) {
  uint64_t kinit = gen_stream_key(seed, kind_init, r, l, sub);
  uint64_t knoise = gen_stream_key(seed, kind_noise, r, l, sub);
  double c = sqrt(1.0 - a * a);
  double q[1024];
  if (dim > 1024) return;
  for (int32_t d = 0; d < dim; ++d) q[d] = gen_normal_at(kinit, d);
  for (int32_t s = 0; s < n_steps; ++s) {
    for (int32_t d = 0; d < dim; ++d) out[(int64_t)s * dim + d] = gen_f32_to_bf16((float)q[d]);
    for (int32_t d = 0; d < dim; ++d)
      q[d] = a * q[d] + c * gen_normal_at(knoise, (int64_t)s * dim + d);
  }
}
