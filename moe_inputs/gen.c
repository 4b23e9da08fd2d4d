/*
 * Seeded synthetic inputs for the MoE-layer forward: a counter-based normal
 * generator and nothing else.
 *
 * This file holds no arithmetic of the MoE method itself (no projection, no
 * scoring, no selection): it only turns (seed, tensor id, element index) into a
 * standard-normal draw, scales it, and rounds it to bf16.  Both the CUDA path
 * and the fp64 oracle consume the bytes it writes.
 *
 * Generator definition (stated here so that it can be re-implemented
 * anywhere):
 *   splitmix64(z): z += 0x9E3779B97F4A7C15; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
 *                  z = (z ^ z>>27) * 0x94D049BB133111EB; return z ^ z>>31
 *                  (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *                  generators", OOPSLA 2014; constants as published by Vigna).
 *   key(seed, tid)  = splitmix64(seed ^ splitmix64(tid))
 *   U(seed, tid, c) = ((splitmix64(key + c) >> 11) + 0.5) * 2^-53   in (0, 1)
 *   N(seed, tid, i) = sqrt(-2 ln U(2i)) * cos(2 pi U(2i+1))         (Box-Muller)
 *   value           = bf16_rne(fp32_rne(scale * N))
 *
 * Rows of x that were redrawn by the input recipe use the tensor id
 * (TID_X | attempt << 32) for that row, with the same element indices.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static inline uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
    return splitmix64(seed ^ splitmix64(tid));
}

static inline double uniform01(uint64_t key, uint64_t counter) {
    uint64_t r = splitmix64(key + counter);
    return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0); /* 2^-53 */
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = uniform01(key, 2 * i);
    double u2 = uniform01(key, 2 * i + 1);
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

/* Round to fp32 (C conversion, round-to-nearest-even), then to bf16 with
 * round-to-nearest-even on the bit pattern.  Inputs are finite. */
static inline uint16_t to_bf16(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[i] = bf16(scale * N(seed, tid, start + i)), i in [0, n). */
void gen_normal_bf16(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n,
                     double scale, uint16_t *out) {
    const uint64_t key = stream_key(seed, tid);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nn; ++i)
        out[i] = to_bf16(scale * normal_at(key, start + (uint64_t)i));
}

/* out[i] = scale * N(seed, tid, start + i) in fp64 (used by statistics tests). */
void gen_normal_f64(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n,
                    double scale, double *out) {
    const uint64_t key = stream_key(seed, tid);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nn; ++i)
        out[i] = scale * normal_at(key, start + (uint64_t)i);
}

/* x[t, :] for rows t in [row0, row0 + rows): row t is drawn from the stream
 * (tid_x | attempt[t] << 32) at element indices t*D .. t*D + D - 1.
 * attempt may be NULL (all zero).  out holds rows*D values. */
void gen_rows_bf16(uint64_t seed, uint64_t tid_x, int64_t row0, int64_t rows,
                   int64_t D, const int32_t *attempt, double scale, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t t = row0 + r;
        uint64_t a = attempt ? (uint64_t)attempt[t] : 0u;
        uint64_t key = stream_key(seed, tid_x | (a << 32));
        for (int64_t d = 0; d < D; ++d)
            out[r * D + d] = to_bf16(scale * normal_at(key, (uint64_t)(t * D + d)));
    }
}

int gen_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
