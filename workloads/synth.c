/*
 * Seeded, counter-based synthetic input generator.
 *
 * This file is shared test/bench infrastructure: it produces the inputs that
 * both the CUDA library and the fp64 oracle consume.  It contains no step of
 * the Gated DeltaNet method itself -- only random-number generation, the
 * distribution transforms of the workload recipe and the rounding of values
 * to their storage type.
 *
 * Definition (also restated in workloads/gen.py, which pins this file):
 *   mix(z)      = SplitMix64 finaliser (Steele, Lea, Flood 2014):
 *                   z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *                   z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   key(s, id)  = mix(mix(s) ^ (id * 0xD1B54A32D192ED03))
 *   draw(k, i)  = mix(k + (i + 1) * 0x9E3779B97F4A7C15)    (i-th SplitMix64 output)
 *   unif(k, i)  = ((draw(k, i) >> 11) + 0.5) * 2^-53         in (0, 1)
 *   normal(k,i) = Box-Muller on the pair p = i / 2:
 *                   r = sqrt(-2 ln unif(k, 2p)), th = 2 pi unif(k, 2p + 1)
 *                   even i -> r cos th, odd i -> r sin th
 * Element (row t, column c) of a tensor whose rows hold `row_len` values has
 * counter index i = t * row_len + c, so any sub-block can be generated alone.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t syn_mix(uint64_t z) {
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27; z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

uint64_t synth_key(uint64_t seed, uint64_t tensor_id) {
    return syn_mix(syn_mix(seed) ^ (tensor_id * 0xD1B54A32D192ED03ULL));
}

static inline double syn_unif(uint64_t key, uint64_t i) {
    uint64_t x = syn_mix(key + (i + 1) * SYN_GOLDEN);
    return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double syn_normal(uint64_t key, uint64_t i) {
    uint64_t p = i >> 1;
    double u1 = syn_unif(key, 2 * p), u2 = syn_unif(key, 2 * p + 1);
    double r = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925287 * u2;
    return (i & 1) ? r * sin(th) : r * cos(th);
}

/* float -> bf16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t syn_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

enum { SYN_F32 = 0, SYN_BF16 = 1, SYN_F64 = 2 };
enum { SYN_NORMAL = 0, SYN_SIGMOID = 1, SYN_NEG_SOFTPLUS = 2, SYN_UNIFORM = 3 };

static inline double syn_value(uint64_t key, uint64_t i, int kind, double a, double b) {
    if (kind == SYN_UNIFORM) return a + b * syn_unif(key, i);
    double z = a + b * syn_normal(key, i);
    if (kind == SYN_SIGMOID) return 1.0 / (1.0 + exp(-z));
    if (kind == SYN_NEG_SOFTPLUS) return -(z > 30.0 ? z : log1p(exp(z)));
    return z;
}

static inline void syn_store(void *out, int dtype, int64_t j, double x) {
    if (dtype == SYN_F64) ((double *)out)[j] = x;
    else if (dtype == SYN_F32) ((float *)out)[j] = (float)x;
    else ((uint16_t *)out)[j] = syn_f32_to_bf16((float)x);
}

/*
 * Fill out[nrows, ncols] (dense) with elements (row0 + r, col0 + c) of a
 * tensor whose rows hold `row_len` values, drawn as `kind`:
 *   NORMAL:        a + b z
 *   SIGMOID:       1 / (1 + exp(-(a + b z)))
 *   NEG_SOFTPLUS:  -log(1 + exp(a + b z))
 *   UNIFORM:       a + b u
 */
void synth_fill(uint64_t seed, uint64_t tensor_id, int64_t row_len,
                int64_t row0, int64_t nrows, int64_t col0, int64_t ncols,
                int kind, double a, double b, int dtype, void *out) {
    uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        uint64_t base = (uint64_t)(row0 + r) * (uint64_t)row_len + (uint64_t)col0;
        for (int64_t c = 0; c < ncols; ++c)
            syn_store(out, dtype, r * ncols + c, syn_value(key, base + (uint64_t)c, kind, a, b));
    }
}

/*
 * Rows that are uniform on the unit sphere: each group of `group` consecutive
 * values of a row is a standard-normal vector divided by its Euclidean norm
 * (in double), then rounded to `dtype`.  Used for query/key inputs that the
 * workload recipe states as "N(0,1), then normalised per head".
 * out[nrows, ncols]; col0 and ncols must be multiples of `group`.
 */
void synth_fill_sphere(uint64_t seed, uint64_t tensor_id, int64_t row_len,
                       int64_t row0, int64_t nrows, int64_t col0, int64_t ncols,
                       int64_t group, int dtype, void *out) {
    uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        uint64_t base = (uint64_t)(row0 + r) * (uint64_t)row_len + (uint64_t)col0;
        for (int64_t g0 = 0; g0 < ncols; g0 += group) {
            double ss = 0.0;
            for (int64_t c = 0; c < group; ++c) {
                double z = syn_normal(key, base + (uint64_t)(g0 + c));
                ss += z * z;
            }
            double inv = 1.0 / sqrt(ss);
            for (int64_t c = 0; c < group; ++c)
                syn_store(out, dtype, r * ncols + g0 + c,
                          syn_normal(key, base + (uint64_t)(g0 + c)) * inv);
        }
    }
}

/* Raw 64-bit draws, for pinning this file against its Python restatement. */
void synth_draws(uint64_t seed, uint64_t tensor_id, int64_t start, int64_t n, uint64_t *out) {
    uint64_t key = synth_key(seed, tensor_id);
    for (int64_t i = 0; i < n; ++i) out[i] = syn_mix(key + ((uint64_t)(start + i) + 1) * SYN_GOLDEN);
}
