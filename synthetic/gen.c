/*
 * Seeded synthetic inputs for the DiLoCo outer-synchronisation step.
 *
 * This file holds no arithmetic of the method itself: it only fills host
 * buffers with reproducible random numbers. Both the CUDA path (through an
 * upload) and the CPU oracle read the same bits, so parity tests compare the
 * two on identical inputs.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based
 * generator. A stream key k yields the 64-bit word for element i as the
 * (i+1)-th SplitMix64 output of a generator seeded with k, i.e.
 * mix(k + (i+1) * gamma). Any element can therefore be produced on its own,
 * in any order and on any thread, with the same bits.
 *
 * Normal variates: Box-Muller (G. Box, M. Muller, 1958) in double precision
 * from one 64-bit word (top and bottom 32 bits as two uniforms in (0,1)),
 * using the cosine branch only.
 *
 * Student-t with 3 degrees of freedom: Z / sqrt(chi2_3 / 3) with
 * chi2_3 = -2 ln U + Z'^2 (the sum of an exponential of mean 2, which is a
 * chi-square with 2 degrees of freedom, and one squared normal), where Z and
 * Z' are the cosine and sine Box-Muller branches of one word and U comes from
 * a second word.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -ffp-contract=off gen.c -lm
 */
#include <math.h>
#include <stdint.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Word i of the stream with key `key`. */
static inline uint64_t sm_word(uint64_t key, uint64_t i) {
    return sm_mix(key + (i + 1ULL) * SM_GAMMA);
}

/* Uniform in the open interval (0, 1) from 32 bits. */
static inline double u01_from32(uint32_t x) {
    return ((double)x + 0.5) * (1.0 / 4294967296.0);
}

static const double TWO_PI = 6.283185307179586476925286766559;

static inline double normal_from_word(uint64_t w) {
    double u1 = u01_from32((uint32_t)(w >> 32));
    double u2 = u01_from32((uint32_t)(w & 0xFFFFFFFFULL));
    return sqrt(-2.0 * log(u1)) * cos(TWO_PI * u2);
}

static inline double student_t3_from_words(uint64_t w, uint64_t w2) {
    double u1 = u01_from32((uint32_t)(w >> 32));
    double u2 = u01_from32((uint32_t)(w & 0xFFFFFFFFULL));
    double r = sqrt(-2.0 * log(u1));
    double z = r * cos(TWO_PI * u2);
    double z2 = r * sin(TWO_PI * u2);
    double u3 = u01_from32((uint32_t)(w2 >> 32));
    double chi2 = -2.0 * log(u3) + z2 * z2;
    return z / sqrt(chi2 / 3.0);
}

/* Derive a stream key from a seed and up to three integer labels. */
uint64_t synth_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c) {
    uint64_t k = sm_mix(seed + SM_GAMMA);
    k = sm_mix(k ^ (a + 0x632BE59BD9B4E019ULL));
    k = sm_mix(k ^ (b + 0x85157AF5ULL * 0x100000001ULL));
    k = sm_mix(k ^ (c + 0xD6E8FEB86659FD93ULL));
    return k;
}

/* Raw 64-bit words of a stream (used by tests of the generator). */
void synth_words(uint64_t key, int64_t start, int64_t n, uint64_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = sm_word(key, (uint64_t)(start + i));
}

/* Uniform doubles in (0,1): out[i] from word start+i. */
void synth_uniform(uint64_t key, int64_t start, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = u01_from32((uint32_t)(sm_word(key, (uint64_t)(start + i)) >> 32));
}

/* out[i] = (float)(mean + std * Z_{start+i}), Z standard normal. */
void synth_normal_f32(uint64_t key, int64_t start, int64_t n, double mean, double std,
                      float* out) {
#pragma omp parallel for schedule(static) if (n > 65536)
    for (int64_t i = 0; i < n; ++i) {
        double z = normal_from_word(sm_word(key, (uint64_t)(start + i)));
        out[i] = (float)(mean + std * z);
    }
}

/*
 * A learner replica built from the global parameters:
 * out[i] = (float)((double)base[i] - scale * X_{start+i})
 * with X standard normal (dist = 0) or Student-t(3) (dist = 1). Element i of
 * the Student-t stream reads words 2*(start+i) and 2*(start+i)+1.
 */
void synth_replica_f32(uint64_t key, int64_t start, int64_t n, const float* base,
                       double scale, int32_t dist, float* out) {
#pragma omp parallel for schedule(static) if (n > 65536)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t j = (uint64_t)(start + i);
        double x;
        if (dist == 1)
            x = student_t3_from_words(sm_word(key, 2 * j), sm_word(key, 2 * j + 1));
        else
            x = normal_from_word(sm_word(key, j));
        out[i] = (float)((double)base[i] - scale * x);
    }
}
