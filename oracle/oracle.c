/*
 * CPU oracle of the DiLoCo outer synchronisation step (test infrastructure).
 *
 * This is the plain, slow, obviously-correct statement of what the CUDA path
 * computes. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the product path never does, and it shares no code with
 * the CUDA library. Floating point is fp64 except where the method itself
 * fixes fp32 (pseudo-gradients, codebook values, the fp32 accumulation and
 * the fp32 outer update). Build with -ffp-contract=off so that no a*b+c is
 * silently fused: every fused multiply-add below is an explicit fmaf().
 *
 * Sources (web pages on the method):
 *  [INTELLECT-1 notes] "INTELLECT-1: Training a 10B Model Across 3 Continents",
 *      section 3.2 (worked example: pseudo-gradient, per-tensor mu/sigma,
 *      +-6 sigma range, 256 buckets, mean over 3 workers accumulated in fp32,
 *      Nesterov outer step with lr 0.7 and momentum 0.9), section 4.1
 *      (uniform quantisation with clipping, steps 1-4: per-tensor mu and
 *      sigma, clip to [mu-6sigma, mu+6sigma], 256 uniform buckets, codebook
 *      value = mean of the data in each bucket), section 4.2 (dequantise to
 *      fp32 and accumulate there; never add in code space).
 *  [Decoupled DiLoCo note] "Decoupled DiLoCo: Resilient, Distributed AI
 *      Training at Scale", architecture item 4 (P=24 fragments; tensors
 *      packed into balanced fragments in the manner of greedy bin-packing;
 *      minimum quorum) and fault-tolerance items 1 and 3 (merge once at least
 *      K learners reported; token-weighted merge).
 *
 * Readings where the pages are silent (the same choices are stated in the
 * design notes):
 *  - Delta_k = fl32(theta_g - theta_k), start point minus learner (sec. 3.2
 *    step 4 defines Delta as start-of-round weights minus current weights).
 *  - sigma is the population standard deviation, two-pass in fp64.
 *  - bucket b = clamp(floor(((double)d - lo) * s), 0, 255), s = 256/(hi-lo)
 *    in fp64; a value on an interior edge goes to the upper bucket.
 *  - the bucket mean is taken over clipped values clamp(d, lo, hi).
 *  - an empty bucket's codebook value is its midpoint lo + (b + 1/2) w.
 *  - degenerate range (hi - lo < 256 * FLT_MIN, which includes sigma = 0):
 *    every code is 0 and every codebook value is (float)mu.
 *  - a segment with any non-finite Delta is invalid: mu, sigma, lo, hi are
 *    NaN, every code is 0 and every codebook value is NaN.
 *  - merge weights are normalised over the present learners in fp64 and
 *    rounded to fp32; the weighted mean is accumulated as
 *    acc = fmaf(w_k, value_k, acc) over present k in increasing order.
 *  - outer Nesterov: m' = fmaf(mu, m, D); g = fmaf(mu, m', D);
 *    theta' = fmaf(-lr, g, theta).
 *  - planner: longest-processing-time greedy; tensors sorted by size
 *    descending (index ascending on ties), each placed on the least-loaded
 *    fragment (lowest index on ties).
 *
 * Pins: every function is checked by the tests against what the pages and
 * the mathematics fix, except oracle_rda_merge_outer_step, which is PARITY
 * UNPINNED (the page names Radial-Directional Averaging without a formula;
 * its tests check only the defining properties of the reading taken).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    OR_OK = 0,
    OR_ERR_ARG = -1,
    OR_ERR_QUORUM = -3,
};

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the later parallel loops (n >= 1); timing only, no effect on
 * any result (every parallel loop writes disjoint outputs). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Fragment planner (Decoupled DiLoCo note, architecture item 4).           */

typedef struct {
    int64_t numel;
    int32_t index;
} or_item;

static int cmp_items(const void* a, const void* b) {
    const or_item* x = (const or_item*)a;
    const or_item* y = (const or_item*)b;
    if (x->numel != y->numel) return x->numel > y->numel ? -1 : 1;
    return x->index < y->index ? -1 : (x->index > y->index);
}

int oracle_plan_fragments(const int64_t* numel, int32_t n_tensors, int32_t n_frags,
                          int32_t* frag_of_tensor, int64_t* frag_load) {
    if (n_tensors < 0 || n_frags <= 0) return OR_ERR_ARG;
    for (int32_t t = 0; t < n_tensors; ++t)
        if (numel[t] < 0) return OR_ERR_ARG;
    or_item* items = (or_item*)malloc(sizeof(or_item) * (size_t)(n_tensors > 0 ? n_tensors : 1));
    for (int32_t t = 0; t < n_tensors; ++t) {
        items[t].numel = numel[t];
        items[t].index = t;
    }
    qsort(items, (size_t)n_tensors, sizeof(or_item), cmp_items);
    for (int32_t p = 0; p < n_frags; ++p) frag_load[p] = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        int32_t best = 0;
        for (int32_t p = 1; p < n_frags; ++p)
            if (frag_load[p] < frag_load[best]) best = p;
        frag_of_tensor[items[i].index] = best;
        frag_load[best] += items[i].numel;
    }
    free(items);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Pseudo-gradient and per-tensor statistics (INTELLECT-1 notes, sec. 3.2   */
/* step 4 and sec. 4.1 steps 1-2).                                          */

static inline float pseudo_grad(float theta_g, float theta_k) {
    return theta_g - theta_k; /* one IEEE fp32 subtraction */
}

/*
 * Per (learner k, tensor t): count, non-finite count, mean, std, lo, hi.
 * Outputs are [K * T] arrays indexed k * T + t.
 */
void oracle_stats(const float* theta_g, const float* const* theta_k, int32_t K,
                  const int64_t* offsets, int32_t T, double clip_sigmas, int64_t* count,
                  int64_t* nonfinite, double* mean, double* std, double* lo, double* hi) {
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int32_t k = 0; k < K; ++k) {
        for (int32_t t = 0; t < T; ++t) {
            const int64_t a = offsets[t], b = offsets[t + 1], n = b - a;
            const int64_t o = (int64_t)k * T + t;
            int64_t bad = 0;
            double sum = 0.0;
            for (int64_t i = a; i < b; ++i) {
                float d = pseudo_grad(theta_g[i], theta_k[k][i]);
                if (!isfinite(d)) ++bad;
                sum += (double)d;
            }
            count[o] = n;
            nonfinite[o] = bad;
            if (bad > 0) {
                mean[o] = std[o] = lo[o] = hi[o] = NAN;
                continue;
            }
            if (n == 0) {
                mean[o] = std[o] = lo[o] = hi[o] = 0.0;
                continue;
            }
            double mu = sum / (double)n;
            double ss = 0.0;
            for (int64_t i = a; i < b; ++i) {
                double c = (double)pseudo_grad(theta_g[i], theta_k[k][i]) - mu;
                ss += c * c;
            }
            double sigma = sqrt(ss / (double)n);
            mean[o] = mu;
            std[o] = sigma;
            lo[o] = mu - clip_sigmas * sigma;
            hi[o] = mu + clip_sigmas * sigma;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Quantisation (INTELLECT-1 notes, sec. 4.1 steps 2-4).                    */

#define NB 256

static int degenerate_range(double lo, double hi) {
    return !(hi - lo >= (double)NB * (double)FLT_MIN);
}

/* Bucket of one value; lo < hi, s = 256 / (hi - lo). */
static inline int bucket_of(float d, double lo, double s) {
    double u = ((double)d - lo) * s;
    if (u < 0.0) return 0;
    if (u >= (double)NB) return NB - 1;
    int b = (int)floor(u);
    return b > NB - 1 ? NB - 1 : b;
}

/* Bucket coordinate u of each listed element (for boundary diagnostics). */
void oracle_bucket_coord(const float* theta_g, const float* theta_k, const int64_t* idx,
                         int64_t n, double lo, double hi, double* u_out) {
    double s = (double)NB / (hi - lo);
    for (int64_t j = 0; j < n; ++j) {
        float d = pseudo_grad(theta_g[idx[j]], theta_k[idx[j]]);
        u_out[j] = ((double)d - lo) * s;
    }
}

/*
 * Codes, codebook and bucket counts per (k, t).
 * codes: K pointers to uint8[n_elems]; codebook: [K*T*256] float;
 * counts: [K*T*256] uint32 (may be NULL).
 */
void oracle_quantize(const float* theta_g, const float* const* theta_k, int32_t K,
                     const int64_t* offsets, int32_t T, const double* mean, const double* lo,
                     const double* hi, const int64_t* nonfinite, uint8_t* const* codes,
                     float* codebook, uint32_t* counts) {
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int32_t k = 0; k < K; ++k) {
        for (int32_t t = 0; t < T; ++t) {
            const int64_t a = offsets[t], b = offsets[t + 1];
            const int64_t o = (int64_t)k * T + t;
            float* cb = codebook + o * NB;
            uint32_t* cnt_out = counts ? counts + o * NB : NULL;
            double sum[NB];
            int64_t cnt[NB];
            for (int j = 0; j < NB; ++j) {
                sum[j] = 0.0;
                cnt[j] = 0;
            }
            if (nonfinite[o] > 0) {
                for (int64_t i = a; i < b; ++i) codes[k][i] = 0;
                for (int j = 0; j < NB; ++j) cb[j] = NAN;
                if (cnt_out)
                    for (int j = 0; j < NB; ++j) cnt_out[j] = 0;
                continue;
            }
            const double L = lo[o], H = hi[o];
            if (degenerate_range(L, H)) {
                for (int64_t i = a; i < b; ++i) codes[k][i] = 0;
                for (int j = 0; j < NB; ++j) cb[j] = (float)mean[o];
                if (cnt_out) {
                    for (int j = 0; j < NB; ++j) cnt_out[j] = 0;
                    cnt_out[0] = (uint32_t)(b - a);
                }
                continue;
            }
            const double s = (double)NB / (H - L);
            for (int64_t i = a; i < b; ++i) {
                float d = pseudo_grad(theta_g[i], theta_k[k][i]);
                int q = bucket_of(d, L, s);
                double v = (double)d;
                if (v < L) v = L; /* clip (sec. 4.1 step 2) */
                if (v > H) v = H;
                sum[q] += v;
                cnt[q] += 1;
                codes[k][i] = (uint8_t)q;
            }
            for (int j = 0; j < NB; ++j) {
                if (cnt[j] > 0)
                    cb[j] = (float)(sum[j] / (double)cnt[j]);
                else
                    cb[j] = (float)(L + ((double)j + 0.5) * (H - L) / (double)NB);
                if (cnt_out) cnt_out[j] = (uint32_t)cnt[j];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Merge and outer Nesterov step (INTELLECT-1 notes, sec. 3.2 steps 6-7 and */
/* sec. 4.2; Decoupled DiLoCo note, fault-tolerance items 1 and 3).         */

/*
 * Normalised fp32 weights of the present learners; returns the number present
 * or a negative status.
 */
int oracle_merge_weights(const float* weights, const uint8_t* present, int32_t K,
                         int32_t min_quorum, float* w_hat) {
    if (K <= 0) return OR_ERR_ARG;
    int32_t n_present = 0;
    double total = 0.0;
    for (int32_t k = 0; k < K; ++k) {
        w_hat[k] = 0.0f;
        if (present && !present[k]) continue;
        double w = weights ? (double)weights[k] : 1.0;
        if (!(w >= 0.0) || !isfinite(w)) return OR_ERR_ARG;
        total += w;
        ++n_present;
    }
    int32_t need = min_quorum > 1 ? min_quorum : 1;
    if (n_present < need) return OR_ERR_QUORUM;
    if (!(total > 0.0)) return OR_ERR_ARG;
    for (int32_t k = 0; k < K; ++k) {
        if (present && !present[k]) continue;
        double w = weights ? (double)weights[k] : 1.0;
        w_hat[k] = (float)(w / total);
    }
    return n_present;
}

/*
 * One merge + outer Nesterov step over a fragment, in place on theta_g and
 * momentum. codes == NULL selects the unquantised mode (values are the fp32
 * pseudo-gradients themselves, read from theta_k). delta_bar_out may be NULL.
 */
int oracle_merge_outer_step(float* theta_g, float* momentum, const uint8_t* const* codes,
                            const float* codebook, const float* const* theta_k, int32_t K,
                            const int64_t* offsets, int32_t T, const float* weights,
                            const uint8_t* present, int32_t min_quorum, float lr, float mu,
                            float* delta_bar_out) {
    float w_hat[256];
    if (K > 256) return OR_ERR_ARG;
    int np = oracle_merge_weights(weights, present, K, min_quorum, w_hat);
    if (np < 0) return np;
    for (int32_t t = 0; t < T; ++t) {
        const int64_t a = offsets[t], b = offsets[t + 1];
#pragma omp parallel for schedule(static)
        for (int64_t i = a; i < b; ++i) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {
                if (present && !present[k]) continue; /* absent: never read */
                float v;
                if (codes)
                    v = codebook[((int64_t)k * T + t) * NB + codes[k][i]];
                else
                    v = pseudo_grad(theta_g[i], theta_k[k][i]);
                acc = fmaf(w_hat[k], v, acc);
            }
            float m_new = fmaf(mu, momentum[i], acc);
            float g = fmaf(mu, m_new, acc);
            float th = fmaf(-lr, g, theta_g[i]);
            if (delta_bar_out) delta_bar_out[i] = acc;
            momentum[i] = m_new;
            theta_g[i] = th;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Ring accumulation with re-quantisation at every hop (INTELLECT-1 notes,  */
/* sec. 4.2: what a node receives is dequantised, added to in fp32, and     */
/* quantised again before it is sent on).                                   */

/*
 * The present learners, in increasing order, form the ring s = 0 .. S-1; the
 * partial sum P travels along it:
 *   P_0 = w_0 * Delta_0                                   (fp32 product)
 *   P_s = fmaf(w_s, Delta_s, dec(Q(P_{s-1})))            s = 1 .. S-1
 * where Q is the per-tensor quantiser of sec. 4.1 (oracle_stats and
 * oracle_quantize applied to P itself) and dec its codebook lookup. The
 * last holder keeps its fp32 sum: D = P_{S-1} feeds the outer Nesterov step
 * exactly as in oracle_merge_outer_step. A present learner of weight 0 is
 * still a hop (it re-quantises what passes through). delta_bar_out may be
 * NULL. Returns the merge-weight status.
 */
int oracle_ring_outer_step(float* theta_g, float* momentum, const float* const* theta_k,
                           int32_t K, const int64_t* offsets, int32_t T, const float* weights,
                           const uint8_t* present, int32_t min_quorum, double clip_sigmas,
                           float lr, float mu, float* delta_bar_out) {
    float w_hat[256];
    if (K > 256) return OR_ERR_ARG;
    int np = oracle_merge_weights(weights, present, K, min_quorum, w_hat);
    if (np < 0) return np;
    const int64_t n = T > 0 ? offsets[T] : 0;
    const size_t nn = (size_t)(n > 0 ? n : 1);
    float* P = (float*)malloc(sizeof(float) * nn);
    float* zero = (float*)calloc(nn, sizeof(float));
    uint8_t* code = (uint8_t*)malloc(nn);
    float* cb = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1) * NB);
    const size_t tt = (size_t)(T > 0 ? T : 1);
    int64_t* cnt = (int64_t*)malloc(sizeof(int64_t) * tt);
    int64_t* bad = (int64_t*)malloc(sizeof(int64_t) * tt);
    double* mean = (double*)malloc(sizeof(double) * tt);
    double* sd = (double*)malloc(sizeof(double) * tt);
    double* lo = (double*)malloc(sizeof(double) * tt);
    double* hi = (double*)malloc(sizeof(double) * tt);
    if (!P || !zero || !code || !cb || !cnt || !bad || !mean || !sd || !lo || !hi) {
        free(P); free(zero); free(code); free(cb); free(cnt); free(bad);
        free(mean); free(sd); free(lo); free(hi);
        return OR_ERR_ARG;
    }
    const float* zp[1] = {zero};
    uint8_t* cp[1] = {code};
    int first = 1;
    for (int32_t k = 0; k < K; ++k) {
        if (present && !present[k]) continue; /* absent: never read */
        if (first) {
            for (int64_t i = 0; i < n; ++i) P[i] = w_hat[k] * pseudo_grad(theta_g[i], theta_k[k][i]);
            first = 0;
            continue;
        }
        /* the partial sum is quantised for sending, then decoded on arrival;
           P - 0 is P exactly, so the quantiser sees P itself */
        oracle_stats(P, zp, 1, offsets, T, clip_sigmas, cnt, bad, mean, sd, lo, hi);
        oracle_quantize(P, zp, 1, offsets, T, mean, lo, hi, bad, cp, cb, NULL);
        for (int32_t t = 0; t < T; ++t)
            for (int64_t i = offsets[t]; i < offsets[t + 1]; ++i)
                P[i] = fmaf(w_hat[k], pseudo_grad(theta_g[i], theta_k[k][i]),
                            cb[(int64_t)t * NB + code[i]]);
    }
    for (int64_t i = 0; i < n; ++i) {
        const float acc = P[i];
        const float m_new = fmaf(mu, momentum[i], acc);
        const float g = fmaf(mu, m_new, acc);
        if (delta_bar_out) delta_bar_out[i] = acc;
        momentum[i] = m_new;
        theta_g[i] = fmaf(-lr, g, theta_g[i]);
    }
    free(P); free(zero); free(code); free(cb); free(cnt); free(bad);
    free(mean); free(sd); free(lo); free(hi);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Radial-Directional Averaging merge (Decoupled DiLoCo note, architecture */
/* item 4: the outer gradients' norms and directions are averaged apart).  */
/* PARITY UNPINNED: the page gives no formula; the reading taken, per      */
/* tensor t:                                                               */
/*   n_k = ||v_k|| over t (v_k the decoded values of learner k),            */
/*   r   = sum_k w_k n_k                  (radial: mean norm)               */
/*   u   = sum_k (w_k / n_k) v_k          (directional: mean unit vector)   */
/*   D   = r u / ||u||                                                      */
/* Norms from the codebook and the bucket counts, sum_b count_b cb_b^2,    */
/* in fp64; ||u||^2 summed over the tensor's elements in fp64. D is formed */
/* in fp32 from scaled codebooks: c_k = (float)((w_k / n_k) r / ||u||),    */
/* acc = acc + (float)(c_k * cb_k[code]) over present k ascending. A      */
/* learner with n_k = 0 has no direction (c_k = 0); ||u|| = 0 gives D = 0. */

int oracle_rda_merge_outer_step(float* theta_g, float* momentum, const uint8_t* const* codes,
                                const float* codebook, const uint32_t* counts, int32_t K,
                                const int64_t* offsets, int32_t T, const float* weights,
                                const uint8_t* present, int32_t min_quorum, float lr, float mu,
                                float* delta_bar_out) {
    float w_hat[256];
    if (K > 256) return OR_ERR_ARG;
    int np = oracle_merge_weights(weights, present, K, min_quorum, w_hat);
    if (np < 0) return np;
    for (int32_t t = 0; t < T; ++t) {
        const int64_t a = offsets[t], b = offsets[t + 1];
        double nrm[256], coef[256];
        double r = 0.0;
        for (int32_t k = 0; k < K; ++k) {
            nrm[k] = coef[k] = 0.0;
            if (present && !present[k]) continue;
            const float* cb = codebook + ((int64_t)k * T + t) * NB;
            const uint32_t* cnt = counts + ((int64_t)k * T + t) * NB;
            double ss = 0.0;
            for (int j = 0; j < NB; ++j) ss += (double)cnt[j] * (double)cb[j] * (double)cb[j];
            nrm[k] = sqrt(ss);
            r += (double)w_hat[k] * nrm[k];
            coef[k] = nrm[k] > 0.0 ? (double)w_hat[k] / nrm[k] : 0.0;
        }
        double uu = 0.0;
        for (int64_t i = a; i < b; ++i) {
            double x = 0.0;
            for (int32_t k = 0; k < K; ++k) {
                if (present && !present[k]) continue;
                x += coef[k] * (double)codebook[((int64_t)k * T + t) * NB + codes[k][i]];
            }
            uu += x * x;
        }
        const double scale = uu > 0.0 ? r / sqrt(uu) : 0.0;
        float c[256];
        for (int32_t k = 0; k < K; ++k) c[k] = (float)(coef[k] * scale);
        for (int64_t i = a; i < b; ++i) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {
                if (present && !present[k]) continue;
                const float v = codebook[((int64_t)k * T + t) * NB + codes[k][i]];
                acc = acc + c[k] * v;
            }
            const float m_new = fmaf(mu, momentum[i], acc);
            const float g = fmaf(mu, m_new, acc);
            if (delta_bar_out) delta_bar_out[i] = acc;
            momentum[i] = m_new;
            theta_g[i] = fmaf(-lr, g, theta_g[i]);
        }
    }
    return OR_OK;
}
