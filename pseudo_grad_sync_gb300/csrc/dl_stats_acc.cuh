// Exact one-pass statistics accumulation shared by the statistics kernel and
// the fused ring hop: per-thread float-float sums of y = value - c (c a
// per-tensor shift) and of y^2 on a power-of-two offset with exact error
// terms, an fp64 side path for values outside the fast range, the
// block-level flush into one fp64 partial per (block, tensor), and the shift
// rule. The finalisation (partials -> mu, sigma, lo, hi) is stats_finish.
#pragma once

#include "dl_common.cuh"

namespace dl {

// fp64 partial sums of one (block, tensor)
struct Partial {
    double s1, s2;
    long long bad;
    long long pad;
};


// y values in this range take the fast float-float path: their squares,
// error terms and offsets stay normal and finite (smaller values lose at
// most 2^-149); NaN fails the test
__device__ __forceinline__ bool fast_range(float ay) {
    return ay <= 0x1p48f && (ay >= 0x1p-50f || ay == 0.0f);
}

// fp64 contribution of one value (small tensors, huge or non-finite values)
__device__ __forceinline__ void side_add(float d, float c, double& s1, double& s2, int& bad) {
    if (!isfinite(d)) {
        ++bad;
        return;
    }
    const double y = static_cast<double>(d) - static_cast<double>(c);
    s1 += y;
    s2 = fma(y, y, s2);
}

// Per-thread sums. y^2 is summed on an offset: (s2h, s2l) holds H0 + the
// squares since the last rebase, with H0 = yt^2 and yt a power of two at
// least as large as every |y| this thread has summed since then; (c2h, c2l)
// holds the squares summed before it (see sq_add and rebase).
struct Acc {
    float s1h, s1l;  // float-float sum of y
    float s2h, s2l;  // float-float H0 + sum of y^2 since the last rebase
    float s2hb, s2lb;  // a second such sum: the odd lane of packed (fp32x2) squares
    float c2h, c2l;  // float-float sum of y^2 before it
    float yt, h0;    // current bound on |y| and H0 = yt^2
    double s1d, s2d; // fp64 side sums
    int bad;
    bool side;
    __device__ __forceinline__ void reset() {
        s1h = s1l = s2h = s2l = s2hb = s2lb = c2h = c2l = yt = h0 = 0.f;
        s1d = s2d = 0.0;
        bad = 0;
        side = false;
    }
};

// Join the squares of one offset sum (hi, lo) = H0 + squares into (c2h, c2l):
// hi >= H0 and H0 is a power of two on hi's ulp grid, so hi - H0 is exact.
__device__ __forceinline__ void join_squares(float& c2h, float& c2l, float hi, float lo, float h0) {
    ff_add_ff(c2h, c2l, __fsub_rn(hi, h0), lo);
}

// The odd-lane sum holds squares only where the packed path ran; elsewhere
// it stays at (H0, 0) and is left out, so that kernels which never use it
// keep their sums bit for bit.
__device__ __forceinline__ bool odd_lane_used(const Acc& acc) {
    return acc.s2hb != acc.h0 || acc.s2lb != 0.f;
}

// Reduction over the kThreads accumulating threads (named barrier 1) of the
// per-thread sums of one tensor into the partial slot *dst. Fixed order
// everywhere, so the result is deterministic.
static __device__ void flush_partial(Acc& acc, Partial* dst, float (*red_ff)[4],
                                     double (*red_side)[2], int* red_bad) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // remove the offsets (s2h >= H0, a power of two on its ulp grid, so the
    // difference is exact) and join the squares summed before the last rebase
    join_squares(acc.c2h, acc.c2l, acc.s2h, acc.s2l, acc.h0);
    if (odd_lane_used(acc)) join_squares(acc.c2h, acc.c2l, acc.s2hb, acc.s2lb, acc.h0);
    acc.s2h = acc.c2h;
    acc.s2l = acc.c2l;
#pragma unroll
    for (int sh = 16; sh; sh >>= 1) {
        const float o1h = __shfl_xor_sync(kFull, acc.s1h, sh);
        const float o1l = __shfl_xor_sync(kFull, acc.s1l, sh);
        const float o2h = __shfl_xor_sync(kFull, acc.s2h, sh);
        const float o2l = __shfl_xor_sync(kFull, acc.s2l, sh);
        ff_add_ff(acc.s1h, acc.s1l, o1h, o1l);
        ff_add_ff(acc.s2h, acc.s2l, o2h, o2l);
    }
    if (__any_sync(kFull, acc.side)) {
        for (int sh = 16; sh; sh >>= 1) {
            acc.s1d += __shfl_xor_sync(kFull, acc.s1d, sh);
            acc.s2d += __shfl_xor_sync(kFull, acc.s2d, sh);
            acc.bad += __shfl_xor_sync(kFull, acc.bad, sh);
        }
    } else {
        acc.s1d = acc.s2d = 0.0;
        acc.bad = 0;
    }
    if (lane == 0) {
        red_ff[warp][0] = acc.s1h;
        red_ff[warp][1] = acc.s1l;
        red_ff[warp][2] = acc.s2h;
        red_ff[warp][3] = acc.s2l;
        red_side[warp][0] = acc.s1d;
        red_side[warp][1] = acc.s2d;
        red_bad[warp] = acc.bad;
    }
    consumer_sync();
    if (threadIdx.x == 0) {
        double s1 = 0.0, s2 = 0.0;
        long long bad = 0;
        for (int w = 0; w < kConsumerWarps; ++w) {
            s1 += static_cast<double>(red_ff[w][0]) + static_cast<double>(red_ff[w][1]) + red_side[w][0];
            s2 += static_cast<double>(red_ff[w][2]) + static_cast<double>(red_ff[w][3]) + red_side[w][1];
            bad += red_bad[w];
        }
        Partial p;
        p.s1 = s1;
        p.s2 = s2;
        p.bad = bad;
        p.pad = 0;
        *dst = p;
    }
    consumer_sync();
}

// y^2 added to the float-float sum (hi, lo) = H0 + squares, for |y| <= yt:
// then y^2 <= H0 <= hi, the sum s = fl(hi + y^2) stays within [hi, 2 hi],
// hi - s is exact, and fma(y, y, hi - s) is the rounding error of s, itself
// rounded once (within 2^-25 ulp(s)). The error goes to lo. Plain fp32
// squares are not enough: when Delta carries few significant bits relative to
// sigma (|mu| >> sigma), y is a short integer times a power of two, and the
// bits that rounding drops from its square follow the pattern of squares (an
// odd square ends in ...001), so every rounding goes the same way; the error
// terms keep those bits. As H0 <= 4 max y^2, the ulps involved stay within a
// factor 2^-21 of the squares themselves.
__device__ __forceinline__ void sq_add(float& hi, float& lo, float y) {
    const float s = __fmaf_rn(y, y, hi);
    const float err = __fmaf_rn(y, y, __fsub_rn(hi, s));
    hi = s;
    lo = __fadd_rn(lo, err);
}

// |y| up to mx (positive, normal) is about to be summed and exceeds yt: move
// the offset sums into (c2h, c2l) and restart them on yt = the power of two
// >= mx. Taken at a thread's first non-zero group of a tensor and then only
// when a value exceeds every earlier one by enough to cross a power of two.
__device__ __forceinline__ void rebase(Acc& acc, float mx) {
    join_squares(acc.c2h, acc.c2l, acc.s2h, acc.s2l, acc.h0);
    if (odd_lane_used(acc)) join_squares(acc.c2h, acc.c2l, acc.s2hb, acc.s2lb, acc.h0);
    acc.yt = __int_as_float((__float_as_int(mx) + 0x7FFFFF) & static_cast<int>(0xFF800000u));
    acc.h0 = __fmul_rn(acc.yt, acc.yt);
    acc.s2h = acc.s2hb = acc.h0;
    acc.s2l = acc.s2lb = 0.f;
}

// Two squares at once (fp32x2 instructions, each lane rounded as the scalar
// ones): y.x goes to (s2h, s2l), y.y to (s2hb, s2lb), with sq_add's exact
// error terms.
__device__ __forceinline__ void sq_add2(Acc& acc, float2 y) {
    const float2 hi = make_float2(acc.s2h, acc.s2hb);
    const float2 s = __ffma2_rn(y, y, hi);
    const float2 err = __ffma2_rn(y, y, __ffma2_rn(s, make_float2(-1.f, -1.f), hi));
    const float2 lo = __fadd2_rn(make_float2(acc.s2l, acc.s2lb), err);
    acc.s2h = s.x;
    acc.s2hb = s.y;
    acc.s2l = lo.x;
    acc.s2lb = lo.y;
}

// fold lo into hi (|lo| <= ulp(hi) afterwards), so that the roundings of
// later additions to lo stay below 2^-24 ulp(hi)
__device__ __forceinline__ void renorm(float& hi, float& lo) {
    const float s = __fadd_rn(hi, lo);
    lo = __fsub_rn(lo, __fsub_rn(s, hi));
    hi = s;
}

// max(|a|, b) that returns NaN if either input is NaN (fmaxf would drop it)
__device__ __forceinline__ float absmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(a)), "f"(b));
    return r;
}


// Shift of one tensor from up to 64 of its first values (v0 at lane, v1 at
// lane + 32; h0 / h1 whether they exist, m how many there are), computed by
// the whole warp; every lane returns it. The mean in fp64, snapped to a
// power-of-two grid no finer than sd/8 (sd the samples' spread): the shift
// then has no bits below the ulp of any typical y = value - c, so rounding y
// to fp32 is unbiased.
__device__ __forceinline__ float warp_shift(double v0, double v1, bool h0, bool h1, int m) {
    double s = (h0 ? v0 : 0.0) + (h1 ? v1 : 0.0);
    for (int sh = 16; sh; sh >>= 1) s += __shfl_xor_sync(kFull, s, sh);
    const double mean = m > 0 ? s / m : 0.0;
    double q = (h0 ? (v0 - mean) * (v0 - mean) : 0.0) + (h1 ? (v1 - mean) * (v1 - mean) : 0.0);
    for (int sh = 16; sh; sh >>= 1) q += __shfl_xor_sync(kFull, q, sh);
    const double sd = m > 0 ? sqrt(q / m) : 0.0;
    double c = mean;
    if (sd > 0.0 && isfinite(sd) && isfinite(mean)) {
        int ex;
        frexp(sd, &ex);  // sd in [2^(ex-1), 2^ex)
        const double grid = ldexp(1.0, ex - 3);
        c = rint(mean / grid) * grid;
    }
    return static_cast<float>(c);
}

// Enqueue the finalisation on s: for each of the K*T (learner, tensor) pairs,
// the fixed-order fp64 sum of its J partials part[(k*T + t)*J + j], then
// mu = shift + S1/N, sigma^2 = S2/N - (S1/N)^2 (population), lo/hi = mu -+
// clip sigma, into out[k*T + t]. d_off is the device copy of the offsets.
int stats_finish(const int64_t* d_off, int T, int K, int J, const float* shift,
                 const Partial* part, double clip, dl_stats* out, cudaStream_t s);

}  // namespace dl
