// Per-(learner, tensor) pseudo-gradient statistics (INTELLECT-1 notes,
// section 4.1 step 1: one mu and one sigma per tensor; step 2: the clip
// range mu +- 6 sigma).
//
// Three launches on the caller's stream:
//  k_shift     one warp per (k, t): c = mean of the first min(N, 64) values
//              of Delta in fp64, snapped to a power-of-two grid below their
//              spread and rounded to fp32. Every block later sums
//              y = Delta - c, which keeps the one-pass variance free of
//              cancellation when |mu| >> sigma; c is computed once so all
//              chunks of a tensor share it. The snapping keeps the fp32
//              rounding of y unbiased (a shift with low-order bits below
//              ulp(y) biases every rounding the same way).
//  k_stats     persistent blocks over 8192-element chunks of the fragment.
//              theta_g's chunk is staged in shared memory by one bulk (TMA)
//              copy and reused for all K learners; each learner's chunk is
//              streamed with 128-bit loads. Per thread: fp32 sums over
//              groups of four, folded into float-float (hi + lo) sums;
//              per warp: a float-float butterfly; per block: an fp64 sum of
//              the 8 warps, written as one partial per (k, chunk, tensor)
//              piece. Tensors shorter than 4096 elements and groups of rare
//              huge, tiny (squares would leave the fp32 normal range) or
//              non-finite values take an fp64 path.
//  k_stats_fin one warp per (k, t): fixed-order fp64 sum of its pieces, then
//              mu = c + S1/N, sigma^2 = S2/N - (S1/N)^2 (population).
// The result is deterministic: every sum has a fixed order.
#include "dl_common.cuh"

namespace dl {
namespace {

struct Partial {
    double s1, s2;
    long long bad;
    long long pad;
};

struct StatsArgs {
    const float* g;
    const float* r[DL_MAX_LEARNERS];
    const int64_t* off;
    float* shift;
    Partial* part;
    dl_stats* out;
    uint32_t* status;
    int64_t n;
    int64_t n_chunks;
    int64_t P;  // partial slots per learner: n_chunks + T
    int T;
    int K;
    double clip;
};

__global__ void __launch_bounds__(kThreads) k_shift(StatsArgs a) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= a.K * a.T) return;
    const int k = w / a.T, t = w % a.T;
    const int64_t o = a.off[t];
    const int64_t N = a.off[t + 1] - o;
    const int m = N < 64 ? static_cast<int>(N) : 64;
    const bool h0 = lane < m, h1 = lane + 32 < m;
    const double v0 = h0 ? static_cast<double>(__fsub_rn(a.g[o + lane], a.r[k][o + lane])) : 0.0;
    const double v1 = h1 ? static_cast<double>(__fsub_rn(a.g[o + lane + 32], a.r[k][o + lane + 32])) : 0.0;
    double s = v0 + v1;
    for (int sh = 16; sh; sh >>= 1) s += __shfl_xor_sync(kFull, s, sh);
    const double mean = m > 0 ? s / m : 0.0;
    double q = (h0 ? (v0 - mean) * (v0 - mean) : 0.0) + (h1 ? (v1 - mean) * (v1 - mean) : 0.0);
    for (int sh = 16; sh; sh >>= 1) q += __shfl_xor_sync(kFull, q, sh);
    if (lane != 0) return;
    const double sd = m > 0 ? sqrt(q / m) : 0.0;
    double c = mean;
    if (sd > 0.0 && isfinite(sd) && isfinite(mean)) {
        // snap to a power-of-two grid no finer than sd/8: the shift then has
        // no bits below the ulp of any typical y = Delta - c, so rounding
        // y to fp32 is unbiased
        int ex;
        frexp(sd, &ex);  // sd in [2^(ex-1), 2^ex)
        const double grid = ldexp(1.0, ex - 3);
        c = rint(mean / grid) * grid;
    }
    a.shift[w] = static_cast<float>(c);
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

__global__ void __launch_bounds__(kThreads) k_stats(StatsArgs a) {
    extern __shared__ __align__(16) float sg[];  // kChunk floats of theta_g
    __shared__ uint64_t bar;
    __shared__ int flag;
    __shared__ float red_ff[DL_MAX_LEARNERS][kWarps][4];
    __shared__ double red_side[DL_MAX_LEARNERS][kWarps][2];
    __shared__ int red_bad[DL_MAX_LEARNERS][kWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();

    uint32_t iter = 0;
    for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x, ++iter) {
        const int64_t base = c * kChunk;
        const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
        if (!stage_chunk(sg, a.g + base, cn, &bar, iter, &flag, a.status)) return;
        const int64_t cend = base + cn;
        for (int t = tensor_containing(a.off, a.T, base); t < a.T; ++t) {
            const int64_t o0 = __ldg(a.off + t), o1 = __ldg(a.off + t + 1);
            if (o0 >= cend) break;
            const int64_t pa = o0 > base ? o0 : base;
            const int64_t pb = o1 < cend ? o1 : cend;
            if (pa >= pb) continue;
            const bool small = (o1 - o0) < kSmallTensor;
            const bool full = (pa == base) && (pb == base + kChunk);
            const int la = static_cast<int>(pa - base), lb = static_cast<int>(pb - base);

            for (int k = 0; k < a.K; ++k) {
                const float csh = __ldg(a.shift + k * a.T + t);
                const float* rk = a.r[k] + base;
                float s1h = 0.f, s1l = 0.f, s2h = 0.f, s2l = 0.f;
                double s1d = 0.0, s2d = 0.0;
                int bad = 0;
                bool side = false;
                if (full && !small) {
                    float4 v[kGroups];
#pragma unroll
                    for (int j = 0; j < kGroups; ++j)
                        v[j] = __ldcs(reinterpret_cast<const float4*>(rk) + tid + j * kThreads);
#pragma unroll
                    for (int j = 0; j < kGroups; ++j) {
                        const float4 gg = reinterpret_cast<const float4*>(sg)[tid + j * kThreads];
                        const float d0 = __fsub_rn(gg.x, v[j].x), d1 = __fsub_rn(gg.y, v[j].y);
                        const float d2 = __fsub_rn(gg.z, v[j].z), d3 = __fsub_rn(gg.w, v[j].w);
                        const float y0 = __fsub_rn(d0, csh), y1 = __fsub_rn(d1, csh);
                        const float y2 = __fsub_rn(d2, csh), y3 = __fsub_rn(d3, csh);
                        const float mx = fmaxf(fmaxf(fabsf(y0), fabsf(y1)), fmaxf(fabsf(y2), fabsf(y3)));
                        // fp32 squares stay normal and finite for 2^-60 <= |y| <= 2^48
                        if (mx <= 0x1p48f && (mx >= 0x1p-60f || mx == 0.0f)) {  // false for NaN
                            const float b1 = __fadd_rn(__fadd_rn(y0, y1), __fadd_rn(y2, y3));
                            const float b2 = __fmaf_rn(
                                y3, y3, __fmaf_rn(y2, y2, __fmaf_rn(y1, y1, __fmul_rn(y0, y0))));
                            ff_add(s1h, s1l, b1);
                            ff_add(s2h, s2l, b2);
                        } else {
                            side = true;
                            side_add(d0, csh, s1d, s2d, bad);
                            side_add(d1, csh, s1d, s2d, bad);
                            side_add(d2, csh, s1d, s2d, bad);
                            side_add(d3, csh, s1d, s2d, bad);
                        }
                    }
                } else {
                    for (int j = 0; j < kGroups; ++j) {
                        const int e0 = 4 * (tid + j * kThreads);
                        if (e0 >= lb || e0 + 4 <= la) continue;
                        for (int i = 0; i < 4; ++i) {
                            const int e = e0 + i;
                            if (e < la || e >= lb) continue;
                            const float d = __fsub_rn(sg[e], __ldcs(rk + e));
                            const float y = __fsub_rn(d, csh);
                            const float ay = fabsf(y);
                            if (!small && ay <= 0x1p48f && (ay >= 0x1p-60f || ay == 0.0f)) {
                                ff_add(s1h, s1l, y);
                                ff_add(s2h, s2l, __fmul_rn(y, y));
                            } else {
                                side = true;
                                side_add(d, csh, s1d, s2d, bad);
                            }
                        }
                    }
                }
                // warp: float-float butterfly (symmetric, so every lane ends equal)
#pragma unroll
                for (int sh = 16; sh; sh >>= 1) {
                    const float o1h = __shfl_xor_sync(kFull, s1h, sh);
                    const float o1l = __shfl_xor_sync(kFull, s1l, sh);
                    const float o2h = __shfl_xor_sync(kFull, s2h, sh);
                    const float o2l = __shfl_xor_sync(kFull, s2l, sh);
                    ff_add_ff(s1h, s1l, o1h, o1l);
                    ff_add_ff(s2h, s2l, o2h, o2l);
                }
                if (__any_sync(kFull, side)) {
                    for (int sh = 16; sh; sh >>= 1) {
                        s1d += __shfl_xor_sync(kFull, s1d, sh);
                        s2d += __shfl_xor_sync(kFull, s2d, sh);
                        bad += __shfl_xor_sync(kFull, bad, sh);
                    }
                } else {
                    s1d = s2d = 0.0;
                    bad = 0;
                }
                if (lane == 0) {
                    red_ff[k][warp][0] = s1h;
                    red_ff[k][warp][1] = s1l;
                    red_ff[k][warp][2] = s2h;
                    red_ff[k][warp][3] = s2l;
                    red_side[k][warp][0] = s1d;
                    red_side[k][warp][1] = s2d;
                    red_bad[k][warp] = bad;
                }
            }
            __syncthreads();
            if (tid < a.K) {
                double s1 = 0.0, s2 = 0.0;
                long long bad = 0;
                for (int w = 0; w < kWarps; ++w) {
                    s1 += static_cast<double>(red_ff[tid][w][0]) + static_cast<double>(red_ff[tid][w][1]) +
                          red_side[tid][w][0];
                    s2 += static_cast<double>(red_ff[tid][w][2]) + static_cast<double>(red_ff[tid][w][3]) +
                          red_side[tid][w][1];
                    bad += red_bad[tid][w];
                }
                Partial p;
                p.s1 = s1;
                p.s2 = s2;
                p.bad = bad;
                p.pad = 0;
                a.part[static_cast<int64_t>(tid) * a.P + c + t] = p;
            }
            __syncthreads();
        }
        __syncthreads();  // the staged chunk is about to be overwritten
    }
}

__global__ void __launch_bounds__(kThreads) k_stats_fin(StatsArgs a) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= a.K * a.T) return;
    const int k = w / a.T, t = w % a.T;
    const int64_t o0 = a.off[t], o1 = a.off[t + 1];
    const int64_t N = o1 - o0;
    double s1 = 0.0, s2 = 0.0;
    long long bad = 0;
    if (N > 0) {
        const int64_t c0 = o0 / kChunk, c1 = (o1 - 1) / kChunk;
        const Partial* pk = a.part + static_cast<int64_t>(k) * a.P + t;
        for (int64_t c = c0 + lane; c <= c1; c += 32) {
            const Partial p = pk[c];
            s1 += p.s1;
            s2 += p.s2;
            bad += p.bad;
        }
    }
    for (int sh = 16; sh; sh >>= 1) {
        s1 += __shfl_xor_sync(kFull, s1, sh);
        s2 += __shfl_xor_sync(kFull, s2, sh);
        bad += __shfl_xor_sync(kFull, bad, sh);
    }
    if (lane != 0) return;
    dl_stats st;
    st.count = N;
    st.nonfinite = bad;
    if (bad > 0) {
        st.mean = st.std = st.lo = st.hi = __longlong_as_double(0x7ff8000000000000LL);
    } else if (N == 0) {
        st.mean = st.std = st.lo = st.hi = 0.0;
    } else {
        const double inv = 1.0 / static_cast<double>(N);
        const double mrel = s1 * inv;
        double var = s2 * inv - mrel * mrel;
        if (!(var > 0.0)) var = 0.0;
        const double sigma = sqrt(var);
        const double mu = static_cast<double>(a.shift[w]) + mrel;
        st.mean = mu;
        st.std = sigma;
        st.lo = mu - a.clip * sigma;
        st.hi = mu + a.clip * sigma;
    }
    a.out[w] = st;
}

size_t shift_bytes(int K, int T) { return align256(sizeof(float) * static_cast<size_t>(K) * T); }

}  // namespace
}  // namespace dl

using namespace dl;

extern "C" size_t dl_stats_workspace_bytes(const dl_fragment* frag, int32_t K) {
    HostFrag f;
    if (check_fragment(frag, &f) != DL_OK || K <= 0 || K > DL_MAX_LEARNERS) return 0;
    const int64_t P = n_chunks_of(f.n) + f.T;
    return kWsHeader + shift_bytes(K, f.T) + align256(sizeof(Partial) * static_cast<size_t>(K) * P);
}

extern "C" int dl_pseudograd_stats(const float* theta_g, const float* const* theta_k, int32_t K,
                                   const dl_fragment* frag, double clip_sigmas, dl_stats* d_stats,
                                   void* d_workspace, size_t workspace_bytes, void* stream) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    if (K <= 0 || K > DL_MAX_LEARNERS || !theta_k || !(clip_sigmas > 0.0) ||
        !(clip_sigmas < 1e300))
        return DL_ERR_ARG;
    if (f.T == 0) return DL_OK;
    if (!d_stats) return DL_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_stats) & 7u) != 0) return DL_ERR_ALIGN;
    if (f.n > 0) {
        if (!theta_g) return DL_ERR_ARG;
        if (!aligned16(theta_g)) return DL_ERR_ALIGN;
        for (int k = 0; k < K; ++k) {
            if (!theta_k[k]) return DL_ERR_ARG;
            if (!aligned16(theta_k[k])) return DL_ERR_ALIGN;
        }
    }
    const size_t need = dl_stats_workspace_bytes(frag, K);
    if (!d_workspace || workspace_bytes < need) return DL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0) return DL_ERR_ALIGN;

    StatsArgs a;
    memset(&a, 0, sizeof(a));
    a.g = theta_g;
    for (int k = 0; k < K; ++k) a.r[k] = theta_k[k];
    a.off = f.d_offsets;
    char* ws = static_cast<char*>(d_workspace);
    a.status = reinterpret_cast<uint32_t*>(ws);
    a.shift = reinterpret_cast<float*>(ws + kWsHeader);
    a.part = reinterpret_cast<Partial*>(ws + kWsHeader + shift_bytes(K, f.T));
    a.out = d_stats;
    a.n = f.n;
    a.n_chunks = n_chunks_of(f.n);
    a.P = a.n_chunks + f.T;
    a.T = f.T;
    a.K = K;
    a.clip = clip_sigmas;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int warps = K * f.T;
    const int small_grid = (warps * 32 + kThreads - 1) / kThreads;
    k_shift<<<small_grid, kThreads, 0, s>>>(a);
    if ((st = launch_status()) != DL_OK) return st;
    if (a.n_chunks > 0) {
        const size_t smem = sizeof(float) * kChunk;
        const int grid = grid_for(reinterpret_cast<const void*>(k_stats), kThreads, smem, a.n_chunks);
        k_stats<<<grid, kThreads, smem, s>>>(a);
        if ((st = launch_status()) != DL_OK) return st;
    }
    k_stats_fin<<<small_grid, kThreads, 0, s>>>(a);
    return launch_status();
}
