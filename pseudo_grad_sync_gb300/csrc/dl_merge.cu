// Dequantise, merge over the present learners in fp32 and apply the outer
// Nesterov step in place (INTELLECT-1 notes, section 3.2 steps 6-7 and
// section 4.2; Decoupled DiLoCo note, fault-tolerance items 1 and 3).
//
// k_merge_q<NPM>  persistent blocks over 8192-element chunks. The codebooks
//                 of the present learners for the current tensor sit in
//                 shared memory (NPM x 1 KB at most); per 4-element group a
//                 thread issues one 32-bit code load per present learner plus
//                 128-bit loads of theta and m, decodes through the shared
//                 codebooks, accumulates fmaf(w_k, value, acc) over present k
//                 in ascending order, and stores theta and m back with
//                 128-bit stores. Each byte of codes, theta and m crosses HBM
//                 once.
// k_merge_u       the unquantised variant: values are the fp32 Delta_k read
//                 from the learner replicas.
#include <math.h>

#include "dl_common.cuh"

namespace dl {
namespace {

struct MergeArgs {
    float* g;
    float* m;
    const uint8_t* cp[DL_MAX_LEARNERS];  // codes of the s-th present learner
    const float* rp[DL_MAX_LEARNERS];    // replica of the s-th present learner
    int kidx[DL_MAX_LEARNERS];           // learner index of slot s
    float w[DL_MAX_LEARNERS];            // normalised weight of slot s
    const float* cb;
    const int64_t* off;
    float* dbar;
    int64_t n;
    int64_t n_chunks;
    int np;
    int T;
    float lr;
    float mu;
};

__device__ __forceinline__ void outer_update(float acc, float& th, float& mm, float lr, float mu) {
    const float m1 = __fmaf_rn(mu, mm, acc);
    const float gg = __fmaf_rn(mu, m1, acc);
    th = __fmaf_rn(-lr, gg, th);
    mm = m1;
}

template <int NPM>
__global__ void __launch_bounds__(kThreads) k_merge_q(MergeArgs a) {
    extern __shared__ float scb[];  // [np][256]
    const int tid = threadIdx.x;
    const int np = a.np;
    int cur_t = -1;
    for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
        const int64_t base = c * kChunk;
        const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
        const int64_t cend = base + cn;
        for (int t = tensor_containing(a.off, a.T, base); t < a.T; ++t) {
            const int64_t o0 = __ldg(a.off + t), o1 = __ldg(a.off + t + 1);
            if (o0 >= cend) break;
            const int64_t pa = o0 > base ? o0 : base;
            const int64_t pb = o1 < cend ? o1 : cend;
            if (pa >= pb) continue;
            if (t != cur_t) {
                __syncthreads();
                for (int i = tid; i < np * kNB; i += kThreads)
                    scb[i] = __ldg(a.cb + (static_cast<int64_t>(a.kidx[i >> 8]) * a.T + t) * kNB + (i & (kNB - 1)));
                __syncthreads();
                cur_t = t;
            }
            if (pa == base && pb == base + kChunk) {
                float4* g4 = reinterpret_cast<float4*>(a.g + base);
                float4* m4 = reinterpret_cast<float4*>(a.m + base);
#pragma unroll 1
                for (int j = 0; j < kGroups; j += 2) {
                    uint32_t cw[2][NPM];
                    float4 th[2], mm[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int gi = tid + (j + u) * kThreads;
                        th[u] = g4[gi];
                        mm[u] = m4[gi];
#pragma unroll
                        for (int s = 0; s < NPM; ++s)
                            if (s < np)
                                cw[u][s] = __ldcs(reinterpret_cast<const unsigned int*>(a.cp[s] + base) + gi);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                        for (int s = 0; s < NPM; ++s) {
                            if (s < np) {
                                const float* cbs = scb + s * kNB;
                                const uint32_t w4 = cw[u][s];
                                const float ws = a.w[s];
                                a0 = __fmaf_rn(ws, cbs[w4 & 255u], a0);
                                a1 = __fmaf_rn(ws, cbs[(w4 >> 8) & 255u], a1);
                                a2 = __fmaf_rn(ws, cbs[(w4 >> 16) & 255u], a2);
                                a3 = __fmaf_rn(ws, cbs[w4 >> 24], a3);
                            }
                        }
                        const int gi = tid + (j + u) * kThreads;
                        outer_update(a0, th[u].x, mm[u].x, a.lr, a.mu);
                        outer_update(a1, th[u].y, mm[u].y, a.lr, a.mu);
                        outer_update(a2, th[u].z, mm[u].z, a.lr, a.mu);
                        outer_update(a3, th[u].w, mm[u].w, a.lr, a.mu);
                        g4[gi] = th[u];
                        m4[gi] = mm[u];
                        if (a.dbar)
                            reinterpret_cast<float4*>(a.dbar + base)[gi] = make_float4(a0, a1, a2, a3);
                    }
                }
            } else {
                for (int64_t i = pa + tid; i < pb; i += kThreads) {
                    float acc = 0.f;
                    for (int s = 0; s < np; ++s)
                        acc = __fmaf_rn(a.w[s], scb[s * kNB + a.cp[s][i]], acc);
                    float th = a.g[i], mm = a.m[i];
                    outer_update(acc, th, mm, a.lr, a.mu);
                    a.g[i] = th;
                    a.m[i] = mm;
                    if (a.dbar) a.dbar[i] = acc;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads) k_merge_u(MergeArgs a) {
    const int tid = threadIdx.x;
    const int np = a.np;
    const int64_t nvec = a.n >> 2;
    float4* g4 = reinterpret_cast<float4*>(a.g);
    float4* m4 = reinterpret_cast<float4*>(a.m);
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * kThreads + tid; gi < nvec;
         gi += static_cast<int64_t>(gridDim.x) * kThreads) {
        float4 th = g4[gi], mm = m4[gi];
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        for (int s = 0; s < np; ++s) {
            const float4 r = __ldcs(reinterpret_cast<const float4*>(a.rp[s]) + gi);
            const float ws = a.w[s];
            a0 = __fmaf_rn(ws, __fsub_rn(th.x, r.x), a0);
            a1 = __fmaf_rn(ws, __fsub_rn(th.y, r.y), a1);
            a2 = __fmaf_rn(ws, __fsub_rn(th.z, r.z), a2);
            a3 = __fmaf_rn(ws, __fsub_rn(th.w, r.w), a3);
        }
        outer_update(a0, th.x, mm.x, a.lr, a.mu);
        outer_update(a1, th.y, mm.y, a.lr, a.mu);
        outer_update(a2, th.z, mm.z, a.lr, a.mu);
        outer_update(a3, th.w, mm.w, a.lr, a.mu);
        g4[gi] = th;
        m4[gi] = mm;
        if (a.dbar) reinterpret_cast<float4*>(a.dbar)[gi] = make_float4(a0, a1, a2, a3);
    }
    // trailing 0..3 elements
    if (blockIdx.x == 0 && tid < (a.n & 3)) {
        const int64_t i = nvec * 4 + tid;
        float th = a.g[i], mm = a.m[i], acc = 0.f;
        for (int s = 0; s < np; ++s) acc = __fmaf_rn(a.w[s], __fsub_rn(th, a.rp[s][i]), acc);
        outer_update(acc, th, mm, a.lr, a.mu);
        a.g[i] = th;
        a.m[i] = mm;
        if (a.dbar) a.dbar[i] = acc;
    }
}

template <int NPM>
int launch_q(const MergeArgs& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * kNB * a.np;
    const int grid = grid_for(reinterpret_cast<const void*>(k_merge_q<NPM>), kThreads, smem, a.n_chunks);
    k_merge_q<NPM><<<grid, kThreads, smem, s>>>(a);
    return launch_status();
}

}  // namespace
}  // namespace dl

using namespace dl;

extern "C" int dl_merge_outer_step(float* theta_g, float* momentum, const uint8_t* const* codes,
                                   const float* d_codebook, const float* const* theta_k, int32_t K,
                                   const dl_fragment* frag, const float* weights,
                                   const uint8_t* present, int32_t min_quorum, float lr, float mu,
                                   float* delta_bar_out, void* stream) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    if (K <= 0 || K > DL_MAX_LEARNERS) return DL_ERR_ARG;
    const bool quant = codes != nullptr;
    if (!quant && !theta_k) return DL_ERR_ARG;

    // quorum and weight normalisation over the present learners (fp64, then fp32)
    MergeArgs a;
    memset(&a, 0, sizeof(a));
    double total = 0.0;
    int np = 0;
    for (int k = 0; k < K; ++k) {
        if (present && !present[k]) continue;
        const double w = weights ? static_cast<double>(weights[k]) : 1.0;
        if (!(w >= 0.0) || !isfinite(w)) return DL_ERR_ARG;
        total += w;
        a.kidx[np++] = k;
    }
    if (np < (min_quorum > 1 ? min_quorum : 1)) return DL_ERR_QUORUM;
    if (!(total > 0.0)) return DL_ERR_ARG;
    for (int s = 0; s < np; ++s) {
        const int k = a.kidx[s];
        const double w = weights ? static_cast<double>(weights[k]) : 1.0;
        a.w[s] = static_cast<float>(w / total);
    }
    a.np = np;
    if (f.n == 0) return DL_OK;

    if (!theta_g || !momentum) return DL_ERR_ARG;
    if (!aligned16(theta_g) || !aligned16(momentum) || (delta_bar_out && !aligned16(delta_bar_out)))
        return DL_ERR_ALIGN;
    for (int s = 0; s < np; ++s) {
        const int k = a.kidx[s];
        if (quant) {
            if (!codes[k]) return DL_ERR_ARG;
            if (!aligned16(codes[k])) return DL_ERR_ALIGN;
            a.cp[s] = codes[k];
        } else {
            if (!theta_k[k]) return DL_ERR_ARG;
            if (!aligned16(theta_k[k])) return DL_ERR_ALIGN;
            a.rp[s] = theta_k[k];
        }
    }
    if (quant) {
        if (!d_codebook) return DL_ERR_ARG;
        if (!aligned16(d_codebook)) return DL_ERR_ALIGN;
    }
    a.g = theta_g;
    a.m = momentum;
    a.cb = d_codebook;
    a.off = f.d_offsets;
    a.dbar = delta_bar_out;
    a.n = f.n;
    a.n_chunks = n_chunks_of(f.n);
    a.T = f.T;
    a.lr = lr;
    a.mu = mu;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!quant) {
        const int grid = grid_for(reinterpret_cast<const void*>(k_merge_u), kThreads, 0,
                                  ((f.n >> 2) + kThreads - 1) / kThreads + 1);
        k_merge_u<<<grid, kThreads, 0, s>>>(a);
        return launch_status();
    }
    if (np <= 4) return launch_q<4>(a, s);
    if (np <= 8) return launch_q<8>(a, s);
    if (np <= 16) return launch_q<16>(a, s);
    return launch_q<32>(a, s);
}
