// Ring accumulation with re-quantisation at every hop, then the outer Nesterov
// step (INTELLECT-1 notes, section 4.2: what a node receives is dequantised,
// added to in fp32, and quantised again before it is sent on; section 4.1
// for the quantiser; section 3.2 step 7 for the outer step).
//
// On one GPU the ring's S present learners, in increasing order, are visited
// one after another; the partial sum P lives in the workspace:
//   hop 0:        P = w_0 * Delta_0
//   hop s >= 1:   quantise P (dl_pseudograd_stats + dl_quantize in values
//                 mode: the vector quantised is P itself), then
//                 P = fmaf(w_s, Delta_s, cb[code])
//   last hop:     instead of storing P, apply the outer Nesterov step with
//                 D = P (and write D out if asked).
// k_ring_hop<DECODE, FINAL> does one hop's element work: persistent blocks
// over 8192-element chunks, the previous codebook of the current tensor in
// shared memory, 128-bit loads and stores, 32-bit code loads.
#include <math.h>
#include <string.h>

#include "dl_common.cuh"

namespace dl {
namespace {

static_assert(kThreads == kNB, "one codebook entry per thread");

struct RingArgs {
    float* g;               // theta_g (written at the last hop only)
    const float* r;         // this hop's learner replica
    float* P;               // partial sum (written unless FINAL)
    float* m;               // momentum (FINAL)
    const uint8_t* codes;   // codes of the previous partial sum (DECODE)
    const float* cb;        // its codebook [T][256] (DECODE)
    const int64_t* off;
    float* dbar;            // optional D (FINAL)
    int64_t n;
    int64_t n_chunks;
    int T;
    float w;
    float lr;
    float mu;
};

template <bool DECODE>
__device__ __forceinline__ float hop_value(float g, float r, float dec, float w) {
    const float d = __fsub_rn(g, r);
    return DECODE ? __fmaf_rn(w, d, dec) : __fmul_rn(w, d);
}

__device__ __forceinline__ void nesterov(float acc, float& th, float& mm, float lr, float mu) {
    const float m1 = __fmaf_rn(mu, mm, acc);
    const float gg = __fmaf_rn(mu, m1, acc);
    th = __fmaf_rn(-lr, gg, th);
    mm = m1;
}

template <bool DECODE, bool FINAL>
__global__ void __launch_bounds__(kThreads) k_ring_hop(RingArgs a) {
    __shared__ float scb[kNB];
    const int tid = threadIdx.x;
    int cur_t = -1;
    for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
        const int64_t base = c * kChunk;
        const int64_t cend = min(base + static_cast<int64_t>(kChunk), a.n);
        for (int t = tensor_containing(a.off, a.T, base); t < a.T; ++t) {
            const int64_t o0 = __ldg(a.off + t), o1 = __ldg(a.off + t + 1);
            if (o0 >= cend) break;
            const int64_t pa = o0 > base ? o0 : base;
            const int64_t pb = o1 < cend ? o1 : cend;
            if (pa >= pb) continue;
            if (DECODE && t != cur_t) {
                __syncthreads();
                scb[tid] = __ldg(a.cb + static_cast<int64_t>(t) * kNB + tid);
                __syncthreads();
                cur_t = t;
            }
            if (pa == base && pb == base + kChunk) {
                const float4* g4 = reinterpret_cast<const float4*>(a.g + base);
                const float4* r4 = reinterpret_cast<const float4*>(a.r + base);
                const uint32_t* c4 = reinterpret_cast<const uint32_t*>(a.codes + base);
#pragma unroll 2
                for (int j = 0; j < kGroups; ++j) {
                    const int gi = tid + j * kThreads;
                    float4 gv = FINAL ? g4[gi] : __ldg(g4 + gi);  // the last hop writes theta_g
                    const float4 rv = __ldcs(r4 + gi);
                    float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
                    if (DECODE) {
                        const uint32_t cw = __ldcs(c4 + gi);
                        e0 = scb[cw & 255u];
                        e1 = scb[(cw >> 8) & 255u];
                        e2 = scb[(cw >> 16) & 255u];
                        e3 = scb[cw >> 24];
                    }
                    const float v0 = hop_value<DECODE>(gv.x, rv.x, e0, a.w);
                    const float v1 = hop_value<DECODE>(gv.y, rv.y, e1, a.w);
                    const float v2 = hop_value<DECODE>(gv.z, rv.z, e2, a.w);
                    const float v3 = hop_value<DECODE>(gv.w, rv.w, e3, a.w);
                    if (FINAL) {
                        float4* m4 = reinterpret_cast<float4*>(a.m + base);
                        float4 mv = m4[gi];
                        nesterov(v0, gv.x, mv.x, a.lr, a.mu);
                        nesterov(v1, gv.y, mv.y, a.lr, a.mu);
                        nesterov(v2, gv.z, mv.z, a.lr, a.mu);
                        nesterov(v3, gv.w, mv.w, a.lr, a.mu);
                        reinterpret_cast<float4*>(a.g + base)[gi] = gv;
                        m4[gi] = mv;
                        if (a.dbar)
                            reinterpret_cast<float4*>(a.dbar + base)[gi] = make_float4(v0, v1, v2, v3);
                    } else {
                        reinterpret_cast<float4*>(a.P + base)[gi] = make_float4(v0, v1, v2, v3);
                    }
                }
            } else {
                for (int64_t i = pa + tid; i < pb; i += kThreads) {
                    float gv = a.g[i];
                    const float dec = DECODE ? scb[a.codes[i]] : 0.f;
                    const float v = hop_value<DECODE>(gv, a.r[i], dec, a.w);
                    if (FINAL) {
                        float mm = a.m[i];
                        nesterov(v, gv, mm, a.lr, a.mu);
                        a.g[i] = gv;
                        a.m[i] = mm;
                        if (a.dbar) a.dbar[i] = v;
                    } else {
                        a.P[i] = v;
                    }
                }
            }
        }
    }
}

template <bool DECODE, bool FINAL>
int launch_hop(const RingArgs& a, cudaStream_t s) {
    const void* k = reinterpret_cast<const void*>(k_ring_hop<DECODE, FINAL>);
    const int grid = grid_for(k, kThreads, 0, a.n_chunks);
    k_ring_hop<DECODE, FINAL><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

struct RingLayout {
    size_t stats_ws, quant_ws, stats_arr, cb, part, codes;
    size_t off_quant_ws, off_stats_arr, off_cb, off_part, off_codes, total;
};

int ring_layout(const dl_fragment* frag, RingLayout* L) {
    HostFrag f;
    const int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    L->stats_ws = align256(dl_stats_workspace_bytes(frag, 1));
    L->quant_ws = align256(dl_quantize_workspace_bytes(frag, 1));
    L->stats_arr = align256(sizeof(dl_stats) * static_cast<size_t>(f.T > 0 ? f.T : 1));
    L->cb = align256(sizeof(float) * kNB * static_cast<size_t>(f.T > 0 ? f.T : 1));
    L->part = align256(sizeof(float) * static_cast<size_t>(f.n));
    L->codes = align256(static_cast<size_t>(f.n));
    size_t o = L->stats_ws;  // the stats workspace first: its status word is ours
    L->off_quant_ws = o;
    o += L->quant_ws;
    L->off_stats_arr = o;
    o += L->stats_arr;
    L->off_cb = o;
    o += L->cb;
    L->off_part = o;
    o += L->part;
    L->off_codes = o;
    o += L->codes;
    L->total = o;
    return DL_OK;
}

}  // namespace
}  // namespace dl

using namespace dl;

extern "C" size_t dl_ring_workspace_bytes(const dl_fragment* frag) {
    RingLayout L;
    if (ring_layout(frag, &L) != DL_OK) return 0;
    return L.total;
}

extern "C" int dl_ring_outer_step(float* theta_g, float* momentum, const float* const* theta_k,
                                  int32_t K, const dl_fragment* frag, const float* weights,
                                  const uint8_t* present, int32_t min_quorum, double clip_sigmas,
                                  float lr, float mu, float* delta_bar_out, void* d_workspace,
                                  size_t workspace_bytes, void* stream) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    if (K <= 0 || K > DL_MAX_LEARNERS || !theta_k || !(clip_sigmas > 0.0) ||
        !(clip_sigmas < 1e300))
        return DL_ERR_ARG;

    // ring order and weights: the present learners ascending, w normalised
    // over them in fp64 and rounded to fp32 (as for the merge)
    int idx[DL_MAX_LEARNERS];
    float w_hat[DL_MAX_LEARNERS];
    int S = 0;
    double total = 0.0;
    for (int k = 0; k < K; ++k) {
        if (present && !present[k]) continue;
        const double w = weights ? static_cast<double>(weights[k]) : 1.0;
        if (!(w >= 0.0) || !isfinite(w)) return DL_ERR_ARG;
        total += w;
        idx[S++] = k;
    }
    if (S < (min_quorum > 1 ? min_quorum : 1)) return DL_ERR_QUORUM;
    if (!(total > 0.0)) return DL_ERR_ARG;
    for (int s = 0; s < S; ++s) {
        const double w = weights ? static_cast<double>(weights[idx[s]]) : 1.0;
        w_hat[s] = static_cast<float>(w / total);
    }
    if (f.n == 0) return DL_OK;
    if (!theta_g || !momentum) return DL_ERR_ARG;
    if (!aligned16(theta_g) || !aligned16(momentum) ||
        (delta_bar_out && !aligned16(delta_bar_out)))
        return DL_ERR_ALIGN;
    for (int s = 0; s < S; ++s) {
        if (!theta_k[idx[s]]) return DL_ERR_ARG;
        if (!aligned16(theta_k[idx[s]])) return DL_ERR_ALIGN;
    }
    RingLayout L;
    if ((st = ring_layout(frag, &L)) != DL_OK) return st;
    if (!d_workspace || workspace_bytes < L.total) return DL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0) return DL_ERR_ALIGN;

    char* ws = static_cast<char*>(d_workspace);
    dl_stats* stats = reinterpret_cast<dl_stats*>(ws + L.off_stats_arr);
    float* cb = reinterpret_cast<float*>(ws + L.off_cb);
    uint8_t* codes = reinterpret_cast<uint8_t*>(ws + L.off_codes);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);

    RingArgs a;
    memset(&a, 0, sizeof(a));
    a.g = theta_g;
    a.m = momentum;
    a.P = reinterpret_cast<float*>(ws + L.off_part);
    a.codes = codes;
    a.cb = cb;
    a.off = f.d_offsets;
    a.dbar = delta_bar_out;
    a.n = f.n;
    a.n_chunks = n_chunks_of(f.n);
    a.T = f.T;
    a.lr = lr;
    a.mu = mu;

    a.r = theta_k[idx[0]];
    a.w = w_hat[0];
    st = S == 1 ? launch_hop<false, true>(a, strm) : launch_hop<false, false>(a, strm);
    for (int s = 1; s < S && st == DL_OK; ++s) {
        // send: quantise the partial sum P itself (values mode)
        const float* P = a.P;
        st = dl_pseudograd_stats(P, nullptr, 1, frag, clip_sigmas, stats, ws, L.stats_ws, strm);
        if (st != DL_OK) break;
        uint8_t* cp[1] = {codes};
        st = dl_quantize(P, nullptr, 1, frag, stats, cp, cb, nullptr, ws + L.off_quant_ws,
                         L.quant_ws, strm);
        if (st != DL_OK) break;
        // receive: decode and add this learner's weighted pseudo-gradient
        a.r = theta_k[idx[s]];
        a.w = w_hat[s];
        st = s == S - 1 ? launch_hop<true, true>(a, strm) : launch_hop<true, false>(a, strm);
    }
    return st;
}
