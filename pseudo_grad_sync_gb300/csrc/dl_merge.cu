// Dequantise, merge over the present learners in fp32 and apply the outer
// Nesterov step in place (INTELLECT-1 notes, section 3.2 steps 6-7 and
// section 4.2; Decoupled DiLoCo note, fault-tolerance items 1 and 3).
//
// k_merge_q<NPM, RDA> persistent blocks over 8192-element chunks (block b takes
//                 chunks b, b + grid, ...: all blocks stay in one region of
//                 the arrays, which measured faster than contiguous runs).
//                 The codebooks
//                 of the present learners for the current tensor sit in
//                 shared memory (NPM x 1 KB at most); per 4-element group a
//                 thread issues one 32-bit code load per present learner plus
//                 128-bit loads of theta and m, decodes through the shared
//                 codebooks, accumulates fmaf(w_k, value, acc) over present k
//                 in ascending order, and stores theta and m back with
//                 128-bit stores. Each byte of codes, theta and m crosses HBM
//                 once.
// k_merge_tma<NPM, TILE, STAGES, MINB, RDA>  the same merge with theta, m and the
//                 codes staged through shared memory by bulk copies (producer
//                 warp, bounded waits); instances for up to 4, 8, 16 and 32
//                 present learners, each sized to keep 2 blocks per SM; used
//                 for the mean merge and the RDA merge whatever the number of
//                 learners, bitwise equal to k_merge_q (which
//                 DL_MERGE_UNSTAGED=1 selects, for tests).
// k_merge_u       the unquantised variant: values are the fp32 Delta_k read
//                 from the learner replicas.
//
// Radial-Directional Averaging (Decoupled DiLoCo note, architecture item 4:
// the outer gradients' norms and directions are averaged apart; the page has
// no formula, the reading is stated with dl_rda_merge_outer_step). Per tensor:
// k_rda_norms     one block per tensor: each present learner's norm from its
//                 codebook and bucket counts (fp64), the weighted mean norm r
//                 and the direction coefficients w_k / n_k;
// k_rda_u         one pass over the codes (each block over a contiguous run of
//                 chunks, so it rescales codebooks rarely): ||u||^2 of
//                 u = sum_k (w_k/n_k) v_k,
//                 one fp64 partial per warp and (chunk, tensor) piece, in
//                 slots (chunk + tensor) * 8 + warp (unique, so no clearing
//                 and a fixed order);
// k_rda_coef      one block per tensor: fixed-order sum of its partials, then
//                 c_k = (w_k / n_k) r / ||u|| per learner;
// k_merge_q<NPM, true> then decodes through codebooks scaled by c_k and adds
//                 the values in fp32 in ascending k.
#include <math.h>
#include <stdlib.h>

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
    const float* rda_c;  // RDA: [np][T] codebook scales (else unused)
    uint32_t* status;    // staged merge: workspace status word (bounded waits)
};

__device__ __forceinline__ void outer_update(float acc, float& th, float& mm, float lr, float mu) {
    const float m1 = __fmaf_rn(mu, mm, acc);
    const float gg = __fmaf_rn(mu, m1, acc);
    th = __fmaf_rn(-lr, gg, th);
    mm = m1;
}

template <int NPM, bool RDA>
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
                for (int i = tid; i < np * kNB; i += kThreads) {
                    float v = __ldg(a.cb + (static_cast<int64_t>(a.kidx[i >> 8]) * a.T + t) * kNB + (i & (kNB - 1)));
                    if (RDA) v = __fmul_rn(__ldg(a.rda_c + (i >> 8) * a.T + t), v);
                    scb[i] = v;
                }
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
                                if (RDA) {  // values already scaled
                                    a0 = __fadd_rn(a0, cbs[w4 & 255u]);
                                    a1 = __fadd_rn(a1, cbs[(w4 >> 8) & 255u]);
                                    a2 = __fadd_rn(a2, cbs[(w4 >> 16) & 255u]);
                                    a3 = __fadd_rn(a3, cbs[w4 >> 24]);
                                } else {
                                    a0 = __fmaf_rn(ws, cbs[w4 & 255u], a0);
                                    a1 = __fmaf_rn(ws, cbs[(w4 >> 8) & 255u], a1);
                                    a2 = __fmaf_rn(ws, cbs[(w4 >> 16) & 255u], a2);
                                    a3 = __fmaf_rn(ws, cbs[w4 >> 24], a3);
                                }
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
                    for (int s = 0; s < np; ++s) {
                        const float v = scb[s * kNB + a.cp[s][i]];
                        acc = RDA ? __fadd_rn(acc, v) : __fmaf_rn(a.w[s], v, acc);
                    }
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

// Staged variant of k_merge_q for up to NPM present learners: a producer warp
// streams tiles of theta, m and every present learner's codes into a
// STAGES-deep shared-memory ring with bulk copies (bounded waits; an abort
// stops the pipeline as dl_common.cuh describes), 8 consumer warps decode from
// shared memory and store theta and m back with 128-bit stores. Per element
// the arithmetic is k_merge_q's, in the same order, so the results are
// bitwise the same. Dynamic shared memory: the present learners' codebooks
// [np][256] f32, then STAGES stages of theta [TILE] f32 | m [TILE] f32 |
// codes [np][TILE] u8, all sized by the actual np.
template <int NPM, int TILE, int STAGES, int MINB, bool RDA>
__global__ void __launch_bounds__(kPipeThreads, MINB) k_merge_tma(MergeArgs a) {
    static_assert(TILE % (4 * kThreads) == 0, "whole float4 groups per consumer thread");
    extern __shared__ __align__(128) unsigned char mbuf[];
    __shared__ PipeBarriers pb;
    const int tid = threadIdx.x, lane = tid & 31;
    const int np = a.np;
    float* scb = reinterpret_cast<float*>(mbuf);
    unsigned char* stages = mbuf + np * kNB * 4;
    const int stage_bytes = TILE * (8 + np);
    pipe_init<STAGES>(&pb);

    if ((tid >> 5) == kConsumerWarps) {  // producer warp
        if (lane == 0) {
            uint32_t it = 0;
            bool live = true;
            for (int64_t c = blockIdx.x; live && c < a.n_chunks; c += gridDim.x) {
                const int64_t base = c * kChunk;
                const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
                for (int o = 0; o < cn; o += TILE) {
                    if (!producer_acquire<STAGES>(&pb, it, a.status)) {
                        live = false;
                        break;
                    }
                    const int s = static_cast<int>(it % STAGES);
                    const int tn = min(TILE, cn - o);
                    const uint32_t fbytes = static_cast<uint32_t>(tn >> 2) * 16u;  // whole float4s
                    const uint32_t cbytes = static_cast<uint32_t>(tn >> 4) * 16u;  // whole 16-byte runs
                    unsigned char* st = stages + s * stage_bytes;
                    fence_proxy_async();
                    mbar_arrive_expect_tx(&pb.full[s], 2u * fbytes + static_cast<uint32_t>(np) * cbytes);
                    const int64_t e0 = base + o;
                    if (fbytes) {
                        bulk_copy_g2s(st, a.g + e0, fbytes, &pb.full[s]);
                        bulk_copy_g2s(st + TILE * 4, a.m + e0, fbytes, &pb.full[s]);
                    }
                    if (cbytes)
                        for (int k = 0; k < np; ++k)
                            bulk_copy_g2s(st + TILE * 8 + k * TILE, a.cp[k] + e0, cbytes, &pb.full[s]);
                    ++it;
                }
            }
            producer_drain<STAGES>(&pb, it, a.status);
        }
        return;
    }

    int cur_t = -1;
    uint32_t it = 0;
    TensorCursor tc;
    for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
        const int64_t base = c * kChunk;
        const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
        for (int o = 0; o < cn; o += TILE, ++it) {
            const int s = static_cast<int>(it % STAGES);
            const int64_t tb = base + o;
            const int tn = min(TILE, cn - o);
            const int fvec = tn & ~3, cvec = tn & ~15;  // elements staged
            const int64_t tend = tb + tn;
            const bool ok = consumer_wait<STAGES>(&pb, it, a.status);
            const unsigned char* st = stages + s * stage_bytes;
            const float* sg = reinterpret_cast<const float*>(st);
            const float* sm = reinterpret_cast<const float*>(st + TILE * 4);
            const unsigned char* sc = st + TILE * 8;
            // the tensors of the tile, from the one holding its first element
            for (int t = tc.seek(a.off, a.T, tb); t < a.T; ++t) {
                tc.load(a.off, t);
                const int64_t o0 = tc.o0, o1 = tc.o1;
                const int64_t pa = o0 > tb ? o0 : tb;
                const int64_t pe = o1 < tend ? o1 : tend;
                if (pa >= pe) continue;  // empty tensor
                if (t != cur_t) {  // consumer-uniform
                    consumer_sync();
                    for (int i = tid; i < np * kNB; i += kThreads) {
                        float v = __ldg(a.cb + (static_cast<int64_t>(a.kidx[i >> 8]) * a.T + t) * kNB +
                                        (i & (kNB - 1)));
                        if (RDA) v = __fmul_rn(__ldg(a.rda_c + (i >> 8) * a.T + t), v);
                        scb[i] = v;
                    }
                    consumer_sync();
                    cur_t = t;
                }
                if (!ok) {  // aborted: the stage is not read
                    if (o1 >= tend) break;
                    continue;
                }
                if (pa == tb && pe == tb + TILE) {
#pragma unroll
                    for (int q = 0; q < TILE / 4 / kThreads; ++q) {
                        const int gi = tid + q * kThreads;  // float4 group in the tile
                        float4 th = reinterpret_cast<const float4*>(sg)[gi];
                        float4 mm = reinterpret_cast<const float4*>(sm)[gi];
                        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                        for (int k = 0; k < NPM; ++k) {
                            if (k < np) {
                                const uint32_t w4 = reinterpret_cast<const uint32_t*>(sc + k * TILE)[gi];
                                const float* cbs = scb + k * kNB;
                                const float ws = a.w[k];
                                if (RDA) {  // values already scaled
                                    a0 = __fadd_rn(a0, cbs[w4 & 255u]);
                                    a1 = __fadd_rn(a1, cbs[(w4 >> 8) & 255u]);
                                    a2 = __fadd_rn(a2, cbs[(w4 >> 16) & 255u]);
                                    a3 = __fadd_rn(a3, cbs[w4 >> 24]);
                                } else {
                                    a0 = __fmaf_rn(ws, cbs[w4 & 255u], a0);
                                    a1 = __fmaf_rn(ws, cbs[(w4 >> 8) & 255u], a1);
                                    a2 = __fmaf_rn(ws, cbs[(w4 >> 16) & 255u], a2);
                                    a3 = __fmaf_rn(ws, cbs[w4 >> 24], a3);
                                }
                            }
                        }
                        outer_update(a0, th.x, mm.x, a.lr, a.mu);
                        outer_update(a1, th.y, mm.y, a.lr, a.mu);
                        outer_update(a2, th.z, mm.z, a.lr, a.mu);
                        outer_update(a3, th.w, mm.w, a.lr, a.mu);
                        reinterpret_cast<float4*>(a.g + tb)[gi] = th;
                        reinterpret_cast<float4*>(a.m + tb)[gi] = mm;
                        if (a.dbar) reinterpret_cast<float4*>(a.dbar + tb)[gi] = make_float4(a0, a1, a2, a3);
                    }
                } else {
                    for (int64_t e = pa + tid; e < pe; e += kThreads) {
                        const int l = static_cast<int>(e - tb);
                        float th = l < fvec ? sg[l] : a.g[e];
                        float mm = l < fvec ? sm[l] : a.m[e];
                        float acc = 0.f;
                        for (int k = 0; k < np; ++k) {
                            const uint32_t code = l < cvec ? sc[k * TILE + l] : a.cp[k][e];
                            const float v = scb[k * kNB + code];
                            acc = RDA ? __fadd_rn(acc, v) : __fmaf_rn(a.w[k], v, acc);
                        }
                        outer_update(acc, th, mm, a.lr, a.mu);
                        a.g[e] = th;
                        a.m[e] = mm;
                        if (a.dbar) a.dbar[e] = acc;
                    }
                }
                if (o1 >= tend) break;  // the next tensor starts at or after the tile's end
            }
            consumer_release<STAGES>(&pb, it, ok);
        }
    }
}

// Tile, stage count and blocks per SM of the staged merge by the number of
// present learners it is instantiated for: blocks of 288 threads (2 or 3 per SM), each with
// at most ~112 KB of dynamic shared memory (codebooks + stages).
template <int NPM> struct MergeShape;
template <> struct MergeShape<4> { static constexpr int kTile = 2048, kStages = 3, kMinB = 2; };   //  76 KB
template <> struct MergeShape<8> { static constexpr int kTile = 2048, kStages = 2, kMinB = 3; };   //  72 KB
template <> struct MergeShape<16> { static constexpr int kTile = 2048, kStages = 2, kMinB = 2; };  // 112 KB
template <> struct MergeShape<32> { static constexpr int kTile = 1024, kStages = 2, kMinB = 2; };  // 112 KB

template <int NPM, bool RDA>
int launch_tma(const MergeArgs& a, cudaStream_t s) {
    constexpr int TILE = MergeShape<NPM>::kTile, STAGES = MergeShape<NPM>::kStages;
    constexpr int MINB = MergeShape<NPM>::kMinB;
    const void* k = reinterpret_cast<const void*>(k_merge_tma<NPM, TILE, STAGES, MINB, RDA>);
    const size_t smem = static_cast<size_t>(a.np) * kNB * 4 +
                        static_cast<size_t>(STAGES) * TILE * (8 + a.np);
    int st = cuda_status(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem)));
    if (st != DL_OK) return st;
    const int grid = grid_for(k, kPipeThreads, smem, a.n_chunks);
    k_merge_tma<NPM, TILE, STAGES, MINB, RDA><<<grid, kPipeThreads, smem, s>>>(a);
    return launch_status();
}

// The staged merge for any number of present learners.
template <bool RDA>
int launch_staged(const MergeArgs& a, cudaStream_t s) {
    if (a.np <= 4) return launch_tma<4, RDA>(a, s);
    if (a.np <= 8) return launch_tma<8, RDA>(a, s);
    if (a.np <= 16) return launch_tma<16, RDA>(a, s);
    return launch_tma<32, RDA>(a, s);
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

template <int NPM, bool RDA>
int launch_q(const MergeArgs& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * kNB * a.np;
    const int grid =
        grid_for(reinterpret_cast<const void*>(k_merge_q<NPM, RDA>), kThreads, smem, a.n_chunks);
    k_merge_q<NPM, RDA><<<grid, kThreads, smem, s>>>(a);
    return launch_status();
}

// DL_MERGE_UNSTAGED=1 (environment) selects k_merge_q instead of the staged
// merge; the two are bitwise equal, and tests use this to compare them.
bool merge_unstaged() {
    const char* v = getenv("DL_MERGE_UNSTAGED");
    return v && v[0] == '1';
}

template <bool RDA>
int launch_quantised(const MergeArgs& a, cudaStream_t s) {
    if (a.np <= 4) return launch_q<4, RDA>(a, s);
    if (a.np <= 8) return launch_q<8, RDA>(a, s);
    if (a.np <= 16) return launch_q<16, RDA>(a, s);
    return launch_q<32, RDA>(a, s);
}

// ---------------------------------------------------------------------------
// RDA kernels

struct RdaArgs {
    const float* cb;          // [K][T][256]
    const uint32_t* counts;   // [K][T][256]
    const uint8_t* cp[DL_MAX_LEARNERS];
    int kidx[DL_MAX_LEARNERS];
    float w[DL_MAX_LEARNERS];
    int np;
    int T;
    const int64_t* off;
    int64_t n;
    int64_t n_chunks;
    double* coef;  // [np][T]  w_k / n_k
    double* r;     // [T]      sum_k w_k n_k
    double* part;  // [(n_chunks + T) * 8] ||u||^2 per piece and warp
    float* c;      // [np][T]  final codebook scales
};

// one block per tensor; warp w takes learners w, w + 8, ...
__global__ void __launch_bounds__(kThreads) k_rda_norms(RdaArgs a) {
    __shared__ double nrm_s[DL_MAX_LEARNERS];
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int s = warp; s < a.np; s += kWarps) {
        const int64_t base = (static_cast<int64_t>(a.kidx[s]) * a.T + t) * kNB;
        double ss = 0.0;
#pragma unroll
        for (int j = 0; j < kNB / 32; ++j) {
            const int b = lane * (kNB / 32) + j;
            const double v = static_cast<double>(__ldg(a.cb + base + b));
            ss = fma(static_cast<double>(__ldg(a.counts + base + b)) * v, v, ss);
        }
        for (int sh = 16; sh; sh >>= 1) ss += __shfl_xor_sync(kFull, ss, sh);
        const double nrm = sqrt(ss);
        if (lane == 0) {
            nrm_s[s] = nrm;
            a.coef[s * a.T + t] = nrm > 0.0 ? static_cast<double>(a.w[s]) / nrm : 0.0;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double rr = 0.0;
        for (int s = 0; s < a.np; ++s) rr = fma(static_cast<double>(a.w[s]), nrm_s[s], rr);
        a.r[t] = rr;
    }
}

template <int NPM>
__global__ void __launch_bounds__(kThreads) k_rda_u(RdaArgs a) {
    extern __shared__ float scu[];  // [np][256] codebooks scaled by w_k / n_k
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int np = a.np;
    int cur_t = -1;
    int64_t c0, c1;
    block_chunks(a.n_chunks, c0, c1);
    for (int64_t c = c0; c < c1; ++c) {
        const int64_t base = c * kChunk;
        const int64_t cend = min(base + static_cast<int64_t>(kChunk), a.n);
        for (int t = tensor_containing(a.off, a.T, base); t < a.T; ++t) {
            const int64_t o0 = __ldg(a.off + t), o1 = __ldg(a.off + t + 1);
            if (o0 >= cend) break;
            const int64_t pa = o0 > base ? o0 : base;
            const int64_t pb = o1 < cend ? o1 : cend;
            if (pa >= pb) continue;
            if (t != cur_t) {
                __syncthreads();
                for (int i = tid; i < np * kNB; i += kThreads) {
                    const int s = i >> 8;
                    const float v = __ldg(a.cb + (static_cast<int64_t>(a.kidx[s]) * a.T + t) * kNB + (i & (kNB - 1)));
                    scu[i] = __fmul_rn(static_cast<float>(a.coef[s * a.T + t]), v);
                }
                __syncthreads();
                cur_t = t;
            }
            // squares of x = sum_k coef_k v_k, four at a time in fp32, summed per
            // thread as a float-float pair (exact two-sums; fp64 is scarce on
            // this part), then in fp64 once per piece
            float ah = 0.f, al = 0.f;
            if (pa == base && pb == base + kChunk) {  // 32-bit code words, 4 elements each
#pragma unroll 1
                for (int j = 0; j < kGroups; j += 2) {
                    uint32_t cw[2][NPM];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int s = 0; s < NPM; ++s)
                            if (s < np)
                                cw[u][s] = __ldcs(reinterpret_cast<const unsigned int*>(a.cp[s] + base) +
                                                  tid + (j + u) * kThreads);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
                        for (int s = 0; s < NPM; ++s) {
                            if (s < np) {
                                const uint32_t w4 = cw[u][s];
                                const float* cs = scu + s * kNB;
                                x0 = __fadd_rn(x0, cs[w4 & 255u]);
                                x1 = __fadd_rn(x1, cs[(w4 >> 8) & 255u]);
                                x2 = __fadd_rn(x2, cs[(w4 >> 16) & 255u]);
                                x3 = __fadd_rn(x3, cs[w4 >> 24]);
                            }
                        }
                        ff_add(ah, al,
                               __fmaf_rn(x3, x3, __fmaf_rn(x2, x2, __fmaf_rn(x1, x1, __fmul_rn(x0, x0)))));
                    }
                }
            } else {
                for (int64_t i = pa + tid; i < pb; i += kThreads) {
                    float x = 0.f;
                    for (int s = 0; s < np; ++s) x = __fadd_rn(x, scu[s * kNB + a.cp[s][i]]);
                    ff_add(ah, al, __fmul_rn(x, x));
                }
            }
            double acc = static_cast<double>(ah) + static_cast<double>(al);
            for (int sh = 16; sh; sh >>= 1) acc += __shfl_xor_sync(kFull, acc, sh);
            if (lane == 0) a.part[(c + t) * kWarps + warp] = acc;
        }
    }
}

template <int NPM>
int launch_rda_u(const RdaArgs& r, cudaStream_t s) {
    const size_t smem = sizeof(float) * kNB * r.np;
    const int grid = grid_for(reinterpret_cast<const void*>(k_rda_u<NPM>), kThreads, smem, r.n_chunks);
    k_rda_u<NPM><<<grid, kThreads, smem, s>>>(r);
    return launch_status();
}

// one block per tensor: its pieces' per-warp partials summed in a fixed order
__global__ void __launch_bounds__(kThreads) k_rda_coef(RdaArgs a) {
    __shared__ double red[kThreads];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int64_t o0 = a.off[t], o1 = a.off[t + 1];
    double uu = 0.0;
    if (o1 > o0) {
        const int64_t s0 = (o0 / kChunk + t) * kWarps, s1 = ((o1 - 1) / kChunk + t + 1) * kWarps;
        for (int64_t i = s0 + tid; i < s1; i += kThreads) uu += a.part[i];
    }
    red[tid] = uu;
    __syncthreads();
    for (int h = kThreads / 2; h > 0; h >>= 1) {
        if (tid < h) red[tid] += red[tid + h];
        __syncthreads();
    }
    uu = red[0];
    const double scale = uu > 0.0 ? a.r[t] / sqrt(uu) : 0.0;
    for (int s = tid; s < a.np; s += kThreads)
        a.c[s * a.T + t] = static_cast<float>(a.coef[s * a.T + t] * scale);
}

}  // namespace
}  // namespace dl

using namespace dl;

namespace dl {
namespace {

// Validation shared by the merges: quorum and weight normalisation over the
// present learners (fp64, then fp32), pointers and alignment; fills `a`.
// Returns DL_OK with a.n == 0 for an empty fragment (nothing to launch).
int prepare_merge(MergeArgs& a, float* theta_g, float* momentum, const uint8_t* const* codes,
                  const float* d_codebook, const float* const* theta_k, int32_t K,
                  const dl_fragment* frag, const float* weights, const uint8_t* present,
                  int32_t min_quorum, float lr, float mu, float* delta_bar_out) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    if (K <= 0 || K > DL_MAX_LEARNERS) return DL_ERR_ARG;
    const bool quant = codes != nullptr;
    if (!quant && !theta_k) return DL_ERR_ARG;

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
    a.T = f.T;
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
    a.lr = lr;
    a.mu = mu;
    return DL_OK;
}

struct RdaLayout {
    size_t coef, r, part, c, total;
};

RdaLayout rda_layout(const HostFrag& f, int K) {
    RdaLayout L;
    L.coef = kWsHeader;
    L.r = L.coef + align256(sizeof(double) * static_cast<size_t>(K) * f.T);
    L.part = L.r + align256(sizeof(double) * static_cast<size_t>(f.T));
    L.c = L.part + align256(sizeof(double) * kWarps * static_cast<size_t>(n_chunks_of(f.n) + f.T));
    L.total = L.c + align256(sizeof(float) * static_cast<size_t>(K) * f.T);
    return L;
}

}  // namespace
}  // namespace dl

// The library's own device status word: bounded waits of calls that take no
// workspace (the staged merge of dl_merge_outer_step) report here, and
// dl_read_device_status(NULL, ...) reads it. One per device; its address on
// the current device is looked up on every call (a cached address would go
// stale after a device reset or a new primary context).
static __device__ uint32_t g_library_status;

namespace dl {
int library_status_word(uint32_t** out) {
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_library_status) != cudaSuccess || !q) return DL_ERR_CUDA;
    *out = static_cast<uint32_t*>(q);
    return DL_OK;
}

int merge_outer_step_status(float* theta_g, float* momentum, const uint8_t* const* codes,
                            const float* d_codebook, const float* const* theta_k, int32_t K,
                            const dl_fragment* frag, const float* weights, const uint8_t* present,
                            int32_t min_quorum, float lr, float mu, float* delta_bar_out,
                            uint32_t* status, void* stream) {
    MergeArgs a;
    const int st = prepare_merge(a, theta_g, momentum, codes, d_codebook, theta_k, K, frag,
                                 weights, present, min_quorum, lr, mu, delta_bar_out);
    if (st != DL_OK || a.n == 0) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (codes == nullptr) {
        const int grid = grid_for(reinterpret_cast<const void*>(k_merge_u), kThreads, 0,
                                  ((a.n >> 2) + kThreads - 1) / kThreads + 1);
        k_merge_u<<<grid, kThreads, 0, s>>>(a);
        return launch_status();
    }
    if (merge_unstaged()) return launch_quantised<false>(a, s);
    int st2 = DL_OK;
    if (!status) st2 = library_status_word(&status);
    if (st2 != DL_OK) return st2;
    a.status = status;
    return launch_staged<false>(a, s);
}
}  // namespace dl

extern "C" int dl_merge_outer_step(float* theta_g, float* momentum, const uint8_t* const* codes,
                                   const float* d_codebook, const float* const* theta_k, int32_t K,
                                   const dl_fragment* frag, const float* weights,
                                   const uint8_t* present, int32_t min_quorum, float lr, float mu,
                                   float* delta_bar_out, void* stream) {
    return merge_outer_step_status(theta_g, momentum, codes, d_codebook, theta_k, K, frag,
                                   weights, present, min_quorum, lr, mu, delta_bar_out, nullptr,
                                   stream);
}

extern "C" size_t dl_rda_workspace_bytes(const dl_fragment* frag, int32_t K) {
    HostFrag f;
    if (check_fragment(frag, &f) != DL_OK || K <= 0 || K > DL_MAX_LEARNERS) return 0;
    return rda_layout(f, K).total;
}

extern "C" int dl_rda_merge_outer_step(float* theta_g, float* momentum,
                                       const uint8_t* const* codes, const float* d_codebook,
                                       const uint32_t* d_counts, int32_t K,
                                       const dl_fragment* frag, const float* weights,
                                       const uint8_t* present, int32_t min_quorum, float lr,
                                       float mu, float* delta_bar_out, void* d_workspace,
                                       size_t workspace_bytes, void* stream) {
    if (!codes) return DL_ERR_ARG;
    MergeArgs a;
    int st = prepare_merge(a, theta_g, momentum, codes, d_codebook, nullptr, K, frag, weights,
                           present, min_quorum, lr, mu, delta_bar_out);
    if (st != DL_OK) return st;
    HostFrag f;
    check_fragment(frag, &f);
    const RdaLayout L = rda_layout(f, K);
    if (a.n == 0) return DL_OK;
    if (!d_counts) return DL_ERR_ARG;
    if (!aligned16(d_counts)) return DL_ERR_ALIGN;
    if (!d_workspace || workspace_bytes < L.total) return DL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0) return DL_ERR_ALIGN;

    char* ws = static_cast<char*>(d_workspace);
    RdaArgs r;
    memset(&r, 0, sizeof(r));
    r.cb = d_codebook;
    r.counts = d_counts;
    r.np = a.np;
    for (int s = 0; s < a.np; ++s) {
        r.cp[s] = a.cp[s];
        r.kidx[s] = a.kidx[s];
        r.w[s] = a.w[s];
    }
    r.T = f.T;
    r.off = f.d_offsets;
    r.n = f.n;
    r.n_chunks = a.n_chunks;
    r.coef = reinterpret_cast<double*>(ws + L.coef);
    r.r = reinterpret_cast<double*>(ws + L.r);
    r.part = reinterpret_cast<double*>(ws + L.part);
    r.c = reinterpret_cast<float*>(ws + L.c);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    k_rda_norms<<<f.T, kThreads, 0, s>>>(r);
    if ((st = launch_status()) != DL_OK) return st;
    st = a.np <= 4 ? launch_rda_u<4>(r, s)
         : a.np <= 8 ? launch_rda_u<8>(r, s)
         : a.np <= 16 ? launch_rda_u<16>(r, s) : launch_rda_u<32>(r, s);
    if (st != DL_OK) return st;
    k_rda_coef<<<f.T, kThreads, 0, s>>>(r);
    if ((st = launch_status()) != DL_OK) return st;
    a.rda_c = r.c;
    if (merge_unstaged()) return launch_quantised<true>(a, s);
    a.status = reinterpret_cast<uint32_t*>(ws);  // staged, as the mean merge
    return launch_staged<true>(a, s);
}
