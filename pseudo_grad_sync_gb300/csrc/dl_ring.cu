// Ring accumulation with re-quantisation at every hop, then the outer Nesterov
// step (INTELLECT-1 notes, section 4.2: what a node receives is dequantised,
// added to in fp32, and quantised again before it is sent on; section 4.1
// for the quantiser; section 3.2 step 7 for the outer step).
//
// On one GPU the ring's S present learners, in increasing order, are visited
// one after another; the partial sum P lives in the workspace:
//   hop 0:        P = w_0 * Delta_0
//   hop s >= 1:   quantise P (dl_quantize in values mode: the vector
//                 quantised is P itself), then P = fmaf(w_s, Delta_s, cb[code])
//   last hop:     instead of storing P, apply the outer Nesterov step with
//                 D = P (and write D out if asked).
// k_ring_hop<DECODE, FINAL, STATS> does one hop's element work: persistent
// blocks, each over one contiguous run of 8192-element chunks (so a block
// meets few tensors), the previous codebook of the current tensor in shared
// memory, 128-bit loads and stores, 32-bit code loads. A
// hop whose P is quantised next (STATS) also accumulates P's per-tensor
// statistics as it writes P, with the exact scheme of the statistics kernel
// (float-float sums of y = P - c and of y^2 on a power-of-two offset, fp64
// for values outside the fast range): the quantiser's statistics then cost
// no extra pass over P. Rings of two or more learners run their hops staged
// through shared memory by bulk copies (k_ring_mid_tma for the hops that
// write P, k_ring_last_tma for the last one); k_ring_hop, the same work with
// plain loads, runs the one-learner ring. Each block entering a tensor
// computes its shift c
// (one warp, from the hop's own formula at the tensor's first 64 elements,
// with the statistics kernel's rule; every block gets the same value), and
// stats_finish turns the partials into mu, sigma, lo, hi.
#include <math.h>
#include <string.h>

#include "dl_stats_acc.cuh"

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
    float* shift;           // [T] shifts of the new P, for the finalisation (STATS)
    Partial* part;          // [T][gridDim.x] partial sums of the new P (STATS)
    int64_t n;
    int64_t n_chunks;
    int T;
    float w;
    float lr;
    float mu;
    uint32_t* status;       // workspace status word (staged last hop)
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

// The shift of tensor t of the P this hop writes, computed by one warp from
// P at the tensor's first min(N, 64) elements (the hop's formula, bit for
// bit) with the statistics kernel's rule; every lane returns it. Each block
// entering the tensor computes the same value.
template <bool DECODE>
__device__ __forceinline__ float ring_shift(const RingArgs& a, int t, int64_t o, int64_t N) {
    const int lane = threadIdx.x & 31;
    const int m = N < 64 ? static_cast<int>(N) : 64;
    const bool h0 = lane < m, h1 = lane + 32 < m;
    const float* cbt = a.cb + static_cast<int64_t>(t) * kNB;
    double v[2] = {0.0, 0.0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (!(h ? h1 : h0)) continue;
        const int64_t i = o + lane + 32 * h;
        const float dec = DECODE ? __ldg(cbt + __ldg(a.codes + i)) : 0.f;
        v[h] = static_cast<double>(hop_value<DECODE>(__ldg(a.g + i), __ldg(a.r + i), dec, a.w));
    }
    return warp_shift(v[0], v[1], h0, h1, m);
}

// Statistics of four P values of one group (the fast path when all four are
// in range, else fp64 for the four)
__device__ __forceinline__ void acc_group(Acc& acc, float v0, float v1, float v2, float v3,
                                          float csh, bool small) {
    const float y0 = __fsub_rn(v0, csh), y1 = __fsub_rn(v1, csh);
    const float y2 = __fsub_rn(v2, csh), y3 = __fsub_rn(v3, csh);
    const float mx = absmax_nan(y3, absmax_nan(y2, absmax_nan(y1, absmax_nan(y0, 0.f))));
    if (!small && fast_range(mx)) {
        if (mx > acc.yt) rebase(acc, mx);
        ff_add(acc.s1h, acc.s1l, __fadd_rn(__fadd_rn(y0, y1), __fadd_rn(y2, y3)));
        sq_add(acc.s2h, acc.s2l, y0);
        sq_add(acc.s2h, acc.s2l, y1);
        sq_add(acc.s2h, acc.s2l, y2);
        sq_add(acc.s2h, acc.s2l, y3);
    } else {
        acc.side = true;
        side_add(v0, csh, acc.s1d, acc.s2d, acc.bad);
        side_add(v1, csh, acc.s1d, acc.s2d, acc.bad);
        side_add(v2, csh, acc.s1d, acc.s2d, acc.bad);
        side_add(v3, csh, acc.s1d, acc.s2d, acc.bad);
    }
}

template <bool DECODE, bool FINAL, bool STATS>
__global__ void __launch_bounds__(kThreads) k_ring_hop(RingArgs a) {
    static_assert(!(FINAL && STATS), "the last hop's sum is not quantised");
    __shared__ float scb[kNB];
    __shared__ float s_shift;
    __shared__ float red_ff[kWarps][4];
    __shared__ double red_side[kWarps][2];
    __shared__ int red_bad[kWarps];
    const int tid = threadIdx.x;
    int cur_t = -1;
    float csh = 0.f;
    bool small = false;
    Acc acc;
    acc.reset();
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
                if (STATS && cur_t >= 0)
                    flush_partial(acc, a.part + static_cast<int64_t>(cur_t) * gridDim.x + blockIdx.x,
                                  red_ff, red_side, red_bad);
                if (DECODE || STATS) {
                    __syncthreads();  // every read of the previous tensor's scb / s_shift is done
                    if (DECODE) scb[tid] = __ldg(a.cb + static_cast<int64_t>(t) * kNB + tid);
                    if (STATS && tid < 32) {
                        const float cs = ring_shift<DECODE>(a, t, o0, o1 - o0);
                        if (tid == 0) {
                            s_shift = cs;
                            if (pa == o0) a.shift[t] = cs;  // the one block holding element o0
                        }
                    }
                    __syncthreads();
                }
                if (STATS) {
                    acc.reset();
                    csh = s_shift;
                    small = (o1 - o0) < kSmallTensor;
                }
                cur_t = t;
            }
            if (pa == base && pb == base + kChunk) {
                const float4* g4 = reinterpret_cast<const float4*>(a.g + base);
                const float4* r4 = reinterpret_cast<const float4*>(a.r + base);
                const uint32_t* c4 = reinterpret_cast<const uint32_t*>(a.codes + base);
#pragma unroll 4
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
                        if (STATS) {
                            acc_group(acc, v0, v1, v2, v3, csh, small);
                            if ((j & 3) == 3) renorm(acc.s2h, acc.s2l);
                        }
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
                        if (STATS) {
                            const float y = __fsub_rn(v, csh);
                            const float ay = fabsf(y);
                            if (!small && fast_range(ay)) {
                                if (ay > acc.yt)
                                    rebase(acc, ay);
                                ff_add(acc.s1h, acc.s1l, y);
                                sq_add(acc.s2h, acc.s2l, y);
                            } else {
                                acc.side = true;
                                side_add(v, csh, acc.s1d, acc.s2d, acc.bad);
                            }
                        }
                    }
                }
                if (STATS) renorm(acc.s2h, acc.s2l);
            }
        }
    }
    if (STATS && cur_t >= 0)
        flush_partial(acc, a.part + static_cast<int64_t>(cur_t) * gridDim.x + blockIdx.x, red_ff,
                      red_side, red_bad);
}

// The last hop staged through shared memory: a producer warp streams
// 2048-element tiles of theta_g, the replica, m and the previous codes into a
// 3-stage ring with bulk copies (bounded waits), 8 consumer warps apply the
// hop and the outer step with k_ring_hop's arithmetic and store theta_g, m
// (and D) with 128-bit stores. Blocks take contiguous chunk runs.
constexpr int kRTile = 2048;
constexpr int kRStages = 3;
constexpr int kRStageBytes = kRTile * 13;  // theta_g, r, m (f32) + codes (u8)

__global__ void __launch_bounds__(kPipeThreads, 2) k_ring_last_tma(RingArgs a) {
    extern __shared__ __align__(128) unsigned char rbuf[];
    __shared__ float scb[kNB];
    __shared__ PipeBarriers pb;
    const int tid = threadIdx.x, lane = tid & 31;
    int64_t c0, c1;
    block_chunks(a.n_chunks, c0, c1);
    pipe_init<kRStages>(&pb);

    if ((tid >> 5) == kConsumerWarps) {  // producer warp
        if (lane == 0) {
            uint32_t it = 0;
            bool live = true;
            for (int64_t c = c0; live && c < c1; ++c) {
                const int64_t base = c * kChunk;
                const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
                for (int o = 0; o < cn; o += kRTile, ++it) {
                    if (!producer_acquire<kRStages>(&pb, it, a.status)) {
                        live = false;
                        break;
                    }
                    const int s = static_cast<int>(it % kRStages);
                    const int tn = min(kRTile, cn - o);
                    const uint32_t fbytes = static_cast<uint32_t>(tn >> 2) * 16u;
                    const uint32_t cbytes = static_cast<uint32_t>(tn >> 4) * 16u;
                    unsigned char* st = rbuf + s * kRStageBytes;
                    const int64_t e0 = base + o;
                    fence_proxy_async();
                    mbar_arrive_expect_tx(&pb.full[s], 3u * fbytes + cbytes);
                    if (fbytes) {
                        bulk_copy_g2s(st, a.g + e0, fbytes, &pb.full[s]);
                        bulk_copy_g2s(st + kRTile * 4, a.r + e0, fbytes, &pb.full[s]);
                        bulk_copy_g2s(st + kRTile * 8, a.m + e0, fbytes, &pb.full[s]);
                    }
                    if (cbytes) bulk_copy_g2s(st + kRTile * 12, a.codes + e0, cbytes, &pb.full[s]);
                }
            }
            producer_drain<kRStages>(&pb, it, a.status);
        }
        return;
    }

    int cur_t = -1;
    TensorCursor tc;
    uint32_t it = 0;
    for (int64_t c = c0; c < c1; ++c) {
        const int64_t base = c * kChunk;
        const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
        for (int o = 0; o < cn; o += kRTile, ++it) {
            const int s = static_cast<int>(it % kRStages);
            const int64_t tb = base + o;
            const int tn = min(kRTile, cn - o);
            const int fvec = tn & ~3, cvec = tn & ~15;
            const int64_t tend = tb + tn;
            const bool ok = consumer_wait<kRStages>(&pb, it, a.status);
            const unsigned char* st = rbuf + s * kRStageBytes;
            const float* sg = reinterpret_cast<const float*>(st);
            const float* sr = reinterpret_cast<const float*>(st + kRTile * 4);
            const float* sm = reinterpret_cast<const float*>(st + kRTile * 8);
            const unsigned char* sc = st + kRTile * 12;
            // the tensors of the tile, from the one holding its first element
            for (int t = tc.seek(a.off, a.T, tb); t < a.T; ++t) {
                tc.load(a.off, t);
                const int64_t o0 = tc.o0, o1 = tc.o1;
                const int64_t pa = o0 > tb ? o0 : tb;
                const int64_t pe = o1 < tend ? o1 : tend;
                if (pa >= pe) continue;  // empty tensor
                if (t != cur_t) {  // consumer-uniform
                    consumer_sync();
                    scb[tid] = __ldg(a.cb + static_cast<int64_t>(t) * kNB + tid);
                    consumer_sync();
                    cur_t = t;
                }
                if (!ok) {  // aborted: the stage is not read
                    if (o1 >= tend) break;
                    continue;
                }
                if (pa == tb && pe == tb + kRTile) {
#pragma unroll
                    for (int q = 0; q < kRTile / 4 / kThreads; ++q) {
                        const int gi = tid + q * kThreads;
                        float4 gv = reinterpret_cast<const float4*>(sg)[gi];
                        const float4 rv = reinterpret_cast<const float4*>(sr)[gi];
                        float4 mv = reinterpret_cast<const float4*>(sm)[gi];
                        const uint32_t cw = reinterpret_cast<const uint32_t*>(sc)[gi];
                        const float v0 = hop_value<true>(gv.x, rv.x, scb[cw & 255u], a.w);
                        const float v1 = hop_value<true>(gv.y, rv.y, scb[(cw >> 8) & 255u], a.w);
                        const float v2 = hop_value<true>(gv.z, rv.z, scb[(cw >> 16) & 255u], a.w);
                        const float v3 = hop_value<true>(gv.w, rv.w, scb[cw >> 24], a.w);
                        nesterov(v0, gv.x, mv.x, a.lr, a.mu);
                        nesterov(v1, gv.y, mv.y, a.lr, a.mu);
                        nesterov(v2, gv.z, mv.z, a.lr, a.mu);
                        nesterov(v3, gv.w, mv.w, a.lr, a.mu);
                        reinterpret_cast<float4*>(a.g + tb)[gi] = gv;
                        reinterpret_cast<float4*>(a.m + tb)[gi] = mv;
                        if (a.dbar)
                            reinterpret_cast<float4*>(a.dbar + tb)[gi] = make_float4(v0, v1, v2, v3);
                    }
                } else {
                    for (int64_t e = pa + tid; e < pe; e += kThreads) {
                        const int l = static_cast<int>(e - tb);
                        float gv = l < fvec ? sg[l] : a.g[e];
                        const float rv = l < fvec ? sr[l] : a.r[e];
                        float mm = l < fvec ? sm[l] : a.m[e];
                        const uint32_t code = l < cvec ? sc[l] : a.codes[e];
                        const float v = hop_value<true>(gv, rv, scb[code], a.w);
                        nesterov(v, gv, mm, a.lr, a.mu);
                        a.g[e] = gv;
                        a.m[e] = mm;
                        if (a.dbar) a.dbar[e] = v;
                    }
                }
                if (o1 >= tend) break;  // the next tensor starts at or after the tile's end
            }
            consumer_release<kRStages>(&pb, it, ok);
        }
    }
}

int launch_last_tma(const RingArgs& a, cudaStream_t s) {
    const void* k = reinterpret_cast<const void*>(k_ring_last_tma);
    const size_t smem = static_cast<size_t>(kRStages) * kRStageBytes;
    int st = cuda_status(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem)));
    if (st != DL_OK) return st;
    const int grid = grid_for(k, kPipeThreads, smem, a.n_chunks);
    k_ring_last_tma<<<grid, kPipeThreads, smem, s>>>(a);
    return launch_status();
}

// A hop before the last one, staged the same way: tiles of theta_g, the
// replica and (DECODE) the previous codes in a 3-stage ring; the consumers
// write P and accumulate its statistics as k_ring_hop does (the same scheme,
// per (block, tensor) partials, the block's shift from the tensor's first 64
// elements).
constexpr int kRMidStageBytes = kRTile * 9;  // theta_g, r (f32) + codes (u8)

template <bool DECODE>
__global__ void __launch_bounds__(kPipeThreads, 2) k_ring_mid_tma(RingArgs a) {
    extern __shared__ __align__(128) unsigned char rbuf[];
    __shared__ float scb[kNB];
    __shared__ float s_shift;
    __shared__ float red_ff[kWarps][4];
    __shared__ double red_side[kWarps][2];
    __shared__ int red_bad[kWarps];
    __shared__ PipeBarriers pb;
    const int tid = threadIdx.x, lane = tid & 31;
    int64_t c0, c1;
    block_chunks(a.n_chunks, c0, c1);
    pipe_init<kRStages>(&pb);

    if ((tid >> 5) == kConsumerWarps) {  // producer warp
        if (lane == 0) {
            uint32_t it = 0;
            bool live = true;
            for (int64_t c = c0; live && c < c1; ++c) {
                const int64_t base = c * kChunk;
                const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
                for (int o = 0; o < cn; o += kRTile, ++it) {
                    if (!producer_acquire<kRStages>(&pb, it, a.status)) {
                        live = false;
                        break;
                    }
                    const int s = static_cast<int>(it % kRStages);
                    const int tn = min(kRTile, cn - o);
                    const uint32_t fbytes = static_cast<uint32_t>(tn >> 2) * 16u;
                    const uint32_t cbytes = DECODE ? static_cast<uint32_t>(tn >> 4) * 16u : 0u;
                    unsigned char* st = rbuf + s * kRMidStageBytes;
                    const int64_t e0 = base + o;
                    fence_proxy_async();
                    mbar_arrive_expect_tx(&pb.full[s], 2u * fbytes + cbytes);
                    if (fbytes) {
                        bulk_copy_g2s(st, a.g + e0, fbytes, &pb.full[s]);
                        bulk_copy_g2s(st + kRTile * 4, a.r + e0, fbytes, &pb.full[s]);
                    }
                    if (cbytes) bulk_copy_g2s(st + kRTile * 8, a.codes + e0, cbytes, &pb.full[s]);
                }
            }
            producer_drain<kRStages>(&pb, it, a.status);
        }
        return;
    }

    int cur_t = -1;
    TensorCursor tc;
    float csh = 0.f;
    bool small = false;
    Acc acc;
    acc.reset();
    uint32_t it = 0;
    for (int64_t c = c0; c < c1; ++c) {
        const int64_t base = c * kChunk;
        const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
        for (int o = 0; o < cn; o += kRTile, ++it) {
            const int s = static_cast<int>(it % kRStages);
            const int64_t tb = base + o;
            const int tn = min(kRTile, cn - o);
            const int fvec = tn & ~3, cvec = tn & ~15;
            const int64_t tend = tb + tn;
            const bool ok = consumer_wait<kRStages>(&pb, it, a.status);
            const unsigned char* st = rbuf + s * kRMidStageBytes;
            const float* sg = reinterpret_cast<const float*>(st);
            const float* sr = reinterpret_cast<const float*>(st + kRTile * 4);
            const unsigned char* sc = st + kRTile * 8;
            // the tensors of the tile, from the one holding its first element
            for (int t = tc.seek(a.off, a.T, tb); t < a.T; ++t) {
                tc.load(a.off, t);
                const int64_t o0 = tc.o0, o1 = tc.o1;
                const int64_t pa = o0 > tb ? o0 : tb;
                const int64_t pe = o1 < tend ? o1 : tend;
                if (pa >= pe) continue;  // empty tensor
                if (t != cur_t) {  // consumer-uniform
                    if (cur_t >= 0)
                        flush_partial(acc, a.part + static_cast<int64_t>(cur_t) * gridDim.x + blockIdx.x,
                                      red_ff, red_side, red_bad);
                    consumer_sync();  // every read of the previous tensor's scb / s_shift is done
                    if (DECODE) scb[tid] = __ldg(a.cb + static_cast<int64_t>(t) * kNB + tid);
                    if (tid < 32) {
                        const float cs = ring_shift<DECODE>(a, t, o0, o1 - o0);
                        if (tid == 0) {
                            s_shift = cs;
                            if (pa == o0) a.shift[t] = cs;  // the one block holding element o0
                        }
                    }
                    consumer_sync();
                    acc.reset();
                    csh = s_shift;
                    small = (o1 - o0) < kSmallTensor;
                    cur_t = t;
                }
                if (!ok) {  // aborted: the stage is not read
                    if (o1 >= tend) break;
                    continue;
                }
                if (pa == tb && pe == tb + kRTile) {
#pragma unroll
                    for (int q = 0; q < kRTile / 4 / kThreads; ++q) {
                        const int gi = tid + q * kThreads;
                        const float4 gv = reinterpret_cast<const float4*>(sg)[gi];
                        const float4 rv = reinterpret_cast<const float4*>(sr)[gi];
                        float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
                        if (DECODE) {
                            const uint32_t cw = reinterpret_cast<const uint32_t*>(sc)[gi];
                            e0 = scb[cw & 255u];
                            e1 = scb[(cw >> 8) & 255u];
                            e2 = scb[(cw >> 16) & 255u];
                            e3 = scb[cw >> 24];
                        }
                        const float v0 = hop_value<DECODE>(gv.x, rv.x, e0, a.w);
                        const float v1 = hop_value<DECODE>(gv.y, rv.y, e1, a.w);
                        const float v2 = hop_value<DECODE>(gv.z, rv.z, e2, a.w);
                        const float v3 = hop_value<DECODE>(gv.w, rv.w, e3, a.w);
                        reinterpret_cast<float4*>(a.P + tb)[gi] = make_float4(v0, v1, v2, v3);
                        acc_group(acc, v0, v1, v2, v3, csh, small);
                    }
                    renorm(acc.s2h, acc.s2l);
                } else {
                    for (int64_t e = pa + tid; e < pe; e += kThreads) {
                        const int l = static_cast<int>(e - tb);
                        const float gv = l < fvec ? sg[l] : a.g[e];
                        const float rv = l < fvec ? sr[l] : a.r[e];
                        const float dec = DECODE ? scb[l < cvec ? sc[l] : a.codes[e]] : 0.f;
                        const float v = hop_value<DECODE>(gv, rv, dec, a.w);
                        a.P[e] = v;
                        const float y = __fsub_rn(v, csh);
                        const float ay = fabsf(y);
                        if (!small && fast_range(ay)) {
                            if (ay > acc.yt) rebase(acc, ay);
                            ff_add(acc.s1h, acc.s1l, y);
                            sq_add(acc.s2h, acc.s2l, y);
                        } else {
                            acc.side = true;
                            side_add(v, csh, acc.s1d, acc.s2d, acc.bad);
                        }
                    }
                    renorm(acc.s2h, acc.s2l);
                }
                if (o1 >= tend) break;  // the next tensor starts at or after the tile's end
            }
            consumer_release<kRStages>(&pb, it, ok);
        }
    }
    if (cur_t >= 0)
        flush_partial(acc, a.part + static_cast<int64_t>(cur_t) * gridDim.x + blockIdx.x, red_ff,
                      red_side, red_bad);
}

template <bool DECODE>
int launch_mid_tma(const RingArgs& a, cudaStream_t s, int* grid_out) {
    const void* k = reinterpret_cast<const void*>(k_ring_mid_tma<DECODE>);
    const size_t smem = static_cast<size_t>(kRStages) * kRMidStageBytes;
    int st = cuda_status(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem)));
    if (st != DL_OK) return st;
    int grid = grid_for(k, kPipeThreads, smem, a.n_chunks);
    if (grid > kMaxBlocksTotal) grid = kMaxBlocksTotal;  // partial slots per tensor
    const size_t part_bytes = sizeof(Partial) * static_cast<size_t>(a.T) * grid;
    if ((st = cuda_status(cudaMemsetAsync(a.part, 0, part_bytes, s))) != DL_OK) return st;
    k_ring_mid_tma<DECODE><<<grid, kPipeThreads, smem, s>>>(a);
    *grid_out = grid;
    return launch_status();
}

// One hop on s. With STATS, the partials of the new P are zeroed first, and
// *grid_out is the hop's grid (the partials' J).
template <bool DECODE, bool FINAL, bool STATS>
int launch_hop(const RingArgs& a, cudaStream_t s, int* grid_out = nullptr) {
    const void* k = reinterpret_cast<const void*>(k_ring_hop<DECODE, FINAL, STATS>);
    int grid = grid_for(k, kThreads, 0, a.n_chunks);
    if (grid > kMaxBlocksTotal) grid = kMaxBlocksTotal;  // partial slots per tensor
    int st;
    if (STATS) {
        const size_t part_bytes = sizeof(Partial) * static_cast<size_t>(a.T) * grid;
        if ((st = cuda_status(cudaMemsetAsync(a.part, 0, part_bytes, s))) != DL_OK) return st;
    }
    k_ring_hop<DECODE, FINAL, STATS><<<grid, kThreads, 0, s>>>(a);
    if (grid_out) *grid_out = grid;
    return launch_status();
}

// Workspace: status header | shifts [T] | partials [T][kMaxBlocksTotal] |
// quantiser scratch | statistics [T] | codebook [T][256] | P [n] | codes [n]
struct RingLayout {
    size_t shift, part, quant_ws, stats_arr, cb, P, codes;
    size_t off_shift, off_part, off_quant_ws, off_stats_arr, off_cb, off_P, off_codes, total;
};

int ring_layout(const dl_fragment* frag, RingLayout* L) {
    HostFrag f;
    const int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    const size_t T1 = static_cast<size_t>(f.T > 0 ? f.T : 1);
    L->shift = align256(sizeof(float) * T1);
    L->part = align256(sizeof(Partial) * T1 * kMaxBlocksTotal);
    L->quant_ws = align256(dl_quantize_workspace_bytes(frag, 1));
    L->stats_arr = align256(sizeof(dl_stats) * T1);
    L->cb = align256(sizeof(float) * kNB * T1);
    L->P = align256(sizeof(float) * static_cast<size_t>(f.n));
    L->codes = align256(static_cast<size_t>(f.n));
    size_t o = kWsHeader;  // the status word first
    L->off_shift = o;
    o += L->shift;
    L->off_part = o;
    o += L->part;
    L->off_quant_ws = o;
    o += L->quant_ws;
    L->off_stats_arr = o;
    o += L->stats_arr;
    L->off_cb = o;
    o += L->cb;
    L->off_P = o;
    o += L->P;
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
                                  float lr, float mu, float* delta_bar_out,
                                  dl_stats* hop_stats_out, void* d_workspace,
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
    if (hop_stats_out && (reinterpret_cast<uintptr_t>(hop_stats_out) & 7u) != 0)
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
    float* cb = reinterpret_cast<float*>(ws + L.off_cb);
    uint8_t* codes = reinterpret_cast<uint8_t*>(ws + L.off_codes);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);

    RingArgs a;
    memset(&a, 0, sizeof(a));
    a.g = theta_g;
    a.m = momentum;
    a.P = reinterpret_cast<float*>(ws + L.off_P);
    a.codes = codes;
    a.cb = cb;
    a.off = f.d_offsets;
    a.dbar = delta_bar_out;
    a.shift = reinterpret_cast<float*>(ws + L.off_shift);
    a.part = reinterpret_cast<Partial*>(ws + L.off_part);
    a.n = f.n;
    a.n_chunks = n_chunks_of(f.n);
    a.T = f.T;
    a.lr = lr;
    a.mu = mu;
    a.status = reinterpret_cast<uint32_t*>(ws);

    // statistics of P_s (quantised at hop s + 1): the caller's row s, or the
    // workspace's
    auto stats_of = [&](int s) {
        return hop_stats_out ? hop_stats_out + static_cast<int64_t>(s) * f.T
                             : reinterpret_cast<dl_stats*>(ws + L.off_stats_arr);
    };
    a.r = theta_k[idx[0]];
    a.w = w_hat[0];
    int J = 0;
    if (S == 1) return launch_hop<false, true, false>(a, strm);
    if ((st = launch_mid_tma<false>(a, strm, &J)) != DL_OK) return st;
    for (int s = 1; s < S; ++s) {
        // send: finish P_{s-1}'s statistics and quantise it (values mode)
        dl_stats* sp = stats_of(s - 1);
        if ((st = stats_finish(a.off, f.T, 1, J, a.shift, a.part, clip_sigmas, sp, strm)) != DL_OK)
            return st;
        uint8_t* cp[1] = {codes};
        st = dl_quantize(a.P, nullptr, 1, frag, sp, cp, cb, nullptr, ws + L.off_quant_ws,
                         L.quant_ws, strm);
        if (st != DL_OK) return st;
        // receive: decode and add this learner's weighted pseudo-gradient
        a.r = theta_k[idx[s]];
        a.w = w_hat[s];
        st = s == S - 1 ? launch_last_tma(a, strm)
                        : launch_mid_tma<true>(a, strm, &J);
        if (st != DL_OK) return st;
    }
    return DL_OK;
}
