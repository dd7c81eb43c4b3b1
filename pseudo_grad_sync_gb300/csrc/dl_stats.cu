// Per-(learner, tensor) pseudo-gradient statistics (INTELLECT-1 notes,
// section 4.1 step 1: one mu and one sigma per tensor; step 2: the clip
// range mu +- 6 sigma).
//
// One launch (after a small memset of the per-(k, t) tickets):
//  k_stats     learner-major persistent grid: block b serves learner
//              k = b % K and the j-th of J contiguous runs of 8192-element
//              chunks (j = b / K), so the K blocks that read one chunk of
//              theta_g run together and theta_g comes from HBM once, then
//              from L2. A producer warp streams the (theta_g, theta_k) tiles
//              into a 2-stage shared-memory ring with bulk copies (TMA
//              engine), 8 consumer warps compute from shared memory; 3
//              blocks per SM. Entering a tensor, one warp derives the tensor's shift c from
//              its first min(N, 64) values of Delta (their fp64 mean,
//              snapped to a power-of-two grid below their spread, rounded to
//              fp32); every block entering the tensor derives the same c.
//              The sums are of y = Delta - c, which keeps the one-pass
//              variance free of cancellation when |mu| >> sigma; the
//              snapping keeps the fp32 rounding of y unbiased (a shift with
//              low-order bits below ulp(y) biases every rounding the same
//              way). Per thread: fp32 sums over groups of four, folded into
//              float-float (hi + lo) sums that persist across all chunks of
//              a tensor, squares two at a time with fp32x2 instructions on a
//              power-of-two offset with exact error terms (so no rounding of
//              a square biases the sum); the block reduces them
//              (float-float butterfly, fp64 over the 8 warps) when it leaves
//              the tensor, into partial slot (k, t, run), and counts it on
//              the (k, t) ticket. The block whose count completes the
//              tensor's runs sums the partials in a fixed order (fp64) and
//              writes mu = c + S1/N, sigma^2 = S2/N - (S1/N)^2 (population),
//              lo/hi = mu -+ clip sigma. Tensors shorter than 4096 elements
//              and groups of rare huge, tiny (squares would leave the fp32
//              normal range) or non-finite values take an fp64 path.
// The result is deterministic: every sum has a fixed order.
#include "dl_stats_acc.cuh"

namespace dl {
namespace {

struct StatsArgs {
    const float* g;
    const float* r[DL_MAX_LEARNERS];
    const int64_t* off;
    float* shift;
    Partial* part;
    unsigned int* ticket;  // [K*T] partials written so far (zeroed per call)
    dl_stats* out;
    uint32_t* status;
    int64_t n;
    int64_t n_chunks;
    int T;
    int K;
    int J;    // chunk runs per learner: the partition of the sums, fixed per fragment and K
    int RPB;  // runs per block: block j takes runs j * RPB .. (j + 1) * RPB - 1
    double clip;
};

constexpr int kTile = 4096;  // elements per pipeline tile

// One thread's share of a full tile: kGroupsPerTile groups of four values.
// All y are formed first so that one range check and at most one rebase
// cover the whole share; a share with a value outside the fast range (or a
// non-finite one) goes to the fp64 path as a whole.
constexpr int kGroupsPerTile = kTile / 4 / kThreads;

template <bool VALUES>
__device__ __forceinline__ void add_tile(Acc& acc, const float* tg, const float* tr, int tid,
                                         float csh) {
    // y = fl(fl(g - r) - c) two at a time: fma(r, -1, g) and fl(d + (-c)) round
    // exactly as the scalar subtractions
    const float2 m1 = make_float2(-1.f, -1.f);
    const float2 nc = make_float2(-csh, -csh);
    float2 y[kGroupsPerTile][2];  // (y0, y1), (y2, y3) of each group of four
    float mx = 0.f;
#pragma unroll
    for (int q = 0; q < kGroupsPerTile; ++q) {
        const float4 gv = reinterpret_cast<const float4*>(tg)[tid + q * kThreads];
        const float4 rv = VALUES ? make_float4(0.f, 0.f, 0.f, 0.f)
                                 : reinterpret_cast<const float4*>(tr)[tid + q * kThreads];
        y[q][0] = __fadd2_rn(__ffma2_rn(make_float2(rv.x, rv.y), m1, make_float2(gv.x, gv.y)), nc);
        y[q][1] = __fadd2_rn(__ffma2_rn(make_float2(rv.z, rv.w), m1, make_float2(gv.z, gv.w)), nc);
        mx = absmax_nan(y[q][0].x, mx);
        mx = absmax_nan(y[q][0].y, mx);
        mx = absmax_nan(y[q][1].x, mx);
        mx = absmax_nan(y[q][1].y, mx);
    }
    // squares, their error terms and H0 stay normal and finite for
    // 2^-50 <= |y| <= 2^48 (smaller values lose at most 2^-149); mx is NaN if
    // any y is, so the fp64 path (which counts it) takes that share
    if (fast_range(mx)) {
        if (mx > acc.yt) rebase(acc, mx);
#pragma unroll
        for (int q = 0; q < kGroupsPerTile; ++q) {
            // (y0 + y1, y2 + y3) in one paired add, then their sum
            const float2 p = __fadd2_rn(make_float2(y[q][0].x, y[q][1].x),
                                        make_float2(y[q][0].y, y[q][1].y));
            ff_add(acc.s1h, acc.s1l, __fadd_rn(p.x, p.y));
            sq_add2(acc, y[q][0]);
            sq_add2(acc, y[q][1]);
        }
        renorm(acc.s2h, acc.s2l);
        renorm(acc.s2hb, acc.s2lb);
    } else {
        acc.side = true;
#pragma unroll 1
        for (int q = 0; q < kGroupsPerTile; ++q) {
            const float4 gv = reinterpret_cast<const float4*>(tg)[tid + q * kThreads];
            const float4 rv = VALUES ? make_float4(0.f, 0.f, 0.f, 0.f)
                                     : reinterpret_cast<const float4*>(tr)[tid + q * kThreads];
            side_add(__fsub_rn(gv.x, rv.x), csh, acc.s1d, acc.s2d, acc.bad);
            side_add(__fsub_rn(gv.y, rv.y), csh, acc.s1d, acc.s2d, acc.bad);
            side_add(__fsub_rn(gv.z, rv.z), csh, acc.s1d, acc.s2d, acc.bad);
            side_add(__fsub_rn(gv.w, rv.w), csh, acc.s1d, acc.s2d, acc.bad);
        }
    }
}

// The run (of the J runs of chunks) that holds chunk c: the largest r with
// floor(n_chunks r / J) <= c. Every run has a chunk (J <= n_chunks).
__device__ __forceinline__ int64_t run_of_chunk(int64_t c, int64_t n_chunks, int J) {
    return ((c + 1) * J - 1) / n_chunks;
}

// The statistics of (k, t) from the partials of every run that meets tensor t,
// summed by one warp in a fixed order (lane-strided, then a fixed butterfly):
// mu = shift + S1/N, sigma^2 = S2/N - (S1/N)^2 (population), lo/hi = mu -+
// clip sigma. Called by the warp of the block that wrote the last partial;
// the partials and the shift come from other blocks, so they are read past L1.
__device__ void finish_stats(const StatsArgs& a, int k, int t, int64_t o0, int64_t o1) {
    const int lane = threadIdx.x & 31;
    const int64_t N = o1 - o0;
    const int64_t rf = run_of_chunk(o0 / kChunk, a.n_chunks, a.J);
    const int64_t rl = run_of_chunk((o1 - 1) / kChunk, a.n_chunks, a.J);
    const Partial* pk = a.part + (static_cast<int64_t>(k) * a.T + t) * a.J;
    double s1 = 0.0, s2 = 0.0;
    long long bad = 0;
    for (int64_t r = rf + lane; r <= rl; r += 32) {
        s1 += __ldcg(&pk[r].s1);
        s2 += __ldcg(&pk[r].s2);
        bad += __ldcg(&pk[r].bad);
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
    } else {
        const double inv = 1.0 / static_cast<double>(N);
        const double mrel = s1 * inv;
        double var = s2 * inv - mrel * mrel;
        if (!(var > 0.0)) var = 0.0;
        const double sigma = sqrt(var);
        const double mu = static_cast<double>(__ldcg(a.shift + static_cast<int64_t>(k) * a.T + t)) + mrel;
        st.mean = mu;
        st.std = sigma;
        st.lo = mu - a.clip * sigma;
        st.hi = mu + a.clip * sigma;
    }
    a.out[static_cast<int64_t>(k) * a.T + t] = st;
}

// Learner-major persistent grid: block b serves learner k = b % K and the
// j-th contiguous run of chunks, j = b / K. The K blocks that read the same chunk
// of theta_g run side by side, so theta_g crosses HBM once and is served to
// the other K - 1 from L2. A producer warp streams the (theta_g, theta_k)
// tiles of those chunks into a STAGES-deep shared-memory ring with bulk
// copies; 8 consumer warps compute from shared memory. Each consumer thread
// keeps its sums across every tile of a tensor; the consumers reduce them
// only when they move to another tensor. Launched as 2 stages with 3 blocks
// per SM.
// VALUES: values mode (no replica; Delta is theta_g itself, K = 1)
template <int STAGES, int MINB, bool VALUES>
__global__ void __launch_bounds__(kPipeThreads, MINB) k_stats(StatsArgs a) {
    constexpr int kStages = STAGES;
    extern __shared__ __align__(128) float smem[];  // [kStages][kTile] theta_g, then theta_k
    float* sg = smem;
    float* sr = smem + kStages * kTile;
    __shared__ PipeBarriers pb;
    __shared__ float red_ff[kConsumerWarps][4];
    __shared__ double red_side[kConsumerWarps][2];
    __shared__ int red_bad[kConsumerWarps];
    __shared__ float s_shift;
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31;
    const int k = blockIdx.x % a.K, j = blockIdx.x / a.K;
    // chunk run r is [n_chunks r / J, n_chunks (r + 1) / J); block j takes the
    // adjacent runs [j RPB, (j + 1) RPB) (the same for every learner, so the K
    // blocks of one j read the same theta_g chunks). The sums restart at every
    // run, so the result depends on J only, not on how many blocks share them.
    const int r_lo = j * a.RPB, r_hi = min(a.J, r_lo + a.RPB);
    const float* __restrict__ rk = a.r[k];
    const float* __restrict__ g = a.g;
    pipe_init<kStages>(&pb);

    if ((tid >> 5) == kConsumerWarps) {  // producer warp
        if (lane == 0) {
            uint32_t it = 0;
            bool live = true;
            for (int r = r_lo; live && r < r_hi; ++r) {
                const int64_t c_hi = a.n_chunks * (r + 1) / a.J;
                for (int64_t c = a.n_chunks * r / a.J; live && c < c_hi; ++c) {
                    const int64_t base = c * kChunk;
                    const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
                    for (int o = 0; live && o < cn; o += kTile) {
                        live = pipe_produce<kTile, kStages>(&pb, sg, sr, g, rk, base + o,
                                                            min(kTile, cn - o), it, a.status);
                        if (live) ++it;
                    }
                }
            }
            producer_drain<kStages>(&pb, it, a.status);
        }
        return;
    }

    // the first block of each learner writes the statistics of its empty
    // tensors (no partial ever reaches them)
    if (j == 0)
        for (int t = tid; t < a.T; t += kThreads)
            if (__ldg(a.off + t + 1) == __ldg(a.off + t)) {
                dl_stats st;
                st.count = st.nonfinite = 0;
                st.mean = st.std = st.lo = st.hi = 0.0;
                a.out[static_cast<int64_t>(k) * a.T + t] = st;
            }

    // The partial of (k, t) for run r goes to its slot; thread 0 then counts
    // it on the (k, t) ticket, and the block that completes the count
    // finishes the statistics of (k, t).
    auto flush_and_count = [&](Acc& acc_, Partial* slot, int t) {
        flush_partial(acc_, slot, red_ff, red_side, red_bad);
        const int64_t o0 = __ldg(a.off + t), o1 = __ldg(a.off + t + 1);
        if (tid == 0) {
            __threadfence();  // the partial (and any shift) before the count
            const int64_t expect = run_of_chunk((o1 - 1) / kChunk, a.n_chunks, a.J) -
                                   run_of_chunk(o0 / kChunk, a.n_chunks, a.J) + 1;
            const unsigned int done = atomicAdd(a.ticket + static_cast<int64_t>(k) * a.T + t, 1u) + 1u;
            s_last = static_cast<int64_t>(done) == expect;
        }
        consumer_sync();
        if (s_last && tid < 32) {
            __threadfence();
            finish_stats(a, k, t, o0, o1);
        }
    };

    TensorCursor cur;
    uint32_t it = 0;
    for (int r = r_lo; r < r_hi; ++r) {
        // slot (k, t, r) of this run's sums sits at part_k + t * J
        Partial* part_k = a.part + static_cast<int64_t>(k) * a.T * a.J + r;
        int cur_t = -1;
        float csh = 0.f;
        bool small = false;
        Acc acc;
        acc.reset();
        const int64_t c_lo = a.n_chunks * r / a.J, c_hi = a.n_chunks * (r + 1) / a.J;
        for (int64_t c = c_lo; c < c_hi; ++c) {
            const int64_t base = c * kChunk;
            const int cn = static_cast<int>(min(static_cast<int64_t>(kChunk), a.n - base));
            for (int o = 0; o < cn; o += kTile, ++it) {
                const int s = static_cast<int>(it % kStages);
                const int64_t tb = base + o;
                const int tn = min(kTile, cn - o);
                const int tvec = tn & ~3;  // elements staged in shared memory
                const int64_t tend = tb + tn;
                const bool ok = consumer_wait<kStages>(&pb, it, a.status);
                const float* tg = sg + s * kTile;
                const float* tr = sr + s * kTile;
                // the tensors of the tile, from the one holding its first element
                for (int t = cur.seek(a.off, a.T, tb); t < a.T; ++t) {
                    cur.load(a.off, t);
                    const int64_t o0 = cur.o0, o1 = cur.o1;
                    const int64_t pa = o0 > tb ? o0 : tb;
                    const int64_t pe = o1 < tend ? o1 : tend;
                    if (pa >= pe) continue;  // empty tensor
                    if (t != cur_t) {
                        if (cur_t >= 0) flush_and_count(acc, part_k + cur_t * a.J, cur_t);
                        // the shift of (k, t), from the tensor's first values:
                        // every block entering the tensor derives the same one
                        if (tid < 32) {
                            const int64_t N = o1 - o0;
                            const int m = N < 64 ? static_cast<int>(N) : 64;
                            const bool h0 = tid < m, h1 = tid + 32 < m;
                            const double v0 = h0 ? static_cast<double>(__fsub_rn(
                                                       __ldg(g + o0 + tid), VALUES ? 0.f : __ldg(rk + o0 + tid)))
                                                 : 0.0;
                            const double v1 = h1 ? static_cast<double>(__fsub_rn(
                                                       __ldg(g + o0 + tid + 32),
                                                       VALUES ? 0.f : __ldg(rk + o0 + tid + 32)))
                                                 : 0.0;
                            const float cs = warp_shift(v0, v1, h0, h1, m);
                            if (tid == 0) {
                                s_shift = cs;
                                if (pa == o0) a.shift[static_cast<int64_t>(k) * a.T + t] = cs;
                            }
                        }
                        consumer_sync();
                        cur_t = t;
                        csh = s_shift;
                        small = (o1 - o0) < kSmallTensor;
                        acc.reset();
                    }
                    if (!ok) {  // aborted: the stage is not read
                        if (o1 >= tend) break;
                        continue;
                    }
                    if (pa == tb && pe == tb + kTile && !small) {
                        add_tile<VALUES>(acc, tg, tr, tid, csh);
                    } else {
                        for (int64_t e = pa + tid; e < pe; e += kThreads) {
                            const int l = static_cast<int>(e - tb);
                            const float gv = l < tvec ? tg[l] : __ldg(g + e);
                            const float rv = VALUES ? 0.f : (l < tvec ? tr[l] : __ldg(rk + e));
                            const float d = __fsub_rn(gv, rv);
                            const float y = __fsub_rn(d, csh);
                            const float ay = fabsf(y);
                            if (!small && fast_range(ay)) {
                                if (ay > acc.yt)
                                    rebase(acc, ay);
                                ff_add(acc.s1h, acc.s1l, y);
                                sq_add(acc.s2h, acc.s2l, y);
                            } else {
                                acc.side = true;
                                side_add(d, csh, acc.s1d, acc.s2d, acc.bad);
                            }
                        }
                        renorm(acc.s2h, acc.s2l);
                    }
                    if (o1 >= tend) break;  // the next tensor starts at or after the tile's end
                }
                consumer_release<kStages>(&pb, it, ok);
            }
        }
        if (cur_t >= 0) flush_and_count(acc, part_k + cur_t * a.J, cur_t);
    }
}

struct FinArgs {
    const int64_t* off;
    const float* shift;
    const Partial* part;
    dl_stats* out;
    int T, K, J;
    double clip;
};

constexpr int kFinThreads = 128;

// One block per (k, t): thread i sums partials i, i + 128, ... in order, then
// a fixed butterfly per warp and the four warps in order.
__global__ void __launch_bounds__(kFinThreads) k_stats_fin(FinArgs a) {
    __shared__ double r1[kFinThreads / 32], r2[kFinThreads / 32];
    __shared__ long long rb[kFinThreads / 32];
    const int w = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = w % a.T;
    const int64_t N = a.off[t + 1] - a.off[t];
    double s1 = 0.0, s2 = 0.0;
    long long bad = 0;
    const Partial* pw = a.part + static_cast<int64_t>(w) * a.J;
    for (int jj = threadIdx.x; jj < a.J; jj += kFinThreads) {
        const Partial p = pw[jj];
        s1 += p.s1;
        s2 += p.s2;
        bad += p.bad;
    }
    for (int sh = 16; sh; sh >>= 1) {
        s1 += __shfl_xor_sync(kFull, s1, sh);
        s2 += __shfl_xor_sync(kFull, s2, sh);
        bad += __shfl_xor_sync(kFull, bad, sh);
    }
    if (lane == 0) {
        r1[warp] = s1;
        r2[warp] = s2;
        rb[warp] = bad;
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    s1 = r1[0];
    s2 = r2[0];
    bad = rb[0];
    for (int i = 1; i < kFinThreads / 32; ++i) {
        s1 += r1[i];
        s2 += r2[i];
        bad += rb[i];
    }
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

int max_blocks_per_learner(int K) { return kMaxBlocksTotal / K; }

}  // namespace

int stats_finish(const int64_t* d_off, int T, int K, int J, const float* shift,
                 const Partial* part, double clip, dl_stats* out, cudaStream_t s) {
    if (K * T == 0) return DL_OK;
    FinArgs f;
    f.off = d_off;
    f.shift = shift;
    f.part = part;
    f.out = out;
    f.T = T;
    f.K = K;
    f.J = J;
    f.clip = clip;
    k_stats_fin<<<K * T, kFinThreads, 0, s>>>(f);
    return launch_status();
}

}  // namespace dl

using namespace dl;

extern "C" size_t dl_stats_workspace_bytes(const dl_fragment* frag, int32_t K) {
    HostFrag f;
    if (check_fragment(frag, &f) != DL_OK || K <= 0 || K > DL_MAX_LEARNERS) return 0;
    // shifts and tickets per (k, t), then partials for K * T * J runs with
    // J <= kMaxBlocksTotal / K: sized as T * kMaxBlocksTotal so that the need
    // never decreases with K
    return kWsHeader + 2 * shift_bytes(K, f.T) +
           align256(sizeof(Partial) * static_cast<size_t>(f.T) * kMaxBlocksTotal);
}

namespace dl {
// The statistics call; with share_sms the grid has half as many blocks, each
// taking two chunk runs in turn, so that one block per SM leaves registers for
// two quantiser blocks: dl_outer_sync uses it for the statistics of the next
// fragment, which then share each SM with the quantiser of the current one
// instead of taking it whole. The runs (the partition of the sums) are the
// same either way, so the results are bitwise the same.
int pseudograd_stats_shared(const float* theta_g, const float* const* theta_k, int32_t K,
                            const dl_fragment* frag, double clip_sigmas, dl_stats* d_stats,
                            void* d_workspace, size_t workspace_bytes, void* stream,
                            bool share_sms) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    const bool values = theta_k == nullptr;  // Delta is theta_g itself
    if (K <= 0 || K > DL_MAX_LEARNERS || (values && K != 1) || !(clip_sigmas > 0.0) ||
        !(clip_sigmas < 1e300))
        return DL_ERR_ARG;
    if (f.T == 0) return DL_OK;
    if (!d_stats) return DL_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_stats) & 7u) != 0) return DL_ERR_ALIGN;
    if (f.n > 0) {
        if (!theta_g) return DL_ERR_ARG;
        if (!aligned16(theta_g)) return DL_ERR_ALIGN;
        for (int k = 0; k < K && !values; ++k) {
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
    for (int k = 0; k < K; ++k) a.r[k] = values ? nullptr : theta_k[k];
    a.off = f.d_offsets;
    char* ws = static_cast<char*>(d_workspace);
    a.status = reinterpret_cast<uint32_t*>(ws);
    a.shift = reinterpret_cast<float*>(ws + kWsHeader);
    a.ticket = reinterpret_cast<unsigned int*>(ws + kWsHeader + shift_bytes(K, f.T));
    a.part = reinterpret_cast<Partial*>(ws + kWsHeader + 2 * shift_bytes(K, f.T));
    a.out = d_stats;
    a.n = f.n;
    a.n_chunks = n_chunks_of(f.n);
    a.T = f.T;
    a.K = K;
    a.clip = clip_sigmas;
    a.J = 1;
    // 2 stages x 3 blocks per SM: more consumer warps for the same bytes in
    // flight than 3 stages x 2 blocks, which measured slower at every K
    const void* kern = values ? reinterpret_cast<const void*>(k_stats<2, 3, true>)
                              : reinterpret_cast<const void*>(k_stats<2, 3, false>);
    const size_t smem_used = sizeof(float) * 2 * 2 * kTile;
    const size_t smem = smem_used;
    if (a.n_chunks > 0) {
        if ((st = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem)))) != DL_OK)
            return st;
        a.J = blocks_per_learner(kern, kPipeThreads, smem_used, K, a.n_chunks);
        if (a.J > max_blocks_per_learner(K)) a.J = max_blocks_per_learner(K);
    }
    // one block per run, or, sharing the SMs, one per two runs (one block per
    // SM where the full grid has two)
    a.RPB = share_sms && a.J > 1 ? 2 : 1;
    const int JB = (a.J + a.RPB - 1) / a.RPB;  // blocks per learner
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // no elements at all: every (k, t) has N = 0, finished without partials
    if (a.n_chunks == 0) return stats_finish(a.off, f.T, K, 0, a.shift, a.part, a.clip, d_stats, s);
    const size_t ticket_bytes = sizeof(unsigned int) * static_cast<size_t>(K) * f.T;
    if ((st = cuda_status(cudaMemsetAsync(a.ticket, 0, ticket_bytes, s))) != DL_OK) return st;
    if (values)
        k_stats<2, 3, true><<<K * JB, kPipeThreads, smem, s>>>(a);
    else
        k_stats<2, 3, false><<<K * JB, kPipeThreads, smem, s>>>(a);
    return launch_status();
}
}  // namespace dl

extern "C" int dl_pseudograd_stats(const float* theta_g, const float* const* theta_k, int32_t K,
                                   const dl_fragment* frag, double clip_sigmas, dl_stats* d_stats,
                                   void* d_workspace, size_t workspace_bytes, void* stream) {
    return pseudograd_stats_shared(theta_g, theta_k, K, frag, clip_sigmas, d_stats, d_workspace,
                                   workspace_bytes, stream, false);
}
