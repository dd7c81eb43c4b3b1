// Shared device helpers and host-side validation for the outer-sync kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "diloco_sync.h"

namespace dl {

// ---------------------------------------------------------------------------
// work decomposition: a fragment is cut into fixed chunks of kChunk elements;
// a chunk meets one or more tensors ("pieces"). Chunk c starts at c * kChunk,
// so every chunk start is 32 KB aligned in an fp32 buffer.
constexpr int kChunk = 8192;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGroups = kChunk / 4 / kThreads;  // float4 groups per thread
constexpr int kNB = DL_NBUCKETS;
constexpr unsigned kFull = 0xffffffffu;

// device failure bits (workspace status word)
constexpr uint32_t kDevErrCopyTimeout = 1u;

// bounded spin on an mbarrier: ~2^22 try_wait polls, each of which may
// suspend for a short hardware-chosen time; far longer than any bulk copy.
constexpr long kSpinLimit = 1L << 22;

// tensors shorter than this take the fp64 per-element statistics path
constexpr int64_t kSmallTensor = 4096;

// workspace header: status word and padding
constexpr size_t kWsHeader = 256;

// learner-major grids (statistics, ring hops): block b serves learner b % K
// and the (b / K)-th run of contiguous chunks; at most this many blocks per
// learner, and in all
constexpr int kMaxBlocksPerLearner = 1024;
constexpr int kMaxBlocksTotal = 2048;

__host__ __device__ inline int64_t n_chunks_of(int64_t n) { return (n + kChunk - 1) / kChunk; }

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier + bulk (TMA engine) copies, sm_90+ forms.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// make the initialised barrier visible to the async (bulk copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// order this thread's earlier generic-proxy shared accesses before later
// async-proxy writes into the same buffer
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; false after `limit` polls (the caller records the failure).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long limit = kSpinLimit) {
    for (long i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---------------------------------------------------------------------------
// Tile pipeline: a producer warp streams tiles into a ring of STAGES
// shared-memory stages with bulk copies; consumer warps wait on the stage's
// "full" mbarrier and release it through its "empty" mbarrier (one arrival
// per consumer warp). Every wait is bounded. A wait that runs out aborts the
// block's pipeline: it records kDevErrCopyTimeout in the status word and sets
// the block's abort flag; from then on the producer issues no copy, the
// consumers read no stage (they still pass every named barrier, so no warp
// waits for one that left), and before the block retires the producer waits
// (bounded) until every copy it issued has landed, so no bulk copy is left
// writing into the shared memory of a retired block. The call's outputs are
// then undefined; the status word says so.
constexpr int kConsumerWarps = kWarps;
constexpr int kPipeThreads = kThreads + 32;  // + one producer warp
constexpr int kMaxStages = 4;

struct PipeBarriers {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int abort;  // set once a bounded wait ran out
};

template <int STAGES>
__device__ __forceinline__ void pipe_init(PipeBarriers* pb) {
    static_assert(STAGES <= kMaxStages, "too many stages");
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&pb->full[s], 1);
            mbar_init(&pb->empty[s], kConsumerWarps);
        }
        pb->abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
}

__device__ __forceinline__ bool pipe_aborted(const PipeBarriers* pb) {
    return *reinterpret_cast<const volatile int*>(&pb->abort) != 0;
}

__device__ __forceinline__ void pipe_abort(PipeBarriers* pb, uint32_t* status) {
    if (!pipe_aborted(pb)) {
        *reinterpret_cast<volatile int*>(&pb->abort) = 1;
        atomicOr(status, kDevErrCopyTimeout);
    }
}

// Bounded wait that also gives up once the block's pipeline is aborted.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t* bar, uint32_t parity,
                                                    const PipeBarriers* pb, long limit) {
    for (long i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31) == 31 && pipe_aborted(pb)) return false;
    }
    return false;
}

// Consumer warp (all lanes): wait until the stage of tile `it` holds it.
// Warp-uniform result; false once the pipeline is aborted, and then the stage
// must not be read.
template <int STAGES>
__device__ __forceinline__ bool consumer_wait(PipeBarriers* pb, uint32_t it, uint32_t* status,
                                              long limit = kSpinLimit) {
    bool ok = !pipe_aborted(pb) &&
              mbar_wait_abortable(&pb->full[it % STAGES], (it / STAGES) & 1u, pb, limit);
    ok = __all_sync(kFull, ok);
    if (!ok) pipe_abort(pb, status);
    return ok;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Consumer warp (all lanes): done with the stage of tile `it`. After an
// abort the stage is not released, so that no copy can be issued into it.
template <int STAGES>
__device__ __forceinline__ void consumer_release(PipeBarriers* pb, uint32_t it, bool ok) {
    __syncwarp();
    if (ok && (threadIdx.x & 31) == 0) mbar_arrive(&pb->empty[it % STAGES]);
}

// Producer lane: wait until the stage of tile `it` is free to be written;
// false once the pipeline is aborted (no copy may be issued then).
template <int STAGES>
__device__ __forceinline__ bool producer_acquire(PipeBarriers* pb, uint32_t it, uint32_t* status,
                                                 long limit = kSpinLimit) {
    if (pipe_aborted(pb)) return false;
    if (it < STAGES) return true;
    if (mbar_wait_abortable(&pb->empty[it % STAGES], ((it / STAGES) - 1) & 1u, pb, limit))
        return true;
    pipe_abort(pb, status);
    return false;
}

// Producer lane, after its last tile or an abort: `issued` tiles were issued;
// wait (bounded) until the copies of the last tile of every stage have
// landed, so that the block never retires with a copy in flight.
template <int STAGES>
__device__ __forceinline__ void producer_drain(PipeBarriers* pb, uint32_t issued, uint32_t* status,
                                               long limit = kSpinLimit) {
    for (uint32_t s = 0; s < STAGES && s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % STAGES);  // last tile of stage s
        if (!mbar_wait_bounded(&pb->full[s], (last / STAGES) & 1u, limit))
            atomicOr(status, kDevErrCopyTimeout);
    }
}

// barrier among the consumer warps only (named barrier 1)
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kThreads) : "memory");
}

// Producer side: lane 0 of the producer warp issues the bulk copies of tile
// number `it` (its stage is it % STAGES) covering [tb, tb + tn) of two arrays
// (of one when gb is null: values mode, the second array is never staged).
// false once the pipeline is aborted: nothing was issued.
template <int TILE, int STAGES>
__device__ __forceinline__ bool pipe_produce(PipeBarriers* pb, float* sa, float* sb, const float* ga,
                                             const float* gb, int64_t tb, int tn, uint32_t it,
                                             uint32_t* status) {
    if (!producer_acquire<STAGES>(pb, it, status)) return false;
    const int s = static_cast<int>(it % STAGES);
    const uint32_t bytes = static_cast<uint32_t>(tn >> 2) * 16u;
    fence_proxy_async();
    mbar_arrive_expect_tx(&pb->full[s], gb ? 2u * bytes : bytes);
    if (bytes) {
        bulk_copy_g2s(sa + s * TILE, ga + tb, bytes, &pb->full[s]);
        if (gb) bulk_copy_g2s(sb + s * TILE, gb + tb, bytes, &pb->full[s]);
    }
    return true;
}

// ---------------------------------------------------------------------------
// Contiguous chunk range [c0, c1) of this block: the chunks split as evenly as
// possible over the grid. A block then meets few tensors, so per-tensor
// set-up (codebooks staged in shared memory) is rarely repeated.
__device__ __forceinline__ void block_chunks(int64_t n_chunks, int64_t& c0, int64_t& c1) {
    const int64_t G = gridDim.x, b = blockIdx.x;
    c0 = n_chunks * b / G;
    c1 = n_chunks * (b + 1) / G;
}

// ---------------------------------------------------------------------------
// Tensor lookup: smallest t with off[t+1] > pos (empty tensors are skipped).
__device__ __forceinline__ int tensor_containing(const int64_t* __restrict__ off, int T,
                                                 int64_t pos) {
    int lo = 0, hi = T - 1;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (__ldg(off + mid + 1) > pos)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// First tensor at or after lo whose end lies past pos (lo <= T - 1): a binary
// search, kept out of line (it runs once per tensor boundary).
static __device__ __noinline__ int tensor_from(const int64_t* __restrict__ off, int lo, int T, int64_t pos) {
    int hi = T - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(off + mid + 1) > pos)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// Bounds [o0, o1) of tensor t held in registers while a block walks forward
// through the fragment: a tile inside the tensor of the previous tile loads no
// offsets, whose load latency would otherwise sit on every tile's critical
// path.
struct TensorCursor {
    int t = -1;
    int64_t o0 = 0, o1 = 0;
    __device__ __forceinline__ void load(const int64_t* __restrict__ off, int tt) {
        if (tt != t) {
            o0 = __ldg(off + tt);
            o1 = __ldg(off + tt + 1);
            t = tt;
        }
    }
    // The tensor holding pos (< off[T]), for a pos at or past the start of
    // the cursor's tensor: the current one while pos is inside it, else the
    // first later tensor that holds it; the result is loaded into the cursor.
    __device__ __forceinline__ int seek(const int64_t* __restrict__ off, int T, int64_t pos) {
        if (t < 0 || pos >= o1) load(off, tensor_from(off, t < 0 ? 0 : min(t + 1, T - 1), T, pos));
        return t;
    }
};

// ---------------------------------------------------------------------------
// float-float (unevaluated sum hi + lo) accumulation, fp32 operations only.
__device__ __forceinline__ void ff_add(float& hi, float& lo, float b) {
    float s = __fadd_rn(hi, b);
    float v = __fsub_rn(s, hi);
    float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, v)), __fsub_rn(b, v));
    lo = __fadd_rn(lo, e);
    hi = s;
}

__device__ __forceinline__ void ff_add_ff(float& ahi, float& alo, float bhi, float blo) {
    float s = __fadd_rn(ahi, bhi);
    float v = __fsub_rn(s, ahi);
    float e = __fadd_rn(__fsub_rn(ahi, __fsub_rn(s, v)), __fsub_rn(bhi, v));
    e = __fadd_rn(e, __fadd_rn(alo, blo));
    float h = __fadd_rn(s, e);
    alo = __fsub_rn(e, __fsub_rn(h, s));
    ahi = h;
}

// ---------------------------------------------------------------------------
// Quantiser parameters of one segment, derived identically by the encode
// kernel and the codebook finalisation from (lo, hi, nonfinite).
struct SegQuant {
    int kind;         // 0 fast, 1 slow (all elements in fp64), 2 degenerate, 3 invalid
    double lo, hi, s; // s = 256 / (hi - lo)
    float lo_f, w_f, s_f, guard;
    float c_f;        // fl32(-lo_f * s_f): u is evaluated as fmaf(d, s_f, c_f)
    float scale;      // 2^ks as fp32 (fast kind only)
    float qoff;       // 2^23 + kResBias as fp32 (fast kind only)
    int ks;           // residual fixed-point exponent
    double ref0, refw; // slow kind: residual reference ref0 + b * refw (fp64)
};

constexpr int kSegFast = 0, kSegSlow = 1, kSegDegenerate = 2, kSegInvalid = 3;
// Residual fixed point: q = rint(r * 2^ks) + 2^19 with w * 2^ks in
// [2^21, 2^22). For the fast kind the reference edge e_b = fmaf(b, w_f, lo_f)
// misses the exact edge lo + b w by at most 2^-23 (|lo| + 256 w) + 2^-16 w,
// which the fast-kind condition (|lo| / w < 2^19) keeps below w / 16 (up to
// 2^-15 w): r lies in (-w/16, 17 w / 16), so q lies in (2^18, 2^23) and the
// fp32 sum fmaf(r, 2^ks, 2^23 + 2^19) falls in [2^23, 2^24), where fp32 holds
// every integer - its low 23 bits are q, rounded once to nearest even.
constexpr int kResBits = 21;
constexpr int64_t kResBias = int64_t(1) << 19;

__device__ __forceinline__ SegQuant seg_quant(double lo, double hi, long long nonfinite) {
    SegQuant q;
    q.lo = lo;
    q.hi = hi;
    q.s = 0.0;
    q.lo_f = q.w_f = q.s_f = q.guard = q.scale = q.qoff = q.c_f = 0.f;
    q.ks = 0;
    q.ref0 = q.refw = 0.0;
    if (nonfinite > 0) {
        q.kind = kSegInvalid;
        return q;
    }
    if (!(hi - lo >= 256.0 * 1.17549435082228750797e-38)) {  // 256 * FLT_MIN
        q.kind = kSegDegenerate;
        return q;
    }
    q.s = 256.0 / (hi - lo);
    const double w = (hi - lo) / 256.0;
    q.lo_f = static_cast<float>(lo);
    q.w_f = static_cast<float>(w);
    q.s_f = static_cast<float>(q.s);
    q.c_f = static_cast<float>(-static_cast<double>(q.lo_f) * static_cast<double>(q.s_f));
    // u_f = fl(d * s_f + c_f) against u = (d - lo) s: s_f, lo_f and c_f each
    // carry one fp32 rounding and the fma one more, so for u_f in [-1, 257]
    // |u_f - u| <= (4 s|lo| + 2 * 258) 2^-24; the guard is twice that
    const double g = (4.0 * q.s * fabs(lo) + 520.0) * 0x1p-23;
    q.guard = static_cast<float>(g);
    int e_w;
    frexp(static_cast<double>(q.w_f), &e_w);  // w_f = f * 2^e_w, f in [0.5, 1)
    q.ks = kResBits + 1 - e_w;                  // w_f * 2^ks in [2^21, 2^22)
    const bool fast = isfinite(q.lo_f) && isfinite(q.s_f) && q.w_f > 0.f && g < 0.25 &&
                      q.ks >= -126 && q.ks <= 127 && fabs(hi) < 1e37 && fabs(lo) < 1e37;
    if (fast) {
        q.kind = kSegFast;
        q.scale = ldexpf(1.0f, q.ks);
        q.qoff = static_cast<float>((int64_t(1) << 23) + kResBias);
    } else {
        q.kind = kSegSlow;
        q.ref0 = lo;
        q.refw = w;
        e_w = 0;
        frexp(w, &e_w);
        q.ks = kResBits + 1 - e_w;
    }
    return q;
}

// Residual reference of bucket b: the fp32 edge fmaf(b, w_f, lo_f) for the
// fast kind (the element minus it is exact or within 2^-24 of a bucket width),
// lo + b * w in fp64 for the slow kind. Encoder and finaliser both call this.
__device__ __forceinline__ double seg_ref(const SegQuant& q, int b) {
    if (q.kind == kSegFast) return static_cast<double>(__fmaf_rn(static_cast<float>(b), q.w_f, q.lo_f));
    return fma(static_cast<double>(b), q.refw, q.ref0);
}

}  // namespace dl

// ---------------------------------------------------------------------------
// host side (defined in dl_host.cu)
namespace dl {
struct HostFrag {
    const int64_t* offsets;
    const int64_t* d_offsets;
    int T;
    int64_t n;
};
int check_fragment(const dl_fragment* frag, HostFrag* out);
bool aligned16(const void* p);
int sm_count();
int grid_for(const void* kernel, int threads, size_t smem, int64_t work_items);
int blocks_per_learner(const void* kernel, int threads, size_t smem, int K, int64_t n_chunks);
int cuda_status(cudaError_t e);
int launch_status();
// the library's device status word (for calls without a workspace)
int library_status_word(uint32_t** out);
// dl_merge_outer_step reporting bounded-wait failures to `status` (NULL: the
// library's word)
int merge_outer_step_status(float* theta_g, float* momentum, const uint8_t* const* codes,
                            const float* d_codebook, const float* const* theta_k, int32_t K,
                            const dl_fragment* frag, const float* weights, const uint8_t* present,
                            int32_t min_quorum, float lr, float mu, float* delta_bar_out,
                            uint32_t* status, void* stream);
// dl_pseudograd_stats; share_sms: at most one of its blocks resident per SM
// (same grid, same results)
int pseudograd_stats_shared(const float* theta_g, const float* const* theta_k, int32_t K,
                            const dl_fragment* frag, double clip_sigmas, dl_stats* d_stats,
                            void* d_workspace, size_t workspace_bytes, void* stream,
                            bool share_sms);
}  // namespace dl
