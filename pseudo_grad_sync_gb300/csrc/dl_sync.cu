// Whole-model outer step: every fragment of a model through statistics,
// quantisation and merge in one call, with the statistics of the next
// fragment running beside the quantisation and merge of the current one.
//
// Decoupled DiLoCo note (architecture items 3-4): the model is split into
// fragments that are synchronised one after another while work continues, so
// that transfer and compute overlap. Here the overlap is between kernels of
// consecutive fragments on one GPU: fragment f+1's statistics (pure HBM
// streaming) run on a side stream while fragment f's quantisation (bound by
// instruction issue) and merge run on the caller's stream, and the idle
// gaps around each call's small set-up and finalising kernels get filled.
//
// Schedule (b = f mod 2 selects one of two statistics buffers):
//   side: wait quantize(f-2) done; stats(f) -> S[b]; record stats_done[b]
//   main: wait stats_done[b]; quantize(f) from S[b]; record quant_done[b];
//         merge(f)
// The side stream forks from the caller's stream at entry and joins it at
// exit, so on return every effect of the call is ordered on `stream`. From
// the second fragment on, the statistics run at one block per SM (two chunk
// runs per block, the same runs as the full grid, so the same sums): a
// statistics block then leaves room on its SM for two quantiser blocks of the
// fragment before, and the kernels share the SMs instead of taking turns. The
// first fragment's statistics, with nothing beside them, take the full grid.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "dl_common.cuh"

namespace dl {
namespace {

// Per-device side stream and event ring, created on first use and kept
// until dl_shutdown. The mutex serialises enqueueing: two callers
// never interleave their records and waits on the shared events.
struct SideResources {
    std::mutex mu;
    bool ready = false;
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaEvent_t stats_done[2] = {nullptr, nullptr};
    cudaEvent_t quant_done[2] = {nullptr, nullptr};
};
SideResources g_side[64];

int side_resources(SideResources** out, int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= 64) return DL_ERR_CUDA;
    *out = &g_side[*dev];
    return DL_OK;
}

// Releases one device's side stream and events (the caller holds r.mu).
int destroy_side(SideResources& r, int dev) {
    // handles from a create_side that failed part way count too
    if (!r.side && !r.fork && !r.join && !r.stats_done[0] && !r.stats_done[1] &&
        !r.quant_done[0] && !r.quant_done[1])
        return DL_OK;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess)
        return DL_ERR_CUDA;
    // the side stream's queued work (and so every event it records) finishes
    // first, so no pending wait on the caller's stream refers to a dead event
    bool ok = !r.side || cudaStreamSynchronize(r.side) == cudaSuccess;
    cudaEvent_t* evs[] = {&r.fork, &r.join, &r.stats_done[0], &r.stats_done[1],
                          &r.quant_done[0], &r.quant_done[1]};
    for (cudaEvent_t* e : evs) {
        if (*e && cudaEventDestroy(*e) != cudaSuccess) ok = false;
        *e = nullptr;
    }
    if (r.side && cudaStreamDestroy(r.side) != cudaSuccess) ok = false;
    r.side = nullptr;
    r.ready = false;
    if (cudaSetDevice(prev) != cudaSuccess) ok = false;
    return ok ? DL_OK : DL_ERR_CUDA;
}

int create_side(SideResources& r, int dev) {
    if (r.ready) return DL_OK;
    if (destroy_side(r, dev) != DL_OK) return DL_ERR_CUDA;  // leftovers of a failed attempt
    const unsigned fl = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&r.side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&r.fork, fl) != cudaSuccess ||
        cudaEventCreateWithFlags(&r.join, fl) != cudaSuccess)
        return DL_ERR_CUDA;
    for (int b = 0; b < 2; ++b)
        if (cudaEventCreateWithFlags(&r.stats_done[b], fl) != cudaSuccess ||
            cudaEventCreateWithFlags(&r.quant_done[b], fl) != cudaSuccess)
            return DL_ERR_CUDA;
    r.ready = true;
    return DL_OK;
}

constexpr int32_t kSyncFlags = DL_SYNC_UNQUANTIZED | DL_SYNC_SERIAL | DL_SYNC_RDA | DL_SYNC_RING;

// Flags that make sense together: RDA and the ring are quantised modes, and
// one excludes the other.
bool flags_valid(int32_t flags) {
    if ((flags & ~kSyncFlags) != 0) return false;
    const bool unq = (flags & DL_SYNC_UNQUANTIZED) != 0;
    const bool rda = (flags & DL_SYNC_RDA) != 0, ring = (flags & DL_SYNC_RING) != 0;
    return !(rda && ring) && !(unq && (rda || ring));
}

// Workspace layout (every part 256-byte aligned). The statistics workspace
// comes first, so its status word is the outer workspace's first word and
// dl_read_device_status reads it; in ring mode the ring's own workspace is
// the whole layout (its status word first, too).
struct SyncLayout {
    size_t stats_ws = 0, stats_arr = 0, quant_ws = 0, codebook = 0, codes_each = 0;
    size_t counts = 0, rda_ws = 0, ring_ws = 0;
    size_t off_stats_arr[2] = {0, 0}, off_quant_ws = 0, off_codebook = 0, off_codes = 0;
    size_t off_counts = 0, off_rda_ws = 0;
    size_t total = 0;
    int T_max = 0;
    int64_t n_max = 0;
};

// Scratch sizes depend on the number of present learners, which may be any
// value in 1..K; the layout takes the largest over all of them.
int sync_layout(const dl_fragment_job* jobs, int32_t n_jobs, int32_t K, int32_t flags,
                SyncLayout* L) {
    if (n_jobs < 0 || K <= 0 || K > DL_MAX_LEARNERS || (n_jobs > 0 && !jobs) ||
        !flags_valid(flags))
        return DL_ERR_ARG;
    *L = SyncLayout();
    if (flags & DL_SYNC_RING) {
        for (int32_t j = 0; j < n_jobs; ++j) {
            HostFrag f;
            const int st = check_fragment(jobs[j].frag, &f);
            if (st != DL_OK) return st;
            const size_t r = dl_ring_workspace_bytes(jobs[j].frag);
            if (r > L->ring_ws) L->ring_ws = r;
        }
        L->ring_ws = align256(L->ring_ws > kWsHeader ? L->ring_ws : kWsHeader);
        L->total = L->ring_ws;
        return DL_OK;
    }
    for (int32_t j = 0; j < n_jobs; ++j) {
        HostFrag f;
        const int st = check_fragment(jobs[j].frag, &f);
        if (st != DL_OK) return st;
        if (f.T > L->T_max) L->T_max = f.T;
        if (f.n > L->n_max) L->n_max = f.n;
        if (f.T == 0) continue;
        for (int np = 1; np <= K; ++np) {
            const size_t s = dl_stats_workspace_bytes(jobs[j].frag, np);
            const size_t q = dl_quantize_workspace_bytes(jobs[j].frag, np);
            if (s > L->stats_ws) L->stats_ws = s;
            if (q > L->quant_ws) L->quant_ws = q;
            if (flags & DL_SYNC_RDA) {
                const size_t r = dl_rda_workspace_bytes(jobs[j].frag, np);
                if (r > L->rda_ws) L->rda_ws = r;
            }
        }
    }
    L->stats_ws = align256(L->stats_ws > kWsHeader ? L->stats_ws : kWsHeader);
    L->stats_arr = align256(sizeof(dl_stats) * static_cast<size_t>(K) * L->T_max);
    L->quant_ws = align256(L->quant_ws);
    L->codebook = align256(sizeof(float) * static_cast<size_t>(K) * L->T_max * kNB);
    L->codes_each = align256(static_cast<size_t>(L->n_max));
    size_t o = L->stats_ws;
    L->off_stats_arr[0] = o;
    o += L->stats_arr;
    L->off_stats_arr[1] = o;
    o += L->stats_arr;
    L->off_quant_ws = o;
    o += L->quant_ws;
    L->off_codebook = o;
    o += L->codebook;
    L->off_codes = o;
    o += L->codes_each * static_cast<size_t>(K);
    if (flags & DL_SYNC_RDA) {
        L->counts = align256(sizeof(uint32_t) * static_cast<size_t>(K) * L->T_max * kNB);
        L->rda_ws = align256(L->rda_ws);
        L->off_counts = o;
        o += L->counts;
        L->off_rda_ws = o;
        o += L->rda_ws;
    }
    L->total = o;
    return DL_OK;
}

// The present learners of one job, in ascending order, with their buffers
// and weights gathered so that every call below sees them as learners 0..np-1.
struct Present {
    int np = 0;
    const float* rep[DL_MAX_LEARNERS];
    float w[DL_MAX_LEARNERS];
};

int gather_present(const dl_fragment_job& job, int32_t K, int32_t min_quorum, Present* p) {
    HostFrag f;
    int st = check_fragment(job.frag, &f);
    if (st != DL_OK) return st;
    p->np = 0;
    double total = 0.0;
    for (int k = 0; k < K; ++k) {
        if (job.present && !job.present[k]) continue;
        const double w = job.weights ? static_cast<double>(job.weights[k]) : 1.0;
        if (!(w >= 0.0) || !(w < 1e300)) return DL_ERR_ARG;
        total += w;
        p->rep[p->np] = job.theta_k ? job.theta_k[k] : nullptr;
        p->w[p->np] = static_cast<float>(w);
        ++p->np;
    }
    if (p->np < (min_quorum > 1 ? min_quorum : 1)) return DL_ERR_QUORUM;
    if (!(total > 0.0)) return DL_ERR_ARG;
    if (f.n == 0) return DL_OK;
    if (!job.theta_g || !job.momentum || !job.theta_k) return DL_ERR_ARG;
    if (!aligned16(job.theta_g) || !aligned16(job.momentum) ||
        (job.delta_bar_out && !aligned16(job.delta_bar_out)))
        return DL_ERR_ALIGN;
    for (int s = 0; s < p->np; ++s) {
        if (!p->rep[s]) return DL_ERR_ARG;
        if (!aligned16(p->rep[s])) return DL_ERR_ALIGN;
    }
    return DL_OK;
}

}  // namespace
}  // namespace dl

using namespace dl;

extern "C" int dl_shutdown(void) {
    int st = DL_OK;
    for (int dev = 0; dev < 64; ++dev) {
        std::lock_guard<std::mutex> lock(g_side[dev].mu);
        const int s = destroy_side(g_side[dev], dev);
        if (st == DL_OK) st = s;
    }
    return st;
}

extern "C" size_t dl_outer_sync_workspace_bytes(const dl_fragment_job* jobs, int32_t n_jobs,
                                                int32_t K, int32_t flags) {
    SyncLayout L;
    if (sync_layout(jobs, n_jobs, K, flags, &L) != DL_OK) return 0;
    return L.total;
}

extern "C" int dl_outer_sync(const dl_fragment_job* jobs, int32_t n_jobs, int32_t K,
                             double clip_sigmas, int32_t min_quorum, float lr, float mu,
                             int32_t flags, void* d_workspace, size_t workspace_bytes,
                             void* stream) {
    if (!flags_valid(flags)) return DL_ERR_ARG;
    const bool quantized = (flags & DL_SYNC_UNQUANTIZED) == 0;
    const bool serial = (flags & DL_SYNC_SERIAL) != 0;
    const bool rda = (flags & DL_SYNC_RDA) != 0, ring = (flags & DL_SYNC_RING) != 0;
    if (quantized && (!(clip_sigmas > 0.0) || !(clip_sigmas < 1e300))) return DL_ERR_ARG;
    SyncLayout L;
    int st = sync_layout(jobs, n_jobs, K, flags, &L);
    if (st != DL_OK) return st;
    if (n_jobs == 0) return DL_OK;
    // every job is validated before anything is enqueued
    for (int32_t j = 0; j < n_jobs; ++j) {
        Present p;
        if ((st = gather_present(jobs[j], K, min_quorum, &p)) != DL_OK) return st;
    }
    cudaStream_t main_s = static_cast<cudaStream_t>(stream);

    if (!quantized) {
        for (int32_t j = 0; j < n_jobs; ++j) {
            const dl_fragment_job& job = jobs[j];
            Present p;
            gather_present(job, K, min_quorum, &p);
            st = dl_merge_outer_step(job.theta_g, job.momentum, nullptr, nullptr, p.rep, p.np,
                                     job.frag, job.weights ? p.w : nullptr, nullptr, min_quorum,
                                     lr, mu, job.delta_bar_out, main_s);
            if (st != DL_OK) return st;
        }
        return DL_OK;
    }

    if (!d_workspace || workspace_bytes < L.total) return DL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0) return DL_ERR_ALIGN;
    if (ring) {  // each fragment's ring runs its hops in order on `stream`
        for (int32_t j = 0; j < n_jobs; ++j) {
            const dl_fragment_job& job = jobs[j];
            Present p;
            gather_present(job, K, min_quorum, &p);
            st = dl_ring_outer_step(job.theta_g, job.momentum, p.rep, p.np, job.frag,
                                    job.weights ? p.w : nullptr, nullptr, min_quorum, clip_sigmas,
                                    lr, mu, job.delta_bar_out, nullptr, d_workspace, L.ring_ws,
                                    main_s);
            if (st != DL_OK) return st;
        }
        return DL_OK;
    }
    char* ws = static_cast<char*>(d_workspace);
    void* stats_ws = ws;
    dl_stats* stats_arr[2] = {reinterpret_cast<dl_stats*>(ws + L.off_stats_arr[0]),
                              reinterpret_cast<dl_stats*>(ws + L.off_stats_arr[1])};
    void* quant_ws = ws + L.off_quant_ws;
    float* codebook = reinterpret_cast<float*>(ws + L.off_codebook);
    uint8_t* codes[DL_MAX_LEARNERS];
    for (int k = 0; k < K; ++k)
        codes[k] = reinterpret_cast<uint8_t*>(ws + L.off_codes + L.codes_each * static_cast<size_t>(k));

    SideResources* R = nullptr;
    std::unique_lock<std::mutex> lock;
    cudaStream_t side_s = main_s;
    if (!serial) {
        int dev = 0;
        if ((st = side_resources(&R, &dev)) != DL_OK) return st;
        lock = std::unique_lock<std::mutex>(R->mu);
        if ((st = create_side(*R, dev)) != DL_OK) return st;
        side_s = R->side;
        if ((st = cuda_status(cudaEventRecord(R->fork, main_s))) != DL_OK) return st;
        if ((st = cuda_status(cudaStreamWaitEvent(side_s, R->fork, 0))) != DL_OK) return st;
    }

    for (int32_t j = 0; j < n_jobs && st == DL_OK; ++j) {
        const dl_fragment_job& job = jobs[j];
        const int b = j & 1;
        Present p;
        gather_present(job, K, min_quorum, &p);
        // side: statistics of fragment j, once quantize(j-2) has read buffer b
        if (!serial && j >= 2 &&
            (st = cuda_status(cudaStreamWaitEvent(side_s, R->quant_done[b], 0))) != DL_OK)
            break;
        // the first fragment's statistics run alone: the full grid; later ones
        // share each SM with the quantiser of the fragment before (same runs,
        // so the same sums either way)
        st = pseudograd_stats_shared(job.theta_g, p.rep, p.np, job.frag, clip_sigmas, stats_arr[b],
                                     stats_ws, L.stats_ws, side_s, !serial && j >= 1);
        if (st != DL_OK) break;
        if (!serial) {
            if ((st = cuda_status(cudaEventRecord(R->stats_done[b], side_s))) != DL_OK) break;
            if ((st = cuda_status(cudaStreamWaitEvent(main_s, R->stats_done[b], 0))) != DL_OK)
                break;
        }
        // main: quantise and merge fragment j
        uint32_t* counts = rda ? reinterpret_cast<uint32_t*>(ws + L.off_counts) : nullptr;
        st = dl_quantize(job.theta_g, p.rep, p.np, job.frag, stats_arr[b], codes, codebook,
                         counts, quant_ws, L.quant_ws, main_s);
        if (st != DL_OK) break;
        if (!serial && (st = cuda_status(cudaEventRecord(R->quant_done[b], main_s))) != DL_OK)
            break;
        if (rda)
            st = dl_rda_merge_outer_step(job.theta_g, job.momentum, codes, codebook, counts,
                                         p.np, job.frag, job.weights ? p.w : nullptr, nullptr,
                                         min_quorum, lr, mu, job.delta_bar_out,
                                         ws + L.off_rda_ws, L.rda_ws, main_s);
        else
            st = merge_outer_step_status(job.theta_g, job.momentum, codes, codebook, nullptr,
                                         p.np, job.frag, job.weights ? p.w : nullptr, nullptr,
                                         min_quorum, lr, mu, job.delta_bar_out,
                                         reinterpret_cast<uint32_t*>(ws), main_s);
    }
    if (!serial) {
        // join even after a failure, so that the caller's stream stays ordered
        const int js = cuda_status(cudaEventRecord(R->join, side_s));
        const int jw = js == DL_OK ? cuda_status(cudaStreamWaitEvent(main_s, R->join, 0)) : js;
        if (st == DL_OK) st = jw;
    }
    return st;
}
