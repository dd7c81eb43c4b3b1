// Host-side pieces of the C ABI: status strings, the fragment planner,
// argument validation and launch sizing.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <queue>
#include <utility>
#include <vector>

#include "dl_common.cuh"

extern "C" int dl_version(void) { return 200; }

extern "C" const char* dl_status_string(int status) {
    switch (status) {
        case DL_OK: return "DL_OK";
        case DL_ERR_ARG: return "DL_ERR_ARG: invalid argument";
        case DL_ERR_ALIGN: return "DL_ERR_ALIGN: buffer not 16-byte (workspace: 256-byte) aligned";
        case DL_ERR_QUORUM: return "DL_ERR_QUORUM: fewer present learners than the minimum quorum";
        case DL_ERR_CUDA: return "DL_ERR_CUDA: CUDA runtime call or launch failed";
        case DL_ERR_SHAPE: return "DL_ERR_SHAPE: offsets must start at 0 and not decrease";
        case DL_ERR_WORKSPACE: return "DL_ERR_WORKSPACE: workspace missing or too small";
        case DL_ERR_DEVICE: return "DL_ERR_DEVICE: a kernel reported a failure";
        default: return "unknown status";
    }
}

// Balanced tensor fragmentation, longest-processing-time greedy (Decoupled
// DiLoCo note, architecture item 4). Fragments are kept in a min-heap keyed
// by (load, index) so that ties go to the lowest fragment index.
extern "C" int dl_plan_fragments(const int64_t* numel, int32_t n_tensors, int32_t n_frags,
                                 int32_t* frag_of_tensor, int64_t* frag_load) {
    if (n_frags <= 0 || n_tensors < 0 || !frag_load) return DL_ERR_ARG;
    if (n_tensors > 0 && (!numel || !frag_of_tensor)) return DL_ERR_ARG;
    for (int32_t t = 0; t < n_tensors; ++t)
        if (numel[t] < 0) return DL_ERR_ARG;
    std::vector<int32_t> order(static_cast<size_t>(n_tensors));
    for (int32_t t = 0; t < n_tensors; ++t) order[t] = t;
    std::sort(order.begin(), order.end(), [numel](int32_t a, int32_t b) {
        return numel[a] != numel[b] ? numel[a] > numel[b] : a < b;
    });
    using Slot = std::pair<int64_t, int32_t>;  // (load, fragment)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t p = 0; p < n_frags; ++p) heap.push(Slot(0, p));
    for (int32_t t : order) {
        Slot s = heap.top();
        heap.pop();
        frag_of_tensor[t] = s.second;
        s.first += numel[t];
        heap.push(s);
    }
    while (!heap.empty()) {
        frag_load[heap.top().second] = heap.top().first;
        heap.pop();
    }
    return DL_OK;
}

extern "C" int dl_read_device_status(void* d_workspace, uint32_t* status_out, void* stream) {
    if (!status_out) return DL_ERR_ARG;
    if (!d_workspace) {  // the library's own word (calls without a workspace)
        uint32_t* w = nullptr;
        const int st = dl::library_status_word(&w);
        if (st != DL_OK) return st;
        d_workspace = w;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, d_workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_workspace, 0, sizeof(v), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return DL_ERR_CUDA;
    *status_out = v;
    return DL_OK;
}

namespace dl {

int check_fragment(const dl_fragment* frag, HostFrag* out) {
    if (!frag || frag->n_tensors < 0) return DL_ERR_ARG;
    out->T = frag->n_tensors;
    out->offsets = frag->offsets;
    out->d_offsets = frag->d_offsets;
    out->n = 0;
    if (frag->n_tensors == 0) return DL_OK;
    if (!frag->offsets || !frag->d_offsets) return DL_ERR_ARG;
    if (frag->offsets[0] != 0) return DL_ERR_SHAPE;
    for (int32_t t = 0; t < frag->n_tensors; ++t)
        if (frag->offsets[t + 1] < frag->offsets[t]) return DL_ERR_SHAPE;
    out->n = frag->offsets[frag->n_tensors];
    return DL_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 1;
        cache[dev] = v;
    }
    return cache[dev];
}

// Persistent grid: as many blocks as fit on every SM at once, never more than
// there are work items. DL_GRID_LIMIT (environment) caps it further; tests
// use that to make single blocks cover many chunks.
int grid_for(const void* kernel, int threads, size_t smem, int64_t work_items) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
            cudaSuccess ||
        per_sm <= 0)
        per_sm = 1;
    int64_t g = static_cast<int64_t>(per_sm) * sm_count();
    if (const char* cap = getenv("DL_GRID_LIMIT")) {
        const long v = strtol(cap, nullptr, 10);
        if (v > 0 && v < g) g = v;
    }
    if (work_items < g) g = work_items;
    return static_cast<int>(g < 1 ? 1 : g);
}

// Learner-major persistent grid: J blocks per learner, K * J blocks in all,
// as many as fit on the GPU at once (never more than there are chunks).
int blocks_per_learner(const void* kernel, int threads, size_t smem, int K, int64_t n_chunks) {
    const int total = grid_for(kernel, threads, smem, int64_t(1) << 40);
    int64_t j = total / K;
    if (j < 1) j = 1;
    if (j > kMaxBlocksPerLearner) j = kMaxBlocksPerLearner;
    if (j > n_chunks) j = n_chunks;
    return static_cast<int>(j < 1 ? 1 : j);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DL_OK : DL_ERR_CUDA; }

int launch_status() { return cudaGetLastError() == cudaSuccess ? DL_OK : DL_ERR_CUDA; }

}  // namespace dl

// ---------------------------------------------------------------------------
// Self-test of the bounded-wait failure path: one thread waits on a
// shared-memory mbarrier that expects one arrival nobody makes, so the wait
// runs out after `polls` polls; the kernel then records the failure in the
// workspace status word, exactly as a stalled bulk copy would, and returns.
namespace {
__global__ void k_selftest_wait(uint32_t* status, long polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    dl::mbar_init(&bar, 1);
    dl::fence_barrier_init();
    if (!dl::mbar_wait_bounded(&bar, 0u, polls)) atomicOr(status, dl::kDevErrCopyTimeout);
}

// Self-test of the tile pipeline's abort path (dl_common.cuh): one block, a
// producer warp streaming 1024-float tiles of `src` into two stages with bulk
// copies and eight consumer warps summing each tile into out[tile]. The
// producer issues tiles 0 .. stall-1 only, as a stalled copy engine would,
// then drains the copies it issued. The consumers' bounded waits for tile
// `stall` run out after `polls` polls: the block's pipeline aborts, the
// status word gets kDevErrCopyTimeout, the remaining tiles are not read
// (out[tile] = NaN) and the kernel ends. stall = n_tiles: the normal path.
constexpr int kSelfTile = 1024;
constexpr int kSelfStages = 2;

__global__ void __launch_bounds__(dl::kPipeThreads) k_selftest_pipeline(const float* src, int n_tiles,
                                                                        int stall, long polls,
                                                                        float* out, uint32_t* status) {
    extern __shared__ __align__(128) float sbuf[];
    __shared__ dl::PipeBarriers pb;
    __shared__ float red[dl::kConsumerWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    dl::pipe_init<kSelfStages>(&pb);
    if (warp == dl::kConsumerWarps) {  // producer warp
        if (lane == 0) {
            uint32_t it = 0;
            for (; it < static_cast<uint32_t>(stall); ++it) {
                if (!dl::producer_acquire<kSelfStages>(&pb, it, status, polls)) break;
                const int s = static_cast<int>(it % kSelfStages);
                dl::fence_proxy_async();
                dl::mbar_arrive_expect_tx(&pb.full[s], kSelfTile * 4);
                dl::bulk_copy_g2s(sbuf + s * kSelfTile, src + static_cast<int64_t>(it) * kSelfTile,
                                  kSelfTile * 4, &pb.full[s]);
            }
            dl::producer_drain<kSelfStages>(&pb, it, status, polls);
        }
        return;
    }
    for (uint32_t it = 0; it < static_cast<uint32_t>(n_tiles); ++it) {
        const bool ok = dl::consumer_wait<kSelfStages>(&pb, it, status, polls);
        float v = 0.f;
        if (ok) {
            const float4 x = reinterpret_cast<const float4*>(sbuf + (it % kSelfStages) * kSelfTile)[tid];
            v = (x.x + x.y) + (x.z + x.w);
        }
        for (int sh = 16; sh; sh >>= 1) v += __shfl_xor_sync(dl::kFull, v, sh);
        if (lane == 0) red[warp] = ok ? v : __int_as_float(0x7fc00000);
        dl::consumer_release<kSelfStages>(&pb, it, ok);
        dl::consumer_sync();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < dl::kConsumerWarps; ++w) t += red[w];
            out[it] = t;
        }
        dl::consumer_sync();
    }
}
}  // namespace

extern "C" int dl_selftest_pipeline(void* d_workspace, const float* d_src, int32_t n_tiles,
                                    int32_t stall_tile, int32_t polls, float* d_out,
                                    void* stream) {
    if (!d_workspace || !d_src || !d_out || n_tiles <= 0 || n_tiles > 4096 || stall_tile < 0 ||
        stall_tile > n_tiles || polls <= 0 || polls > dl::kSpinLimit)
        return DL_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0 || !dl::aligned16(d_src) ||
        (reinterpret_cast<uintptr_t>(d_out) & 3u) != 0)
        return DL_ERR_ALIGN;
    k_selftest_pipeline<<<1, dl::kPipeThreads, kSelfStages * kSelfTile * sizeof(float),
                          static_cast<cudaStream_t>(stream)>>>(
        d_src, n_tiles, stall_tile, static_cast<long>(polls), d_out,
        static_cast<uint32_t*>(d_workspace));
    return dl::launch_status();
}

extern "C" int dl_selftest_wait_timeout(void* d_workspace, int32_t polls, void* stream) {
    if (!d_workspace || polls <= 0 || polls > dl::kSpinLimit) return DL_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0) return DL_ERR_ALIGN;
    k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint32_t*>(d_workspace), static_cast<long>(polls));
    return dl::launch_status();
}
