// Uniform quantisation with clipping and a bucket-mean codebook (INTELLECT-1
// notes, section 4.1 steps 2-4), fused with the uint8 encode.
//
// k_quantize   persistent blocks over 8192-element chunks; theta_g's chunk is
//              staged in shared memory by one bulk (TMA) copy and reused for
//              all K learners. Per element of learner k:
//                * bucket: u = (Delta - lo) * 256 / (hi - lo) is evaluated in
//                  fp32; when u is within a proven error guard of an integer
//                  (or outside (0, 256)) the element is redone in fp64 with
//                  the exact definition, so codes equal the fp64 rule;
//                * codebook sum: the residual r = clamp(Delta) - e_b, e_b the
//                  fp32 bucket edge fmaf(b, w_f, lo_f), is exact or within
//                  2^-24 bucket widths; it becomes a fixed-point integer (2^26 steps per bucket
//                  width) and added, together with a count of one, as a single
//                  64-bit shared-memory atomic into the block's histogram
//                  (count in bits 44..63). Integer sums make the result
//                  independent of the order of the additions;
//                * the code byte is written with 32-bit stores (4 per store).
//              Block histograms are flushed into a [K][T][256] global
//              (count, residual-sum) table with integer atomics whenever the
//              block moves to another tensor or may reach 2^16 elements.
// k_cb_fin     one thread per (k, t, b): codebook value = reference + mean
//              residual (fp64, rounded once to fp32), midpoint for an empty
//              bucket, and the optional counts.
#include <mutex>

#include "dl_common.cuh"

namespace dl {
namespace {

struct QuantArgs {
    const float* g;
    const float* r[DL_MAX_LEARNERS];
    uint8_t* codes[DL_MAX_LEARNERS];
    const int64_t* off;
    const dl_stats* stats;
    unsigned long long* acc;  // [K*T*256] x (count, residual sum)
    float* cb;
    uint32_t* counts;
    uint32_t* status;
    int64_t n;
    int64_t n_chunks;
    int T;
    int K;
};

// elements a block may add to one bucket between flushes: every packed
// value is < 2^28 and the low field holds 44 bits
constexpr int kFlushLimit = 1 << 16;

struct SegRt {  // per-(k, current tensor) parameters kept in shared memory
    SegQuant q;
    float hi_g;   // 256 - guard
    float mid_g;  // 0.5 - guard
};

__device__ __forceinline__ void rare_code(float d, const SegQuant& q, int& b, int& qv) {
    const double u = __dmul_rn(__dsub_rn(static_cast<double>(d), q.lo), q.s);
    int bb = u < 0.0 ? 0 : (u >= 256.0 ? 255 : static_cast<int>(floor(u)));
    if (bb > 255) bb = 255;
    double v = static_cast<double>(d);
    if (v < q.lo) v = q.lo;
    if (v > q.hi) v = q.hi;
    const double r = __dsub_rn(v, seg_ref(q, bb));
    b = bb;
    qv = static_cast<int>(llrint(ldexp(r, q.ks))) + static_cast<int>(kResBias);
}

// bucket of one value and its histogram update; returns the code
__device__ __forceinline__ uint32_t encode_one(float d, const SegRt& p,
                                               unsigned long long* __restrict__ hk) {
    int b, qv;
    const float t = __fsub_rn(d, p.q.lo_f);
    const float uf = __fmul_rn(t, p.q.s_f);
    const float bf = floorf(uf);
    const float fr = __fsub_rn(uf, bf);
    if (p.q.kind == kSegFast && uf >= p.q.guard && uf <= p.hi_g &&
        fabsf(__fsub_rn(fr, 0.5f)) <= p.mid_g) {
        b = static_cast<int>(bf);
        const float r = __fsub_rn(d, __fmaf_rn(bf, p.q.w_f, p.q.lo_f));
        qv = __float2int_rn(__fmul_rn(r, p.q.scale)) + static_cast<int>(kResBias);
    } else {
        rare_code(d, p.q, b, qv);
    }
    atomicAdd(hk + b, (1ull << kCountShift) + static_cast<unsigned long long>(static_cast<unsigned>(qv)));
    return static_cast<uint32_t>(b);
}

__device__ void flush_hist(unsigned long long* hist, const QuantArgs& a, int t) {
    __syncthreads();
    for (int i = threadIdx.x; i < a.K * kNB; i += kThreads) {
        const unsigned long long v = hist[i];
        if (v) {
            const int k = i >> 8, b = i & (kNB - 1);
            unsigned long long* dst =
                a.acc + ((static_cast<int64_t>(k) * a.T + t) * kNB + b) * 2;
            atomicAdd(dst, v >> kCountShift);
            atomicAdd(dst + 1, v & ((1ull << kCountShift) - 1));
            hist[i] = 0ull;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) k_quantize(QuantArgs a) {
    extern __shared__ __align__(16) float sg[];  // kChunk floats, then K*256 u64
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(sg + kChunk);
    __shared__ uint64_t bar;
    __shared__ int flag;
    __shared__ SegRt seg[DL_MAX_LEARNERS];

    const int tid = threadIdx.x;
    for (int i = tid; i < a.K * kNB; i += kThreads) hist[i] = 0ull;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();

    int cur_t = -1;
    int acc_elems = 0;
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
            const int plen = static_cast<int>(pb - pa);
            if (t != cur_t || acc_elems + plen > kFlushLimit) {
                if (cur_t >= 0) flush_hist(hist, a, cur_t);
                if (t != cur_t) {
                    if (tid < a.K) {
                        const dl_stats st = a.stats[static_cast<int64_t>(tid) * a.T + t];
                        SegRt p;
                        p.q = seg_quant(st.lo, st.hi, st.nonfinite);
                        p.hi_g = 256.0f - p.q.guard;
                        p.mid_g = 0.5f - p.q.guard;
                        seg[tid] = p;
                    }
                    __syncthreads();
                }
                cur_t = t;
                acc_elems = 0;
            }
            acc_elems += plen;
            const bool full = (pa == base) && (pb == base + kChunk);
            const int la = static_cast<int>(pa - base), lb = static_cast<int>(pb - base);

            for (int k = 0; k < a.K; ++k) {
                const SegRt p = seg[k];
                uint8_t* ck = a.codes[k] + base;
                const float* rk = a.r[k] + base;
                unsigned long long* hk = hist + k * kNB;
                if (p.q.kind >= kSegDegenerate) {  // every code is 0
                    if (full) {
#pragma unroll
                        for (int j = 0; j < kGroups; ++j)
                            reinterpret_cast<uint32_t*>(ck)[tid + j * kThreads] = 0u;
                    } else {
                        for (int e = la + tid; e < lb; e += kThreads) ck[e] = 0;
                    }
                    continue;
                }
                if (full) {
                    float4 v[kGroups];
#pragma unroll
                    for (int j = 0; j < kGroups; ++j)
                        v[j] = __ldcs(reinterpret_cast<const float4*>(rk) + tid + j * kThreads);
#pragma unroll
                    for (int j = 0; j < kGroups; ++j) {
                        const float4 gg = reinterpret_cast<const float4*>(sg)[tid + j * kThreads];
                        const uint32_t b0 = encode_one(__fsub_rn(gg.x, v[j].x), p, hk);
                        const uint32_t b1 = encode_one(__fsub_rn(gg.y, v[j].y), p, hk);
                        const uint32_t b2 = encode_one(__fsub_rn(gg.z, v[j].z), p, hk);
                        const uint32_t b3 = encode_one(__fsub_rn(gg.w, v[j].w), p, hk);
                        reinterpret_cast<uint32_t*>(ck)[tid + j * kThreads] =
                            b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
                    }
                } else {
                    for (int e = la + tid; e < lb; e += kThreads) {
                        const float d = __fsub_rn(sg[e], __ldcs(rk + e));
                        ck[e] = static_cast<uint8_t>(encode_one(d, p, hk));
                    }
                }
            }
        }
        __syncthreads();  // the staged chunk is about to be overwritten
    }
    if (cur_t >= 0) flush_hist(hist, a, cur_t);
}

__global__ void __launch_bounds__(kThreads) k_cb_fin(QuantArgs a) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(a.K) * a.T * kNB) return;
    const int64_t kt = idx >> 8;
    const int b = static_cast<int>(idx & (kNB - 1));
    const dl_stats st = a.stats[kt];
    const SegQuant q = seg_quant(st.lo, st.hi, st.nonfinite);
    float v;
    unsigned long long cnt = 0;
    if (q.kind == kSegInvalid) {
        v = __int_as_float(0x7fc00000);
    } else if (q.kind == kSegDegenerate) {
        v = static_cast<float>(st.mean);
        cnt = b == 0 ? static_cast<unsigned long long>(st.count) : 0ull;
    } else {
        cnt = a.acc[idx * 2];
        if (cnt > 0) {
            const long long net = static_cast<long long>(a.acc[idx * 2 + 1]) -
                                  static_cast<long long>(cnt) * kResBias;
            const double mean_r = ldexp(static_cast<double>(net), -q.ks) / static_cast<double>(cnt);
            const double ref = seg_ref(q, b);
            v = static_cast<float>(__dadd_rn(ref, mean_r));
        } else {  // empty bucket: its midpoint
            const double mid = __ddiv_rn(__dmul_rn(static_cast<double>(b) + 0.5, __dsub_rn(q.hi, q.lo)), 256.0);
            v = static_cast<float>(__dadd_rn(q.lo, mid));
        }
    }
    a.cb[idx] = v;
    if (a.counts) a.counts[idx] = static_cast<uint32_t>(cnt);
}

size_t acc_bytes(int K, int T) {
    return align256(sizeof(unsigned long long) * 2 * static_cast<size_t>(K) * T * kNB);
}

}  // namespace
}  // namespace dl

using namespace dl;

extern "C" size_t dl_quantize_workspace_bytes(const dl_fragment* frag, int32_t K) {
    HostFrag f;
    if (check_fragment(frag, &f) != DL_OK || K <= 0 || K > DL_MAX_LEARNERS) return 0;
    return kWsHeader + acc_bytes(K, f.T);
}

extern "C" int dl_quantize(const float* theta_g, const float* const* theta_k, int32_t K,
                           const dl_fragment* frag, const dl_stats* d_stats, uint8_t* const* codes,
                           float* d_codebook, uint32_t* d_counts, void* d_workspace,
                           size_t workspace_bytes, void* stream) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    if (K <= 0 || K > DL_MAX_LEARNERS || !theta_k || !codes) return DL_ERR_ARG;
    if (f.T == 0) return DL_OK;
    if (!d_stats || !d_codebook) return DL_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_stats) & 7u) != 0 || !aligned16(d_codebook) ||
        (d_counts && !aligned16(d_counts)))
        return DL_ERR_ALIGN;
    if (f.n > 0) {
        if (!theta_g) return DL_ERR_ARG;
        if (!aligned16(theta_g)) return DL_ERR_ALIGN;
        for (int k = 0; k < K; ++k) {
            if (!theta_k[k] || !codes[k]) return DL_ERR_ARG;
            if (!aligned16(theta_k[k]) || !aligned16(codes[k])) return DL_ERR_ALIGN;
        }
    }
    const size_t need = dl_quantize_workspace_bytes(frag, K);
    if (!d_workspace || workspace_bytes < need) return DL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0) return DL_ERR_ALIGN;

    QuantArgs a;
    memset(&a, 0, sizeof(a));
    a.g = theta_g;
    for (int k = 0; k < K; ++k) {
        a.r[k] = theta_k[k];
        a.codes[k] = codes[k];
    }
    a.off = f.d_offsets;
    a.stats = d_stats;
    char* ws = static_cast<char*>(d_workspace);
    a.status = reinterpret_cast<uint32_t*>(ws);
    a.acc = reinterpret_cast<unsigned long long*>(ws + kWsHeader);
    a.cb = d_codebook;
    a.counts = d_counts;
    a.n = f.n;
    a.n_chunks = n_chunks_of(f.n);
    a.T = f.T;
    a.K = K;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if ((st = cuda_status(cudaMemsetAsync(a.acc, 0, acc_bytes(K, f.T), s))) != DL_OK) return st;
    if (a.n_chunks > 0) {
        const size_t smem = sizeof(float) * kChunk + sizeof(unsigned long long) * kNB * K;
        if ((st = cuda_status(cudaFuncSetAttribute(k_quantize, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem)))) != DL_OK)
            return st;
        const int grid = grid_for(reinterpret_cast<const void*>(k_quantize), kThreads, smem, a.n_chunks);
        k_quantize<<<grid, kThreads, smem, s>>>(a);
        if ((st = launch_status()) != DL_OK) return st;
    }
    const int64_t cells = static_cast<int64_t>(K) * f.T * kNB;
    k_cb_fin<<<static_cast<unsigned>((cells + kThreads - 1) / kThreads), kThreads, 0, s>>>(a);
    return launch_status();
}

// ---------------------------------------------------------------------------
// dl_quantize for callers that cannot allocate: the workspace is this static
// device array (one per device, alive until the process exits). In host code
// the symbol is only a stand-in; its device address comes from
// cudaGetSymbolAddress, looked up once per device on the first call.

namespace {
static __device__ __align__(256) unsigned char g_quant_scratch[DL_QUANTIZE_NOALLOC_MAX_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DL_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_quant_scratch) != cudaSuccess || !p) return DL_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DL_OK;
}
}  // namespace

extern "C" int dl_quantize_noalloc(const float* theta_g, const float* const* theta_k, int32_t K,
                                   const dl_fragment* frag, const dl_stats* d_stats,
                                   uint8_t* const* codes, float* d_codebook, uint32_t* d_counts,
                                   void* stream) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    if (K <= 0 || K > DL_MAX_LEARNERS) return DL_ERR_ARG;
    if (dl_quantize_workspace_bytes(frag, K) > DL_QUANTIZE_NOALLOC_MAX_BYTES) return DL_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != DL_OK) return st;
    return dl_quantize(theta_g, theta_k, K, frag, d_stats, codes, d_codebook, d_counts, scratch,
                       DL_QUANTIZE_NOALLOC_MAX_BYTES, stream);
}
