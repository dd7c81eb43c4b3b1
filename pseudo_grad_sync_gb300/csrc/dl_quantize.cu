// Uniform quantisation with clipping and a bucket-mean codebook (INTELLECT-1
// notes, section 4.1 steps 2-4), fused with the uint8 encode.
//
// k_quantize   learner-group grid: the K learners form near-equal groups of at
//              most 7; a block serves one group and takes batches of
//              contiguous 8192-element chunks from its group's counter, so
//              the blocks of all groups sweep the fragment together
//              (theta_g crosses HBM once, then comes from L2) and each
//              theta_g value a block loads serves every learner of its group;
//              a block entering a tensor loads its learners' quantiser
//              parameters (derived by k_quant_setup); each chunk is loaded
//              in two halves with 128-bit loads. Per element of learner k:
//                * bucket: u = (Delta - lo) * 256 / (hi - lo) is evaluated in
//                  fp32 with one fma; an element clipped well outside the
//                  range (fp32 u below -1/2 or above 256.5) takes bucket 0
//                  or 255 with its segment's constant residual; when u is
//                  within a proven error guard of an integer (or of the range
//                  ends) the element is redone in fp64 with the exact
//                  definition, so codes equal the fp64 rule;
//                * codebook sum: the residual r = clamp(Delta) - e_b, e_b the
//                  fp32 bucket edge fmaf(b, w_f, lo_f), is exact or within
//                  2^-24 bucket widths; it becomes a biased fixed-point
//                  integer q (2^21 to 2^22 steps per bucket width, below
//                  2^23) that is added with two 32-bit shared-memory atomics:
//                  word A gets (1 << 18) + (q >> 19) (count in bits 18..31),
//                  word B gets q & (2^19 - 1). Both stay exact for up to 8192
//                  elements;
//                * no float-to-integer conversions on this path: floor(u) is
//                  read from the bits of u + 1.5 * 2^23 added rounding down,
//                  and q from the bits of fmaf(r, 2^ks, 2^23 + bias), both
//                  full-rate fp32 operations;
//                * the code byte is written with 32-bit stores (4 per store).
//              After each piece (chunk x tensor; one block barrier) thread b
//              folds bin b of the histogram into 64-bit per-bin sums it owns
//              (the histograms are double-buffered, so one barrier suffices);
//              a block serving one learner alone keeps 8 copies of its
//              histogram (fewer bank conflicts) and folds them every 8
//              pieces. The sums go to a [K][T][256] (count, residual-sum)
//              table with integer atomics when the block moves to another
//              tensor.
//              Integer sums make the result independent of addition order.
// k_quant_setup  before k_quantize: zeroes the per-bin sums and batch
//              counters and derives each (k, t)'s quantiser parameters once,
//              in fp64, from its statistics.
// k_cb_fin     one thread per (k, t, b): codebook value = reference + mean
//              residual (fp64, rounded once to fp32), midpoint for an empty
//              bucket, and the optional counts.
#include "dl_common.cuh"

namespace dl {
namespace {

struct SegRt {  // quantiser parameters of one (k, t) segment
    SegQuant q;
    float mid_g;   // 0.5 - guard
    uint32_t qb_lo, qb_hi;  // histogram words of an element clipped to lo / hi
};

// Learners per block at most: 7 learners' histograms (8 KB each) with the
// static and reserved shared memory keep three blocks within a 196 KB
// shared-memory carveout, which leaves about 60 KB of L1 for the kernel's
// in-flight 128-bit loads; 8 would need the 228 KB carveout (28 KB of L1),
// measured 4-5% slower at K = 8 and K = 16.
constexpr int kQMaxL = 7;
constexpr int kQMaxG = (DL_MAX_LEARNERS + kQMaxL - 1) / kQMaxL;  // learner groups at most

// One-learner blocks (K = 1: the learner-side quantiser, values mode) spread
// the learner's histogram over kOneCopies copies, copy = lane mod kOneCopies,
// laid out [bin][copy]: lane i's word for bin b sits in bank
// 8 (b mod 4) + i mod 8, so only the four lanes of one class can meet in a
// bank (for Gaussian codes about 2.8 instead of 3.5 passes per warp-wide
// atomic). A copy then takes at most 32 threads x 32 values = 1024 values per
// piece, so its words stay exact over kOneFoldEvery pieces between folds.
// Blocks serving several learners keep one copy per learner: the copies'
// shared memory would crowd out the L1 space their loads need.
constexpr int kOneCopies = 8;
constexpr int kOneFoldEvery = 8;

struct QuantArgs {
    const float* g;
    const float* r[DL_MAX_LEARNERS];
    uint8_t* codes[DL_MAX_LEARNERS];
    const int64_t* off;
    const dl_stats* stats;
    SegRt* seg;               // [K*T] quantiser parameters, derived once per call by k_quant_setup
    unsigned long long* acc;  // [K*T*256] x (count, biased residual sum)
    float* cb;
    uint32_t* counts;
    uint32_t* status;
    int64_t n;
    int64_t n_chunks;
    int T;
    int K;
    int G;                 // learner groups
    int gk0[kQMaxG + 1];   // first learner of group g; gk0[G] = K
    int gb0[kQMaxG + 1];   // first block of group g; gb0[G] = grid size
    unsigned int* work;    // [G] chunk-batch counters (zeroed with the sums)
    int batch;             // contiguous chunks per batch
};

constexpr uint32_t kLoMask = (1u << 19) - 1;
constexpr uint32_t kCountOne = 1u << 18;
constexpr uint32_t kQMax = (1u << 23) - 1;
constexpr float kFloorMagic = 12582912.0f;    // 1.5 * 2^23
constexpr int kFloorMagicBits = 0x4B400000;  // its fp32 bit pattern

// residual fixed point of the (clamped) value v in bucket bb, fp64
__device__ __forceinline__ uint32_t residual_q(const SegQuant& q, int bb, double v) {
    const double r = __dsub_rn(v, seg_ref(q, bb));
    long long x = llrint(ldexp(r, q.ks)) + kResBias;
    x = x < 0 ? 0 : (x > static_cast<long long>(kQMax) ? static_cast<long long>(kQMax) : x);
    return static_cast<uint32_t>(x);
}

// fp64 path of one element: the exact bucket rule and residual
__device__ __forceinline__ void rare_code(float d, const SegQuant& q, int& b, uint32_t& qv) {
    const double u = __dmul_rn(__dsub_rn(static_cast<double>(d), q.lo), q.s);
    int bb = u < 0.0 ? 0 : (u >= 256.0 ? 255 : static_cast<int>(floor(u)));
    if (bb > 255) bb = 255;
    double v = static_cast<double>(d);
    if (v < q.lo) v = q.lo;
    if (v > q.hi) v = q.hi;
    b = bb;
    qv = residual_q(q, bb, v);
}

// q (< 2^23) enters the histogram as qb = 0x4B000000 + q, the bit pattern of
// the fp32 value 2^23 + q
constexpr uint32_t kQBits = 0x4B000000u;

__device__ __forceinline__ SegRt seg_params(const dl_stats& st) {
    SegRt p;
    p.q = seg_quant(st.lo, st.hi, st.nonfinite);
    p.mid_g = 0.5f - p.q.guard;
    // an element clipped to lo (hi) lands in bucket 0 (255) with the value lo
    // (hi), so its residual is one constant per segment: what rare_code gives
    p.qb_lo = p.qb_hi = kQBits;
    if (p.q.kind == kSegFast) {
        p.qb_lo = kQBits + residual_q(p.q, 0, p.q.lo);
        p.qb_hi = kQBits + residual_q(p.q, 255, p.q.hi);
    }
    return p;
}

// word A of bin b gets one count plus q >> 19, word B gets the low 19 bits
// of q (those of qb, as 0x4B000000 has none); with R copies the lane's copy
// of each word
template <int R>
__device__ __forceinline__ void hist_add(uint32_t* __restrict__ hA, int b, uint32_t qb) {
    const int i = R == 1 ? b : b * R + static_cast<int>(threadIdx.x & (R - 1));
    atomicAdd(hA + i, (qb >> 19) + (kCountOne - (kQBits >> 19)));
    atomicAdd(hA + R * kNB + i, qb & kLoMask);
}

// Folds the R copies of bin b (words A at h[R b ..], words B R * kNB further)
// into the 64-bit sums l2l[b] (count) and l2l[kNB + b] (biased residual sum)
// and zeroes them. The 16-byte reads are staggered by b so that a warp's
// reads spread over all banks.
template <int R>
__device__ __forceinline__ void fold_copies(uint32_t* __restrict__ h, unsigned long long* __restrict__ l2l,
                                            int b) {
    constexpr int kVec = R / 4;  // 16-byte vectors per bin and word
    static_assert(kVec == 1 || kVec == 2 || kVec == 4 || kVec == 8, "R in {4, 8, 16, 32}");
    constexpr int kShift = kVec == 1 ? 3 : (kVec == 2 ? 2 : (kVec == 4 ? 1 : 0));
    uint4* pa = reinterpret_cast<uint4*>(h + b * R);
    uint4* pb = reinterpret_cast<uint4*>(h + R * kNB + b * R);
    unsigned long long cnt = 0, hi = 0, lo = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int jj = (j + (b >> kShift)) & (kVec - 1);
        const uint4 va = pa[jj], vb = pb[jj];
        cnt += (va.x >> 18) + (va.y >> 18) + (va.z >> 18) + (va.w >> 18);
        hi += (va.x & (kCountOne - 1)) + (va.y & (kCountOne - 1)) + (va.z & (kCountOne - 1)) +
              (va.w & (kCountOne - 1));
        lo += static_cast<unsigned long long>(vb.x) + vb.y + vb.z + vb.w;
        pa[jj] = make_uint4(0u, 0u, 0u, 0u);
        pb[jj] = make_uint4(0u, 0u, 0u, 0u);
    }
    l2l[b] += cnt;
    l2l[kNB + b] += (hi << 19) + lo;
}

// four codes as one 32-bit word, b0 in the lowest byte
__device__ __forceinline__ uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
    return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// bucket of one value and its histogram update; returns the code
template <int R>
__device__ __forceinline__ uint32_t encode_fast(float d, const SegRt& p, uint32_t* __restrict__ hA) {
    const float uf = __fmaf_rn(d, p.q.s_f, p.q.c_f);
    // floor(uf) for |uf| < 2^22: adding 1.5 * 2^23 rounding down lands on the
    // integer grid of [2^23, 2^24); any other uf gives b far outside [0, 256)
    const float tf = __fadd_rd(uf, kFloorMagic);
    int b = __float_as_int(tf) - kFloorMagicBits;
    const float bf = __fsub_rn(tf, kFloorMagic);
    const float fr = __fsub_rn(uf, bf);
    uint32_t qb;  // q on the bit grid of [2^23, 2^24): 0x4B000000 + q
    if (static_cast<unsigned>(b) < 256u && fabsf(__fsub_rn(fr, 0.5f)) <= p.mid_g) {
        const float r = __fsub_rn(d, __fmaf_rn(bf, p.q.w_f, p.q.lo_f));
        qb = __float_as_uint(__fmaf_rn(r, p.q.scale, p.q.qoff));
    } else if (uf < -0.5f) {
        // clipped below: for the fast kind |uf - u| <= 2^-23 |u| + 2^-23 s |lo|
        // + ... with 2^-23 s |lo| < guard / 4 < 1/16, so u < 0 and d < lo
        b = 0;
        qb = p.qb_lo;
    } else if (uf > 256.5f) {  // clipped above: likewise u > 256 and d > hi
        b = 255;
        qb = p.qb_hi;
    } else {
        uint32_t qv;
        rare_code(d, p.q, b, qv);
        qb = kQBits + qv;
    }
    hist_add<R>(hA, b, qb);
    return static_cast<uint32_t>(b);
}

template <int R>
__device__ __forceinline__ uint32_t encode_one(float d, const SegRt& p, uint32_t* __restrict__ hA) {
    if (p.q.kind == kSegFast) return encode_fast<R>(d, p, hA);
    int b;
    uint32_t qv;
    rare_code(d, p.q, b, qv);
    hist_add<R>(hA, b, kQBits + qv);
    return static_cast<uint32_t>(b);
}

__device__ __forceinline__ void flush_bin(const QuantArgs& a, int k, int t, int b,
                                          unsigned long long* l2) {
    if (l2[b] != 0ull) {
        unsigned long long* dst = a.acc + ((static_cast<int64_t>(k) * a.T + t) * kNB + b) * 2;
        atomicAdd(dst, l2[b]);
        atomicAdd(dst + 1, l2[kNB + b]);
    }
    l2[b] = 0ull;
    l2[kNB + b] = 0ull;
}

// The fast-path parameters of one segment, packed into three 16-byte words
// so that a block reloads them per learner with three broadcast loads.
struct __align__(16) FastParams {
    float s_f, c_f, w_f, lo_f;
    float scale, qoff, mid_g;
    uint32_t qb_lo, qb_hi;
    int kind;
    int pad0, pad1;
};

__device__ __forceinline__ FastParams fast_params(const SegRt& p) {
    FastParams f;
    f.s_f = p.q.s_f;
    f.c_f = p.q.c_f;
    f.w_f = p.q.w_f;
    f.lo_f = p.q.lo_f;
    f.scale = p.q.scale;
    f.qoff = p.q.qoff;
    f.mid_g = p.mid_g;
    f.qb_lo = p.qb_lo;
    f.qb_hi = p.qb_hi;
    f.kind = p.q.kind;
    f.pad0 = f.pad1 = 0;
    return f;
}

// bucket of one value of a fast-kind segment and its histogram update (the
// same arithmetic as encode_fast; the fp64 rule from the full parameters)
template <int R>
__device__ __forceinline__ uint32_t encode_fp(float d, const FastParams& f, const SegRt* full,
                                              uint32_t* __restrict__ hA) {
    const float uf = __fmaf_rn(d, f.s_f, f.c_f);
    const float tf = __fadd_rd(uf, kFloorMagic);
    int b = __float_as_int(tf) - kFloorMagicBits;
    const float bf = __fsub_rn(tf, kFloorMagic);
    const float fr = __fsub_rn(uf, bf);
    uint32_t qb;
    if (static_cast<unsigned>(b) < 256u && fabsf(__fsub_rn(fr, 0.5f)) <= f.mid_g) {
        const float r = __fsub_rn(d, __fmaf_rn(bf, f.w_f, f.lo_f));
        qb = __float_as_uint(__fmaf_rn(r, f.scale, f.qoff));
    } else if (uf < -0.5f) {
        b = 0;
        qb = f.qb_lo;
    } else if (uf > 256.5f) {
        b = 255;
        qb = f.qb_hi;
    } else {
        uint32_t qv;
        rare_code(d, full->q, b, qv);
        qb = kQBits + qv;
    }
    hist_add<R>(hA, b, qb);
    return static_cast<uint32_t>(b);
}

// Four values of a fast-kind segment, packed codes returned. When all four
// values of every lane take encode_fp's first branch (the common case), the
// warp runs that branch's arithmetic straight through, with the four
// histogram updates back to back; otherwise each value goes through
// encode_fp. Both routes give the same codes and sums.
template <int R>
__device__ __forceinline__ uint32_t encode4_fp(float4 gq, float4 rq, const FastParams& f,
                                               const SegRt* full, uint32_t* __restrict__ hA) {
    const float d[4] = {__fsub_rn(gq.x, rq.x), __fsub_rn(gq.y, rq.y), __fsub_rn(gq.z, rq.z),
                        __fsub_rn(gq.w, rq.w)};
    float bf[4];
    int b[4];
    bool ok = true;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float uf = __fmaf_rn(d[e], f.s_f, f.c_f);
        const float tf = __fadd_rd(uf, kFloorMagic);
        b[e] = __float_as_int(tf) - kFloorMagicBits;
        bf[e] = __fsub_rn(tf, kFloorMagic);
        const float fr = __fsub_rn(uf, bf[e]);
        ok = ok && static_cast<unsigned>(b[e]) < 256u && fabsf(__fsub_rn(fr, 0.5f)) <= f.mid_g;
    }
    if (__all_sync(kFull, ok)) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float r = __fsub_rn(d[e], __fmaf_rn(bf[e], f.w_f, f.lo_f));
            hist_add<R>(hA, b[e], __float_as_uint(__fmaf_rn(r, f.scale, f.qoff)));
        }
        return pack4(b[0], b[1], b[2], b[3]);
    }
    const uint32_t c0 = encode_fp<R>(d[0], f, full, hA);
    const uint32_t c1 = encode_fp<R>(d[1], f, full, hA);
    const uint32_t c2 = encode_fp<R>(d[2], f, full, hA);
    const uint32_t c3 = encode_fp<R>(d[3], f, full, hA);
    return pack4(c0, c1, c2, c3);
}

constexpr int kBatchesPerBlock = 32;  // chunk batches a block takes, about
constexpr int kMaxBatch = 16;         // chunks per batch at most

// 32-bit histogram words of a quantiser block: serving L learners, the
// double-buffered [2][L][word A bins | word B bins]; serving one learner
// alone, [word A bins x copies | word B bins x copies].
__host__ __device__ constexpr size_t quant_hist_words(int L, bool one) {
    return one ? static_cast<size_t>(2) * kOneCopies * kNB : static_cast<size_t>(L) * 2 * 2 * kNB;
}

// Dynamic shared memory of a quantiser block: the histogram words and the
// 64-bit per-bin sums [L][count bins | residual-sum bins].
__host__ __device__ constexpr size_t quant_smem(int L, bool one) {
    return quant_hist_words(L, one) * 4 + static_cast<size_t>(L) * 2 * kNB * 8;
}

// Learner-group grid: the K learners form G near-equal groups of at most
// kQMaxL; group g has blocks gb0[g] .. gb0[g+1]-1, as many as its share of the
// learners. A block takes batches of contiguous chunks (about 32 per block,
// 1 to 16 chunks each) from its group's counter until none is left, so
// blocks that meet costly chunks (many small tensors) take fewer, and the
// blocks of all groups sweep the fragment together (the theta_g they read is
// shared through L2). Per half-chunk a thread loads its
// theta_g values once and then, learner by learner, that learner's replica
// values: theta_g is read once per group, not once per learner, and each
// piece's block barrier and histogram fold serve L learners.
// VALUES: values mode (no replica; Delta is theta_g itself, K = 1). ONE: one
// learner per block (K = 1): its parameters stay in registers, each block
// takes one static contiguous run of chunks, and its histogram has
// kOneCopies copies, folded every kOneFoldEvery pieces and when the block
// moves to another tensor.
template <bool VALUES, bool ONE>
__global__ void __launch_bounds__(kThreads, 3) k_quantize(QuantArgs a) {
    extern __shared__ __align__(16) unsigned char qsm[];
    __shared__ SegRt s_seg[kQMaxL];       // parameters of the current tensor, per learner
    __shared__ FastParams s_fp[kQMaxL];
    __shared__ unsigned int s_item;
    int grp = 0;
    while (grp + 1 < a.G && static_cast<int>(blockIdx.x) >= a.gb0[grp + 1]) ++grp;
    const int k0 = a.gk0[grp];
    const int L = ONE ? 1 : a.gk0[grp + 1] - k0;
    constexpr int R = ONE ? kOneCopies : 1;  // histogram copies per learner
    const int hist_words = static_cast<int>(quant_hist_words(L, ONE));
    uint32_t* l1 = reinterpret_cast<uint32_t*>(qsm);
    unsigned long long* l2 = reinterpret_cast<unsigned long long*>(qsm + static_cast<size_t>(hist_words) * 4);

    const int tid = threadIdx.x;
    const float* __restrict__ g = a.g;
    for (int i = tid; i < hist_words; i += kThreads) l1[i] = 0u;
    for (int i = tid; i < L * 2 * kNB; i += kThreads) l2[i] = 0ull;
    __syncthreads();

    int cur_t = -1;  // tensor whose sums are in l2
    int seg_t = -1;  // tensor whose parameters are in s_seg
    int par = 0;     // learner groups: the histogram buffer of this piece
    int since = 0;   // one learner: pieces since the copies were folded
    FastParams f_one;  // ONE: the learner's parameters for the current tensor
    // Learner groups: thread 0 fetches the next batch while the block works on
    // the current one. One learner per block (no group to share theta_g with):
    // one static contiguous run of chunks per block, no fetches.
    unsigned int next = (!ONE && tid == 0) ? atomicAdd(a.work + grp, 1u) : 0u;
    for (int round = 0;; ++round) {
    int64_t c_lo, c_hi;
    if (ONE) {
        if (round > 0) break;
        c_lo = a.n_chunks * blockIdx.x / gridDim.x;
        c_hi = a.n_chunks * (blockIdx.x + 1) / gridDim.x;
    } else {
        if (tid == 0) s_item = next;
        __syncthreads();
        c_lo = static_cast<int64_t>(s_item) * a.batch;
        __syncthreads();  // every thread has read s_item
        if (c_lo >= a.n_chunks) break;
        if (tid == 0) next = atomicAdd(a.work + grp, 1u);
        c_hi = min(c_lo + a.batch, a.n_chunks);
    }
    for (int64_t c = c_lo; c < c_hi; ++c) {
        const int64_t base = c * kChunk;
        const int64_t cend = min(base + kChunk, a.n);
        for (int t = tensor_containing(a.off, a.T, base); t < a.T; ++t) {
            const int64_t o0 = __ldg(a.off + t), o1 = __ldg(a.off + t + 1);
            if (o0 >= cend) break;
            const int64_t pa = o0 > base ? o0 : base;
            const int64_t pb = o1 < cend ? o1 : cend;
            if (pa >= pb) continue;
            if (t != seg_t) {  // block-uniform: threads 0..L-1 load the parameters
                __syncthreads();  // every read of the previous ones is done
                if (tid < L) {
                    s_seg[tid] = a.seg[static_cast<int64_t>(k0 + tid) * a.T + t];
                    s_fp[tid] = fast_params(s_seg[tid]);
                }
                __syncthreads();
                if (ONE) f_one = s_fp[0];
                seg_t = t;
            }
            if constexpr (ONE) {
                if (t != cur_t || since == kOneFoldEvery) {  // block-uniform
                    __syncthreads();  // every update so far is in the copies
                    if (cur_t >= 0) {
                        fold_copies<R>(l1, l2, tid);
                        if (t != cur_t) flush_bin(a, k0, cur_t, tid, l2);
                    }
                    cur_t = t;
                    since = 0;
                    __syncthreads();  // the copies are zero again
                }
            }
            const bool full = (pa == base) && (pb == base + kChunk);
            uint32_t* hpar = ONE ? l1 : l1 + static_cast<size_t>(par) * L * 2 * kNB;
            if (full) {
                const float4* g4 = reinterpret_cast<const float4*>(g + base);
#pragma unroll 1
                for (int h = 0; h < kGroups; h += kGroups / 2) {  // two halves: fewer registers
                    float4 gv[kGroups / 2];
#pragma unroll
                    for (int q = 0; q < kGroups / 2; ++q) gv[q] = __ldg(g4 + tid + (h + q) * kThreads);
#pragma unroll 1
                    for (int l = 0; l < L; ++l) {
                        const FastParams f = ONE ? f_one : s_fp[l];
                        uint32_t* c4 = reinterpret_cast<uint32_t*>(a.codes[k0 + l] + base);
                        if (f.kind >= kSegDegenerate) {  // every code is 0, no sums
#pragma unroll
                            for (int q = 0; q < kGroups / 2; ++q) c4[tid + (h + q) * kThreads] = 0u;
                            continue;
                        }
                        uint32_t* hA = hpar + l * 2 * R * kNB;
                        const float4* r4 = reinterpret_cast<const float4*>(a.r[k0 + l] + base);
                        float4 rv[kGroups / 2];
#pragma unroll
                        for (int q = 0; q < kGroups / 2; ++q)
                            rv[q] = VALUES ? make_float4(0.f, 0.f, 0.f, 0.f)
                                           : __ldcs(r4 + tid + (h + q) * kThreads);
                        if (f.kind == kSegFast) {
#pragma unroll
                            for (int q = 0; q < kGroups / 2; ++q)
                                c4[tid + (h + q) * kThreads] = encode4_fp<R>(gv[q], rv[q], f, s_seg + l, hA);
                        } else {
                            const SegRt p = s_seg[l];
#pragma unroll
                            for (int q = 0; q < kGroups / 2; ++q) {
                                const uint32_t b0 = encode_one<R>(__fsub_rn(gv[q].x, rv[q].x), p, hA);
                                const uint32_t b1 = encode_one<R>(__fsub_rn(gv[q].y, rv[q].y), p, hA);
                                const uint32_t b2 = encode_one<R>(__fsub_rn(gv[q].z, rv[q].z), p, hA);
                                const uint32_t b3 = encode_one<R>(__fsub_rn(gv[q].w, rv[q].w), p, hA);
                                c4[tid + (h + q) * kThreads] = pack4(b0, b1, b2, b3);
                            }
                        }
                    }
                }
            } else {
                for (int l = 0; l < L; ++l) {
                    uint8_t* __restrict__ ck = a.codes[k0 + l];
                    const SegRt p = s_seg[l];
                    if (p.q.kind >= kSegDegenerate) {
                        for (int64_t e = pa + tid; e < pb; e += kThreads) ck[e] = 0;
                        continue;
                    }
                    const float* __restrict__ rk = a.r[k0 + l];
                    uint32_t* hA = hpar + l * 2 * R * kNB;
                    for (int64_t e = pa + tid; e < pb; e += kThreads) {
                        const float d = __fsub_rn(__ldg(g + e), VALUES ? 0.f : __ldcs(rk + e));
                        ck[e] = static_cast<uint8_t>(encode_one<R>(d, p, hA));
                    }
                }
            }
            if constexpr (ONE) {
                ++since;
                continue;
            }
            __syncthreads();  // every update of this piece is in l1[par]
            if (cur_t != t) {
                if (cur_t >= 0)
                    for (int l = 0; l < L; ++l) flush_bin(a, k0 + l, cur_t, tid, l2 + l * 2 * kNB);
                cur_t = t;
            }
            for (int l = 0; l < L; ++l) {
                uint32_t* hA = hpar + l * 2 * kNB;
                unsigned long long* l2l = l2 + l * 2 * kNB;
                const uint32_t va = hA[tid], vb = hA[kNB + tid];
                if (va != 0u) {
                    l2l[tid] += va >> 18;
                    l2l[kNB + tid] += (static_cast<unsigned long long>(va & ((1u << 18) - 1)) << 19) + vb;
                    hA[tid] = 0u;
                    hA[kNB + tid] = 0u;
                }
            }
            par ^= 1;
        }
    }
    }
    if constexpr (ONE) {
        __syncthreads();  // every update is in the copies
        if (cur_t >= 0) fold_copies<R>(l1, l2, tid);
    }
    if (cur_t >= 0)
        for (int l = 0; l < L; ++l) flush_bin(a, k0 + l, cur_t, tid, l2 + l * 2 * kNB);
}

// Before the quantiser: zeroes the workspace's zeroed part (per-bin sums and
// batch counters, n16 16-byte words at zero) and derives the quantiser
// parameters of every (learner, tensor) once from its statistics, for the
// quantiser blocks to load when they enter a tensor and for k_cb_fin. (Derived
// in each block instead, this fp64 work sat on the critical path of every
// block at every tensor it entered.)
__global__ void __launch_bounds__(kThreads) k_quant_setup(QuantArgs a, uint4* zero, int64_t n16) {
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = i0; i < n16; i += stride) zero[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t i = i0; i < static_cast<int64_t>(a.K) * a.T; i += stride) a.seg[i] = seg_params(a.stats[i]);
}

__global__ void __launch_bounds__(kThreads) k_cb_fin(QuantArgs a) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(a.K) * a.T * kNB) return;
    const int64_t kt = idx >> 8;
    const int b = static_cast<int>(idx & (kNB - 1));
    const dl_stats st = a.stats[kt];
    const SegQuant q = a.seg[kt].q;
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

// the workspace's zeroed part: the sums, then the groups' batch counters
size_t zeroed_bytes(int K, int T) { return acc_bytes(K, T) + 256; }

// the per-(learner, tensor) quantiser parameters, after the zeroed part
size_t seg_bytes(int K, int T) { return align256(sizeof(SegRt) * static_cast<size_t>(K) * T); }

// The no-allocation entry point's static array holds the workspace of its
// largest fragment (DL_QUANTIZE_NOALLOC_MAX_SEGMENTS (learner, tensor) pairs).
static_assert(sizeof(SegRt) <= 96, "per-segment parameters grew");
static_assert(kWsHeader + 2 * 8 * 256 * static_cast<size_t>(DL_QUANTIZE_NOALLOC_MAX_SEGMENTS) + 256 +
                      96 * static_cast<size_t>(DL_QUANTIZE_NOALLOC_MAX_SEGMENTS) <=
                  DL_QUANTIZE_NOALLOC_MAX_BYTES,
              "the no-allocation scratch no longer holds its largest fragment");

// Learner groups of the quantiser grid (see k_quantize) for K learners and a
// grid of `blocks`: G near-equal groups, blocks shared in proportion.
void plan_groups(QuantArgs& a, int K, int blocks) {
    const int G = (K + kQMaxL - 1) / kQMaxL;
    a.G = G;
    a.gk0[0] = 0;
    for (int g = 0; g < G; ++g) a.gk0[g + 1] = a.gk0[g] + K / G + (g < K % G ? 1 : 0);
    a.gb0[0] = 0;
    for (int g = 0; g < G; ++g) {
        const int64_t share = static_cast<int64_t>(blocks) * a.gk0[g + 1] / K;
        a.gb0[g + 1] = static_cast<int>(share > a.gb0[g] ? share : a.gb0[g] + 1);
    }
}

}  // namespace
}  // namespace dl

using namespace dl;

extern "C" size_t dl_quantize_workspace_bytes(const dl_fragment* frag, int32_t K) {
    HostFrag f;
    if (check_fragment(frag, &f) != DL_OK || K <= 0 || K > DL_MAX_LEARNERS) return 0;
    return kWsHeader + zeroed_bytes(K, f.T) + seg_bytes(K, f.T);
}

extern "C" int dl_quantize(const float* theta_g, const float* const* theta_k, int32_t K,
                           const dl_fragment* frag, const dl_stats* d_stats, uint8_t* const* codes,
                           float* d_codebook, uint32_t* d_counts, void* d_workspace,
                           size_t workspace_bytes, void* stream) {
    HostFrag f;
    int st = check_fragment(frag, &f);
    if (st != DL_OK) return st;
    const bool values = theta_k == nullptr;  // Delta is theta_g itself
    if (K <= 0 || K > DL_MAX_LEARNERS || (values && K != 1) || !codes) return DL_ERR_ARG;
    if (f.T == 0) return DL_OK;
    if (!d_stats || !d_codebook) return DL_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_stats) & 7u) != 0 || !aligned16(d_codebook) ||
        (d_counts && !aligned16(d_counts)))
        return DL_ERR_ALIGN;
    if (f.n > 0) {
        if (!theta_g) return DL_ERR_ARG;
        if (!aligned16(theta_g)) return DL_ERR_ALIGN;
        for (int k = 0; k < K; ++k) {
            if ((!values && !theta_k[k]) || !codes[k]) return DL_ERR_ARG;
            if ((!values && !aligned16(theta_k[k])) || !aligned16(codes[k])) return DL_ERR_ALIGN;
        }
    }
    const size_t need = dl_quantize_workspace_bytes(frag, K);
    if (!d_workspace || workspace_bytes < need) return DL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0) return DL_ERR_ALIGN;

    QuantArgs a;
    memset(&a, 0, sizeof(a));
    a.g = theta_g;
    for (int k = 0; k < K; ++k) {
        a.r[k] = values ? nullptr : theta_k[k];
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

    a.work = reinterpret_cast<unsigned int*>(ws + kWsHeader + acc_bytes(K, f.T));
    a.seg = reinterpret_cast<SegRt*>(ws + kWsHeader + zeroed_bytes(K, f.T));
    {
        const int64_t n16 = static_cast<int64_t>(zeroed_bytes(K, f.T) / 16);
        const int64_t items = n16 > static_cast<int64_t>(K) * f.T ? n16 : static_cast<int64_t>(K) * f.T;
        const int64_t blocks = (items + kThreads - 1) / kThreads;
        k_quant_setup<<<static_cast<unsigned>(blocks < 1024 ? blocks : 1024), kThreads, 0, s>>>(
            a, reinterpret_cast<uint4*>(a.acc), n16);
        if ((st = launch_status()) != DL_OK) return st;
    }
    if (a.n_chunks > 0) {
        const void* kern = values ? reinterpret_cast<const void*>(k_quantize<true, true>)
                           : K == 1 ? reinterpret_cast<const void*>(k_quantize<false, true>)
                                    : reinterpret_cast<const void*>(k_quantize<false, false>);
        const int Lmax = (K + (K + kQMaxL - 1) / kQMaxL - 1) / ((K + kQMaxL - 1) / kQMaxL);
        const size_t smem = quant_smem(Lmax, K == 1);
        // the instance's largest need, whatever K this call has
        const size_t smem_max = K == 1 ? quant_smem(1, true) : quant_smem(kQMaxL, false);
        if ((st = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem_max)))) != DL_OK)
            return st;
        plan_groups(a, K, grid_for(kern, kThreads, smem, a.n_chunks * ((K + kQMaxL - 1) / kQMaxL)));
        const int grid = a.gb0[a.G];
        // batches of contiguous chunks, about kBatchesPerBlock per block: short
        // enough that the last ones finish together, long enough that a block
        // rarely changes tensor between batches
        const int64_t per_block = a.n_chunks * a.G / (static_cast<int64_t>(grid) * kBatchesPerBlock);
        a.batch = static_cast<int>(per_block < 1 ? 1 : (per_block > kMaxBatch ? kMaxBatch : per_block));
        if (values)
            k_quantize<true, true><<<grid, kThreads, smem, s>>>(a);
        else if (K == 1)
            k_quantize<false, true><<<grid, kThreads, smem, s>>>(a);
        else
            k_quantize<false, false><<<grid, kThreads, smem, s>>>(a);
        if ((st = launch_status()) != DL_OK) return st;
    }
    const int64_t cells = static_cast<int64_t>(K) * f.T * kNB;
    k_cb_fin<<<static_cast<unsigned>((cells + kThreads - 1) / kThreads), kThreads, 0, s>>>(a);
    return launch_status();
}

// ---------------------------------------------------------------------------
// dl_quantize for callers that cannot allocate: the workspace is this static
// device array (one per device, alive until the process exits). In host code
// the symbol is only a stand-in; its device address on the current device
// comes from cudaGetSymbolAddress, looked up on every call (a cached address
// would go stale after a device reset or a new primary context).

namespace {
static __device__ __align__(256) unsigned char g_quant_scratch[DL_QUANTIZE_NOALLOC_MAX_BYTES];

int scratch_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_quant_scratch) != cudaSuccess || !p) return DL_ERR_CUDA;
    *out = p;
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
    if (static_cast<int64_t>(K) * f.T > DL_QUANTIZE_NOALLOC_MAX_SEGMENTS ||
        dl_quantize_workspace_bytes(frag, K) > DL_QUANTIZE_NOALLOC_MAX_BYTES)
        return DL_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != DL_OK) return st;
    return dl_quantize(theta_g, theta_k, K, frag, d_stats, codes, d_codebook, d_counts, scratch,
                       DL_QUANTIZE_NOALLOC_MAX_BYTES, stream);
}
