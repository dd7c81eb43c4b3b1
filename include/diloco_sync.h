/*
 * diloco_sync.h - C ABI of the GB300 DiLoCo outer-synchronisation library.
 *
 * One call sequence syncs one fragment of a model whose K learner replicas
 * already sit in this GPU's memory:
 *
 *   dl_plan_fragments      (host, once)  tensors -> P balanced fragments
 *   dl_pseudograd_stats    (device)      per-(learner, tensor) mu / sigma
 *   dl_quantize            (device)      uint8 codes + bucket-mean codebooks
 *   dl_merge_outer_step    (device)      decode, weighted fp32 mean, Nesterov
 *
 * dl_outer_sync runs that sequence over every fragment of a model in one
 * call, overlapping consecutive fragments on two streams; flags select the
 * RDA merge or the re-quantising ring in place of the mean merge.
 *
 * Sources: the INTELLECT-1 paper notes ("INTELLECT-1: Training a 10B Model
 * Across 3 Continents", sections 3.2, 4.1 and 4.2) define the pseudo-gradient,
 * the 6-sigma / 256-bucket quantiser with a bucket-mean codebook, the fp32
 * accumulation rule and the outer Nesterov step (lr 0.7, momentum 0.9); the
 * Decoupled DiLoCo note ("Decoupled DiLoCo: Resilient, Distributed AI
 * Training at Scale", architecture item 4 and fault-tolerance items 1 and 3)
 * defines fragments packed by greedy bin-packing, the minimum quorum and the
 * token-weighted merge.
 *
 * Conventions for every call:
 *  - A fragment is a flat run of n fp32 elements made of T tensors; tensor t
 *    occupies [offsets[t], offsets[t+1]). Every per-fragment buffer (theta_g,
 *    momentum, each learner replica, each learner's codes) is a separate flat
 *    buffer of n elements.
 *  - All buffers are owned by the caller. "d_" pointers and the pointers
 *    inside pointer arrays are device pointers; pointer arrays themselves
 *    (theta_k, codes) and offsets / weights / present are host arrays read
 *    during the call only.
 *  - Device buffers of fp32 or uint8 elements must be 16-byte aligned.
 *    Workspaces must be 256-byte aligned.
 *  - Device work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and runs asynchronously; the call returns once it is
 *    enqueued. Host-side validation happens before anything is enqueued, so
 *    an error return means nothing was launched (DL_ERR_CUDA excepted).
 *  - No call allocates device memory; scratch comes from the caller's
 *    workspace, sized by the matching *_workspace_bytes query. (dl_outer_sync
 *    creates one stream and a few events per device on first use.) The first
 *    4 bytes of a workspace are its device status word: zero them once when
 *    the workspace is allocated; calls only ever set bits in it, and
 *    dl_read_device_status clears it.
 *  - n = 0 is a valid no-op. Outputs must not alias inputs, except that
 *    theta_g and momentum are updated in place by the merge.
 *  - No C++ exception crosses the ABI. Calls are thread-safe as long as
 *    concurrent calls use different workspaces.
 */
#ifndef DILOCO_SYNC_H
#define DILOCO_SYNC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (0 = success, negative = error). */
#define DL_OK 0
#define DL_ERR_ARG (-1)       /* bad argument: null pointer, bad size, bad weight */
#define DL_ERR_ALIGN (-2)     /* a buffer violates the alignment rule */
#define DL_ERR_QUORUM (-3)    /* fewer present learners than the minimum quorum */
#define DL_ERR_CUDA (-4)      /* a CUDA runtime call or launch failed */
#define DL_ERR_SHAPE (-5)     /* offsets not starting at 0 or decreasing */
#define DL_ERR_WORKSPACE (-6) /* workspace missing or too small */
#define DL_ERR_DEVICE (-7)    /* a kernel reported a failure (see dl_read_device_status) */

#define DL_NBUCKETS 256      /* uint8 code space */
#define DL_MAX_LEARNERS 32   /* largest K accepted by every call */

/* Statistics of one (learner k, tensor t) pseudo-gradient segment; arrays of
 * these are laid out [K][T] (index k * T + t). 48 bytes. */
typedef struct dl_stats {
    int64_t count;     /* elements in the tensor */
    int64_t nonfinite; /* elements whose pseudo-gradient is Inf or NaN */
    double mean;       /* mu; NaN when nonfinite > 0; 0 for an empty tensor */
    double std;        /* population sigma */
    double lo;         /* mu - clip_sigmas * sigma */
    double hi;         /* mu + clip_sigmas * sigma */
} dl_stats;

/* Tensor layout of one fragment. offsets (host) and d_offsets (device) hold
 * the same T+1 non-decreasing values with offsets[0] = 0; n = offsets[T]. */
typedef struct dl_fragment {
    const int64_t* offsets;
    const int64_t* d_offsets;
    int32_t n_tensors;
} dl_fragment;

/* Version of this ABI (major * 100 + minor). */
int dl_version(void);

/* Human-readable name of a status code. Never returns NULL. */
const char* dl_status_string(int status);

/*
 * Balanced tensor fragmentation (Decoupled DiLoCo note, architecture item 4:
 * tensors packed into P fragments of similar size, like greedy bin-packing).
 * Host only. Longest-processing-time greedy: tensors taken by numel
 * descending (index ascending on ties), each placed on the fragment with the
 * smallest load so far (lowest fragment index on ties). Tensors are never
 * split, so a tensor larger than the average fragment gets one to itself.
 *   numel          [n_tensors] element counts, each >= 0
 *   frag_of_tensor [n_tensors] out: fragment index of each tensor
 *   frag_load      [n_frags]   out: total elements per fragment
 * Returns DL_ERR_ARG for n_frags <= 0, n_tensors < 0, negative numel or
 * null outputs (when n_tensors > 0).
 */
int dl_plan_fragments(const int64_t* numel, int32_t n_tensors, int32_t n_frags,
                      int32_t* frag_of_tensor, int64_t* frag_load);

/* Workspace bytes needed by dl_pseudograd_stats for this fragment and K.
 * Never decreases with K, so a workspace sized for K serves any K' <= K
 * (a subset of present learners); the same holds for dl_quantize. */
size_t dl_stats_workspace_bytes(const dl_fragment* frag, int32_t K);

/*
 * Per-tensor statistics of every learner's pseudo-gradient (INTELLECT-1
 * notes, section 3.2 step 4 and section 4.1 steps 1-2).
 * Delta_k[i] = fl32(theta_g[i] - theta_k[k][i]) is formed on the fly and
 * never stored. For each (k, t): mean, population std, lo = mean -
 * clip_sigmas * std, hi = mean + clip_sigmas * std, computed to fp64
 * accuracy, plus the element and non-finite counts.
 *   theta_g      device [n] fp32, global parameters at the start of the round
 *   theta_k      host [K] of device [n] fp32, learner replicas; or NULL with
 *                K = 1 for values mode: Delta is theta_g itself (statistics of
 *                any fp32 vector, e.g. a partial sum to be re-quantised)
 *   clip_sigmas  > 0, 6 in the pages
 *   d_stats      device [K*T] dl_stats, out (8-byte aligned)
 *   d_workspace  device scratch of dl_stats_workspace_bytes(frag, K) bytes
 */
int dl_pseudograd_stats(const float* theta_g, const float* const* theta_k, int32_t K,
                        const dl_fragment* frag, double clip_sigmas, dl_stats* d_stats,
                        void* d_workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes needed by dl_quantize for this fragment and K. */
size_t dl_quantize_workspace_bytes(const dl_fragment* frag, int32_t K);

/*
 * Uniform quantisation with clipping and a bucket-mean codebook (INTELLECT-1
 * notes, section 4.1 steps 2-4). For each (k, t) with lo < hi:
 *   code   = clamp(floor((Delta - lo) * 256 / (hi - lo)), 0, 255), decided
 *            exactly as in fp64 (a value on an interior edge goes up);
 *   cb[b]  = mean of clamp(Delta, lo, hi) over the elements with code b, or
 *            the bucket midpoint lo + (b + 1/2)(hi - lo)/256 when empty.
 * A segment whose range is below 256 * FLT_MIN (sigma = 0 included) gets
 * code 0 everywhere and cb[b] = (float)mean; a segment with non-finite
 * elements gets code 0 everywhere and a NaN codebook.
 *   theta_g, theta_k  as for dl_pseudograd_stats (theta_k NULL with K = 1:
 *               values mode, the vector quantised is theta_g itself)
 *   d_stats     device [K*T], as written by dl_pseudograd_stats
 *   codes       host [K] of device [n] uint8, out
 *   d_codebook  device [K*T*256] fp32, out, index (k*T + t)*256 + b
 *   d_counts    device [K*T*256] uint32 bucket populations, out; may be NULL
 *   d_workspace device scratch of dl_quantize_workspace_bytes(frag, K) bytes
 */
int dl_quantize(const float* theta_g, const float* const* theta_k, int32_t K,
                const dl_fragment* frag, const dl_stats* d_stats, uint8_t* const* codes,
                float* d_codebook, uint32_t* d_counts, void* d_workspace,
                size_t workspace_bytes, void* stream);

/*
 * Dequantise, merge and apply the outer Nesterov step (INTELLECT-1 notes,
 * section 3.2 steps 6-7 and section 4.2; Decoupled DiLoCo note,
 * fault-tolerance items 1 and 3), in place on theta_g and momentum:
 *   w_hat_k = weights[k] / sum_{j present} weights[j]   (fp64, then fp32)
 *   D[i]    = sum over present k, ascending, of fmaf(w_hat_k, v_k[i], .)
 *             with v_k = codebook value of code k (fp32, never summed in
 *             code space) or, in unquantised mode, the fp32 Delta_k;
 *   m'      = fmaf(mu, m, D);  g = fmaf(mu, m', D);  theta' = fmaf(-lr, g, theta)
 *   theta_g, momentum  device [n] fp32, in/out
 *   codes       host [K] of device [n] uint8, or NULL for unquantised mode
 *   d_codebook  device [K*T*256] fp32 (ignored in unquantised mode)
 *   theta_k     host [K] of device [n] fp32 (read only in unquantised mode)
 *   weights     host [K] fp32 >= 0 (tokens processed), or NULL for all 1
 *   present     host [K] 0/1, or NULL for all present; absent learners'
 *               buffers are never read and their pointers may be NULL
 *   min_quorum  fewer present learners than max(1, min_quorum) gives
 *               DL_ERR_QUORUM and leaves the state untouched
 *   delta_bar_out device [n] fp32, out (D); may be NULL
 * A zero total weight or a negative / non-finite weight gives DL_ERR_ARG.
 * With up to 4 present learners (quantised mode) the data is staged through
 * shared memory by bulk copies whose waits are bounded; a wait that runs out
 * sets a bit in the library's own status word (this call has no workspace),
 * read with dl_read_device_status(NULL, ...).
 */
int dl_merge_outer_step(float* theta_g, float* momentum, const uint8_t* const* codes,
                        const float* d_codebook, const float* const* theta_k, int32_t K,
                        const dl_fragment* frag, const float* weights, const uint8_t* present,
                        int32_t min_quorum, float lr, float mu, float* delta_bar_out,
                        void* stream);

/* One fragment's share of a whole-model outer step (see dl_outer_sync). */
typedef struct dl_fragment_job {
    const dl_fragment* frag;      /* tensor layout of the fragment */
    float* theta_g;               /* device [n] fp32, in/out */
    float* momentum;              /* device [n] fp32, in/out */
    const float* const* theta_k;  /* host [K] of device [n] fp32 learner replicas */
    const float* weights;         /* host [K] fp32 >= 0, or NULL for all 1 */
    const uint8_t* present;       /* host [K] 0/1, or NULL for all present */
    float* delta_bar_out;         /* device [n] fp32, out (merged D); may be NULL */
} dl_fragment_job;

#define DL_SYNC_UNQUANTIZED 1 /* merge the fp32 Delta_k directly (no stats, no codes) */
#define DL_SYNC_SERIAL 2      /* run every kernel on `stream`, one fragment after another */
#define DL_SYNC_RDA 4         /* merge with dl_rda_merge_outer_step instead of the mean */
#define DL_SYNC_RING 8        /* each fragment through dl_ring_outer_step (on `stream`) */

/* Workspace bytes needed by dl_outer_sync for these jobs, K and flags (0 on a
 * bad argument or an invalid flag combination). Only the jobs' fragments are
 * read. Covers every number of present learners from 1 to K, so one
 * workspace serves any quorum. */
size_t dl_outer_sync_workspace_bytes(const dl_fragment_job* jobs, int32_t n_jobs, int32_t K,
                                     int32_t flags);

/*
 * A whole outer step over the fragments of a model (Decoupled DiLoCo note,
 * architecture items 3-4: fragments synchronised one after another while
 * other work goes on; INTELLECT-1 notes, sections 3.2 and 4.1-4.2 for each
 * fragment's arithmetic). For each job in order it does exactly what
 *   dl_pseudograd_stats -> dl_quantize -> dl_merge_outer_step
 * do over that job's present learners (ascending; absent learners are never
 * read), with codes, codebooks and statistics kept in the workspace, so the
 * results are bitwise those of the three calls.
 *
 * Scheduling: the statistics of fragment j+1 run on a library-owned side
 * stream beside the quantisation and merge of fragment j on `stream`
 * (two statistics buffers); from the second fragment on with half the
 * blocks of a standalone call (each takes two of the same chunk runs, so the
 * sums and results are the same). The side stream forks from `stream` at entry and
 * joins it before return, so all effects are ordered on `stream`. The side
 * stream and its events are created on the current device on first use and
 * live until dl_shutdown (or process exit); enqueueing is serialised per
 * device by a mutex. `stream` must belong to the current device. DL_SYNC_SERIAL keeps
 * everything on `stream` and creates nothing.
 *
 * DL_SYNC_RDA: the merge of each job is dl_rda_merge_outer_step (the
 * quantiser's bucket counts kept in the workspace), bitwise what the four
 * calls stats -> quantize (with counts) -> dl_rda_merge_outer_step give.
 * DL_SYNC_RING: each job is one dl_ring_outer_step call on `stream` (its
 * hops are sequential by definition, so nothing overlaps); bitwise what
 * that call gives. Neither combines with DL_SYNC_UNQUANTIZED, nor with each
 * other (DL_ERR_ARG).
 *   jobs, n_jobs  host array of fragment jobs; fragments must not overlap
 *                 each other's buffers
 *   K             learners per job (1..DL_MAX_LEARNERS)
 *   clip_sigmas   > 0 (6 in the pages); ignored with DL_SYNC_UNQUANTIZED
 *   min_quorum    applied to every job; a job below it fails the whole call
 *   lr, mu        outer Nesterov learning rate and momentum (0.7, 0.9)
 *   flags         0 or DL_SYNC_UNQUANTIZED, DL_SYNC_RDA or DL_SYNC_RING,
 *                 each optionally with DL_SYNC_SERIAL
 *   d_workspace   device scratch of dl_outer_sync_workspace_bytes(..., flags)
 *                 (unused with DL_SYNC_UNQUANTIZED). Its first word is the
 *                 device status word read by dl_read_device_status.
 * Every job is validated before anything is enqueued (quorum, weights,
 * pointers, alignment); a CUDA failure part way returns DL_ERR_CUDA with the
 * earlier fragments enqueued.
 */
int dl_outer_sync(const dl_fragment_job* jobs, int32_t n_jobs, int32_t K, double clip_sigmas,
                  int32_t min_quorum, float lr, float mu, int32_t flags, void* d_workspace,
                  size_t workspace_bytes, void* stream);

/* Releases what the library created on its own: dl_outer_sync's side stream
 * and events, on every device where they exist, after waiting for the work
 * queued on the side stream. The next dl_outer_sync creates them again. Must not run
 * concurrently with a dl_outer_sync call that is enqueueing (it waits for
 * the per-device mutex). Returns DL_OK, or DL_ERR_CUDA if a destroy failed
 * (the handles are dropped either way). */
int dl_shutdown(void);

/* Workspace bytes needed by dl_rda_merge_outer_step for this fragment and K
 * (0 on a bad argument). */
size_t dl_rda_workspace_bytes(const dl_fragment* frag, int32_t K);

/*
 * Radial-Directional Averaging merge, then the outer Nesterov step (Decoupled
 * DiLoCo note, architecture item 4: the outer gradients' norms and directions
 * are averaged apart instead of averaging the vectors). The page gives no
 * formula; the reading implemented, per tensor t over the present learners
 * k with normalised weights w_k (as for the merge) and decoded values v_k:
 *   n_k = ||v_k||  (from the codebook and the bucket counts, fp64)
 *   r   = sum_k w_k n_k                         radial: mean norm
 *   u   = sum_k (w_k / n_k) v_k                 directional: mean unit vector
 *   D   = r u / ||u||   formed in fp32 as sum_k fl(c_k * v_k), ascending k,
 *         with c_k = (float)((w_k / n_k) r / ||u||); c_k = 0 when n_k = 0,
 *         D = 0 when ||u|| = 0
 * then m' = fmaf(mu, m, D); g = fmaf(mu, m', D); theta' = fmaf(-lr, g, theta).
 *   codes, d_codebook  as for dl_merge_outer_step (quantised mode only)
 *   d_counts    device [K*T*256] uint32 bucket populations from dl_quantize
 *   d_workspace device scratch of dl_rda_workspace_bytes(frag, K) bytes
 * Weights, present, min_quorum, lr, mu, delta_bar_out and the errors are as
 * for dl_merge_outer_step.
 */
int dl_rda_merge_outer_step(float* theta_g, float* momentum, const uint8_t* const* codes,
                            const float* d_codebook, const uint32_t* d_counts, int32_t K,
                            const dl_fragment* frag, const float* weights,
                            const uint8_t* present, int32_t min_quorum, float lr, float mu,
                            float* delta_bar_out, void* d_workspace, size_t workspace_bytes,
                            void* stream);

/* Workspace bytes needed by dl_ring_outer_step for this fragment (0 on a bad
 * fragment); independent of K. */
size_t dl_ring_workspace_bytes(const dl_fragment* frag);

/*
 * Ring accumulation with re-quantisation at every hop, then the outer
 * Nesterov step (INTELLECT-1 notes, section 4.2: a node dequantises what it
 * receives, adds in fp32, and quantises again before sending on; section 4.1
 * for the quantiser). The present learners, in increasing order, form the
 * ring s = 0 .. S-1 and the partial sum P passes along it:
 *   P_0 = w_0 * Delta_0                         (fp32)
 *   P_s = fmaf(w_s, Delta_s, dec(Q(P_{s-1})))   s = 1 .. S-1
 *   D = P_{S-1}; then the outer step of dl_merge_outer_step.
 * Q is the per-tensor quantiser of dl_quantize applied to P itself, with
 * clip_sigmas; w_s are the weights normalised over the present learners as
 * for the merge. A present learner of weight 0 is still a hop. Compared with
 * dl_merge_outer_step (one quantisation per learner), the error of D grows
 * with the number of hops: this call measures that.
 *   theta_g, momentum  device [n] fp32, in/out
 *   theta_k     host [K] of device [n] fp32 (absent learners never read)
 *   weights, present, min_quorum, lr, mu, delta_bar_out  as for
 *               dl_merge_outer_step
 *   hop_stats_out  device [S-1][T] dl_stats (8-byte aligned), or NULL: row s
 *               gets the statistics of P_s as quantised at hop s+1 (the
 *               partial sum's range at each hop); untouched when S = 1
 *   d_workspace device scratch of dl_ring_workspace_bytes(frag) bytes (holds
 *               P, its codes and codebooks; its first word is the device
 *               status word)
 * The statistics of each P_s are accumulated by the hop that writes it (no
 * separate pass over P), with the arithmetic of dl_pseudograd_stats.
 */
int dl_ring_outer_step(float* theta_g, float* momentum, const float* const* theta_k, int32_t K,
                       const dl_fragment* frag, const float* weights, const uint8_t* present,
                       int32_t min_quorum, double clip_sigmas, float lr, float mu,
                       float* delta_bar_out, dl_stats* hop_stats_out, void* d_workspace,
                       size_t workspace_bytes, void* stream);

/*
 * dl_quantize without a caller-provided workspace. The pages have no
 * counterpart: this is a library convenience, not part of the method.
 *
 * For callers that cannot allocate device memory - code whose device memory
 * is owned by another allocator or budget (a framework's caching allocator,
 * a plugin host), or code for which cudaMalloc is not allowed or too costly
 * (it may synchronise the device). The scratch lives in one static device
 * array of DL_QUANTIZE_NOALLOC_MAX_BYTES inside the library; every GPU that
 * loads the library holds it until the process exits. Inputs and outputs
 * are the caller's, exactly as for dl_quantize; results are identical.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress; nothing is cached, so the address stays right
 *    after a device reset or a new primary context). The first lookup on a
 *    device may load the library's device code there: make the first call
 *    on each device before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents
 *    (the call clears what must start at zero). Calls whose GPU work may
 *    overlap - on different streams or from different host threads - race
 *    on it and give wrong results; order them on one stream.
 *  - A fragment with K * n_tensors > DL_QUANTIZE_NOALLOC_MAX_SEGMENTS (its
 *    scratch need would not fit the array) gets DL_ERR_WORKSPACE and nothing
 *    is launched.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define DL_QUANTIZE_NOALLOC_MAX_BYTES (8u * 1024u * 1024u)
#define DL_QUANTIZE_NOALLOC_MAX_SEGMENTS 2000
int dl_quantize_noalloc(const float* theta_g, const float* const* theta_k, int32_t K,
                        const dl_fragment* frag, const dl_stats* d_stats, uint8_t* const* codes,
                        float* d_codebook, uint32_t* d_counts, void* stream);

/*
 * Device-side failure word of a workspace (0 = none). Kernels that wait on
 * a bulk copy give up after a bounded time instead of hanging; they then set
 * a bit here and the call's outputs are undefined. Blocks until the stream
 * has finished, then copies the word to the host and clears it.
 *   d_workspace  a workspace previously passed to a call that takes one, or
 *                NULL for the library's own word on the current device (set
 *                by dl_merge_outer_step, which takes no workspace)
 *   status_out   host, out
 */
int dl_read_device_status(void* d_workspace, uint32_t* status_out, void* stream);

/*
 * Self-test of the failure path of the bounded waits (a diagnostic; the pages
 * have no counterpart). Launches one wait on a shared-memory barrier that
 * nothing completes; after `polls` polls (1 .. 2^22) it gives up, sets the
 * same bit in the workspace's status word that a stalled bulk copy would set,
 * and returns - no trap, no hang, the context stays usable. Read the result
 * with dl_read_device_status.
 *   d_workspace  any workspace of this library (256-byte aligned)
 */
int dl_selftest_wait_timeout(void* d_workspace, int32_t polls, void* stream);

/*
 * Self-test of the abort path of the staged kernels' tile pipeline (a
 * diagnostic; the pages have no counterpart). One block streams n_tiles tiles
 * of 1024 floats from d_src through two shared-memory stages and writes each
 * tile's sum to d_out[tile]; its producer issues only tiles 0 .. stall_tile-1,
 * as a stalled copy engine would. The consumers' waits for tile stall_tile
 * give up after `polls` polls (1 .. 2^22): the block's pipeline aborts exactly
 * as in the staged kernels - no further copy issued, no further stage read
 * (d_out[tile] = NaN from stall_tile on), every issued copy waited for before
 * the block retires - and the workspace's status word gets the bit a stalled
 * copy sets. No trap, no hang, no fault. stall_tile = n_tiles runs the normal
 * path (every sum written, status untouched).
 *   d_workspace  any workspace of this library (256-byte aligned)
 *   d_src        device, n_tiles * 1024 floats, 16-byte aligned
 *   n_tiles      1 .. 4096; 0 <= stall_tile <= n_tiles
 *   d_out        device, n_tiles floats
 * Errors: DL_ERR_ARG, DL_ERR_ALIGN, DL_ERR_CUDA (launch).
 */
int dl_selftest_pipeline(void* d_workspace, const float* d_src, int32_t n_tiles,
                         int32_t stall_tile, int32_t polls, float* d_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DILOCO_SYNC_H */
