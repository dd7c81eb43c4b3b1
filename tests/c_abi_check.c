/*
 * A plain C99 user of the library's C ABI (include/diloco_sync.h), built and
 * run by tests/test_c_abi.py on the host. It calls only what answers on the
 * host: the version, the status strings, the fragment planner, the workspace
 * queries, and calls that validation refuses before any device work (the
 * device pointers below are never dereferenced). Prints "ok" and exits 0 when
 * every check holds; otherwise names the first failing check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "diloco_sync.h"

#define CHECK(cond)                                                          \
    do {                                                                     \
        if (!(cond)) {                                                       \
            fprintf(stderr, "failed at line %d: %s\n", __LINE__, #cond);     \
            return 1;                                                        \
        }                                                                    \
    } while (0)

/* a 256-byte aligned device address that no call below dereferences */
#define FAKE ((void*)(uintptr_t)(1u << 20))

int main(void) {
    static const int codes[] = {DL_OK,       DL_ERR_ARG,  DL_ERR_ALIGN,     DL_ERR_QUORUM,
                                DL_ERR_CUDA, DL_ERR_SHAPE, DL_ERR_WORKSPACE, DL_ERR_DEVICE,
                                12345};
    size_t i;
    CHECK(dl_version() == 200);
    for (i = 0; i < sizeof codes / sizeof codes[0]; ++i) {
        const char* s = dl_status_string(codes[i]);
        CHECK(s != NULL && s[0] != '\0');
    }

    /* Longest processing time first: sizes 7, 5, 4, 3, 3 into 2 fragments go
       7 -> 0, 5 -> 1, 4 -> 1, 3 -> 0, 3 -> 1 (the least-loaded fragment, the
       lower index on ties), loads 10 and 12. */
    {
        const int64_t numel[5] = {7, 5, 4, 3, 3};
        int32_t frag[5];
        int64_t load[2];
        CHECK(dl_plan_fragments(numel, 5, 2, frag, load) == DL_OK);
        CHECK(frag[0] == 0 && frag[1] == 1 && frag[2] == 1 && frag[3] == 0 && frag[4] == 1);
        CHECK(load[0] == 10 && load[1] == 12);
        CHECK(dl_plan_fragments(numel, 5, 0, frag, load) == DL_ERR_ARG);
    }

    {
        static const int64_t off[4] = {0, 10, 10, 30};
        dl_fragment f;
        const float* reps[3] = {(const float*)FAKE, (const float*)FAKE, (const float*)FAKE};
        uint8_t* cptr[3] = {(uint8_t*)FAKE, (uint8_t*)FAKE, (uint8_t*)FAKE};
        const uint8_t* ccptr[3] = {(const uint8_t*)FAKE, (const uint8_t*)FAKE,
                                   (const uint8_t*)FAKE};
        const uint8_t none_present[3] = {0, 0, 0};
        const uint8_t two_present[3] = {1, 0, 1};
        const float bad_weights[3] = {1.0f, -1.0f, 1.0f};
        dl_fragment_job job;
        size_t ws1, ws3;
        f.offsets = off;
        f.d_offsets = (const int64_t*)FAKE;
        f.n_tensors = 3;

        /* workspace sizes never decrease with K */
        ws1 = dl_stats_workspace_bytes(&f, 1);
        ws3 = dl_stats_workspace_bytes(&f, 3);
        CHECK(ws1 > 0 && ws3 >= ws1);
        CHECK(dl_quantize_workspace_bytes(&f, 3) >= dl_quantize_workspace_bytes(&f, 1));
        CHECK(dl_rda_workspace_bytes(&f, 3) >= dl_rda_workspace_bytes(&f, 1));
        CHECK(dl_ring_workspace_bytes(&f) > 0);

        /* refused on the host: bad K, short workspace, no quorum, bad weight */
        CHECK(dl_pseudograd_stats((const float*)FAKE, reps, 0, &f, 6.0, (dl_stats*)FAKE, FAKE, ws3,
                                  NULL) == DL_ERR_ARG);
        CHECK(dl_pseudograd_stats((const float*)FAKE, reps, 3, &f, 6.0, (dl_stats*)FAKE, FAKE,
                                  ws3 - 1, NULL) == DL_ERR_WORKSPACE);
        CHECK(dl_quantize_noalloc((const float*)FAKE, reps, 0, &f, (const dl_stats*)FAKE, cptr,
                                  (float*)FAKE, NULL, NULL) == DL_ERR_ARG);
        CHECK(dl_merge_outer_step((float*)FAKE, (float*)FAKE, ccptr, (const float*)FAKE, NULL, 3,
                                  &f, NULL, none_present, 1, 0.7f, 0.9f, NULL,
                                  NULL) == DL_ERR_QUORUM);
        CHECK(dl_merge_outer_step((float*)FAKE, (float*)FAKE, ccptr, (const float*)FAKE, NULL, 3,
                                  &f, NULL, two_present, 3, 0.7f, 0.9f, NULL,
                                  NULL) == DL_ERR_QUORUM);
        CHECK(dl_merge_outer_step((float*)FAKE, (float*)FAKE, ccptr, (const float*)FAKE, NULL, 3,
                                  &f, bad_weights, NULL, 1, 0.7f, 0.9f, NULL,
                                  NULL) == DL_ERR_ARG);

        /* dl_outer_sync checks every job before it enqueues anything */
        memset(&job, 0, sizeof job);
        job.frag = &f;
        job.theta_g = (float*)FAKE;
        job.momentum = (float*)FAKE;
        job.theta_k = reps;
        job.present = none_present;
        CHECK(dl_outer_sync(&job, 1, 3, 6.0, 1, 0.7f, 0.9f, 0, FAKE,
                            dl_outer_sync_workspace_bytes(&job, 1, 3, 0), NULL) == DL_ERR_QUORUM);
    }

    /* offsets must start at 0 and never decrease */
    {
        static const int64_t bad[3] = {0, 10, 5};
        dl_fragment g;
        const float* reps[1] = {(const float*)FAKE};
        g.offsets = bad;
        g.d_offsets = (const int64_t*)FAKE;
        g.n_tensors = 2;
        CHECK(dl_pseudograd_stats((const float*)FAKE, reps, 1, &g, 6.0, (dl_stats*)FAKE, FAKE,
                                  (size_t)1 << 30, NULL) == DL_ERR_SHAPE);
    }

    CHECK(dl_shutdown() == DL_OK); /* nothing was created: no CUDA call */
    printf("ok\n");
    return 0;
}
