/*
 * abi_from_c.c -- uses libqhead.so through include/qhead.h from plain C (no
 * Python, no C++): the version string, and argument errors reported by every
 * entry point before any device work.  Needs no GPU.  Prints "ok" and exits
 * 0 when every check holds; prints the failing check and exits 1 otherwise.
 */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "qhead.h"

static int failures = 0;

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            printf("FAILED: %s (line %d)\n", #cond, __LINE__);       \
            ++failures;                                              \
        }                                                            \
    } while (0)

int main(void) {
    /* Never dereferenced: every call below fails its argument checks first. */
    qhead_head hd;
    memset(&hd, 0, sizeof hd);
    hd.wq = (const uint32_t*)0x10000;
    hd.scales = (const void*)0x20000;
    hd.biases = (const void*)0x30000;
    hd.V = 1000;
    hd.H = 256;
    hd.bits = 4;
    hd.group = 64;
    hd.sb_dtype = QHEAD_SB_F16;
    hd.softcap = 0.f;
    void* h = (void*)0x40000;
    int32_t* t = (int32_t*)0x41000;
    float* f = (float*)0x42000;
    void* ws = (void*)0x60000;

    CHECK(strstr(qhead_version(), "sm_103a") != NULL);

    /* head checks, shared by every entry point */
    qhead_head bad = hd;
    bad.bits = 3;
    CHECK(qhead_fwd(&bad, h, 4, NULL, NULL, NULL, f, NULL, ws, 1 << 20, NULL) ==
          QHEAD_EUNSUPPORTED);
    CHECK(strlen(qhead_last_error()) > 0);
    bad = hd;
    bad.scales = (const void*)0x20002;
    CHECK(qhead_bwd(&bad, h, 4, t, NULL, f, f + 8, f + 16, ws, 1 << 20, NULL) == QHEAD_EINVAL);
    CHECK(qhead_fwd(NULL, h, 4, NULL, NULL, NULL, f, NULL, ws, 1 << 20, NULL) == QHEAD_EINVAL);
    CHECK(qhead_fwd_workspace(&bad, 4) == (size_t)-1);

    /* the element types of scales and biases: fp16, bf16 and fp32 pass the
       head checks (the call then stops at the missing workspace); others are
       unsupported */
    bad = hd;
    bad.sb_dtype = QHEAD_SB_BF16;
    CHECK(qhead_fwd(&bad, h, 4, NULL, NULL, NULL, f, NULL, NULL, 0, NULL) == QHEAD_EINVAL);
    bad.sb_dtype = QHEAD_SB_F32;
    CHECK(qhead_fwd(&bad, h, 4, NULL, NULL, NULL, f, NULL, NULL, 0, NULL) == QHEAD_EINVAL);
    CHECK(strstr(qhead_last_error(), "workspace") != NULL);
    bad.sb_dtype = 3;
    CHECK(qhead_fwd(&bad, h, 4, NULL, NULL, NULL, f, NULL, NULL, 0, NULL) == QHEAD_EUNSUPPORTED);

    /* M == 0 is a no-op everywhere */
    CHECK(qhead_fwd(&hd, NULL, 0, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) == QHEAD_OK);
    CHECK(qhead_bwd(&hd, NULL, 0, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) == QHEAD_OK);
    CHECK(qhead_fwd_workspace(&hd, 0) == 0);

    /* entry-point specific checks */
    CHECK(qhead_fwd(&hd, (void*)0x40004, 4, NULL, NULL, NULL, f, NULL, ws, 1 << 20, NULL) ==
          QHEAD_EINVAL); /* h not 16-byte aligned */
    CHECK(qhead_bwd_filter(&hd, h, 4, t, NULL, f, f + 8, -1.f, f + 16, NULL, ws, 1 << 20,
                           NULL) == QHEAD_EINVAL);
    CHECK(strstr(qhead_last_error(), "eps") != NULL);
    CHECK(qhead_bwd_filter(&hd, h, 4, t, NULL, f, f + 8, NAN, f + 16, NULL, ws, 1 << 20,
                           NULL) == QHEAD_EINVAL);
    CHECK(qhead_bwd_blockskip(&hd, h, 4, t, NULL, f, f + 8, NULL, 1e-5f, f + 16, ws, 1 << 20,
                              NULL) == QHEAD_EINVAL); /* no block_max */
    CHECK(qhead_bwd_dw(&hd, h, 4, t, NULL, f, f + 8, NULL, NULL, ws, 1 << 20, NULL) ==
          QHEAD_EINVAL); /* no dw */
    CHECK(qhead_verify(&hd, h, 2, 0, NULL, NULL, NULL, t, t + 8, NULL, ws, 1 << 20, NULL) ==
          QHEAD_EINVAL); /* W < 1 */
    /* the no-allocation forward looks up the current device first: without a
       device that lookup fails (QHEAD_ECUDA), with one the argument check does */
    {
        const int rc = qhead_fwd_noalloc(&hd, h, -1, NULL, NULL, NULL, f, NULL, NULL);
        CHECK(rc == QHEAD_EINVAL || rc == QHEAD_ECUDA);
    }

    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}
