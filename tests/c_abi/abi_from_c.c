/* A plain C caller of libgdn.so: includes gdn.h with a C compiler, links the library, and checks the
 * host-side argument validation and the status strings.  It makes no call that reaches a kernel, so it
 * runs without a GPU.  Exit status 0 = every check passed. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gdn.h"

static int failures = 0;

#define EXPECT(cond)                                                  \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "FAILED: %s (line %d)\n", #cond, __LINE__); \
            ++failures;                                               \
        }                                                             \
    } while (0)

int main(void) {
    gdn_dims d;
    memset(&d, 0, sizeof d);
    d.B = 4; d.T = 4; d.HK = 2; d.HV = 4; d.DK = 128; d.DV = 128; d.num_slots = 8;
    d.qkv_dtype = GDN_BF16; d.state_dtype = GDN_BF16; d.out_dtype = GDN_BF16;
    d.scale = 1.0f; d.l2_eps = 1e-6f;
    void* p = (void*)(uintptr_t)0x10000; /* aligned, never dereferenced: validation fails first */
    EXPECT(gdn_abi_version() == 1);
    EXPECT(strcmp(gdn_status_string(GDN_OK), "GDN_OK") == 0);
    EXPECT(gdn_mtp_verify(NULL, p, p, p, p, p, p, p, p, p, p, NULL, NULL, NULL) == GDN_ERR_NULL);
    EXPECT(gdn_mtp_verify(&d, NULL, p, p, p, p, p, p, p, p, p, NULL, NULL, NULL) == GDN_ERR_NULL);
    d.DK = 48;
    EXPECT(gdn_decode(&d, p, p, p, p, p, p, p, p, p, p, NULL, NULL) == GDN_ERR_UNSUPPORTED);
    d.DK = 128; d.HK = 3;
    EXPECT(gdn_commit_replay(&d, p, p, p, p, p, p, p, p, p, p, NULL, NULL) == GDN_ERR_SHAPE);
    d.HK = 2;
    EXPECT(gdn_commit(&d, p, p, (void*)(uintptr_t)0x10002, p, NULL, NULL) == GDN_ERR_ALIGN);
    d.B = 0;
    EXPECT(gdn_commit(&d, NULL, NULL, NULL, NULL, NULL, NULL) == GDN_OK);
    /* prefill: T is the packed token count (beyond GDN_MAX_T); the device-side arrays are plain int32 */
    d.B = 4; d.T = 4096;
    EXPECT(gdn_prefill(&d, NULL, p, p, p, p, p, p, p, p, p, NULL, p, NULL, NULL) == GDN_ERR_NULL);
    EXPECT(gdn_prefill(&d, p, p, p, p, p, p, p, p, p, p, (const int32_t*)(uintptr_t)0x10002, p, NULL, NULL) ==
           GDN_ERR_ALIGN);
    d.T = -1;
    EXPECT(gdn_prefill(&d, p, p, p, p, p, p, p, p, p, p, NULL, p, NULL, NULL) == GDN_ERR_SHAPE);
    d.T = 0;
    EXPECT(gdn_prefill(&d, p, p, p, p, p, p, p, p, p, p, NULL, p, NULL, NULL) == GDN_OK);
    /* gated norm: explicit sizes and dtypes */
    EXPECT(gdn_gated_rmsnorm(0, 128, GDN_BF16, GDN_BF16, NULL, NULL, NULL, 1e-6f, NULL, NULL) == GDN_OK);
    EXPECT(gdn_gated_rmsnorm(16, 128, GDN_BF16, GDN_BF16, p, p, p, -1.0f, p, NULL) == GDN_ERR_VALUE);
    EXPECT(gdn_gated_rmsnorm(16, 0, GDN_BF16, GDN_BF16, p, p, p, 1e-6f, p, NULL) == GDN_ERR_SHAPE);
    EXPECT(gdn_gated_rmsnorm(16, 128, 5, GDN_BF16, p, p, p, 1e-6f, p, NULL) == GDN_ERR_DTYPE);
    EXPECT(gdn_gated_rmsnorm(16, 128, GDN_BF16, GDN_BF16, p, NULL, p, 1e-6f, p, NULL) == GDN_ERR_NULL);
    EXPECT(gdn_last_cuda_error() == 0);
    if (failures == 0) printf("abi_from_c: ok\n");
    return failures == 0 ? 0 : 1;
}
