/*
 * The C-ABI used from plain C, with no Python and no GPU: every entry point's
 * host-side argument checks answer before any CUDA call, and the status
 * strings are available.  Built and run by tests/test_abi.py.  Exits 0 when
 * every check holds; otherwise prints the failing check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ce.h"

static int failures = 0;

#define EXPECT(expr, want)                                                          \
    do {                                                                            \
        int got_ = (expr);                                                          \
        if (got_ != (want)) {                                                       \
            fprintf(stderr, "%s:%d: %s returned %d, expected %d\n", __FILE__,      \
                    __LINE__, #expr, got_, (want));                                 \
            ++failures;                                                             \
        }                                                                           \
    } while (0)

int main(void) {
    /* addresses that are never dereferenced: the checks reject the calls first */
    const void *z = (const void *)(uintptr_t)0x10000;
    const int32_t *t = (const int32_t *)(uintptr_t)0x20000;
    float *loss = (float *)(uintptr_t)0x30000;
    void *g = (void *)(uintptr_t)0x40000;

    EXPECT(ce_fwd_bwd(NULL, t, 4, 4, CE_F32, loss, g, NULL), CE_ERR_NULL);
    EXPECT(ce_fwd_bwd(z, t, 0, 4, CE_F32, loss, g, NULL), CE_ERR_SHAPE);
    EXPECT(ce_fwd_bwd(z, t, 4, 4, 7, loss, g, NULL), CE_ERR_DTYPE);
    EXPECT(ce_fwd_bwd((const char *)z + 2, t, 4, 4, CE_F32, loss, g, NULL), CE_ERR_ALIGN);
    EXPECT(ce_fwd_bwd(z, t, 4, 4, CE_F32, loss, (char *)z + 16, NULL), CE_ERR_OVERLAP);
    EXPECT(ce_fwd_bwd_ex(z, t, 4, 4, CE_BF16, 5, NULL, loss, g, NULL), CE_ERR_REDUCTION);
    EXPECT(ce_forward(z, t, 4, 4, CE_F16, CE_REDUCE_MEAN, NULL, NULL), CE_ERR_NULL);
    EXPECT(ce_softmax_fwd(z, 4, 4, CE_F32, NULL, NULL), CE_ERR_NULL);
    EXPECT(ce_softmax_bwd(z, z, 4, 4, 9, g, NULL), CE_ERR_DTYPE);
    EXPECT(ce_fwd_bwd_host(z, t, 4, 4, CE_F32, loss, NULL, NULL), CE_ERR_NULL);
    EXPECT(ce_fwd_bwd_host_grad(z, t, 4, 4, CE_F32, loss, NULL, NULL), CE_ERR_NULL);
    EXPECT(ce_fwd_bwd_host_grad(z, t, 4, 4, CE_F32, loss, (char *)z + 8, NULL), CE_ERR_OVERLAP);
    EXPECT(ce_fwd_bwd_noalloc(z, t, 1LL << 40, 4, CE_F32, loss, g, NULL), CE_ERR_SHAPE);
    if (strcmp(ce_status_string(CE_OK), "unknown status") == 0) ++failures;
    if (strcmp(ce_status_string(12345), "unknown status") != 0) ++failures;
    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}
