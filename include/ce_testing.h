/*
 * ce_testing.h -- test hooks of the softmax cross-entropy library.
 *
 * Not for production use: these entry points exist so that a test suite can
 * reach code paths that a correct run never takes, and see values that the
 * product entry points do not return.  The pages that define the operation
 * have no counterpart; everything else about the call is as in ce.h.
 */
#ifndef CE_TESTING_H
#define CE_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    /* -1: none.  Otherwise the TMA copy that stages row `skip_copy_row` (its
     * tile, slice or first chunk) is never issued, so the kernel's bounded
     * wait for it must give up: the kernel counts a timeout (read it with
     * ce_get_device_errors), makes the batch loss (or that row's loss) NaN,
     * waits for its other copies and returns.  No copy is ever in flight to
     * the skipped slot. */
    int64_t skip_copy_row;
    /* 0: the library's limit (about a second).  Otherwise the number of SM
     * clock cycles after which a wait for a row copy gives up.  The waits for
     * a cluster peer's partial sums and for copies still in flight after a
     * failure keep the library's limit. */
    int64_t wait_limit_cycles;
    /* NULL, or device [B][C] fp32 (4-byte aligned, not overlapping the other
     * arguments): the kernel also writes every gradient element here as the
     * fp32 value it computed before rounding it to the logits' dtype. */
    float *grad_f32_out;
} ce_test_hooks;

/*
 * ce_fwd_bwd_test -- ce_fwd_bwd_path (same arguments, same results) with the
 * test hooks above; hooks may be NULL.  The streaming path (CE_PATH_STREAM)
 * stages nothing and records no fp32 gradient: with any hook set it returns
 * CE_ERR_PATH.  With a hook set the kernels run in their general build (the
 * one ce_fwd_bwd_ex uses), not in the plain call's.
 */
int ce_fwd_bwd_test(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
                    float *loss_out, void *grad_out, void *stream, int path, int split,
                    const ce_test_hooks *hooks);

#ifdef __cplusplus
}
#endif

#endif /* CE_TESTING_H */
