/*
 * moe_b300_testing.h -- test hooks of libmoe_b300.so.  Not for production use.
 *
 * They exist so the failure path of the library's bounded device-side waits
 * can be exercised without faulting, trapping or hanging a GPU: the wait is
 * made to run out on purpose (a status flag that nothing sets) and the test
 * checks that the error is reported and that the context stays usable.
 */
#ifndef MOE_B300_TESTING_H
#define MOE_B300_TESTING_H

#include "moe_b300.h"

#ifdef __cplusplus
extern "C" {
#endif

/* moe_dispatch, except that dispatch tile `stalled_tile` (0-based, tiles of
 * 4096 priority positions) never publishes its per-expert totals.  The tile
 * after it waits for them, gives up after its bounded wait (about one
 * second), records MOE_ERR_DEVICE_TIMEOUT in the workspace error word and
 * finishes; moe_get_device_error() then returns MOE_ERR_DEVICE_TIMEOUT.  The
 * slots written downstream of the stalled tile are not meaningful.  Returns
 * MOE_ERR_INVALID_ARG when stalled_tile is not a tile of this call. */
MOE_API moe_status_t moe_testing_dispatch_stalled(const moe_shape_t* shape, int32_t C, const int32_t* idx,
                                                  const void* x, int32_t* pos, int32_t* counts,
                                                  int32_t* offsets, int64_t* dropped, void* x_perm,
                                                  int32_t stalled_tile, void* ws, size_t ws_bytes,
                                                  void* stream);

/* The first step of the forward's tensor-core router (used for long bf16
 * batches with 32 to 256 logit columns) alone: the fp32 router weights
 * [W_g | W_noise] are split into bf16 parts hi + lo, and one tcgen05 GEMM
 * computes approx[t, c] = sum_j x[t, j] (hi[j, c] + lo[j, c]) in fp32 for
 * every column c < nc (nc = E, or 2E with W_noise).  The router then trusts
 * each approximate logit only to within 2^-10 * 1.25 * ||x_t|| * ||w_c||;
 * this hook lets a test measure the real error of the split and of the
 * tensor cores' accumulation against that margin.
 *   shape   bf16, token choice; d a multiple of 64; nc a multiple of 32, <= 256
 *   x       [T,d] bf16; W_g, W_noise [d,E] fp32 (W_noise may be NULL)
 *   approx  [T,nc] fp32 out
 *   ws, ws_bytes  a workspace of moe_workspace_size(shape, any C)
 * Returns MOE_ERR_UNSUPPORTED for shapes outside that set. */
MOE_API moe_status_t moe_testing_router_filter(const moe_shape_t* shape, const void* x, const float* W_g,
                                               const float* W_noise, float* approx, void* ws, size_t ws_bytes,
                                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_TESTING_H */
