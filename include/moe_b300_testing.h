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

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_TESTING_H */
