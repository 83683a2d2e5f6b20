/*
 * b200norm_testing.h -- hooks for the library's own tests.  Not needed to use
 * the operators; they let tests reach every schedule and the device-side
 * timeout path without faulting or hanging a GPU.
 */
#ifndef B200NORM_TESTING_H
#define B200NORM_TESTING_H

#include "b200norm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launch a two-CTA cooperative kernel whose grid barrier can never complete
 * (it waits for a third CTA).  Both CTAs give up after `limit_ns`
 * nanoseconds and record B200NORM_ERR_DEVICE_TIMEOUT in the workspace, which
 * b200norm_workspace_status() then reports.  The workspace must be
 * re-initialised afterwards.  Never faults; returns within ~limit_ns. */
B200NORM_API b200norm_status b200norm_testing_barrier_timeout(void* workspace,
                                                              size_t workspace_bytes,
                                                              uint64_t limit_ns,
                                                              b200norm_stream_t stream);

/* The same probe on the static scratch of b200norm_skip_group_noalloc (on the
 * current device): its waits give up after `limit_ns` and record
 * B200NORM_ERR_DEVICE_TIMEOUT there, which
 * b200norm_skip_group_noalloc_status() then reports and clears.  The barrier
 * counts are back at zero afterwards.  Never faults. */
B200NORM_API b200norm_status b200norm_testing_noalloc_barrier_timeout(uint64_t limit_ns,
                                                                      b200norm_stream_t stream);

/* Force a schedule on the calling thread (0 = automatic choice):
 *   row_mode:    1 = register-resident schedules only (never the pipelined
 *                    one that automatic choice gives long runs of short
 *                    SkipSimplifiedLayerNormalization rows)
 *                2 = walk each row twice (any row length)
 *                3 = pipelined lane groups (rows of at most 32 16-byte
 *                    vectors with 16-byte aligned tensors; other calls return
 *                    B200NORM_ERR_UNSUPPORTED)
 *   group_route: 2 = NHWC cooperative grid with one bounded grid barrier
 *                3 = two-phase partials -> normalize (any shape)
 *                4 = NHWC through L2 (statistics kernel, then apply kernel)
 *                5 = NHWC through L2 in one cooperative grid (statistics, a
 *                    bounded grid barrier, then a second pass over L2)
 *                6 = NHWC cooperative grid with each CTA's slab of pixels
 *                    resident in shared memory (bulk copies in and out with
 *                    16-byte vectors), one bounded grid barrier
 * Other values are rejected with B200NORM_ERR_INVALID_ARGUMENT.  A later
 * SkipGroupNorm call that the forced route cannot take returns
 * B200NORM_ERR_UNSUPPORTED. */
B200NORM_API b200norm_status b200norm_testing_force(int row_mode, int group_route);

/* Force the row schedule of SkipSimplifiedLayerNormalization and
 * GatedRMSNorm calls on the calling thread to one row per cluster of `csize`
 * CTAs, each thread holding `nv` vectors: csize in {1, 2, 4, 8, 16}, nv in
 * {1, 2, 4, 8}; (0, 0) restores the automatic choice.  A later call whose
 * row would need more than 512 threads per CTA under the forced split
 * returns B200NORM_ERR_UNSUPPORTED; a cluster the device cannot co-schedule
 * falls back to the walking schedule. */
B200NORM_API b200norm_status b200norm_testing_force_split(int csize, int nv);

/* Switch programmatic dependent launch off (0) or on (1, the default) for
 * every later launch of the library, on all threads.  With it on, a kernel
 * may be scheduled while the preceding grid on its stream drains and waits
 * for that grid before touching memory; results are identical either way. */
B200NORM_API b200norm_status b200norm_testing_set_pdl(int on);

/* Stall the pipelined row schedule (process-wide) for later launches: with
 * on = 1 its producer issues no copies, so every consumer wait gives up after
 * limit_ns (in (0, 5 s]) and the kernel records B200NORM_ERR_DEVICE_TIMEOUT
 * (read with b200norm_rows_status) with nothing in flight; outputs are left
 * unwritten.  on = 0 restores normal launches (limit_ns ignored). */
B200NORM_API b200norm_status b200norm_testing_pipe_stall(int on, uint64_t limit_ns);

/* Schedule the automatic planner picks, without launching anything.
 * Rows (SSLN / GatedRMSNorm): out = {mode, ve, tpr, nv, rpg, block, csize, grid}.
 * SkipGroupNorm: out = {route, ve, nv, block, csize, grid, ctas_per_item,
 * pix_per_cta}.  `aligned16` says whether every pointer is 16-byte aligned. */
B200NORM_API b200norm_status b200norm_testing_plan_rows(int64_t rows, int64_t n,
                                                        b200norm_dtype T, int aligned16,
                                                        int64_t out[8]);
/* The same for GatedRMSNorm spans of C elements (b200norm_testing_plan_rows
 * gives SkipSimplifiedLayerNormalization's plan; the two differ for some
 * widths when there are many rows). */
B200NORM_API b200norm_status b200norm_testing_plan_gated(int64_t rows, int64_t C,
                                                         b200norm_dtype T, int aligned16,
                                                         int64_t out[8]);
B200NORM_API b200norm_status b200norm_testing_plan_group(int64_t N, int64_t C, int64_t H,
                                                         int64_t W, int groups, b200norm_dtype T,
                                                         b200norm_dtype M, int channels_last,
                                                         int aligned16, int64_t out[8]);

#ifdef __cplusplus
}
#endif

#endif /* B200NORM_TESTING_H */
