/*
 * mlg_test.h -- test and benchmark hooks of libmlg.  NOT part of the public
 * interface in mlg.h.
 *
 * These hooks exist so that the test suite can steer the decode fold onto
 * each of its kernels and code paths (including a path that only runs when a
 * speculation turns out wrong) and so that launch shapes can be swept while
 * benchmarking.  Results never depend on them: every setting folds the same
 * rows to the same bits.  The settings are process-wide, unsynchronised
 * globals read at launch time: change them only while no other thread
 * enqueues folds, and restore 0 (the automatic choice) afterwards.  A
 * serving process has no reason to include this header.
 */
#ifndef MLG_TEST_H_
#define MLG_TEST_H_

#include "mlg.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Knobs of mlg_test_set_knob; the value 0 restores the automatic choice.
 *   MLG_TEST_GATHER_CLUSTER     CTAs per expert cluster of the cluster decode
 *                               kernel (1, 2, 4, 8): the cluster splits k_in
 *                               (partial h summed on chip) and n_out
 *   MLG_TEST_GATHER_NSPLIT      independent CTAs per expert and cluster rank
 *                               of the cluster decode kernel (1, 2, 4, 8): each
 *                               computes all of h and folds its own n_out slice
 *   MLG_TEST_GROUPED_CTAS       persistent CTAs of the grouped and router folds
 *   MLG_TEST_GATHER_PATH        kernel of the decode folds: 1 = the resident-pair
 *                               kernel (max_rank 16 or 32, n_out <= 2048, the pair
 *                               in half an SM; other shapes return UNSUPPORTED),
 *                               2 = the cluster kernel (any shape)
 *   MLG_TEST_GATHER_SPECULATION row lists of the resident-pair kernel: 1 = found
 *                               only after the preceding kernel completes (no
 *                               speculation), 2 = the early scan deliberately
 *                               reads another expert's rows so that every check
 *                               fails and the rows are requested again -- the
 *                               recovery path a wrong speculation takes; in the
 *                               multi-adapter form the same values pick the first
 *                               cell whose pair loads early (2: another CTA's)
 * Errors: INVALID_ARG for an unknown knob or a value out of range. */
#define MLG_TEST_GATHER_CLUSTER 1
#define MLG_TEST_GROUPED_CTAS 2
#define MLG_TEST_GATHER_NSPLIT 3
#define MLG_TEST_GATHER_PATH 4
#define MLG_TEST_GATHER_SPECULATION 5
MLG_API mlg_status mlg_test_set_knob(int32_t knob, int32_t value);

#ifdef __cplusplus
}
#endif

#endif /* MLG_TEST_H_ */
