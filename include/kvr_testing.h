/*
 * kvr_testing.h -- test hooks of libkvr. Not part of the library's API: they
 * exist so that tests can drive error paths that correct inputs never reach,
 * without faulting, trapping or hanging the GPU.
 */
#ifndef KVR_TESTING_H_
#define KVR_TESTING_H_

#include "kvr.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kvr_testing_tiered_withheld_copy -- kvr_sparse_attend_tiered in which every
 * CTA of the attention kernel never issues the last bulk copy of its window
 * list (it still waits for it), and each wait for a copy gives up after
 * wait_ns nanoseconds instead of the normal one second. The wait for the
 * withheld copy therefore runs out: the kernel sets KVR_DEVERR_TIMEOUT in
 * err_word, stops issuing, waits (bounded) for the copies it did issue and
 * returns; out and window_mass are then invalid. Nothing else is different:
 * the context stays usable and the next call computes normally. The paper
 * has no counterpart: this is a test of the bounded device-side waits.
 * Arguments as kvr_sparse_attend_tiered; wait_ns must be 1..10^10.
 */
kvr_status kvr_testing_tiered_withheld_copy(const kvr_shape *shape, const kvr_tier_state *state,
                                            const void *q, const void *K, const void *V,
                                            const int32_t *seq_len, float scale, float *out,
                                            float *window_mass, void *workspace,
                                            size_t workspace_bytes, int32_t *err_word,
                                            void *stream, int64_t wait_ns);

#ifdef __cplusplus
}
#endif

#endif /* KVR_TESTING_H_ */
