/*
 * dsa_testing.h -- test-only entry points of libdsa.so.
 *
 * Not part of the DSA step: these exist so that tests can drive paths that a
 * correct run never takes.  They have no counterpart on the pages.
 */
#ifndef DSA_TESTING_H_
#define DSA_TESTING_H_

#include "dsa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* dsa_sparse_mla with the kernel's bounded-wait failure path forced: the
 * kernel's producer warps withhold one barrier arrival of the first latent
 * tile, and every wait of the kernel is given a budget of 2^20 cycles (about
 * half a millisecond) instead of the usual 2^30.  The MMA thread's wait for
 * that tile runs out, the kernel unwinds (no MMA or copy left in flight, TMEM
 * released) and stores DSA_ERR_TIMEOUT into *dev_status; the contents of out
 * and lse are then unspecified.
 * Arguments, checks and host-side return values are those of dsa_sparse_mla;
 * the GPU context stays usable, so later calls on the stream run normally. */
dsa_status dsa_test_sparse_mla_wait_timeout(const dsa_batch* batch, const uint16_t* q_lat,
                                           const void* latent_pages, float kv_scale,
                                           float sm_scale, const int32_t* indices, int32_t topk,
                                           uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                                           int32_t* dev_status, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_TESTING_H_ */
