/*
 * gpulz_testing.h -- test hook of the GPULZ library (not part of the coder's
 * API; no counterpart in the paper).
 *
 * The coder places blocks and tiles by a decoupled look-back: each entry of a
 * descriptor array is published by the CTA that owns it, and a CTA waits for
 * its predecessors' entries. Every such wait is bounded: once it has lasted
 * longer than a limit (200 ms in the coder), the kernel stops waiting,
 * records GPULZ_ERR_TIMEOUT in the stream's device status word and returns,
 * instead of hanging the GPU. This hook runs that same look-back on a
 * descriptor array the caller prepared, so a test can make a wait run out
 * (an entry that nothing publishes) and check the status.
 *
 * Descriptor (u64): bits 63..48 epoch (1..65535; the call's tag), bits 47..46
 * kind (0 not published, 1 aggregate = the entry's own value, 2 inclusive =
 * the sum of all entries up to and including it), bits 45..0 value.
 */
#ifndef GPULZ_TESTING_H
#define GPULZ_TESTING_H

#include <stddef.h>
#include <stdint.h>

#include "gpulz.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gpulz_test_lookback -- one warp computes the exclusive prefix of `value`
 * over entries [0, idx) of d_desc (device, at least idx + 1 entries, 8-byte
 * aligned), reading only entries [0, idx], and publishes entry idx as an
 * inclusive descriptor of `epoch`. An entry below idx that does not carry
 * `epoch` with a nonzero kind is waited for; after limit_ns nanoseconds of
 * device time (at most 200 ms) the wait gives up: the stream's status word
 * records GPULZ_ERR_TIMEOUT (read with gpulz_device_status) and entry idx is
 * published with the partial sum. *d_prefix (device, 8-byte aligned) receives
 * the prefix. Asynchronous on `stream`; uses the stream's scratch (status
 * word) like the coder's calls. Returns GPULZ_ERR_INVALID_ARG for null or
 * misaligned pointers, epoch 0 or above 65535, or limit_ns above 200 ms.
 */
gpulz_status gpulz_test_lookback(uint64_t* d_desc, uint32_t idx, uint64_t value, uint32_t epoch,
                                 uint64_t limit_ns, size_t* d_prefix, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GPULZ_TESTING_H */
