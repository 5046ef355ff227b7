/*
 * pagedattn_testing.h -- a hook of libpagedattn.so for tests of its failure
 * handling. Not part of the attention API: the pages have no counterpart.
 *
 * Every wait inside the library's kernels is bounded. When one role of a
 * kernel (a copy producer, the MMA issuer, the softmax or gradient warps,
 * the decode consumers) waits longer than the limit for another, it gives up,
 * ORs PA_DEV_TIMEOUT into err_flag, tells the other roles to give up too,
 * waits (with their own limit) for the copies and MMAs it already started,
 * frees what it holds and returns; the outputs of that call are then
 * undefined, and the GPU context stays usable. The limit is 2 s, far beyond
 * any wait of a working kernel, so the path never runs in normal use. A test
 * shortens the limit with this hook to make the waits of a small call give
 * up on purpose and check that the call ends with the flag raised and that a
 * following normal call is correct.
 */
#ifndef PAGEDATTN_TESTING_H_
#define PAGEDATTN_TESTING_H_

#include "pagedattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Sets the give-up limit, in nanoseconds, of the waits between the roles of
 * the kernels that pa_attn_prefill, pa_attn_prefill_paged,
 * pa_attn_prefill_backward, pa_attn_decode_paged (and its no-allocation
 * variant), pa_attn_decode_paged_fp8 and pa_mla_decode_paged launch from now
 * on in this process, and returns the previous limit. 0, or anything above the
 * default of 2 s, restores the default. Under a limit below 1 ms the waits
 * poll without suspending the waiting threads and read the clock every few
 * polls, so that the limit is seen soon after it runs out. The waits for copies and
 * MMAs already in flight keep their own limit (0.1 s). Host-only: it touches
 * no device and affects launches made after it returns; set it back before
 * other work.
 */
PA_API unsigned long long pa_testing_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_TESTING_H_ */
