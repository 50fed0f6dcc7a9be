/*
 * ea_checked.h - test hooks of the bounds-checked build of the library
 * (libea_checked.so, compiled with -DEA_CHECKS).  The normal build does not
 * export them.  The pages have no counterpart: these exist so that the
 * failure paths of the device code can be tested without a fault.
 */
#ifndef EA_CHECKED_H
#define EA_CHECKED_H

#include <stdint.h>

#include "ea.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * ea_checked_inject_prefill_timeout - make the next prefill attention launch
 * (ea_hybrid_attn_prefill, ea_prefill_attend, ea_hybrid_attn_prefill_varlen,
 * on any thread) leave out the K/V loads of key tile number `skip_load`
 * (0-based, counted over the tiles that each CTA pair's producer loads, in
 * order; every pair that reaches that count skips it) and give every bounded
 * device wait of that launch a limit of `timeout_ns` instead of 2 s.  The consumer of the
 * missing load then waits until the limit, sets EA_ERR_TIMEOUT in the
 * workspace error word, and every role of the kernel leaves within bounded
 * time.  One-shot: later launches are normal again.  Returns
 * EA_ERR_INVALID_ARG for skip_load < 0 or timeout_ns == 0.  Not thread safe.
 */
ea_status ea_checked_inject_prefill_timeout(int64_t skip_load, uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* EA_CHECKED_H */
