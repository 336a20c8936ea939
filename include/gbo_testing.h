/*
 * gbo_testing.h -- test hooks of libgbo.so.  These are not part of the
 * optimizer (the source pages have no counterpart); they let tests exercise
 * the library's failure handling without faulting or hanging a GPU.
 */
#ifndef GBO_TESTING_H
#define GBO_TESTING_H

#include "gbo.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launch one thread that runs the Newton-Schulz kernel's bounded mbarrier
 * wait on a barrier nothing ever arrives on, with a limit of `limit_us`
 * microseconds instead of the kernel's 2 s.  The wait gives up, ORs
 * GBO_STATUS_TIMEOUT into *dev_status (device int32) and the kernel returns;
 * the CUDA context stays usable.  Asynchronous on `stream`.
 * Errors: INVALID_ARG (NULL/misaligned status, limit outside 1..10^7 us),
 * UNSUPPORTED, CUDA.
 */
int gbo_testing_wait_timeout(int32_t *dev_status, uint32_t limit_us, gbo_stream_t stream);

/*
 * Whether Muon plans created from now on (any thread) run the Gram route's
 * p x p iterations of matrices with p <= 192 in bf16 mode as one on-chip
 * chain launch (enable != 0, the default) or as one tensor-core launch per
 * product with every p x p result stored in the workspace (enable == 0).
 * Both round every p x p result to bf16 once; tests compare them.
 * Returns the previous setting.  Plans already created keep theirs.
 */
int32_t gbo_testing_set_small_chain(int32_t enable);

/*
 * Whether Muon plans created from now on (any thread) run the Gram
 * X_0 X_0^T of the chain's wide matrices with p <= 128 inside the chain
 * launch, streaming X_0 through the matrix's shared memory (enable != 0, the
 * default), or as a tensor-core launch of its own that stores A_0 and P_0
 * for the chain to load (enable == 0).  Returns the previous setting.
 * Plans already created keep theirs.
 */
int32_t gbo_testing_set_fused_gram(int32_t enable);

/*
 * Test and A/B switch for plans created after the call: the on-chip Gram of
 * wide matrices of at most 128 rows with bf16 gradients on 16-byte rows
 * also runs their momentum pass (enable != 0): the chain kernel streams G
 * and B, writes B, and forms X_0 = bf16(D) and the pre-normalisation factor
 * itself (OMN page, Muon path: momentum, Nesterov direction, max-abs
 * rescale and Frobenius norm), so X_0 is not read back for the Gram; or
 * their momentum pass runs in the momentum kernel and the chain kernel
 * streams X_0 (enable == 0, the default: on a GB300 the momentum kernel's
 * many warps stream faster than the chain kernel's eight momentum warps).
 * Returns the previous setting.  Plans already created keep theirs.
 */
int32_t gbo_testing_set_fused_momentum(int32_t enable);

/*
 * Test and A/B switch, read at each launch of the bf16 CTA-pair
 * Newton-Schulz kernel: a launch whose last wave of 256 x 256 tiles would
 * occupy at most half of the resident CTA pairs runs those tiles as two
 * 256 x 128 halves each, so the launch ends after half a tile's time
 * (enable != 0, the default), or runs them whole (enable == 0).  Both give
 * the same results: every output element sums the same products in the
 * same order.  Returns the previous setting.
 */
int32_t gbo_testing_set_tail_split(int32_t enable);

/*
 * Test and A/B switch, read at each launch of the momentum pass: where every
 * matrix of a bf16-mode plan has flat momentum tiles (G and B rows on
 * 16-byte boundaries, X in stored orientation), the tiles stream through
 * shared memory by bulk copies, one block per SM with a producer warp
 * running ahead of three groups of eight consumer warps (enable != 0, the
 * default), or take the register kernel, several blocks per SM each loading
 * its own tiles (enable == 0).  Both give bitwise the same B, X_0 and norm partials: each
 * element is computed by the same operations.  Returns the previous setting.
 */
int32_t gbo_testing_set_momentum_stream(int32_t enable);

/*
 * How many CTA pairs (2-CTA clusters) of the bf16 Newton-Schulz kernel the
 * current device holds at once: the persistent grid of its pair launches.
 * Where the device's SMs do not all pair up within their clusters'
 * placement groups, the rest stay free while those launches run.  -1 on a
 * CUDA error (no device).
 */
int32_t gbo_testing_pair_residency(void);

/*
 * Test and A/B switch, read at every launch: whether launches carry the
 * programmatic-dependent-launch attribute, so that each kernel's prologue
 * (barrier set-up, TMEM allocation) runs under the previous kernel's tail:
 * 0 never, 1 always, 2 (the default) only while the stream is being
 * captured into a CUDA graph.  Measured on a GB300: in graph replays it made
 * the one-layer step ~1.7% faster; launched directly on a stream it made the
 * many-small-matrix step 12.7% slower.  Results are the same either way.
 * Returns the previous setting, or -1 for a mode outside 0 .. 2.
 */
int32_t gbo_testing_set_pdl(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* GBO_TESTING_H */
