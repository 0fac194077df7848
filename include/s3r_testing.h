/*
 * s3r_testing.h - a test hook of libs3r.so, not part of the hot path.
 *
 * The kernels' waits on their own copies and on one another are bounded: a
 * wait that runs out sets S3R_DEVERR_TIMEOUT in the workspace's error word,
 * every role of the kernel leaves its loop, waits (again bounded) for the
 * copies it still has in flight, frees the tensor memory it holds and
 * returns, so the CUDA context stays usable.  Nothing in a correct call makes
 * a wait run out; this hook makes one run out on purpose, so that a test can
 * check that path.  It causes no fault, trap or unbounded wait.
 */
#ifndef S3R_TESTING_H
#define S3R_TESTING_H

#include "s3r.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Arm the next s3r_verify_attn / s3r_verify_attn_append call that runs on the
 * tensor-core verify kernel (more than 16 query rows per KV head); the flag
 * is host state of the library and is consumed by that launch.  In that
 * launch, CTA 0 issues no K copies for its first tile and never arrives on
 * that tile's barrier: the score MMA's wait for it runs out after its full
 * spin limit (about 4M probes of the barrier, some seconds), the abort spreads
 * to every role, and the drain's bounded wait for that barrier runs out too.
 * The call then reports S3R_DEVERR_TIMEOUT; its outputs are unspecified and
 * the workspace must be re-zeroed with s3r_workspace_init() before reuse.
 */
S3R_API void s3r_test_stall_next_verify(void);

#ifdef __cplusplus
}
#endif

#endif /* S3R_TESTING_H */
