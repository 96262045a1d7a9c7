/*
 * dsa_policy.h -- score-based KV eviction baselines (TOVA, H2O) in the same
 * gather framework as the diagonal method (part of libdsa.so, CUDA, sm_103a).
 *
 * "Understanding and Exploiting Diagonal Attention Sparsity in
 * Autoregressive Image Generation" (arXiv 2609.19702), section 2 ("KV cache
 * sparsity techniques", Fig. 2) and section 5.1 ("Sparse KV baselines"):
 * score-based methods keep KV pairs by attention scores; TOVA evicts the key
 * with the minimum score at each step, H2O keeps heavy hitters by
 * accumulated attention scores; the prompt KV is always attended in full.
 *
 * Readings taken where the page is silent (per stream = sequence-head, as
 * for the diagonal method):
 *   - budget: step t (0-based) attends the prompt and a_t = min(t + 1, N_att)
 *     decode entries, the current token included; between steps at most
 *     N_att - 1 decode entries are kept (N_att slots per stream);
 *   - TOVA: once a_t = N_att, the attended decode entry with the lowest
 *     logit q_t . k (lowest softmax weight) is evicted after the step, the
 *     current token included; ties go to the oldest position;
 *   - H2O: each decode entry accumulates its normalised attention weight
 *     (softmax over the prompt and the attended decode entries) over the
 *     steps it is attended, from the step it enters; once a_t = N_att, the
 *     n_recent = min(ceil(N_att / 2), N_att - 1) newest entries are kept and
 *     among the others the lowest accumulated weight is evicted, ties to the
 *     oldest.
 *
 * One handle = one layer's `heads` streams stepping together, as dsa_create.
 */
#ifndef DSA_POLICY_H
#define DSA_POLICY_H

#include <stddef.h>
#include <stdint.h>

#include "dsa.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { DSA_POLICY_TOVA = 1, DSA_POLICY_H2O = 2 };

typedef struct dsa_pol_ctx *dsa_pol; /* opaque; library-owned */

/*
 * dsa_pol_create -- a handle of `heads` streams under `policy`
 * (DSA_POLICY_TOVA or DSA_POLICY_H2O) with `N_att` >= 1 attended decode
 * entries, prompt length L_p >= 0, head_dim 64 or 128, dtype DSA_BF16 or
 * DSA_F32 (the type of every K / V row, q, k_new, v_new and out).
 * Allocates the prompt prefix [heads, L_p, 2, head_dim], N_att slots
 * [heads, N_att, 2, head_dim], the position held by each slot and, for H2O,
 * the accumulated weight of each slot (int32 / float [heads, N_att]).
 * Errors: DSA_ERR_ARG, DSA_ERR_OOM, DSA_ERR_CUDA.
 */
int dsa_pol_create(int heads, int head_dim, int L_p, int N_att, int policy, int dtype, dsa_pol *out);

/* Frees the handle (synchronizes the device first).  NULL is accepted. */
int dsa_pol_destroy(dsa_pol h);

/* Prompt K, V: device, [heads, L_p, head_dim] each (ignored when L_p = 0);
 * resets the step to 0 and empties the decode cache.  Asynchronous. */
int dsa_pol_prefill(dsa_pol h, const void *K, const void *V, void *stream);

/*
 * dsa_pol_decode_step -- one decode step: q, k_new, v_new, out device
 * [heads, head_dim] each, 16-byte aligned.  Appends the current token,
 * attends the prompt and the attended decode entries, writes out, and
 * applies the eviction.  Asynchronous on `stream`; advances the step.
 * Errors: DSA_ERR_STATE (invalid handle, no prefill), DSA_ERR_ARG,
 * DSA_ERR_CUDA; device-side faults via dsa_pol_sync_status.
 */
int dsa_pol_decode_step(dsa_pol h, const void *q, const void *k_new, const void *v_new, void *out, void *stream);

/* Positions of the decode entries the cache holds after the last step:
 * host [heads, N_att] int32, -1 for an empty slot (synchronous). */
int dsa_pol_get_positions(dsa_pol h, int32_t *host_dst, void *stream);

/* Position evicted by the last step, per stream: host [heads] int32, -1 if
 * none (synchronous). */
int dsa_pol_get_last_eviction(dsa_pol h, int32_t *host_dst, void *stream);

/* Waits for `stream`; DSA_ERR_TIMEOUT if a bounded wait of the kernel gave
 * up (sticky). */
int dsa_pol_sync_status(dsa_pol h, void *stream);

/* Test knob: polls per bounded wait before giving up (0: at once). */
int dsa_pol_set_wait_limit(dsa_pol h, uint32_t limit);

/* Test knob: force the launch shape, stage size and stages per warp
 * (1: 8 KB x 2, 2: 6 KB x 2, 3: 8 KB x 3, 4: 6 KB x 3, 5: 8 KB x 4, 6: 6 KB
 * x 4), or 0 for the automatic choice: the shape whose resident warps take
 * the streams in the fewest rounds, and among those the deepest pipeline
 * per warp.  DSA_ERR_ARG if the shape cannot launch for this handle.
 * Results do not depend on it. */
int dsa_pol_set_shape(dsa_pol h, int shape);

#ifdef __cplusplus
}
#endif

#endif /* DSA_POLICY_H */
