/*
 * dsa_diag.h -- attention diagnostics of dense decode attention (part of
 * libdsa.so, CUDA, sm_103a).
 *
 * "Understanding and Exploiting Diagonal Attention Sparsity in
 * Autoregressive Image Generation" (arXiv 2609.19702), section 3.4
 * "Attention Sparsity Analysis":
 *   - "Skewed attention toward prompt and local tokens" and Fig. 8: the
 *     attention weight a decode query puts on the prompt tokens, on the
 *     local tokens (the most recent 10 % of the decoded tokens) and on the
 *     middle tokens (the other decoded tokens), averaged over heads and
 *     decode steps;
 *   - "Diagonal attention sparsity pattern" and Fig. 10: the cosine
 *     similarity between the attention score vectors of query i and query
 *     i + d, over the same keys 0..i (vertical) or over the keys shifted by
 *     d, d..i+d (diagonal), averaged over heads and queries, as a function
 *     of the query distance d.
 * Readings taken where the page is open: query i is decode step i and
 * attends the prompt and decode keys 0..i with softmax(q k^T / sqrt(d))
 * (dense decode attention); "the most recent 10 %" of the i + 1 decoded
 * keys is ceil(0.1 (i + 1)) keys, the current one included; the score
 * vectors of the similarity hold the weights on decode keys only (the
 * page's ranges [0, i] and [d, i + d] index the decode region, where the
 * diagonal stripes lie; the prompt keys do not shift with the query); the
 * averages are uniform over every (head, query) pair with i + d < L_dec.
 *
 * The path of the method does not use these: they characterise a trace
 * (e.g. to check that a synthetic or recorded trace shows the diagonal
 * structure the method relies on).
 */
#ifndef DSA_DIAG_H
#define DSA_DIAG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * dsa_diag_trace -- the diagnostics of one layer's dense decode trace.
 *
 * Q:  device, [heads, L_dec, head_dim]  decode queries q_0 .. q_{L_dec-1}
 * Kp: device, [heads, L_p, head_dim]    prompt keys (NULL when L_p = 0)
 * Kd: device, [heads, L_dec, head_dim]  decode keys k_0 .. k_{L_dec-1}
 *     all of `dtype` (DSA_BF16 or DSA_F32), C-contiguous, 16-byte aligned;
 *     head_dim 64 or 128.
 * dist: host, [n_dist] query distances, each in [1, L_dec).
 * step_mass: device, [heads, L_dec, 3] float (prompt, local, middle weight
 *     of every query), or NULL.
 * mass_mean: host, [3]: the three weights averaged over heads and queries.
 * vertical, diagonal: host, [n_dist] each: the mean cosine similarities.
 *
 * Logits and weights are fp32 (bf16 products are exact in fp32).  The call
 * allocates its own scratch (at most about 1 GiB: the weights of a chunk of
 * heads, L_dec x (L_p + L_dec) floats per head), runs on `stream` and
 * returns once the results are on the host (synchronous).  Errors:
 * DSA_ERR_ARG (values, NULL or unaligned pointers), DSA_ERR_OOM, DSA_ERR_CUDA.
 */
int dsa_diag_trace(int heads, int head_dim, int L_p, int L_dec, int dtype, const void *Q, const void *Kp,
                   const void *Kd, int n_dist, const int32_t *dist, float *step_mass, double *mass_mean,
                   double *vertical, double *diagonal, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_DIAG_H */
