/*
 * dsa_proj.h -- the QKV projection with rotary position embedding that feeds
 * a decode step, and the fused layer step built on it (part of libdsa.so,
 * CUDA, sm_103a).
 *
 * "Understanding and Exploiting Diagonal Attention Sparsity in
 * Autoregressive Image Generation" (arXiv 2609.19702), section 2,
 * "LLM-aligned decoding behavior": each decoder layer projects the newest
 * token's hidden state to a query, key and value before causal
 * self-attention; section 5.3, Fig. 16(b), times this QKV projection as one
 * part of every decode step.  For one layer and step:
 *
 *     [q | k | v] = x W^T                 x: [B, hidden]    W: [3 H d, hidden]
 *     q, k <- RoPE(q, pos), RoPE(k, pos)   per head; v is not rotated
 *
 * Readings taken where the page is silent (its models are LLaMA-style
 * decoders): W is a linear layer's weight ([out_features, in_features], row
 * major), the q rows of all heads first (d rows per head), then k, then v,
 * and there is no bias; RoPE is the rotate-half form with base 10000
 * (elements j and j + d/2 of a head turn together by pos * 10000^(-2j/d));
 * outputs are ordered as decode streams, s = b * H + h, each a d-vector; the
 * position of decode token t is L_p + t.
 *
 * The projection runs on the tensor cores (tcgen05.mma, bf16 operands, fp32
 * accumulation in tensor memory), with W and x staged by TMA and RoPE applied
 * in the epilogue; the results are rounded to bf16 once.
 */
#ifndef DSA_PROJ_H
#define DSA_PROJ_H

#include <stddef.h>
#include <stdint.h>

#include "dsa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dsa_proj_ctx *dsa_proj; /* opaque; library-owned */

/*
 * dsa_proj_create -- a projection context for `batch` tokens of `heads`
 * heads of `head_dim`, from `hidden` input features.
 *
 * batch in [1, 256]; head_dim 64 or 128; heads * head_dim a multiple of 128
 * (an even head count at head_dim 64); hidden a positive multiple of 64.
 * Allocates on the current device: the split-reduction scratch (SMs x
 * batch (rounded up to 16) x 128 floats plus one counter per 128 output
 * features) and bf16 staging for one step's q (batch x
 * heads x head_dim), used by dsa_decode_step_fused.  Errors: DSA_ERR_ARG,
 * DSA_ERR_OOM, DSA_ERR_CUDA.
 */
int dsa_proj_create(int batch, int heads, int head_dim, int hidden, dsa_proj *out);

/* Frees the context (synchronizes the device first).  NULL is accepted. */
int dsa_proj_destroy(dsa_proj p);

/*
 * dsa_qkv_rope -- q, k, v of one decode step at position `pos` (>= 0).
 *
 * x: device, [batch, hidden] bf16, row major.
 * W: device, [3 * heads * head_dim, hidden] bf16, row major (see above).
 * q, k, v: device, [batch * heads, head_dim] bf16 each (caller-owned).
 * All 16-byte aligned.  Asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream); launched as a programmatic dependent launch:
 * it starts reading W while the previous kernel in the stream finishes (so
 * W must not be written by that kernel), and touches x, q, k, v and its
 * scratch only after that kernel has completed.  Deterministic: an output
 * tile shared by several CTAs is summed in a fixed order.  Launches that use
 * one context must not overlap (one stream, or ordered streams).
 * Errors: DSA_ERR_STATE (invalid context), DSA_ERR_ARG (NULL, unaligned or
 * negative arguments), DSA_ERR_CUDA (launch).  Device-side faults (a bounded
 * wait that gave up) are reported by dsa_proj_sync_status.
 */
int dsa_qkv_rope(dsa_proj p, const void *x, const void *W, int pos, void *q, void *k, void *v, void *stream);

/*
 * dsa_decode_step_fused -- one decode step of handle h whose q, k_new and
 * v_new come from the projection of x by W at position L_p + t (t = h's
 * step counter).  The projection kernel writes q to p's staging buffer and
 * k_new, v_new straight into the decode state, in its stored form (bf16, or
 * for a DSA_FP8_E4M3 handle the E4M3 codes of fp32(value) / scale with the
 * stream's scales), at the slot the newest token takes at this step (its
 * ring slot, or its prefix row during the sink fill); the decode kernel
 * reads the token there and appends nothing.  The results equal
 * dsa_qkv_rope followed by dsa_decode_step bit for bit.
 *
 * h must be a DSA_BF16 or DSA_FP8_E4M3 handle with heads = batch * heads of
 * p and the same head_dim, not in graph mode (the position and the slot are
 * taken from the host's step counter).  x, W, out as in dsa_qkv_rope /
 * dsa_decode_step.  Asynchronous on `stream`; advances t.  Errors: as
 * dsa_decode_step and dsa_qkv_rope, DSA_ERR_ARG when h and p do not match,
 * DSA_ERR_STATE in graph mode.
 */
int dsa_decode_step_fused(dsa_handle h, dsa_proj p, const void *x, const void *W, void *out, void *stream);

/*
 * Waits for `stream` and reports the projection kernel's sticky device
 * status: DSA_ERR_TIMEOUT if one of its bounded waits gave up (the outputs
 * of that launch are undefined).  Reading an error also resets the status
 * and the split-reduction counters, so the context can be used again.
 */
int dsa_proj_sync_status(dsa_proj p, void *stream);

/* Test knob: the polls each bounded wait of the projection kernel makes
 * before it gives up (0: give up at once; default: unbounded polls, one
 * second of wall time). */
int dsa_proj_set_wait_limit(dsa_proj p, uint32_t limit);

#ifdef __cplusplus
}
#endif

#endif /* DSA_PROJ_H */
