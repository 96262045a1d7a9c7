/*
 * dsa.h -- C ABI of the diagonal-aware sparse decode attention library
 * (libdsa.so, CUDA, sm_103a).
 *
 * The method is from "Understanding and Exploiting Diagonal Attention
 * Sparsity in Autoregressive Image Generation" (arXiv 2609.19702), section 4
 * "Diagonal-Aware Sparse Attention", Algorithm 1 and Fig. 12; the sink
 * variant is "Diagonal+sink4" of section 5.1.  Per decode step and per
 * stream (one sequence x one head of one layer) it attends the whole prompt
 * KV plus N_att of the N_r most recent decode KV entries, grows a per-stream
 * skip set by the argmin of the current logits during phase 2, moves that set
 * along the diagonal every step, and evicts the oldest entry once the window
 * is full.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - A handle holds `heads` independent streams (e.g. batch x heads of one
 *   layer) that all step together with one decode step counter t (0-based).
 *   Use one handle per layer.
 * - Device pointers are plain CUDA device addresses (e.g. a torch tensor's
 *   data_ptr()), C-contiguous, 16-byte aligned.  `stream` is a cudaStream_t
 *   passed as void* (NULL = the legacy default stream).  The library issues
 *   all device work on that stream and never synchronizes it, except in the
 *   functions documented as synchronous.
 * - Element type: DSA_BF16 (q, k, v, out and the stored KV are bf16,
 *   arithmetic in fp32), DSA_F32 (all fp32) or DSA_FP8_E4M3 (the stored KV
 *   is FP8 E4M3 with per-stream scales, see dsa_set_kv_scales; q, k_new,
 *   v_new, the prompt K / V and out are bf16; arithmetic in fp32).
 * - Ownership: the library owns every state buffer of a handle (prompt
 *   prefix, decode ring, skip bitmask, split partials) and frees them in
 *   dsa_destroy.  The caller owns q / k_new / v_new / out / K / V and must
 *   keep them alive until `stream` has passed the call.
 * - Errors: every function returns DSA_OK or a negative dsa_status.  Errors
 *   found on the host are returned at once and leave the handle unchanged;
 *   the message is available from dsa_last_error() on the same thread.
 *   Errors found on the device (a bounded wait that gave up, an internal
 *   consistency check) are recorded in a sticky per-handle status word that
 *   dsa_sync_status() reads.
 * - A handle is not thread-safe: do not call into one handle from two host
 *   threads at once.  Different handles are independent.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dsa_ctx *dsa_handle;

enum dsa_status {
    DSA_OK = 0,
    DSA_ERR_ARG = -1,          /* bad argument (value, size, NULL or unaligned pointer) */
    DSA_ERR_STATE = -2,        /* call out of order (decode before prefill, bad handle) */
    DSA_ERR_OOM = -3,          /* device allocation failed */
    DSA_ERR_CUDA = -4,         /* a CUDA runtime call failed (no device, launch error) */
    DSA_ERR_TIMEOUT = -5,      /* device: a bounded wait in a kernel gave up */
    DSA_ERR_DEVICE_CHECK = -6  /* device: an internal consistency check failed */
};

enum dsa_dtype { DSA_BF16 = 0, DSA_F32 = 1, DSA_FP8_E4M3 = 2 };

/*
 * dsa_create / dsa_create_ex -- allocate the state of `heads` streams.
 *
 * Algorithm 1 inputs (section 4): N_r is the recent-window size (decode KV
 * kept per stream; the page uses N_r = 0.5 L_dec), N_att the number of
 * decode tokens attended per step (sparsity 1 - N_att / L_dec), L_p the
 * prompt length.  `sink` > 0 selects the Diagonal+sink4 variant (section 5.1)
 * with `sink` attention sinks: decode tokens 0..sink-1 are kept and attended
 * at every step; the algorithm runs on the later tokens with a window of
 * N_r - sink and a budget of N_att - sink, so at most N_r decode entries are
 * held and at most N_att attended.  N_r = N_att = L_dec gives dense decode
 * attention; N_att = N_r gives a sliding window (StreamingLLM with sink).
 *
 * Requirements: heads >= 1; head_dim in {64, 128}; L_p >= 0;
 * 1 <= N_att <= N_r <= 65536 (+ sink); sink >= 0 and, if sink > 0,
 * N_att > sink.  dsa_create uses DSA_BF16.  Device memory:
 * dsa_state_bytes() plus split partials.  On success *out receives the
 * handle; on failure *out is set to NULL and nothing stays allocated.
 * Uses the current CUDA device.
 */
int dsa_create(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, dsa_handle *out);
int dsa_create_ex(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype,
                  dsa_handle *out);

/*
 * dsa_prefill -- load the prompt KV and reset the decode state (t = 0, empty
 * skip sets, status cleared).  Section 4, Algorithm 1 inputs K_p, V_p: the
 * prompt KV is always attended in full ("Throughout all phases, the prompt
 * KV is always attended in full").
 *
 * K, V: device, [heads, L_p, head_dim] of the handle's dtype (bf16 for
 * DSA_FP8_E4M3, which stores them as E4M3 codes with the handle's scales;
 * may be NULL when L_p = 0).  Asynchronous on `stream`.
 */
int dsa_prefill(dsa_handle h, const void *K, const void *V, void *stream);

/*
 * dsa_decode_step -- one decode step t for every stream, then t += 1.
 * Section 4, Algorithm 1 (all three phases) in one kernel launch:
 *   - append k_new, v_new as decode entry t (in the ring slot of the entry
 *     evicted at this step once t >= N_r: "K[t - N_r] <- empty");
 *   - attend q over the prompt rows plus the attended window entries
 *     idx = window - skip_idx; softmax and the weighted sum of V in fp32
 *     (a long stream, or one of few streams, is split over several warps
 *     whose partial results a second, small kernel merges);
 *   - in phase 2 (N_att - 1 <= t <= N_r - 2, sink removed) append the
 *     attended decode entry with the lowest logit q.k to the skip set (ties:
 *     the oldest); the entry is skipped from step t + 1 on.  The skip set is
 *     kept as relative offsets r = t - position, which the +1 diagonal shift
 *     leaves unchanged.
 * q, k_new, v_new: device, [heads, head_dim]; out: device, [heads, head_dim]
 * receives softmax(q [K_p; K[idx]]^T / sqrt(head_dim)) [V_p; V[idx]].
 * Asynchronous on `stream`.  Returns DSA_ERR_STATE before dsa_prefill.
 */
int dsa_decode_step(dsa_handle h, const void *q, const void *k_new, const void *v_new, void *out,
                    void *stream);

/* dsa_destroy -- free the handle and its device memory (synchronizes the
 * device first so no launch still uses it).  NULL is accepted. */
int dsa_destroy(dsa_handle h);

/* dsa_get_step -- the next decode step t (number of steps taken). */
int dsa_get_step(dsa_handle h, int *t);

/*
 * dsa_get_skip_mask -- copy the skip sets to host memory (synchronous on
 * `stream`).  host_dst: [heads, ceil((N_r - sink) / 32)] uint32; bit r of
 * stream s is set when relative offset r = t - position (of the decode
 * entries after the sinks) is skipped.  Not on the decode path.
 */
int dsa_get_skip_mask(dsa_handle h, uint32_t *host_dst, void *stream);

/*
 * dsa_get_last_selection -- per stream, the relative offset r* = t - j*
 * appended to the skip set by the last decode step, or -1 for every stream
 * if that step made no selection.  host_dst: [heads] int32.  Synchronous on
 * `stream`.  Not on the decode path.
 */
int dsa_get_last_selection(dsa_handle h, int32_t *host_dst, void *stream);

/*
 * dsa_sync_status -- synchronize `stream` and return the sticky device
 * status: DSA_OK, DSA_ERR_TIMEOUT or DSA_ERR_DEVICE_CHECK (or DSA_ERR_CUDA
 * if the synchronization itself failed).  dsa_prefill clears it.
 */
int dsa_sync_status(dsa_handle h, void *stream);

/* dsa_last_error -- message of the last failed call on this host thread
 * ("" if none).  The pointer stays valid until the next call on the thread. */
const char *dsa_last_error(void);

/*
 * dsa_state_bytes -- device bytes of the persistent state of a handle:
 * prompt prefix (L_p + sink rows) and decode ring (N_r - sink slots) of K
 * and V (1 byte per element for DSA_FP8_E4M3), plus the skip bitmask, per
 * stream.  This is the KV footprint bound
 * N_r + L_p of the cost analysis (section 4).  Split partials are extra.
 * Returns 0 for invalid arguments.
 */
size_t dsa_state_bytes(int heads, int head_dim, int L_p, int N_r, int sink, int dtype);

/*
 * Step plan: what dsa_decode_step does at step t (host computation only).
 * algo_bytes counts, over all streams, the HBM bytes the step must move:
 * the attended K and V rows read from the prefix and the ring (the current
 * token counted once, through k_new / v_new), q, k_new and v_new read, the
 * new entry written and out written.  The skip-bitmask read is excluded.
 */
typedef struct dsa_step_plan {
    int phase;                 /* 0: sink fill, 1 / 2 / 3: Algorithm 1 phases */
    int t_inner;               /* t - sink, or -1 during the sink fill */
    int n_prefix;              /* always-attended rows (prompt plus sinks) */
    int n_decode;              /* attended decode rows, current token included */
    int select;                /* 1 if this step appends to the skip set */
    int nsplit;                /* work items (pieces) per stream */
    int chunk;                 /* rows per work item */
    int grid;                  /* CTAs of the decode launch */
    int pipeline;              /* launch pipeline (1 .. 4, see dsa_set_pipeline) */
    unsigned long long algo_bytes;
    int cta_merge;             /* 1: split streams combined inside the decode launch (see dsa_set_merge) */
} dsa_step_plan;

int dsa_plan_step(dsa_handle h, int t, dsa_step_plan *out);

/*
 * dsa_plan_query -- the plan dsa_plan_step would report for step t of a
 * handle of these sizes on a device with `sm_count` SMs whose decode kernel
 * keeps ctas_per_sm[p] CTAs resident per SM under launch pipeline p + 1
 * (0: the pipeline cannot launch; [0] must be >= 1), cta_merge_ok[p] != 0
 * where the in-CTA merge of split streams keeps that occupancy (NULL: no
 * in-CTA merge).  Host only: touches no device and allocates nothing, so
 * the planning logic (Algorithm 1's step counts, the split and grid sizing,
 * the launch cost model) can be checked without a GPU.  Arrays have 4
 * entries.  DSA_ERR_ARG for sizes dsa_create would reject or bad arguments.
 */
int dsa_plan_query(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype, int t, int sm_count,
                   const int *ctas_per_sm, const int *cta_merge_ok, dsa_step_plan *out);

/*
 * dsa_decode_step_noalloc -- one decode step on state buffers the caller
 * owns, without any device allocation.  The paper has no counterpart: it is
 * an interface for callers that cannot allocate device memory while they
 * decode, e.g. a serving engine that reserves all device memory for its own
 * KV arena up front and does not let libraries take more, or a decode loop
 * that must not call the allocator because allocation can synchronize the
 * device.  It runs the same kernel as dsa_decode_step.
 *
 * The caller passes the configuration (as for dsa_create_ex), the step t
 * (0-based; the caller counts steps) and every buffer, all device pointers:
 *   prefix   [heads, L_p + sink, 2, head_dim]  entry i = K row i then V row i;
 *            rows 0..L_p-1 hold the prompt (the layout dsa_prefill builds),
 *            rows L_p.. are written by the sink fill; 16-byte aligned
 *   ring     [heads, N_r - sink, 2, head_dim]  decode entries; no
 *            initialisation needed; 16-byte aligned
 *   mask     [heads, ceil((N_r - sink) / 32)] uint32, all zero before t = 0
 *   last_sel [heads] int32, written on selection steps
 *   q, k_new, v_new, out  as for dsa_decode_step.
 * The split partials and a status word live in a static 4 MiB device array
 * of this library (every GPU that loads the library holds it until the
 * process exits).  Streams that run as one work item each (the usual case
 * beyond about a thousand streams) need only the status word; split streams
 * need 528 bytes per work item at head_dim 128 (272 at 64), so a step is
 * refused with DSA_ERR_ARG and a message when its streams x work items
 * exceed about 7,900 (15,400 at head_dim 64).  That check comes before the
 * pointers are looked at.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress): make that first call before any
 * stream capture.  Every call shares the array and clears its status word
 * when it starts, so calls that overlap on the GPU (other streams, other
 * threads) race: order them on one stream.  Device-side errors (a bounded
 * wait that gave up, a skip-mask count that disagrees with the step) are
 * recorded in that status word: dsa_decode_step_noalloc_status reads it.
 * Asynchronous on `stream`.
 */
int dsa_decode_step_noalloc(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype, int t,
                            void *prefix, void *ring, uint32_t *mask, int32_t *last_sel, const void *q,
                            const void *k_new, const void *v_new, void *out, void *stream);

/*
 * dsa_decode_step_noalloc_status -- the device status of the last
 * dsa_decode_step_noalloc call on the current device: waits for `stream`
 * (pass the stream of that call) and returns DSA_OK, DSA_ERR_TIMEOUT or
 * DSA_ERR_DEVICE_CHECK (DSA_ERR_CUDA if the copy failed).  Valid until the
 * next dsa_decode_step_noalloc call on the device, which clears the word.
 * Allocates nothing.  The paper has no counterpart.
 */
int dsa_decode_step_noalloc_status(void *stream);

/*
 * dsa_set_kv_scales -- per-stream scales of a DSA_FP8_E4M3 handle.  The
 * paper treats KV quantization as orthogonal to the method and applicable
 * on top of it (section 6, Related Works, "KV quantization for LLM") and
 * fixes no format; this library stores every K and V row (prompt, sinks,
 * decode entries) as OCP FP8 E4M3 codes: the code of an element x is the
 * E4M3 value nearest to fp32(x) * fp32(1 / scale) (ties to even; magnitudes
 * beyond 448 saturate to 448), and the attention uses code * scale.
 * k_scale, v_scale: host, [heads] float, each positive and finite (default
 * 1.0 for every stream).  Synchronizes the device, and discards the stored
 * sequence (its rows were coded with the old scales): dsa_prefill must
 * follow before the next decode step.  DSA_ERR_ARG for other dtypes or bad
 * values.  Not on the decode path.
 */
int dsa_set_kv_scales(dsa_handle h, const float *k_scale, const float *v_scale);

/* Tuning and test knobs (not needed for normal use). */

/* Force the number of work items (pieces) per stream (>= 1), or 0 for the
 * automatic choice.  Grows the partial buffers if needed (allocates; not on
 * the decode path). */
int dsa_set_splits(dsa_handle h, int nsplit);

/* Force the launch pipeline of the decode kernel, or 0 for the automatic
 * choice per step.  1: two 8 KB shared-memory stages per warp and at most
 * 512 decode rows per work item (12 warps per SM); 2: two 6 KB stages, at
 * most 256 rows per item (16 warps per SM); 3 and 4: the stages of 1 and 2,
 * three per warp (8 warps per SM).  Results do not depend on the pipeline
 * beyond fp32 rounding order (selections are identical).  DSA_ERR_ARG for
 * other values or a pipeline the device cannot launch. */
int dsa_set_pipeline(dsa_handle h, int pipeline);

/* How split streams are combined.  0 (default): where a step splits every
 * stream into 2 or 4 pieces and the pipeline has the shared memory to
 * spare, the pieces of a stream run on warps of one CTA and its piece-0
 * warp combines them through shared memory inside the decode launch (no
 * partials in global memory, no merge launch); otherwise a merge launch
 * combines the pieces' partials.  1: always the merge launch.  Both combine
 * the pieces in piece order with the same arithmetic: for the same plan
 * (pipeline and pieces, see dsa_set_pipeline and dsa_set_splits) results
 * are identical bit for bit.  The automatic plan weighs the cost of the
 * merge the mode implies, so the two modes may plan a step differently.
 * DSA_ERR_ARG for other values. */
int dsa_set_merge(dsa_handle h, int mode);

/* Copy the stored KV state to host memory (synchronizes the device): the
 * prompt prefix [heads, L_p + sink, 2, head_dim] and the decode ring
 * [heads, N_r - sink, 2, head_dim] (decode position p in slot (p - sink)
 * mod (N_r - sink)), in the stored element type (E4M3 codes for
 * DSA_FP8_E4M3).  Either pointer may be NULL.  Used by the tests to check
 * stored values bit for bit. */
int dsa_debug_copy_state(dsa_handle h, void *host_prefix, void *host_ring);

/*
 * dsa_debug_set_step -- move a freshly prefilled handle (step 0) to step t
 * without decoding the steps before it.  Only for handles that never
 * select (N_att == N_r: the dense and sliding-window settings, whose skip
 * sets stay empty), so the state at step t is the prompt plus the decode
 * entries alone.  The entries the jump passes over are zero rows (every
 * ring slot and the sink rows of the prefix are cleared; a zero K row
 * scores 0 and a zero V row adds nothing), so the next step attends the
 * prompt plus min(t + 1, N_r) decode rows as a real step t would: the same
 * rows, bytes and launch.  Lets a benchmark time the last steps of a long
 * dense trace without running all the steps before them.  Asynchronous on
 * `stream`.  DSA_ERR_STATE if the handle is not at step 0 after
 * dsa_prefill, or is in graph mode; DSA_ERR_ARG if N_att != N_r or t < 0.
 */
int dsa_debug_set_step(dsa_handle h, int t, void *stream);

/* Poll limit of the bounded waits inside the decode kernel (default: none;
 * every wait still gives up after about one second).  A limit of 0 makes
 * every wait give up at once; the kernel then records DSA_ERR_TIMEOUT, lets
 * its own copies land and returns.  Used to test the timeout path without a
 * real hang. */
int dsa_set_wait_limit(dsa_handle h, uint32_t limit);

/*
 * dsa_set_graph_mode -- CUDA-graph-replayable steady-state steps (not part of
 * the method; a runtime option).  With on != 0 the decode kernel takes the
 * step t from a counter in device memory (started at the handle's current
 * step) and the last CTA of every launch advances it, so a stream capture of
 * one dsa_decode_step per handle (e.g. all layers of one decode step) can be
 * replayed once per step with the same arguments: each replay decodes the
 * next step.  Only the steady state may run in this mode (t - sink >=
 * N_r - sink: every step evicts, none selects); dsa_decode_step returns
 * DSA_ERR_STATE before it.  Replays do not pass through the host, so the
 * handle's host-side step is stale until dsa_sync_step.  The inputs of a
 * replayed step are whatever the captured pointers hold at replay time.
 * Synchronizes the device when switching on.  on == 0 returns to host-side
 * steps (call dsa_sync_step first).  Errors: DSA_ERR_STATE, DSA_ERR_OOM,
 * DSA_ERR_CUDA.
 */
int dsa_set_graph_mode(dsa_handle h, int on);

/* Graph mode: waits for `stream` and sets the handle's step from the device
 * counter (no-op otherwise). */
int dsa_sync_step(dsa_handle h, void *stream);

/* Make the n-th following device allocation of this library fail (n >= 1),
 * or disable with n <= 0.  Host-side; tests the out-of-memory paths. */
int dsa_debug_fail_alloc_after(int n);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
