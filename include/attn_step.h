/*
 * attn_step.h -- a whole decode step of the attention path as one launch.
 *
 * A decode step of Gemma-4-12B runs the attention calls of its 48 layers in
 * order (Gemma-4-12B model page, "Compute-graph nodes": per layer attn.qk_norm,
 * attn.v_norm, attn.rope, then attn.core; layer i is global iff i % 6 == 5).
 * Called one by one, every call costs a host launch and leaves a gap on the
 * GPU.  An attn_step records the calls once, captures them in order into one
 * CUDA graph on the current device, and then replays the whole step with one
 * launch.  Inside the graph consecutive kernels keep their programmatic
 * dependencies, so each call's prologue still overlaps the previous call's
 * tail exactly as with direct calls on one stream.
 *
 * Usage: attn_step_create; any number of attn_step_add_* in execution order;
 * attn_step_finalize; attn_step_launch as often as needed; attn_step_destroy.
 *
 * - Each attn_step_add_X takes the arguments of the function X declared in
 *   attn_decode.h, minus the stream, and runs X's host-side validation at
 *   once (same checks, same return codes and attn_last_error message);
 *   nothing is launched.  A call that fails validation is not recorded.
 * - The arrays are used in place: they must stay allocated, at the same
 *   addresses, until the step is destroyed.  Their contents may change
 *   between launches (the next step's q, seq_lens, block tables, cache).
 * - attn_step_finalize captures the recorded calls on the CUDA current device
 *   of the calling thread; every later launch must use a stream of that
 *   device.  No call may be added after it.
 * - attn_step_launch enqueues the whole step on `stream` (a cudaStream_t as
 *   void*; NULL = legacy default stream) and returns; the step's calls run
 *   in the order added, each after the previous one (as on one stream).  A
 *   step must not be launched again while an earlier launch of it may still
 *   be running on another stream (the calls reuse their outputs and
 *   workspaces).
 *
 * The ATTN_DEV_* status words given to the calls behave as with direct calls.
 * Return values: ATTN_OK or ATTN_ERR_* (attn_decode.h), with a message in
 * attn_last_error().
 */
#ifndef ATTN_STEP_H
#define ATTN_STEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct attn_step attn_step;

/* A new, empty step in *out (host memory owned by the library). */
int32_t attn_step_create(attn_step** out);

/* Frees the step and its graph.  NULL is ignored.  The caller makes sure no
 * launch of it is still running (for instance by synchronising its stream). */
void attn_step_destroy(attn_step* step);

int32_t attn_step_add_decode_sliding(attn_step* step, const void* q, const void* k_pool, const void* v_pool,
                                     const int32_t* block_table, const int32_t* seq_lens, void* o, int32_t batch,
                                     int32_t max_blocks, int64_t num_pages, int32_t max_seq_len, int32_t window,
                                     int32_t out_dtype, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                     int32_t* status);
int32_t attn_step_add_decode_global(attn_step* step, const void* q, const void* k_pool, const void* v_pool,
                                    const int32_t* block_table, const int32_t* seq_lens, void* o, int32_t batch,
                                    int32_t max_blocks, int64_t num_pages, int32_t max_seq_len, int32_t window,
                                    int32_t out_dtype, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                    int32_t* status);
int32_t attn_step_add_decode_global_shared(attn_step* step, const void* q, const void* kv_pool, const void* w_k,
                                           const int32_t* block_table, const int32_t* seq_lens, void* o,
                                           int32_t batch, int32_t max_blocks, int64_t num_pages,
                                           int32_t max_seq_len, int32_t window, int32_t out_dtype,
                                           int32_t num_splits, void* workspace, size_t workspace_bytes,
                                           int32_t* status);
int32_t attn_step_add_kv_append_sliding(attn_step* step, const void* qkv, const void* w_q, const void* w_k,
                                        const int32_t* block_table, const int32_t* positions, void* q_out,
                                        void* k_pool, void* v_pool, int32_t batch, int32_t max_blocks,
                                        int64_t num_pages, int32_t* status);
int32_t attn_step_add_kv_append_global(attn_step* step, const void* qkv, const void* w_q, const void* w_k,
                                       const int32_t* block_table, const int32_t* positions, void* q_out,
                                       void* k_pool, void* v_pool, int32_t batch, int32_t max_blocks,
                                       int64_t num_pages, int32_t* status);

/* Calls recorded so far, and kernels they launch per step. */
int32_t attn_step_num_calls(const attn_step* step);
int32_t attn_step_num_kernels(const attn_step* step);

/* Captures the recorded calls (at least one) into a CUDA graph and
 * instantiates it.  On failure nothing is kept and the step stays open. */
int32_t attn_step_finalize(attn_step* step);

/* One launch of the whole step on `stream`; the step must be finalized. */
int32_t attn_step_launch(attn_step* step, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_STEP_H */
