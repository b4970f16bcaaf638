/*
 * attn_step.h -- a whole decode step of the attention path as one launch.
 *
 * A decode step of Gemma-4-12B runs the attention calls of its 48 layers in
 * order (Gemma-4-12B model page, "Compute-graph nodes": per layer attn.qk_norm,
 * attn.v_norm, attn.rope, then attn.core; layer i is global iff i % 6 == 5).
 * Called one by one, every call costs host work (validation, tensor-map
 * encoding, launches).  An attn_step records the calls once and then replays
 * the whole step with one call, in one of two launch modes:
 *
 * - ATTN_STEP_LAUNCH_GRAPH: the step's kernels are captured in order into
 *   one CUDA graph on the current device; a launch is one cudaGraphLaunch.
 *   Inside the graph consecutive kernels keep their programmatic
 *   dependencies, so each call's prologue overlaps the previous call's tail
 *   as with direct calls on one stream.  Across two graph launches it does
 *   not: a graph's first kernel starts only once the previous graph has
 *   ended.
 * - ATTN_STEP_LAUNCH_DIRECT: the step's kernel launches, with every argument
 *   (tensor maps included) built once at finalize, are enqueued back to back
 *   on the stream, one cudaLaunchKernelEx each.  Programmatic overlap then
 *   also holds between consecutive steps, at the cost of one host launch per
 *   kernel.
 * - ATTN_STEP_LAUNCH_AUTO (the default): DIRECT for steps of at most
 *   ATTN_STEP_DIRECT_MAX_KERNELS kernels, where the boundary between two
 *   graph launches is a measurable share of the step; GRAPH otherwise.
 *
 * Usage: attn_step_create; any number of attn_step_add_* in execution order;
 * optionally attn_step_set_launch_mode; attn_step_finalize; attn_step_launch
 * as often as needed; attn_step_destroy.
 *
 * - Each attn_step_add_X takes the arguments of the function X declared in
 *   attn_decode.h, minus the stream, and runs X's host-side validation at
 *   once (same checks, same return codes and attn_last_error message);
 *   nothing is launched.  A call that fails validation is not recorded.
 * - The arrays are used in place: they must stay allocated, at the same
 *   addresses, until the step is destroyed.  Their contents may change
 *   between launches (the next step's q, seq_lens, block tables, cache).
 * - attn_step_finalize runs every recorded call once more with its kernel
 *   launches recorded instead of enqueued (host validation again, tensor
 *   maps encoded, kernel attributes set), on the CUDA current device of the
 *   calling thread, and in GRAPH mode captures them into a graph.  Every
 *   later launch must use a stream of that device.  No call may be added
 *   after it.
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

/* Launch modes (see above). */
#define ATTN_STEP_LAUNCH_AUTO 0
#define ATTN_STEP_LAUNCH_GRAPH 1
#define ATTN_STEP_LAUNCH_DIRECT 2
/* AUTO picks DIRECT for steps of at most this many kernels (two calls). */
#define ATTN_STEP_DIRECT_MAX_KERNELS 4

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

/* Chooses the launch mode (ATTN_STEP_LAUNCH_*) before attn_step_finalize.
 * ATTN_ERR_INVALID_ARG for an unknown mode or a finalized step. */
int32_t attn_step_set_launch_mode(attn_step* step, int32_t mode);

/* The mode requested so far; after attn_step_finalize, the mode in use
 * (GRAPH or DIRECT).  -1 for a NULL step. */
int32_t attn_step_launch_mode(const attn_step* step);

/* Records the launches of the recorded calls (at least one) and, in GRAPH
 * mode, captures them into a CUDA graph and instantiates it.  On failure
 * nothing is kept and the step stays open. */
int32_t attn_step_finalize(attn_step* step);

/* One replay of the whole step on `stream`; the step must be finalized.  In
 * DIRECT mode the kernels are enqueued on the step's device (made current
 * for the call and restored after it). */
int32_t attn_step_launch(attn_step* step, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_STEP_H */
