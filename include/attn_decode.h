/*
 * attn_decode.h -- C ABI of the GB300 (sm_103a) paged decode-attention library
 * for the Gemma-4-12B text path.
 *
 * Two operations, one per attention node of the model's compute graph
 * (Gemma-4-12B model page, "Compute-graph nodes", the two attn.core rows):
 *
 *   attn_decode_sliding -- node `slidingDecodeGQA`, the 40 sliding-window layers:
 *       16 query heads over 8 KV heads (query head h reads KV head h/2),
 *       head dim 256, window 1024, scale 1.
 *   attn_decode_global  -- node `decodeGQA`, the 8 global layers:
 *       16 query heads over 1 KV head (h/16 = 0), head dim 512, scale 1.
 *
 * Both compute, for every sequence b and query head h with c = h / G,
 *
 *   o[b,h,:] = sum over visible l of softmax_l( <q[b,h,:], k[b,l,c,:]> ) * v[b,l,c,:]
 *
 * where the softmax is normalised over the visible positions only
 * (Attention.lean `softmax`), the query sits at position p = L-1 with
 * L = seq_lens[b] (Attention.lean `decodeGQA`), and position l is visible iff
 * l <= p and, when a window w > 0 is given, p < l + w (Attention.lean
 * `slidingGQA`), i.e. the last min(L, w) positions (Op Specs page, NOTE on
 * slidingDecodeGQA).  The scale is fixed at 1 ("the q/k norms take its
 * place", Gemma-4-12B model page, "What to watch for"); there is no logit
 * soft-cap in attention (only the LM head is capped).  L == 0 gives o = 0.
 *
 * KV cache: pages of 16 token positions (Gemma-4-12B model page, "At a
 * glance", shape domain: page size 16).  A pool is one contiguous array
 * [num_pages, 16, Hkv, D] of bf16 -- each page holds 16 token rows, each row
 * the Hkv heads of one position, the token-major order of the attn.core
 * tensor k[B, S, Hkv, D].  Position l of sequence b lives in page
 * block_table[b * max_blocks + l / 16], row l % 16.  Entries for pages that
 * hold no visible position are never read and may be -1.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All array pointers are DEVICE pointers owned by the caller; each must be
 *   16-byte aligned and the arrays contiguous in the layouts stated.
 * - The library allocates no memory and never synchronises: work is enqueued
 *   on `stream` (a cudaStream_t passed as void*; NULL = legacy default stream)
 *   and the call returns as soon as it is launched.
 * - Host-side validation runs before anything is launched; on any error
 *   nothing is enqueued and the call returns a nonzero ATTN_ERR_* code, with
 *   a message in attn_last_error() (per host thread).
 * - `status` (optional, may be NULL) is a device int32 that the kernels OR
 *   ATTN_DEV_* bits into when they detect a contract violation on the device
 *   (the host cannot see seq_lens or block_table without a synchronisation).
 *   The caller zeroes it and reads it back when it wants to check.  A page id
 *   outside [0, num_pages) on a visible position is never dereferenced: the
 *   copy engine fills that page with zeros and ATTN_DEV_BAD_PAGE is raised.
 * - The device (SM count) is the CUDA current device of the calling thread.
 */
#ifndef ATTN_DECODE_H
#define ATTN_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_DECODE_ABI_VERSION 1

/* return codes */
#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG 1 /* null or misaligned pointer, bad size           */
#define ATTN_ERR_UNSUPPORTED 2 /* outside the model's shape domain               */
#define ATTN_ERR_WORKSPACE 3   /* workspace missing or smaller than required     */
#define ATTN_ERR_CUDA 4        /* a CUDA runtime/driver call or launch failed    */

/* output element type */
#define ATTN_OUT_BF16 0 /* o is bf16, rounded to nearest even                    */
#define ATTN_OUT_F32 1  /* o is fp32                                             */

/* operation kinds (for the planning queries) */
#define ATTN_KIND_SLIDING 0
#define ATTN_KIND_GLOBAL 1

/* device status bits (OR-ed into *status) */
#define ATTN_DEV_WAIT_TIMEOUT 1 /* a copy-pipeline wait exceeded its time limit     */
#define ATTN_DEV_BAD_PAGE 2     /* visible position mapped to page id not in [0,num_pages) */
#define ATTN_DEV_BAD_SEQ_LEN 4  /* seq_lens[b] < 0 or > max_blocks*16 (clamped)      */
#define ATTN_DEV_INTERNAL 8     /* an internal index check failed; the access was skipped */

/* Fixed shapes of the two operations (Gemma-4-12B model page, attn.core rows). */
#define ATTN_SLIDING_HQ 16
#define ATTN_SLIDING_HKV 8
#define ATTN_SLIDING_D 256
#define ATTN_GLOBAL_HQ 16
#define ATTN_GLOBAL_HKV 1
#define ATTN_GLOBAL_D 512
#define ATTN_PAGE_SIZE 16

/* attn.rope of each layer type (model page, "What to watch for" and the
 * attn.rope rows): pairs (i, i + D/2), i < PAIRS, turn by pos * THETA^(-2i/D). */
#define ATTN_SLIDING_ROPE_THETA 10000.0
#define ATTN_SLIDING_ROPE_PAIRS 128
#define ATTN_GLOBAL_ROPE_THETA 1000000.0
#define ATTN_GLOBAL_ROPE_PAIRS 64

/* Shape domain (Gemma-4-12B model page, "At a glance"): B in [1,256],
 * up to 262144 cached positions. */
#define ATTN_MAX_BATCH 256
#define ATTN_MAX_SEQ_LEN 262144

/* The first ATTN_WORKSPACE_ZERO_BYTES of every decode workspace hold the
 * arrival counters of the in-grid merge (see num_splits below).  They must be
 * zero before a workspace is first used; every call leaves them zero.  The
 * rest of the workspace needs no initialisation.  A call that finds a counter
 * above its number of arrivals raises ATTN_DEV_INTERNAL (its sequence may then
 * be left unwritten); a counter left below it cannot be told apart. */
#define ATTN_WORKSPACE_ZERO_BYTES 8192

/*
 * attn_decode_sliding -- slidingDecodeGQA (Gemma-4-12B sliding layers).
 *
 * q            bf16 [batch, 16, 256]
 * k_pool       bf16 [num_pages, 16, 8, 256]
 * v_pool       bf16 [num_pages, 16, 8, 256]
 * block_table  int32 [batch, max_blocks]
 * seq_lens     int32 [batch], 0 <= L <= max_blocks*16
 * o            [batch, 16, 256], bf16 or fp32 per out_dtype (written, never read)
 * batch        1..256
 * max_blocks   >= 1, width of block_table
 * num_pages    >= 1, pages in each pool; num_pages*16 < 2^31
 * max_seq_len  host-side upper bound on seq_lens (0..max_blocks*16); it only
 *              caps how many thread blocks are launched for small problems
 *              and never changes which positions are read
 * window       > 0; the node's value is 1024
 * out_dtype    ATTN_OUT_BF16 or ATTN_OUT_F32
 * num_splits   0 = automatic (one wave of resident thread blocks); > 0 forces
 *              that many thread blocks per KV head (at most 1024).  The
 *              visible pages of all sequences, concatenated, are cut into
 *              that many equal spans; each block of a sequence cut by a span
 *              boundary leaves a partial softmax result.  When the plan
 *              bounds the blocks that can share a sequence to at most 24
 *              (sliding calls whose window, or max_seq_len, caps a sequence
 *              at 92 visible pages or fewer; the node's window of 1024 caps
 *              it at 65 pages, 18 blocks) and expects at most 8 (spans
 *              sized as if every sequence had its cap of visible pages),
 *              the last of them to finish merges the partials inside the
 *              decode kernel;
 *              otherwise a second kernel merges them.  attn_decode_launches
 *              tells which.  The result does not depend on this value beyond
 *              floating-point regrouping.
 * workspace    device scratch of at least attn_decode_workspace_size(...)
 *              bytes for those partial results; its first
 *              ATTN_WORKSPACE_ZERO_BYTES must be zero before its first use
 *              (every call leaves them zero), the rest needs no
 *              initialisation; must not be shared by calls that may overlap
 * status       optional device int32 for ATTN_DEV_* bits, or NULL
 * stream       cudaStream_t, as void*
 * returns      ATTN_OK or ATTN_ERR_*
 */
int32_t attn_decode_sliding(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_table, const int32_t* seq_lens, void* o,
                            int32_t batch, int32_t max_blocks, int64_t num_pages,
                            int32_t max_seq_len, int32_t window, int32_t out_dtype,
                            int32_t num_splits, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream);

/*
 * attn_decode_global -- decodeGQA (Gemma-4-12B global layers).
 *
 * Same arguments as attn_decode_sliding, with shapes
 *   q bf16 [batch, 16, 512];  k_pool, v_pool bf16 [num_pages, 16, 1, 512];
 *   o [batch, 16, 512].
 * window <= 0 is the node as printed (no window, every cached key visible);
 * window > 0 applies the slidingGQA visibility rule.
 * k_pool and v_pool may be the same pointer.
 */
int32_t attn_decode_global(const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_table, const int32_t* seq_lens, void* o,
                           int32_t batch, int32_t max_blocks, int64_t num_pages,
                           int32_t max_seq_len, int32_t window, int32_t out_dtype,
                           int32_t num_splits, void* workspace, size_t workspace_bytes,
                           int32_t* status, void* stream);

/*
 * attn_decode_global_shared -- decodeGQA over a values-only global cache.
 *
 * On global layers keys and values come from one head x (Gemma-4-12B model
 * page, "What to watch for": values = keys; "Compute-graph nodes":
 * attn.qk_norm, attn.v_norm, attn.rope): V = rmsnormUnit(x) and
 * K = rope(rmsnorm(x) * w_k), so K = rope(V * w_k) and the cache need hold
 * V only.  This call reads V pages only (half the bytes of
 * attn_decode_global) and rebuilds each visible key as
 *
 *   k[l] = bf16( rope(v[l] * w_k, l) )     (rounded once, nearest even)
 *
 * with RoPE over pairs (i, i + 256), i < ATTN_GLOBAL_ROPE_PAIRS, angle
 * l * ATTN_GLOBAL_ROPE_THETA^(-2i/512), l the key's own position; then it
 * computes exactly what attn_decode_global computes with that k_pool.
 *
 * kv_pool   bf16 [num_pages, 16, 1, 512]: V, as attn_kv_append_global
 *           writes it with k_pool = NULL
 * w_k       bf16 [512]: the qk_norm weight of the keys (device pointer)
 * Every other argument, the plan and the workspace are attn_decode_global's.
 * The product v * w_k is exact in fp32; the rotation is fp32 with angles
 * accurate to about 1e-7 rad, so a rebuilt key may differ from the fp64
 * definition by one bf16 rounding step.
 */
int32_t attn_decode_global_shared(const void* q, const void* kv_pool, const void* w_k,
                                  const int32_t* block_table, const int32_t* seq_lens, void* o,
                                  int32_t batch, int32_t max_blocks, int64_t num_pages,
                                  int32_t max_seq_len, int32_t window, int32_t out_dtype,
                                  int32_t num_splits, void* workspace, size_t workspace_bytes,
                                  int32_t* status, void* stream);

/*
 * attn_decode_plan -- the launch plan, as pure host arithmetic (no CUDA call).
 *
 * kind         ATTN_KIND_SLIDING or ATTN_KIND_GLOBAL
 * batch, max_seq_len, window, num_splits   as for the operations
 * num_sms      streaming multiprocessors of the target device (>= 1)
 * out_num_splits        receives the thread blocks per KV head (see num_splits)
 * out_workspace_bytes   receives the workspace size the operation requires
 * returns      ATTN_OK or ATTN_ERR_INVALID_ARG
 */
int32_t attn_decode_plan(int32_t kind, int32_t batch, int32_t max_seq_len, int32_t window,
                         int32_t num_splits, int32_t num_sms, int32_t* out_num_splits,
                         size_t* out_workspace_bytes);

/*
 * attn_decode_launches -- kernels one decode call with these arguments
 * launches on a device of num_sms multiprocessors (host arithmetic only, like
 * attn_decode_plan): 1 when the split sequences are merged inside the decode
 * kernel, 2 when a combine kernel follows it; -1 (and attn_last_error) on bad
 * arguments.
 */
int32_t attn_decode_launches(int32_t kind, int32_t batch, int32_t max_seq_len, int32_t window,
                             int32_t num_splits, int32_t num_sms);

/*
 * attn_decode_workspace_size -- attn_decode_plan's workspace size for the
 * current CUDA device.  Returns 0 (and sets attn_last_error) on bad
 * arguments or when no device can be queried.
 */
size_t attn_decode_workspace_size(int32_t kind, int32_t batch, int32_t max_seq_len,
                                  int32_t window, int32_t num_splits);

/*
 * attn_decode_sliding_noalloc -- attn_decode_sliding for callers that cannot
 * allocate device memory.  The pages this library follows have no
 * counterpart for it: it exists for integration, not for the method.
 *
 * Some callers have no way to hand over a workspace: a plugin in a serving
 * runtime that gets device pointers for its inputs and outputs but no
 * allocator, code whose device memory is fixed by a budget set up front, or
 * a caller that must not touch the CUDA allocator on its hot path
 * (cudaMalloc can synchronise the device and stall other streams).  This
 * entry point takes the same arguments as
 * attn_decode_sliding minus the workspace, and keeps the partial results of
 * split sequences in a fixed 8 MiB array compiled into the library, which
 * every GPU that loads the library holds until the process exits.  It calls
 * no cudaMalloc, cudaFree or other allocating routine.
 *
 * - The first call on a device (with that device current) looks up the
 *   array's device address with cudaGetSymbolAddress; make that first call
 *   before any stream capture.  The address is kept for the life of the
 *   process, so this entry point must not be used on a device after
 *   cudaDeviceReset on it (the array may then sit elsewhere).
 * - Calls whose plan needs more than 8 MiB of scratch are rejected with
 *   ATTN_ERR_UNSUPPORTED and a message; nothing is launched.  The automatic
 *   plan (num_splits = 0) fits for every batch up to ATTN_MAX_BATCH; large
 *   forced num_splits may not.
 * - All calls share the one array, which keeps whatever the last call left
 *   there.  Nothing in it needs to start at zero: each call writes the
 *   partial rows it reads.  Calls that may overlap on the GPU (concurrent
 *   streams, or several host threads) race on the array and must be
 *   serialised by the caller.
 * - Everything else (arguments, layouts, errors, status bits, results) is as
 *   for attn_decode_sliding.
 */
int32_t attn_decode_sliding_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                    const int32_t* block_table, const int32_t* seq_lens, void* o,
                                    int32_t batch, int32_t max_blocks, int64_t num_pages,
                                    int32_t max_seq_len, int32_t window, int32_t out_dtype,
                                    int32_t num_splits, int32_t* status, void* stream);

/*
 * attn_kv_append_sliding / attn_kv_append_global -- the steps that feed the
 * decode for one new token per sequence (Gemma-4-12B model page, "Compute-
 * graph nodes": attn.qk_norm, attn.v_norm, attn.rope; "What to watch for":
 * the RoPE constants above and "values = keys" on global layers):
 *
 *   q heads  q_out[b,h] = rope(rmsnorm(x_q[b,h]) * w_q, pos)
 *   key      rope(rmsnorm(x_k) * w_k, pos)  -> k_pool at the token's slot
 *   value    rmsnormUnit(x_v)                -> v_pool at the token's slot
 *
 * with rmsnorm(x)[i] = x[i] / sqrt(sum_j x[j]^2 / D + 1e-6), pos =
 * positions[b], and the token's slot = page block_table[b, pos/16], row
 * pos % 16 (so the caller's next decode call has seq_lens[b] = pos + 1).
 *
 * qkv          bf16 [batch, row]: the attn.qkv_proj output of the token.
 *              Sliding: row = [q 16x256 | k 8x256 | v 8x256] (8192).
 *              Global: row = [q 16x512 | x 512] (8704); x gives both the key
 *              (qk_norm with w_k, then RoPE) and the value (v_norm).
 * w_q, w_k     bf16 [D]: the qk_norm weights, shared by all heads.
 * block_table  int32 [batch, max_blocks]; positions int32 [batch].
 * q_out        bf16 [batch, 16, D] (written): the decode's q.
 * k_pool, v_pool  the decode's pools (one row per sequence written).
 *              attn_kv_append_global only: k_pool may be NULL for a
 *              values-only cache (attn_decode_global_shared), and then
 *              only the value row is written.
 * status       optional device int32: a position outside [0, max_blocks*16)
 *              raises ATTN_DEV_BAD_SEQ_LEN, a page id outside [0, num_pages)
 *              ATTN_DEV_BAD_PAGE; that token's cache row is then not written
 *              (its q is).
 *
 * Computed in fp32 (RoPE angles without the fp32 rounding of pos * freq,
 * see kv_append.cuh), rounded once to bf16 (nearest even).  Asynchronous on
 * `stream`, launched like the decode kernels (programmatic dependent of the
 * previous kernel).  Alignment: qkv, w_q, w_k, q_out and the pools 16 bytes.
 * Returns ATTN_OK or ATTN_ERR_* with nothing launched.
 */
int32_t attn_kv_append_sliding(const void* qkv, const void* w_q, const void* w_k, const int32_t* block_table,
                               const int32_t* positions, void* q_out, void* k_pool, void* v_pool, int32_t batch,
                               int32_t max_blocks, int64_t num_pages, int32_t* status, void* stream);
int32_t attn_kv_append_global(const void* qkv, const void* w_q, const void* w_k, const int32_t* block_table,
                              const int32_t* positions, void* q_out, void* k_pool, void* v_pool, int32_t batch,
                              int32_t max_blocks, int64_t num_pages, int32_t* status, void* stream);

/*
 * attn_prefill_sliding / attn_prefill_global -- multi-query attention over the
 * paged cache, for a chunk of new tokens per sequence whose keys and values
 * are already in the cache (Attention.lean `causalGQA` / `slidingGQA` with
 * S > 1 queries, Op Specs page, "Attention"; shapes and scale 1 as in the
 * decode calls above):
 *
 *   sequence b caches L = seq_lens[b] tokens; its last n = cu_q[b+1] - cu_q[b]
 *   tokens are the queries, packed as rows cu_q[b] .. cu_q[b+1]-1 of q, and
 *   query i sits at position p = L - n + i.  It sees key l iff l <= p (and
 *   p - window < l when window > 0):
 *       o[t, h] = sum over visible l of softmax_l(<q[t, h], k[l, h/G]>) * v[l, h/G]
 *
 * q            bf16 [total_q, 16, D], D = 256 (sliding) or 512 (global)
 * k_pool, v_pool, block_table, num_pages, max_blocks: as for the decode calls
 * seq_lens     int32 [batch], n <= L <= max_blocks*16 for every sequence
 * cu_q         int32 [batch + 1], cu_q[0] = 0, non-decreasing, cu_q[batch] = total_q
 * o            [total_q, 16, D], bf16 (RNE) or fp32 per out_dtype
 * max_q        host-side bound on the per-sequence query count n (sizes the grid)
 * window       sliding: > 0 (1024 for Gemma-4-12B); global: <= 0 none, > 0 a window
 * status       optional device int32: a sequence with n > L, L beyond the
 *              table, n > max_q or rows past total_q raises
 *              ATTN_DEV_BAD_SEQ_LEN and that sequence's rows (or those past
 *              max_q) are not written; a visible page id outside
 *              [0, num_pages) raises ATTN_DEV_BAD_PAGE and is read as zeros.
 *
 * All pointers are device pointers owned by the caller (q and o may be null
 * when total_q is 0); nothing is allocated and nothing synchronises.
 * Alignment: q, o and the pools 16 bytes, the int32
 * arrays 4.  Asynchronous on `stream`, launched as a programmatic dependent of
 * the previous kernel.  Computed with bf16 tensor-core products and fp32
 * accumulation; P is rounded to bf16 for the P*V product.  Returns ATTN_OK
 * (also when max_q is 0: nothing is launched) or ATTN_ERR_* with nothing
 * launched.
 */
int32_t attn_prefill_sliding(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* cu_q, void* o, int32_t batch, int32_t total_q,
                             int32_t max_q, int32_t max_blocks, int64_t num_pages, int32_t window, int32_t out_dtype,
                             int32_t* status, void* stream);
int32_t attn_prefill_global(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
                            const int32_t* seq_lens, const int32_t* cu_q, void* o, int32_t batch, int32_t total_q,
                            int32_t max_q, int32_t max_blocks, int64_t num_pages, int32_t window, int32_t out_dtype,
                            int32_t* status, void* stream);

/*
 * attn_selftest_wait_timeout -- exercises the device-side failure path of the
 * copy pipeline.  It launches one warp that waits, with the same bounded
 * wait and time limit as the decode kernels (1 s), on a shared-memory
 * barrier that nothing arrives at.  The wait gives up, ATTN_DEV_WAIT_TIMEOUT
 * is OR-ed into *status (a device int32, required) and the kernel returns;
 * the CUDA context stays usable.  Asynchronous on `stream`.  For tests of
 * failure detection; the pages have no counterpart for it.
 */
int32_t attn_selftest_wait_timeout(int32_t* status, void* stream);

/*
 * attn_selftest_delayed_copy -- a stand-in for a kernel that rewrites the
 * decode's inputs while the decode is already being scheduled.  It launches
 * one block as a programmatic dependent of the previous kernel in `stream`:
 * the block waits for that kernel, lets its own dependents launch at once,
 * sleeps `delay_ns` (0 to 1,000,000), then copies `bytes` (a multiple of 4,
 * at most 16 MiB) from `src` to `dst` (device pointers, 4-byte aligned, not
 * overlapping).  A decode launched next builds its schedule hints and starts
 * its first copies from the old contents of dst, and must still read the new
 * ones after its wait.  Returns ATTN_OK or ATTN_ERR_INVALID_ARG /
 * ATTN_ERR_CUDA with nothing launched.  For tests of the launch order; the
 * pages have no counterpart for it.
 */
int32_t attn_selftest_delayed_copy(void* dst, const void* src, int64_t bytes, int32_t delay_ns, void* stream);

/* Message of the last error on this host thread ("" if none). */
const char* attn_last_error(void);

/* ATTN_DECODE_ABI_VERSION of the loaded library. */
int32_t attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_DECODE_H */
