// attn_decode.cu -- host side of the C ABI declared in include/attn_decode.h:
// argument validation, the split plan, TMA tensor maps and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <vector>

#include "attn_decode.h"
#include "combine.cuh"
#include "global.cuh"
#include "kv_append.cuh"
#include "prefill_tc.cuh"
#include "prefill_pair.cuh"
#include "sliding.cuh"

namespace {

thread_local char g_err[512] = "";
// Set while attn_step_add_* validates a call: run_decode and run_append
// return after their host checks, before anything is encoded or launched.
thread_local bool g_validate_only = false;
// Kernels the last call validated by run_decode or run_append launches.
thread_local int32_t g_last_launches = 0;
// One kernel launch with all its arguments bound (tensor maps included),
// ready to be enqueued on any stream of its device.
using RecordedLaunch = std::function<cudaError_t(cudaStream_t)>;
// Set while attn_step_finalize records a step: launch_pdl appends each launch
// to this list instead of enqueuing it.
thread_local std::vector<RecordedLaunch>* g_record = nullptr;

int32_t fail(int32_t code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// Launch plan: how many thread blocks share the pages of one KV head.
//
// The decode kernels cut the concatenated visible pages of all sequences
// into grid_x equal spans (the balanced schedule in common.cuh), so grid_x
// only has to fill the GPU once: one wave of resident blocks, 3 per SM for
// the sliding kernel (~75 KB of shared memory each, 8 KV-head columns) and
// 2 per SM for the global kernel (~107 KB each).  max_seq_len bounds the
// total pages, so small problems launch fewer blocks; it never changes
// which positions are read.  The workspace holds one partial row per
// (block, sequence) pair that a span boundary can cut: grid_x + batch slots.
// ---------------------------------------------------------------------------
struct Plan {
  int grid_x;
  int min_pages;
  bool merge_in_grid;  // cut sequences merged by their last block; no combine kernel
  size_t part_o_bytes;
  size_t workspace_bytes;
};

// Cut sequences are merged inside the sliding decode grid when at most this
// many blocks can share one sequence: the last of them reads the others'
// partial rows (2 KB each per KV head) in groups of four.
constexpr int kMergeInGridMax = 24;
// ... and when the blocks that typically share one sequence are few: with
// many, the last block's reads of their partials take longer than the
// combine kernel, whose blocks read every partial of a row at once.
constexpr int kMergeInGridTypical = 8;

// Workspace layout: [counters, ATTN_WORKSPACE_ZERO_BYTES][partial rows][(max, sum) pairs].
static_assert(ATTN_WORKSPACE_ZERO_BYTES >= ATTN_MAX_BATCH * ATTN_SLIDING_HKV * 4, "a counter per (sequence, KV head)");

int32_t make_plan(int32_t kind, int32_t batch, int32_t max_seq_len, int32_t window,
                  int32_t forced_blocks, int32_t num_sms, Plan* out) {
  if (kind != ATTN_KIND_SLIDING && kind != ATTN_KIND_GLOBAL)
    return fail(ATTN_ERR_INVALID_ARG, "unknown kind %d", kind);
  if (batch < 1) return fail(ATTN_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", batch);
  if (max_seq_len < 0) return fail(ATTN_ERR_INVALID_ARG, "max_seq_len must be >= 0");
  if (forced_blocks < 0) return fail(ATTN_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (num_sms < 1) return fail(ATTN_ERR_INVALID_ARG, "num_sms must be >= 1");
  const bool sliding = kind == ATTN_KIND_SLIDING;
  const int D = sliding ? ATTN_SLIDING_D : ATTN_GLOBAL_D;
  const int Hq = sliding ? ATTN_SLIDING_HQ : ATTN_GLOBAL_HQ;
  const int columns = sliding ? ATTN_SLIDING_HKV : 1;
  const int blocks_per_sm = sliding ? pda::sliding::kBlocksPerSm : pda::global::kBlocksPerSm;
  const int min_pages = sliding ? pda::sliding::kMinPages : pda::global::kMinPages;

  // visible pages of one sequence, at most
  int64_t max_pages = (max_seq_len + ATTN_PAGE_SIZE - 1) / ATTN_PAGE_SIZE;
  if (window > 0) {
    const int64_t wpages = (window + ATTN_PAGE_SIZE - 1) / ATTN_PAGE_SIZE + 1;
    if (wpages < max_pages) max_pages = wpages;
  }
  const int64_t total_max = max_pages * batch;
  int64_t gx;
  if (forced_blocks > 0) {
    gx = forced_blocks;
  } else {
    gx = static_cast<int64_t>(num_sms) * blocks_per_sm / columns;
    const int64_t useful = (total_max + min_pages - 1) / min_pages;
    if (gx > useful) gx = useful;
  }
  if (gx > pda::kMaxSplits) gx = pda::kMaxSplits;
  if (gx < 1) gx = 1;
  out->grid_x = static_cast<int>(gx);
  out->min_pages = min_pages;
  // Blocks that can share one sequence of at most max_pages visible pages:
  // every span holds at least min_pages weighted pages, so a run of n pages
  // meets at most (n - 1) / min_pages + 2 spans.
  const int64_t sharing = max_pages > 0 ? (max_pages - 1) / min_pages + 2 : 1;
  // Typical sharing: spans sized as if every sequence had max_pages visible
  // pages (shorter sequences give shorter spans; the bound above still holds).
  const int64_t per_typ = std::max<int64_t>(min_pages, (total_max + gx - 1) / gx);
  const int64_t sharing_typ = max_pages > 0 ? (max_pages - 1) / per_typ + 2 : 1;
  out->merge_in_grid = sliding && sharing <= kMergeInGridMax && sharing_typ <= kMergeInGridTypical;
  const size_t rows = (static_cast<size_t>(gx) + batch) * Hq;
  out->part_o_bytes = align256(rows * D * sizeof(float));
  out->workspace_bytes = ATTN_WORKSPACE_ZERO_BYTES + out->part_o_bytes + align256(rows * sizeof(float2));
  return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Device facts and TMA descriptors
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

int32_t current_device(int* dev, int* num_sms) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device index %d unsupported", *dev);
  static int sms[kMaxDevices] = {0};
  if (sms[*dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
    if (e != cudaSuccess || n < 1)
      return fail(ATTN_ERR_CUDA, "cudaDeviceGetAttribute(SM count): %s", cudaGetErrorString(e));
    sms[*dev] = n;
  }
  *num_sms = sms[*dev];
  return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The pool [num_pages, 16, Hkv, D] viewed as a 2-D tensor of num_pages*16
// token rows by Hkv*D bf16 elements; boxes of 16 rows x box_cols.
int32_t encode_pool_map(CUtensorMap* map, const void* pool, int64_t num_pages, int row_elems,
                        int box_cols, CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_elems),
                              static_cast<cuuint64_t>(num_pages) * ATTN_PAGE_SIZE};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), ATTN_PAGE_SIZE};
  const cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
                   elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return ATTN_OK;
}

// The global pool [num_pages*16 rows][512] seen as a 3-D tensor (x: 64 dims
// of a chunk, y: row, z: chunk of 64 dims, stride 128 bytes), so that one
// box {64, 16, 8} copies a whole page as 8 swizzled tiles of [16 rows][64],
// the layout the consumers read with ldmatrix.
int32_t encode_global_page_map(CUtensorMap* map, const void* pool, int64_t num_pages) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  constexpr int kChunk = pda::global::kChunk;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kChunk), static_cast<cuuint64_t>(num_pages) * ATTN_PAGE_SIZE,
                              static_cast<cuuint64_t>(ATTN_GLOBAL_D / kChunk)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ATTN_GLOBAL_D) * 2, static_cast<cuuint64_t>(kChunk) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kChunk), ATTN_PAGE_SIZE,
                             static_cast<cuuint32_t>(ATTN_GLOBAL_D / kChunk)};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box,
                   elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (page map) failed (%d)", static_cast<int>(r));
  return ATTN_OK;
}

// A pool [num_pages*16 rows][Hkv*D] seen as a 3-D tensor (x: 64 dims of a
// chunk, y: row, z: chunk of 64 dims, stride 128 bytes); a box {64, 16,
// chunks} copies `chunks` consecutive chunks of a page's 16 rows (one KV
// head's D dims at z = c * D / 64) as swizzled [16 rows][64] tiles.
int32_t encode_chunk_map(CUtensorMap* map, const void* pool, int64_t num_pages, int row_elems, int chunks) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(num_pages) * ATTN_PAGE_SIZE,
                              static_cast<cuuint64_t>(row_elems / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_elems) * 2, 128};
  const cuuint32_t box[3] = {64, ATTN_PAGE_SIZE, static_cast<cuuint32_t>(chunks)};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box,
                   elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (chunk map) failed (%d)", static_cast<int>(r));
  return ATTN_OK;
}

// Q or O [total_q, Hq, D] (bf16) as {64 dims, D/64 chunks, total_q queries, Hq heads}:
// a box {64, 1, kQ, G} copies one 64-dim chunk of kQ consecutive queries for
// the G heads of a KV head as [head][query][64 dims], 128-byte swizzled (the
// single-CTA prefill's row order); queries past total_q read as zeros.
int32_t encode_q_map(CUtensorMap* map, const void* q, int32_t total_q, int hq, int d, int g, int nq) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(d / 64), static_cast<cuuint64_t>(total_q),
                              static_cast<cuuint64_t>(hq)};
  const cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(hq) * d * 2, static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(nq), static_cast<cuuint32_t>(g)};
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (q map) failed (%d)", static_cast<int>(r));
  return ATTN_OK;
}

template <typename Kernel>
int32_t ensure_smem(Kernel kernel, size_t bytes, int dev, bool* done) {
  if (done[dev]) return ATTN_OK;
  cudaError_t e = cudaSuccess;
  if (bytes > 0)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  // Every kernel of the library asks for the largest shared-memory carveout,
  // so consecutive launches never wait for an SM to change its L1/shared split.
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  done[dev] = true;
  return ATTN_OK;
}

// Every kernel is launched as a programmatic dependent of the kernel before
// it in the stream.  A decode grid may then be scheduled while that kernel
// finishes: it sets up its shared memory, then waits in griddepcontrol.wait
// before it reads any input or writes any output, and lets its own dependent
// (the combine) launch only after that wait.  The combine runs its schedule
// arithmetic while the decode grid streams, waits for the decode grid's
// results the same way, and lets the next kernel launch once it is merging.
// Following anything but a kernel, the attribute has no effect.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl_now(Kernel kernel, dim3 grid, int threads, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, int threads, size_t smem, cudaStream_t s, Args... args) {
  if (g_record) {
    try {
      g_record->emplace_back(
          [=](cudaStream_t st) { return launch_pdl_now(kernel, grid, threads, smem, st, args...); });
    } catch (...) {  // no exception may leave the C ABI
      return cudaErrorMemoryAllocation;
    }
    return cudaSuccess;
  }
  return launch_pdl_now(kernel, grid, threads, smem, s, args...);
}

// 2*pi as three floats for the additive range reduction (Cody and Waite):
// the first two keep 8 significant bits, so n * part is exact for n < 2^16
// turns; the third is the float nearest to what remains.
pda::TwoPi split_two_pi() {
  const double two_pi = 6.283185307179586476925286766559;
  pda::TwoPi out;
  double rest = two_pi;
  for (int k = 0; k < 2; ++k) {
    int e;
    const double m = std::frexp(rest, &e);  // rest = m * 2^e, 0.5 <= m < 1
    const double part = std::ldexp(std::trunc(std::ldexp(m, 8)), e - 8);
    out.part[k] = static_cast<float>(part);
    rest -= part;
  }
  out.part[2] = static_cast<float>(rest);
  out.inv = static_cast<float>(1.0 / two_pi);
  return out;
}

pda::FloatPair split_float_pair(double f) {
  pda::FloatPair fp;
  fp.hi = static_cast<float>(f);
  fp.lo = static_cast<float>(f - static_cast<double>(fp.hi));
  return fp;
}

// ---------------------------------------------------------------------------
// Common validation + launch
// ---------------------------------------------------------------------------
int32_t run_decode(int32_t kind, const void* q, const void* k_pool, const void* v_pool,
                   const int32_t* block_table, const int32_t* seq_lens, void* o, int32_t batch,
                   int32_t max_blocks, int64_t num_pages, int32_t max_seq_len, int32_t window,
                   int32_t out_dtype, int32_t num_splits, void* workspace, size_t workspace_bytes,
                   int32_t* status, void* stream, const void* w_k = nullptr) {
  g_err[0] = '\0';
  const bool sliding = kind == ATTN_KIND_SLIDING;
  const bool shared = w_k != nullptr;  // values-only global cache (k_pool is v_pool)
  const char* name = sliding ? "attn_decode_sliding" : shared ? "attn_decode_global_shared" : "attn_decode_global";
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !o)
    return fail(ATTN_ERR_INVALID_ARG, "%s: null array pointer", name);
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(block_table) ||
      !aligned16(seq_lens) || !aligned16(o) || (shared && !aligned16(w_k)))
    return fail(ATTN_ERR_INVALID_ARG, "%s: every array must be 16-byte aligned", name);
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "%s: status must be 4-byte aligned", name);
  if (batch < 1) return fail(ATTN_ERR_INVALID_ARG, "%s: batch must be >= 1 (got %d)", name, batch);
  if (batch > ATTN_MAX_BATCH)
    return fail(ATTN_ERR_UNSUPPORTED, "%s: batch %d outside the model's domain [1, %d]", name, batch,
                ATTN_MAX_BATCH);
  if (max_blocks < 1) return fail(ATTN_ERR_INVALID_ARG, "%s: max_blocks must be >= 1", name);
  if (num_pages < 1) return fail(ATTN_ERR_INVALID_ARG, "%s: num_pages must be >= 1", name);
  if (num_pages > (int64_t{1} << 31) / ATTN_PAGE_SIZE - 1)
    return fail(ATTN_ERR_UNSUPPORTED, "%s: num_pages %lld too large (row index must fit in int32)", name,
                static_cast<long long>(num_pages));
  if (max_seq_len < 0 || static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks) * ATTN_PAGE_SIZE)
    return fail(ATTN_ERR_INVALID_ARG, "%s: max_seq_len %d not in [0, max_blocks*16 = %lld]", name,
                max_seq_len, static_cast<long long>(max_blocks) * ATTN_PAGE_SIZE);
  if (max_seq_len > ATTN_MAX_SEQ_LEN)
    return fail(ATTN_ERR_UNSUPPORTED, "%s: max_seq_len %d beyond the model's domain (%d)", name,
                max_seq_len, ATTN_MAX_SEQ_LEN);
  if (sliding && window <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "%s: window must be > 0 (the node's is 1024)", name);
  if (out_dtype != ATTN_OUT_BF16 && out_dtype != ATTN_OUT_F32)
    return fail(ATTN_ERR_INVALID_ARG, "%s: out_dtype must be ATTN_OUT_BF16 or ATTN_OUT_F32", name);
  if (num_splits < 0) return fail(ATTN_ERR_INVALID_ARG, "%s: num_splits must be >= 0", name);

  int dev = 0, num_sms = 0;
  int32_t st = current_device(&dev, &num_sms);
  if (st != ATTN_OK) return st;
  Plan plan;
  st = make_plan(kind, batch, max_seq_len, window, num_splits, num_sms, &plan);
  if (st != ATTN_OK) return st;
  if (!workspace || workspace_bytes < plan.workspace_bytes)
    return fail(ATTN_ERR_WORKSPACE, "%s: workspace of %zu bytes required (got %zu)", name,
                plan.workspace_bytes, workspace ? workspace_bytes : size_t{0});
  if (!aligned16(workspace)) return fail(ATTN_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", name);

  pda::DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.o = o;
  p.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
  p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
  p.counters = static_cast<int32_t*>(workspace);
  p.part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ATTN_WORKSPACE_ZERO_BYTES);
  p.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + ATTN_WORKSPACE_ZERO_BYTES +
                                        plan.part_o_bytes);
  p.merge_in_grid = plan.merge_in_grid;
  p.status = status;
  p.num_pages = num_pages;
  p.batch = batch;
  p.max_blocks = max_blocks;
  p.window = window;
  p.grid_x = plan.grid_x;
  p.min_pages = plan.min_pages;
  p.part_rows = (static_cast<int64_t>(plan.grid_x) + batch) *
                (sliding ? ATTN_SLIDING_HQ : ATTN_GLOBAL_HQ);
  p.out_f32 = out_dtype == ATTN_OUT_F32;

  g_last_launches = plan.merge_in_grid ? 1 : 2;
  if (g_validate_only) return ATTN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tm_k, tm_v;
  cudaError_t e;
  if (sliding) {
    const int row = ATTN_SLIDING_HKV * ATTN_SLIDING_D;
    if ((st = encode_pool_map(&tm_k, k_pool, num_pages, row, ATTN_SLIDING_D, CU_TENSOR_MAP_SWIZZLE_NONE))) return st;
    if ((st = encode_pool_map(&tm_v, v_pool, num_pages, row, ATTN_SLIDING_D, CU_TENSOR_MAP_SWIZZLE_NONE))) return st;
    static bool smem_set[kMaxDevices] = {false};
    if ((st = ensure_smem(pda::sliding::decode_kernel, pda::sliding::kSmemBytes, dev, smem_set))) return st;
    static bool comb_set[kMaxDevices] = {false};
    if ((st = ensure_smem(pda::combine_kernel<ATTN_SLIDING_D>, 0, dev, comb_set))) return st;
    e = launch_pdl(pda::sliding::decode_kernel, dim3(plan.grid_x, ATTN_SLIDING_HKV), pda::sliding::kThreads,
                   pda::sliding::kSmemBytes, s, tm_k, tm_v, p);
    if (e == cudaSuccess && !plan.merge_in_grid)
      e = launch_pdl(pda::combine_kernel<ATTN_SLIDING_D>,
                     dim3(ATTN_SLIDING_HQ * (ATTN_SLIDING_D / pda::kCombineCols), batch), pda::kCombineWarps * 32, 0,
                     s, p);
  } else if (shared) {
    if ((st = encode_global_page_map(&tm_v, v_pool, num_pages))) return st;
    pda::global::KeyRebuild kr;
    kr.w_k = static_cast<const __nv_bfloat16*>(w_k);
    kr.two_pi = split_two_pi();
    for (int j = 0; j < pda::global::kRopePairs; ++j)
      kr.freq[j] = split_float_pair(std::pow(ATTN_GLOBAL_ROPE_THETA, -2.0 * j / ATTN_GLOBAL_D));
    static bool smem_set[kMaxDevices] = {false};
    if ((st = ensure_smem(pda::global::decode_kernel_shared, pda::global::kSharedSmemBytes, dev, smem_set)))
      return st;
    static bool comb_set[kMaxDevices] = {false};
    if ((st = ensure_smem(pda::combine_kernel<ATTN_GLOBAL_D>, 0, dev, comb_set))) return st;
    e = launch_pdl(pda::global::decode_kernel_shared, dim3(plan.grid_x), pda::global::kThreads,
                   pda::global::kSharedSmemBytes, s, tm_v, p, kr);
    if (e == cudaSuccess)
      e = launch_pdl(pda::combine_kernel<ATTN_GLOBAL_D>,
                     dim3(ATTN_GLOBAL_HQ * (ATTN_GLOBAL_D / pda::kCombineCols), batch), pda::kCombineWarps * 32, 0,
                     s, p);
  } else {
    if ((st = encode_global_page_map(&tm_k, k_pool, num_pages))) return st;
    if ((st = encode_global_page_map(&tm_v, v_pool, num_pages))) return st;
    static bool smem_set[kMaxDevices] = {false};
    if ((st = ensure_smem(pda::global::decode_kernel, pda::global::kSmemBytes, dev, smem_set))) return st;
    static bool comb_set[kMaxDevices] = {false};
    if ((st = ensure_smem(pda::combine_kernel<ATTN_GLOBAL_D>, 0, dev, comb_set))) return st;
    e = launch_pdl(pda::global::decode_kernel, dim3(plan.grid_x), pda::global::kThreads, pda::global::kSmemBytes, s,
                   tm_k, tm_v, p);
    if (e == cudaSuccess)
      e = launch_pdl(pda::combine_kernel<ATTN_GLOBAL_D>,
                     dim3(ATTN_GLOBAL_HQ * (ATTN_GLOBAL_D / pda::kCombineCols), batch), pda::kCombineWarps * 32, 0,
                     s, p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "%s: launch failed: %s", name, cudaGetErrorString(e));
  return ATTN_OK;
}

}  // namespace

extern "C" {

int32_t attn_decode_sliding(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_table, const int32_t* seq_lens, void* o,
                            int32_t batch, int32_t max_blocks, int64_t num_pages,
                            int32_t max_seq_len, int32_t window, int32_t out_dtype,
                            int32_t num_splits, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream) {
  return run_decode(ATTN_KIND_SLIDING, q, k_pool, v_pool, block_table, seq_lens, o, batch, max_blocks,
                    num_pages, max_seq_len, window, out_dtype, num_splits, workspace, workspace_bytes,
                    status, stream);
}

int32_t attn_decode_global(const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_table, const int32_t* seq_lens, void* o,
                           int32_t batch, int32_t max_blocks, int64_t num_pages,
                           int32_t max_seq_len, int32_t window, int32_t out_dtype,
                           int32_t num_splits, void* workspace, size_t workspace_bytes,
                           int32_t* status, void* stream) {
  return run_decode(ATTN_KIND_GLOBAL, q, k_pool, v_pool, block_table, seq_lens, o, batch, max_blocks,
                    num_pages, max_seq_len, window, out_dtype, num_splits, workspace, workspace_bytes,
                    status, stream);
}

int32_t attn_decode_global_shared(const void* q, const void* kv_pool, const void* w_k,
                                  const int32_t* block_table, const int32_t* seq_lens, void* o, int32_t batch,
                                  int32_t max_blocks, int64_t num_pages, int32_t max_seq_len, int32_t window,
                                  int32_t out_dtype, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                  int32_t* status, void* stream) {
  if (!w_k) {
    g_err[0] = '\0';
    return fail(ATTN_ERR_INVALID_ARG, "attn_decode_global_shared: null w_k");
  }
  return run_decode(ATTN_KIND_GLOBAL, q, kv_pool, kv_pool, block_table, seq_lens, o, batch, max_blocks, num_pages,
                    max_seq_len, window, out_dtype, num_splits, workspace, workspace_bytes, status, stream, w_k);
}

int32_t attn_decode_plan(int32_t kind, int32_t batch, int32_t max_seq_len, int32_t window,
                         int32_t num_splits, int32_t num_sms, int32_t* out_num_splits,
                         size_t* out_workspace_bytes) {
  g_err[0] = '\0';
  Plan plan;
  const int32_t st = make_plan(kind, batch, max_seq_len, window, num_splits, num_sms, &plan);
  if (st != ATTN_OK) return st;
  if (out_num_splits) *out_num_splits = plan.grid_x;
  if (out_workspace_bytes) *out_workspace_bytes = plan.workspace_bytes;
  return ATTN_OK;
}

int32_t attn_decode_launches(int32_t kind, int32_t batch, int32_t max_seq_len, int32_t window,
                             int32_t num_splits, int32_t num_sms) {
  g_err[0] = '\0';
  Plan plan;
  if (make_plan(kind, batch, max_seq_len, window, num_splits, num_sms, &plan) != ATTN_OK) return -1;
  return plan.merge_in_grid ? 1 : 2;
}

size_t attn_decode_workspace_size(int32_t kind, int32_t batch, int32_t max_seq_len, int32_t window,
                                  int32_t num_splits) {
  g_err[0] = '\0';
  int dev = 0, num_sms = 0;
  if (current_device(&dev, &num_sms) != ATTN_OK) return 0;
  Plan plan;
  if (make_plan(kind, batch, max_seq_len, window, num_splits, num_sms, &plan) != ATTN_OK) return 0;
  return plan.workspace_bytes;
}

const char* attn_last_error(void) { return g_err; }

int32_t attn_abi_version(void) { return ATTN_DECODE_ABI_VERSION; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Norms, RoPE and cache append of one token per sequence
// ---------------------------------------------------------------------------
namespace {

int32_t run_append(int32_t kind, const void* qkv, const void* w_q, const void* w_k, const int32_t* block_table,
                   const int32_t* positions, void* q_out, void* k_pool, void* v_pool, int32_t batch,
                   int32_t max_blocks, int64_t num_pages, int32_t* status, void* stream) {
  g_err[0] = '\0';
  const bool sliding = kind == ATTN_KIND_SLIDING;
  const char* name = sliding ? "attn_kv_append_sliding" : "attn_kv_append_global";
  if (!qkv || !w_q || !w_k || !block_table || !positions || !q_out || (sliding && !k_pool) || !v_pool)
    return fail(ATTN_ERR_INVALID_ARG, "%s: null pointer argument", name);
  auto aligned = [](const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; };
  if (!aligned(qkv, 16) || !aligned(w_q, 16) || !aligned(w_k, 16) || !aligned(q_out, 16) || !aligned(k_pool, 16) ||
      !aligned(v_pool, 16) || !aligned(block_table, 4) || !aligned(positions, 4))
    return fail(ATTN_ERR_INVALID_ARG, "%s: misaligned pointer (qkv, w_q, w_k, q_out and the pools 16 bytes)", name);
  if (status && !aligned(status, 4)) return fail(ATTN_ERR_INVALID_ARG, "%s: status must be 4-byte aligned", name);
  if (batch < 1 || batch > ATTN_MAX_BATCH)
    return fail(ATTN_ERR_UNSUPPORTED, "%s: batch %d outside [1, %d]", name, batch, ATTN_MAX_BATCH);
  if (max_blocks < 1) return fail(ATTN_ERR_INVALID_ARG, "%s: max_blocks must be >= 1", name);
  if (num_pages < 1 || num_pages > (int64_t{1} << 31) / ATTN_PAGE_SIZE - 1)
    return fail(ATTN_ERR_INVALID_ARG, "%s: num_pages %lld out of range", name, static_cast<long long>(num_pages));

  const int D = sliding ? ATTN_SLIDING_D : ATTN_GLOBAL_D;
  const double theta = sliding ? ATTN_SLIDING_ROPE_THETA : ATTN_GLOBAL_ROPE_THETA;
  pda::append::AppendParams p{};
  p.qkv = static_cast<const __nv_bfloat16*>(qkv);
  p.w_q = static_cast<const __nv_bfloat16*>(w_q);
  p.w_k = static_cast<const __nv_bfloat16*>(w_k);
  p.block_table = block_table;
  p.positions = positions;
  p.q_out = static_cast<__nv_bfloat16*>(q_out);
  p.k_pool = static_cast<__nv_bfloat16*>(k_pool);
  p.v_pool = static_cast<__nv_bfloat16*>(v_pool);
  p.status = status;
  p.num_pages = num_pages;
  p.batch = batch;
  p.max_blocks = max_blocks;
  p.eps = 1e-6f;
  p.two_pi = split_two_pi();
  // frequencies theta^(-2i/D), i = V*lane + j, as products of these factors
  const int V = D / 64;
  auto split = split_float_pair;
  for (int k = 0; k < pda::append::kLaneBits; ++k) p.lane_factor[k] = split(std::pow(theta, -2.0 * V * (1 << k) / D));
  for (int j = 0; j < V; ++j) p.dim_factor[j] = split(std::pow(theta, -2.0 * j / D));
  static_assert(ATTN_SLIDING_D / 64 <= pda::append::kMaxV && ATTN_GLOBAL_D / 64 <= pda::append::kMaxV, "dims per lane");
  const int rows = sliding ? ATTN_SLIDING_HQ + 2 * ATTN_SLIDING_HKV : ATTN_GLOBAL_HQ + 1;
  const dim3 grid((batch * rows + 3) / 4);
  g_last_launches = 1;
  if (g_validate_only) return ATTN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (sliding)
    e = launch_pdl(pda::append::append_kernel<ATTN_SLIDING_D, ATTN_SLIDING_HQ, ATTN_SLIDING_HKV,
                                              ATTN_SLIDING_ROPE_PAIRS, false>,
                   grid, 128, 0, s, p);
  else
    e = launch_pdl(pda::append::append_kernel<ATTN_GLOBAL_D, ATTN_GLOBAL_HQ, ATTN_GLOBAL_HKV,
                                              ATTN_GLOBAL_ROPE_PAIRS, true>,
                   grid, 128, 0, s, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "%s: launch failed: %s", name, cudaGetErrorString(e));
  return ATTN_OK;
}

}  // namespace

extern "C" int32_t attn_kv_append_sliding(const void* qkv, const void* w_q, const void* w_k,
                                          const int32_t* block_table, const int32_t* positions, void* q_out,
                                          void* k_pool, void* v_pool, int32_t batch, int32_t max_blocks,
                                          int64_t num_pages, int32_t* status, void* stream) {
  return run_append(ATTN_KIND_SLIDING, qkv, w_q, w_k, block_table, positions, q_out, k_pool, v_pool, batch,
                    max_blocks, num_pages, status, stream);
}

extern "C" int32_t attn_kv_append_global(const void* qkv, const void* w_q, const void* w_k,
                                         const int32_t* block_table, const int32_t* positions, void* q_out,
                                         void* k_pool, void* v_pool, int32_t batch, int32_t max_blocks,
                                         int64_t num_pages, int32_t* status, void* stream) {
  return run_append(ATTN_KIND_GLOBAL, qkv, w_q, w_k, block_table, positions, q_out, k_pool, v_pool, batch,
                    max_blocks, num_pages, status, stream);
}

// One warp waits, with the decode kernels' bounded wait and time limit, on a
// barrier that nothing arrives at; the wait gives up, the timeout bit is
// raised and the kernel returns.  No copy is ever issued.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int32_t* status) {
  __shared__ alignas(8) uint64_t bar;
  if (threadIdx.x == 0) {
    pda::mbar_init(&bar, 1);
    pda::fence_mbar_init();
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, pda::mbar_wait(&bar, 0));
  if (!ok && threadIdx.x == 0) pda::report(status, ATTN_DEV_WAIT_TIMEOUT);
}

extern "C" int32_t attn_selftest_wait_timeout(int32_t* status, void* stream) {
  g_err[0] = '\0';
  if (!status || (reinterpret_cast<uintptr_t>(status) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "attn_selftest_wait_timeout: status must be a 4-byte aligned device int32");
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "attn_selftest_wait_timeout: launch failed: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

namespace {

// Single-CTA prefill grid: one CTA per SM looping over the work items.
constexpr bool kPersistentPrefill = true;

// Multi-query attention over the paged cache (attn_prefill_*): one CTA per
// query tile (prefill_tc.cuh) or CTA pairs sharing each product
// (prefill_pair.cuh, kPair).
template <typename C, bool kPair, typename Kernel>
int32_t run_prefill(Kernel kernel, int32_t kind, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
                    const int32_t* seq_lens, const int32_t* cu_q, void* o, int32_t batch, int32_t total_q,
                    int32_t max_q, int32_t max_blocks, int64_t num_pages, int32_t window, int32_t out_dtype,
                    int32_t* status, void* stream) {
  g_err[0] = '\0';
  const char* name = kind == ATTN_KIND_SLIDING ? "attn_prefill_sliding" : "attn_prefill_global";
  if (!k_pool || !v_pool || !block_table || !seq_lens || !cu_q || (total_q > 0 && (!q || !o)))
    return fail(ATTN_ERR_INVALID_ARG, "%s: null pointer argument", name);
  auto aligned = [](const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; };
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(cu_q, 4) || (status && !aligned(status, 4)))
    return fail(ATTN_ERR_INVALID_ARG, "%s: misaligned pointer (q, o and the pools 16 bytes, tables 4)", name);
  if (batch < 1 || batch > ATTN_MAX_BATCH)
    return fail(ATTN_ERR_UNSUPPORTED, "%s: batch %d outside [1, %d]", name, batch, ATTN_MAX_BATCH);
  if (total_q < 0 || max_q < 0 || max_q > total_q || max_q > ATTN_MAX_SEQ_LEN)
    return fail(ATTN_ERR_INVALID_ARG, "%s: need 0 <= max_q <= total_q and max_q <= %d", name, ATTN_MAX_SEQ_LEN);
  if (static_cast<int64_t>(total_q) * C::kHq * C::kD > (int64_t{1} << 40))
    return fail(ATTN_ERR_INVALID_ARG, "%s: total_q %d too large", name, total_q);
  if (max_blocks < 1) return fail(ATTN_ERR_INVALID_ARG, "%s: max_blocks must be >= 1", name);
  if (num_pages < 1 || num_pages > (int64_t{1} << 31) / ATTN_PAGE_SIZE - 1)
    return fail(ATTN_ERR_INVALID_ARG, "%s: num_pages %lld out of range", name, static_cast<long long>(num_pages));
  if (kind == ATTN_KIND_SLIDING && window <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "%s: window must be > 0", name);
  if (out_dtype != ATTN_OUT_BF16 && out_dtype != ATTN_OUT_F32)
    return fail(ATTN_ERR_INVALID_ARG, "%s: out_dtype must be ATTN_OUT_BF16 or ATTN_OUT_F32", name);
  if (max_q == 0) return ATTN_OK;  // no queries

  int dev = 0, num_sms = 0;
  int32_t st = current_device(&dev, &num_sms);
  if (st != ATTN_OK) return st;
  static bool smem_set[2][kMaxDevices] = {{false}};
  if ((st = ensure_smem(kernel, C::kSmemBytes, dev, smem_set[kind]))) return st;

  // K: a CTA pair with one page per CTA and step copies all D dims of it in
  // one box; otherwise a box is one 64-dim chunk of a page.  V: a page's
  // output dims of the CTA (half of kDS in a pair).
  int k_box_chunks = 1;
  if constexpr (kPair) k_box_chunks = C::kKBoxChunks;
  CUtensorMap tm_k, tm_v;
  if ((st = encode_chunk_map(&tm_k, k_pool, num_pages, C::kHkv * C::kD, k_box_chunks))) return st;
  if ((st = encode_chunk_map(&tm_v, v_pool, num_pages, C::kHkv * C::kD, kPair ? C::kDS / 128 : C::kDS / 64)))
    return st;

  pda::prefill_tc::PrefillParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.cu_q = cu_q;
  p.o = o;
  p.status = status;
  p.num_pages = num_pages;
  p.batch = batch;
  p.max_blocks = max_blocks;
  p.window = window;
  p.total_q = total_q;
  p.max_q = max_q;
  p.out_f32 = out_dtype == ATTN_OUT_F32;
  int tiles = (max_q + C::kQ - 1) / C::kQ;
  if (kPair) tiles += tiles & 1;  // whole clusters of two query tiles
  const dim3 grid(tiles, C::kHkv * C::kSlices, batch);
  cudaError_t e = cudaSuccess;
  if constexpr (kPair) {
    e = launch_pdl(kernel, grid, C::kThreads, C::kSmemBytes, static_cast<cudaStream_t>(stream), tm_k, tm_v, p);
  } else {
    CUtensorMap tm_q, tm_o;  // the tile's Q, and (bf16 output) its O, in one box per 64-dim chunk
    if ((st = encode_q_map(&tm_q, q, total_q, C::kHq, C::kD, C::kG, C::kQ))) return st;
    if (out_dtype == ATTN_OUT_BF16) {
      if ((st = encode_q_map(&tm_o, o, total_q, C::kHq, C::kD, C::kG, C::kQ))) return st;
    } else {
      tm_o = tm_q;  // not used: fp32 output is written by the threads
    }
    // one CTA per SM looping over the work items (query tile, KV head and
    // slice, sequence), or one CTA per item
    const int64_t work = static_cast<int64_t>(tiles) * C::kHkv * C::kSlices * batch;
    const int64_t ctas = kPersistentPrefill ? std::min<int64_t>(work, std::max(1, num_sms)) : work;
    e = launch_pdl(kernel, dim3(static_cast<unsigned>(ctas)), C::kThreads, C::kSmemBytes,
                   static_cast<cudaStream_t>(stream), tm_k, tm_v, tm_q, tm_o, p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "%s: launch failed: %s", name, cudaGetErrorString(e));
  return ATTN_OK;
}

// The prefill kernels in use: global layers on CTA pairs (each SM copies
// half of every K and V tile: 290 -> 462 TFLOP/s on a 4096-token chunk of a
// 32768-token context); sliding layers on single CTAs, which measured faster
// there (609 against 338 TFLOP/s with pairs: their steps are bound by the
// softmax and issue latency, which the pair's cross-SM handshakes lengthen).
constexpr bool kSlidingPair = false;
constexpr bool kGlobalPair = true;
using kSlidingPrefill = pda::prefill_tc::SlidingConfig;
using kGlobalPrefill = pda::prefill_pair::GlobalPairConfig;
template <typename C, bool kPair>
auto prefill_kernel() {
  if constexpr (kPair)
    return pda::prefill_pair::prefill_pair_kernel<C>;
  else
    return pda::prefill_tc::prefill_tc_kernel<C>;
}

}  // namespace

extern "C" int32_t attn_prefill_sliding(const void* q, const void* k_pool, const void* v_pool,
                                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* cu_q,
                                        void* o, int32_t batch, int32_t total_q, int32_t max_q, int32_t max_blocks,
                                        int64_t num_pages, int32_t window, int32_t out_dtype, int32_t* status,
                                        void* stream) {
  return run_prefill<kSlidingPrefill, kSlidingPair>(prefill_kernel<kSlidingPrefill, kSlidingPair>(), ATTN_KIND_SLIDING, q, k_pool, v_pool, block_table, seq_lens, cu_q,
                                                  o, batch, total_q, max_q, max_blocks, num_pages, window, out_dtype,
                                                  status, stream);
}

extern "C" int32_t attn_prefill_global(const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_table, const int32_t* seq_lens, const int32_t* cu_q,
                                       void* o, int32_t batch, int32_t total_q, int32_t max_q, int32_t max_blocks,
                                       int64_t num_pages, int32_t window, int32_t out_dtype, int32_t* status,
                                       void* stream) {
  return run_prefill<kGlobalPrefill, kGlobalPair>(prefill_kernel<kGlobalPrefill, kGlobalPair>(), ATTN_KIND_GLOBAL, q, k_pool, v_pool, block_table, seq_lens, cu_q, o,
                                                 batch, total_q, max_q, max_blocks, num_pages, window, out_dtype,
                                                 status, stream);
}

// Waits for the previous kernel in the stream, lets its own dependents launch
// at once, sleeps `delay_ns` (bounded by the host to 1 ms, and by an
// iteration cap), then copies `words` 32-bit words.  A programmatic dependent
// launched after it therefore runs its pre-wait prologue while dst still
// holds the old values.
__global__ void __launch_bounds__(256) selftest_delayed_copy_kernel(uint32_t* dst, const uint32_t* src, int64_t words,
                                                                    int32_t delay_ns) {
  pda::wait_for_primary_grid();
  pda::allow_dependent_launch();
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int it = 0; it < (1 << 20); ++it) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= static_cast<uint64_t>(delay_ns)) break;
    __nanosleep(256);
  }
  for (int64_t i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
}

extern "C" int32_t attn_selftest_delayed_copy(void* dst, const void* src, int64_t bytes, int32_t delay_ns,
                                              void* stream) {
  g_err[0] = '\0';
  if (!dst || !src || (reinterpret_cast<uintptr_t>(dst) & 3u) || (reinterpret_cast<uintptr_t>(src) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "attn_selftest_delayed_copy: dst and src must be 4-byte aligned device pointers");
  if (bytes < 0 || (bytes & 3) || bytes > (int64_t{1} << 24))
    return fail(ATTN_ERR_INVALID_ARG, "attn_selftest_delayed_copy: bytes must be a multiple of 4 in [0, 16 MiB]");
  if (delay_ns < 0 || delay_ns > 1000000)
    return fail(ATTN_ERR_INVALID_ARG, "attn_selftest_delayed_copy: delay_ns must be in [0, 1000000]");
  const cudaError_t e = launch_pdl(selftest_delayed_copy_kernel, dim3(1), 256, 0, static_cast<cudaStream_t>(stream),
                                   static_cast<uint32_t*>(dst), static_cast<const uint32_t*>(src), bytes / 4, delay_ns);
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, "attn_selftest_delayed_copy: launch failed: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Sliding-window decode with built-in scratch, for callers that cannot
// allocate device memory themselves.
//
// The partial softmax rows that the split sequences leave for the combine
// kernel live in one file-scope device array instead of a caller-provided
// workspace.  Every GPU that loads this library keeps the array for the life
// of the process.  In host code the array's name is only a host-side stand-in
// for the device object and must never be handed to a kernel; the device
// address comes from cudaGetSymbolAddress, taken once per device on the first
// call made with that device current.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t{8} << 20;  // 8 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

int32_t noalloc_scratch(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(ATTN_ERR_CUDA, "attn_decode_sliding_noalloc: cudaGetSymbolAddress of the scratch failed: %s",
                  cudaGetErrorString(e));
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int32_t attn_decode_sliding_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                               const int32_t* block_table, const int32_t* seq_lens, void* o,
                                               int32_t batch, int32_t max_blocks, int64_t num_pages,
                                               int32_t max_seq_len, int32_t window, int32_t out_dtype,
                                               int32_t num_splits, int32_t* status, void* stream) {
  g_err[0] = '\0';
  int dev = 0, num_sms = 0;
  int32_t st = current_device(&dev, &num_sms);
  if (st != ATTN_OK) return st;
  // Size check first; every other argument is validated by the common path below.
  if (window > 0 && batch >= 1 && max_seq_len >= 0 && num_splits >= 0) {
    Plan plan;
    st = make_plan(ATTN_KIND_SLIDING, batch, max_seq_len, window, num_splits, num_sms, &plan);
    if (st != ATTN_OK) return st;
    if (plan.workspace_bytes > kNoAllocScratchBytes)
      return fail(ATTN_ERR_UNSUPPORTED,
                  "attn_decode_sliding_noalloc: this call needs %zu bytes of scratch but the built-in "
                  "scratch holds %zu (batch %d, num_splits %d); use attn_decode_sliding with a workspace",
                  plan.workspace_bytes, kNoAllocScratchBytes, batch, num_splits);
  }
  void* scratch = nullptr;
  if ((st = noalloc_scratch(dev, &scratch)) != ATTN_OK) return st;
  return run_decode(ATTN_KIND_SLIDING, q, k_pool, v_pool, block_table, seq_lens, o, batch, max_blocks,
                    num_pages, max_seq_len, window, out_dtype, num_splits, scratch, kNoAllocScratchBytes,
                    status, stream);
}

#include "step.cuh"
