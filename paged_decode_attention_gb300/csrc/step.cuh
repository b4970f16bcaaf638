// step.cuh -- host side of include/attn_step.h: the attention calls of a
// decode step recorded once and replayed with one call, either as one CUDA
// graph or as the recorded kernel launches enqueued back to back.  Included
// at the end of attn_decode.cu, whose validation (g_validate_only), launch
// recording (g_record) and error reporting it shares.
#pragma once

#include <functional>
#include <new>
#include <utility>
#include <vector>

#include "attn_step.h"

struct attn_step {
  std::vector<std::function<int32_t(void*)>> calls;  // each enqueues one call on the given stream
  int32_t kernels = 0;
  int32_t mode = ATTN_STEP_LAUNCH_AUTO;  // as requested; resolved by attn_step_finalize
  bool finalized = false;
  int device = -1;                       // the device the step was finalized on
  std::vector<RecordedLaunch> launches;  // every kernel launch of the step, arguments bound
  cudaGraph_t graph = nullptr;           // ATTN_STEP_LAUNCH_GRAPH only
  cudaGraphExec_t exec = nullptr;
};

namespace {

// Validates `call` (its launches suppressed) and, if it passes, appends it
// with the number of kernels it launches.
int32_t record(attn_step* step, std::function<int32_t(void*)> call, const char* name) {
  g_err[0] = '\0';
  if (!step) return fail(ATTN_ERR_INVALID_ARG, "%s: null step", name);
  if (step->finalized) return fail(ATTN_ERR_INVALID_ARG, "%s: the step is already finalized", name);
  g_validate_only = true;
  g_last_launches = 0;
  const int32_t st = call(nullptr);
  g_validate_only = false;
  if (st != ATTN_OK) return st;
  const int32_t kernels = g_last_launches;
  try {
    step->calls.push_back(std::move(call));
  } catch (...) {  // no exception may leave the C ABI
    return fail(ATTN_ERR_INVALID_ARG, "%s: out of host memory", name);
  }
  step->kernels += kernels;
  return ATTN_OK;
}

}  // namespace

extern "C" {

int32_t attn_step_create(attn_step** out) {
  g_err[0] = '\0';
  if (!out) return fail(ATTN_ERR_INVALID_ARG, "attn_step_create: null out");
  *out = new (std::nothrow) attn_step();
  if (!*out) return fail(ATTN_ERR_INVALID_ARG, "attn_step_create: out of host memory");
  return ATTN_OK;
}

void attn_step_destroy(attn_step* step) {
  if (!step) return;
  if (step->exec) cudaGraphExecDestroy(step->exec);
  if (step->graph) cudaGraphDestroy(step->graph);
  delete step;
}

int32_t attn_step_add_decode_sliding(attn_step* step, const void* q, const void* k_pool, const void* v_pool,
                                     const int32_t* block_table, const int32_t* seq_lens, void* o, int32_t batch,
                                     int32_t max_blocks, int64_t num_pages, int32_t max_seq_len, int32_t window,
                                     int32_t out_dtype, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                     int32_t* status) {
  return record(step, [=](void* s) {
    return attn_decode_sliding(q, k_pool, v_pool, block_table, seq_lens, o, batch, max_blocks, num_pages,
                               max_seq_len, window, out_dtype, num_splits, workspace, workspace_bytes, status, s);
  }, "attn_step_add_decode_sliding");
}

int32_t attn_step_add_decode_global(attn_step* step, const void* q, const void* k_pool, const void* v_pool,
                                    const int32_t* block_table, const int32_t* seq_lens, void* o, int32_t batch,
                                    int32_t max_blocks, int64_t num_pages, int32_t max_seq_len, int32_t window,
                                    int32_t out_dtype, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                    int32_t* status) {
  return record(step, [=](void* s) {
    return attn_decode_global(q, k_pool, v_pool, block_table, seq_lens, o, batch, max_blocks, num_pages,
                              max_seq_len, window, out_dtype, num_splits, workspace, workspace_bytes, status, s);
  }, "attn_step_add_decode_global");
}

int32_t attn_step_add_decode_global_shared(attn_step* step, const void* q, const void* kv_pool, const void* w_k,
                                           const int32_t* block_table, const int32_t* seq_lens, void* o,
                                           int32_t batch, int32_t max_blocks, int64_t num_pages,
                                           int32_t max_seq_len, int32_t window, int32_t out_dtype,
                                           int32_t num_splits, void* workspace, size_t workspace_bytes,
                                           int32_t* status) {
  return record(step, [=](void* s) {
    return attn_decode_global_shared(q, kv_pool, w_k, block_table, seq_lens, o, batch, max_blocks, num_pages,
                                     max_seq_len, window, out_dtype, num_splits, workspace, workspace_bytes,
                                     status, s);
  }, "attn_step_add_decode_global_shared");
}

int32_t attn_step_add_kv_append_sliding(attn_step* step, const void* qkv, const void* w_q, const void* w_k,
                                        const int32_t* block_table, const int32_t* positions, void* q_out,
                                        void* k_pool, void* v_pool, int32_t batch, int32_t max_blocks,
                                        int64_t num_pages, int32_t* status) {
  return record(step, [=](void* s) {
    return attn_kv_append_sliding(qkv, w_q, w_k, block_table, positions, q_out, k_pool, v_pool, batch, max_blocks,
                                  num_pages, status, s);
  }, "attn_step_add_kv_append_sliding");
}

int32_t attn_step_add_kv_append_global(attn_step* step, const void* qkv, const void* w_q, const void* w_k,
                                       const int32_t* block_table, const int32_t* positions, void* q_out,
                                       void* k_pool, void* v_pool, int32_t batch, int32_t max_blocks,
                                       int64_t num_pages, int32_t* status) {
  return record(step, [=](void* s) {
    return attn_kv_append_global(qkv, w_q, w_k, block_table, positions, q_out, k_pool, v_pool, batch, max_blocks,
                                 num_pages, status, s);
  }, "attn_step_add_kv_append_global");
}

int32_t attn_step_num_calls(const attn_step* step) { return step ? static_cast<int32_t>(step->calls.size()) : 0; }

int32_t attn_step_num_kernels(const attn_step* step) { return step ? step->kernels : 0; }

int32_t attn_step_set_launch_mode(attn_step* step, int32_t mode) {
  g_err[0] = '\0';
  const char* name = "attn_step_set_launch_mode";
  if (!step) return fail(ATTN_ERR_INVALID_ARG, "%s: null step", name);
  if (step->finalized) return fail(ATTN_ERR_INVALID_ARG, "%s: the step is already finalized", name);
  if (mode != ATTN_STEP_LAUNCH_AUTO && mode != ATTN_STEP_LAUNCH_GRAPH && mode != ATTN_STEP_LAUNCH_DIRECT)
    return fail(ATTN_ERR_INVALID_ARG, "%s: unknown mode %d", name, mode);
  step->mode = mode;
  return ATTN_OK;
}

int32_t attn_step_launch_mode(const attn_step* step) { return step ? step->mode : -1; }

int32_t attn_step_finalize(attn_step* step) {
  g_err[0] = '\0';
  const char* name = "attn_step_finalize";
  if (!step) return fail(ATTN_ERR_INVALID_ARG, "%s: null step", name);
  if (step->finalized) return fail(ATTN_ERR_INVALID_ARG, "%s: already finalized", name);
  if (step->calls.empty()) return fail(ATTN_ERR_INVALID_ARG, "%s: no calls recorded", name);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "%s: cudaGetDevice: %s", name, cudaGetErrorString(e));

  // Run every call once more with its launches recorded instead of enqueued:
  // host validation, tensor maps and kernel attributes are done here, once.
  std::vector<RecordedLaunch> launches;
  int32_t st = ATTN_OK;
  g_record = &launches;
  for (size_t i = 0; i < step->calls.size() && st == ATTN_OK; ++i) st = step->calls[i](nullptr);
  g_record = nullptr;
  if (st != ATTN_OK) return st;
  if (launches.size() != static_cast<size_t>(step->kernels))
    return fail(ATTN_ERR_INVALID_ARG, "%s: recorded %zu launches for %d kernels", name, launches.size(),
                step->kernels);

  int32_t mode = step->mode;
  if (mode == ATTN_STEP_LAUNCH_AUTO)
    mode = step->kernels <= ATTN_STEP_DIRECT_MAX_KERNELS ? ATTN_STEP_LAUNCH_DIRECT : ATTN_STEP_LAUNCH_GRAPH;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  if (mode == ATTN_STEP_LAUNCH_GRAPH) {
    cudaStream_t cs = nullptr;
    e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "%s: cudaStreamCreate: %s", name, cudaGetErrorString(e));
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) {
      cudaStreamDestroy(cs);
      return fail(ATTN_ERR_CUDA, "%s: cudaStreamBeginCapture: %s", name, cudaGetErrorString(e));
    }
    // The kernels keep their programmatic-serialisation attribute, so the
    // graph holds programmatic edges between consecutive kernels.
    for (size_t i = 0; i < launches.size() && st == ATTN_OK; ++i) {
      const cudaError_t le = launches[i](cs);
      if (le != cudaSuccess) st = fail(ATTN_ERR_CUDA, "%s: launch %zu: %s", name, i, cudaGetErrorString(le));
    }
    e = cudaStreamEndCapture(cs, &graph);
    if (st == ATTN_OK && e != cudaSuccess)
      st = fail(ATTN_ERR_CUDA, "%s: cudaStreamEndCapture: %s", name, cudaGetErrorString(e));
    if (st == ATTN_OK) {
      e = cudaGraphInstantiate(&exec, graph, 0);
      if (e != cudaSuccess) st = fail(ATTN_ERR_CUDA, "%s: cudaGraphInstantiate: %s", name, cudaGetErrorString(e));
    }
    cudaStreamDestroy(cs);
    if (st != ATTN_OK) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();  // a failed capture leaves no sticky error; clear the non-sticky one
      return st;
    }
  }
  step->launches = std::move(launches);
  step->graph = graph;
  step->exec = exec;
  step->mode = mode;
  step->device = dev;
  step->finalized = true;
  return ATTN_OK;
}

int32_t attn_step_launch(attn_step* step, void* stream) {
  g_err[0] = '\0';
  if (!step) return fail(ATTN_ERR_INVALID_ARG, "attn_step_launch: null step");
  if (!step->finalized) return fail(ATTN_ERR_INVALID_ARG, "attn_step_launch: the step is not finalized");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (step->exec) {
    const cudaError_t e = cudaGraphLaunch(step->exec, s);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "attn_step_launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
  }
  // Direct mode: the recorded launches, back to back, on the step's device.
  int cur = 0;
  cudaError_t e = cudaGetDevice(&cur);
  if (e == cudaSuccess && cur != step->device) e = cudaSetDevice(step->device);
  for (size_t i = 0; i < step->launches.size() && e == cudaSuccess; ++i) e = step->launches[i](s);
  if (cur != step->device) cudaSetDevice(cur);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "attn_step_launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

}  // extern "C"
