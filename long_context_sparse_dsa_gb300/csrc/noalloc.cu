// noalloc.cu -- dsa_layer_fwd for callers that cannot give the library memory.
//
// dsa_layer_fwd needs a caller-provided workspace for the indexer's score
// block.  Some callers cannot provide one: a host framework whose operator
// interface has no workspace argument and whose own caching allocator owns
// all device memory (a plugin must not call cudaMalloc behind its back), or
// a code path where a cudaMalloc is not allowed because it may synchronise
// the device.  dsa_layer_fwd_noalloc serves them: the score block lives in
// one file-scope device array of fixed size, g_noalloc_scores, which every
// GPU that loads this library holds until the process exits.
//
// This file adds only that entry point; it calls the existing public entry
// points in the same order as dsa_layer_fwd, with the array in place of the
// workspace and the query chunk shrunk to fit it.
#include <mutex>

#include "../../include/dsa.h"
#include "common.cuh"

namespace dsa {
void set_last_error_message(const char* msg);  // defined in api.cu
dsa_status check_layer_fwd_args(const dsa_dims* dims, const void* q, const void* k, const void* v,
                                const void* q_idx, const void* k_idx, const float* w, const void* o,
                                const float* lse, const int32_t* idx, const void* kpool);  // api.cu
}

namespace {

constexpr size_t kNoallocScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;

// The score block of one query chunk.  Nothing in it needs to start at zero:
// the indexer writes every entry the top-k reads.
static __device__ __align__(256) float g_noalloc_scores[kNoallocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float* g_scores_dev[kMaxDevices] = {};

// Device address of g_noalloc_scores on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
dsa_status scratch_address(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    dsa::set_last_error_message("dsa_layer_fwd_noalloc: no usable current CUDA device");
    return DSA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scores_dev[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scores);
    if (e != cudaSuccess || ptr == nullptr) {
      dsa::set_last_error_message("dsa_layer_fwd_noalloc: cudaGetSymbolAddress of the scratch array failed");
      return DSA_ERR_CUDA;
    }
    g_scores_dev[dev] = static_cast<float*>(ptr);
  }
  *out = g_scores_dev[dev];
  return DSA_OK;
}

}  // namespace

extern "C" dsa_status dsa_layer_fwd_noalloc(const dsa_dims* dims, const void* q, const void* k, const void* v,
                                            const void* q_idx, const void* k_idx, const float* w, void* o,
                                            float* lse, int32_t* idx, void* kpool, dsa_stream_t stream) {
  // every argument is checked before anything is enqueued (or the scratch
  // array's address is looked up)
  dsa_status st = dsa::check_layer_fwd_args(dims, q, k, v, q_idx, k_idx, w, o, lse, idx, kpool);
  if (st != DSA_OK) return st;
  const int64_t P = dims->L / 4;
  const int64_t rows_fit = (int64_t)(kNoallocScratchBytes / sizeof(float)) / P;
  if (rows_fit < 1) {
    dsa::set_last_error_message(
        "dsa_layer_fwd_noalloc: one score row (L/4 fp32 values) does not fit the fixed scratch array");
    return DSA_ERR_UNSUPPORTED;
  }
  float* scores = nullptr;
  if ((st = scratch_address(&scores)) != DSA_OK) return st;
  const int64_t chunk = dims->q_chunk < rows_fit ? dims->q_chunk : rows_fit;
  if ((st = dsa_pool_keys(dims, k_idx, kpool, stream)) != DSA_OK) return st;
  for (int64_t q0 = 0; q0 < dims->L; q0 += chunk) {
    const int64_t n = dims->L - q0 < chunk ? dims->L - q0 : chunk;
    if ((st = dsa_indexer_score(dims, q_idx, kpool, w, q0, n, scores, stream)) != DSA_OK) return st;
    if ((st = dsa_topk(dims, scores, q0, n, idx, stream)) != DSA_OK) return st;
  }
  return dsa_sparse_attn_fwd(dims, q, k, v, idx, o, lse, nullptr, stream);
}
