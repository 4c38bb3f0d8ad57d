// api.cu -- the C ABI of libdsa_gb300.so (declared in include/dsa.h).
//
// Validation of every argument happens here, before anything is enqueued;
// a shape the kernels do not implement returns DSA_ERR_UNSUPPORTED (never a
// silent switch to another algorithm).  The entry points only enqueue work on
// the caller's stream; they do not allocate, free or synchronise.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/dsa.h"
#include "common.cuh"
#include "launch.h"

namespace dsa {
__device__ unsigned int g_dev_error = 0;
__constant__ unsigned int c_wait_limit = 1u << 20;

// Waits on an mbarrier that nothing ever arrives on; the bounded wait must
// give up after `spins` polls and record a timeout.  Nothing asynchronous is
// in flight, so giving up is safe.
__global__ void selftest_wait_kernel(uint32_t spins) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_n(smem_u32(&bar), 0, nullptr, spins);
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}
}  // namespace dsa

namespace {

thread_local char g_msg[512] = "";
int g_indexer_topk_route = 1;   // see dsa_set_indexer_topk_route
int g_attn_fwd_route = 0;       // see dsa_set_attn_fwd_route

dsa_status fail(dsa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

dsa_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return DSA_OK;
  if (e == cudaErrorNotSupported) return fail(DSA_ERR_UNSUPPORTED, "%s: not supported", what);
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE_PTR(p)                                                             \
  do {                                                                             \
    if ((p) == nullptr) return fail(DSA_ERR_INVALID_ARG, "%s is NULL", #p);        \
    if (!aligned16(p)) return fail(DSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

dsa_status check_dims(const dsa_dims* d, bool with_backward) {
  if (!d) return fail(DSA_ERR_INVALID_ARG, "dims is NULL");
  if (d->pool != 4) return fail(DSA_ERR_UNSUPPORTED, "pool must be 4 (got %d)", d->pool);
  if (d->L < 4 || d->L % 4 != 0) return fail(DSA_ERR_INVALID_ARG, "L must be a positive multiple of 4 (got %lld)", (long long)d->L);
  if (d->L > (int64_t)1 << 31) return fail(DSA_ERR_UNSUPPORTED, "L above 2^31 is not supported");
  if (d->k < 1) return fail(DSA_ERR_INVALID_ARG, "k must be >= 1 (got %d)", d->k);
  if (d->k > 1024) return fail(DSA_ERR_UNSUPPORTED, "k above 1024 is not supported (got %d)", d->k);
  if (d->q_chunk < 1) return fail(DSA_ERR_INVALID_ARG, "q_chunk must be >= 1 (got %d)", d->q_chunk);
  if (!(d->scale > 0.f) || d->scale != d->scale) return fail(DSA_ERR_INVALID_ARG, "scale must be a positive number");
  if (d->d != 64 && d->d != 128) return fail(DSA_ERR_UNSUPPORTED, "head dim d must be 64 or 128 (got %d)", d->d);
  if (d->di != 64 && d->di != 128) return fail(DSA_ERR_UNSUPPORTED, "indexer dim di must be 64 or 128 (got %d)", d->di);
  if (d->dtype == DSA_BF16) {
    if (d->Hq != 16 && d->Hq != 32) return fail(DSA_ERR_UNSUPPORTED, "bf16 layers need Hq in {16,32} (got %d)", d->Hq);
    if (d->Hi != 4 && d->Hi != 8) return fail(DSA_ERR_UNSUPPORTED, "bf16 layers need Hi in {4,8} (got %d)", d->Hi);
  } else if (d->dtype == DSA_FP32) {
    if (d->Hq < 1 || d->Hq > 32) return fail(DSA_ERR_UNSUPPORTED, "fp32 layers need 1 <= Hq <= 32 (got %d)", d->Hq);
    if (d->Hi < 1 || d->Hi > 8) return fail(DSA_ERR_UNSUPPORTED, "fp32 layers need 1 <= Hi <= 8 (got %d)", d->Hi);
    if (with_backward) return fail(DSA_ERR_UNSUPPORTED, "the backward is implemented for bf16 layers only");
  } else {
    return fail(DSA_ERR_INVALID_ARG, "unknown dtype %d", d->dtype);
  }
  return DSA_OK;
}

dsa_status check_range(const dsa_dims* d, int64_t q_begin, int64_t q_count) {
  if (q_begin < 0 || q_count < 1 || q_begin + q_count > d->L)
    return fail(DSA_ERR_INVALID_ARG, "query range [%lld, %lld) outside [0, %lld)", (long long)q_begin,
                (long long)(q_begin + q_count), (long long)d->L);
  return DSA_OK;
}

bool is_bf16(const dsa_dims* d) { return d->dtype == DSA_BF16; }

dsa_status do_pool(const dsa_dims* d, const void* k_idx, void* kpool, cudaStream_t s, const float* gate = nullptr) {
  return cuda_status(dsa::launch_pool_keys(is_bf16(d), d->L, d->di, k_idx, gate, kpool, s), "pool_keys launch");
}

dsa_status do_score(const dsa_dims* d, const void* q_idx, const void* kpool, const float* w, int64_t q_begin,
                    int64_t q_count, float* scores, cudaStream_t s) {
  cudaError_t e;
  if (is_bf16(d))
    e = dsa::launch_indexer_tc_bf16(d->L, d->Hi, d->di, q_idx, kpool, w, q_begin, q_count, scores, s);
  else
    e = dsa::launch_indexer_simt_f32(d->L, d->Hi, d->di, static_cast<const float*>(q_idx),
                                     static_cast<const float*>(kpool), w, q_begin, q_count, scores, s);
  return cuda_status(e, "indexer_score launch");
}

dsa_status do_topk(const dsa_dims* d, const float* scores, int64_t q_begin, int64_t q_count, int32_t* idx,
                   cudaStream_t s) {
  return cuda_status(dsa::launch_topk(d->L, d->k, scores, q_begin, q_count, idx, s), "topk launch");
}

size_t indexer_topk_ws_bytes(const dsa_dims* d, int64_t rows) {
  if (is_bf16(d)) return dsa::fused_indexer_topk_ws_bytes(d->L, rows);
  const size_t bytes = (size_t)rows * (size_t)(d->L / 4) * sizeof(float);   // the score block
  return (bytes + 255) & ~(size_t)255;
}

// Indexer + top-k of one query range: fused (no score block) for bf16 layers,
// the unfused pair through the score block in ws for fp32 layers.
dsa_status do_indexer_topk(const dsa_dims* d, const void* q_idx, const void* kpool, const float* w, int64_t q_begin,
                           int64_t q_count, int32_t* idx, void* ws, cudaStream_t s) {
  if (!is_bf16(d)) {
    dsa_status st = do_score(d, q_idx, kpool, w, q_begin, q_count, static_cast<float*>(ws), s);
    if (st) return st;
    return do_topk(d, static_cast<float*>(ws), q_begin, q_count, idx, s);
  }
  return cuda_status(dsa::launch_indexer_topk_bf16(d->L, d->Hi, d->di, d->k, q_idx, kpool, w, q_begin, q_count, idx,
                                                   ws, g_indexer_topk_route, s),
                     "indexer_topk launch");
}

dsa_status do_fwd(const dsa_dims* d, const void* q, const void* k, const void* v, const int32_t* idx, void* o,
                  float* lse, float* o_acc, cudaStream_t s) {
  cudaError_t e;
  if (is_bf16(d)) {
    if (g_attn_fwd_route == 1 && dsa::attn_fwd_tc_supported(d->Hq, d->d))
      e = dsa::launch_attn_fwd_tc_bf16(d->L, d->Hq, d->d, d->k, d->scale, q, k, v, idx, o, lse, o_acc, s);
    else
      e = dsa::launch_attn_fwd_bf16(d->L, d->Hq, d->d, d->k, d->scale, q, k, v, idx, o, lse, o_acc, s);
  } else {
    e = dsa::launch_attn_fwd_f32(d->L, d->Hq, d->d, d->k, d->scale, static_cast<const float*>(q),
                                 static_cast<const float*>(k), static_cast<const float*>(v), idx,
                                 static_cast<float*>(o), lse, s);
    // an fp32 layer's output already carries P in fp32
    if (e == cudaSuccess && o_acc != nullptr)
      e = cudaMemcpyAsync(o_acc, o, (size_t)d->L * d->Hq * d->d * sizeof(float), cudaMemcpyDeviceToDevice, s);
  }
  return cuda_status(e, "sparse_attn_fwd launch");
}

size_t bwd_ws_bytes(const dsa_dims* d) {
  const size_t bytes = (size_t)d->L * (size_t)d->Hq * sizeof(float);
  return (bytes + 255) & ~(size_t)255;
}

dsa_status do_bwd(const dsa_dims* d, const void* q, const void* k, const void* v, const int32_t* idx,
                  const float* lse, const float* o_acc, const void* dout, float* dq, float* dk, float* dv,
                  float* dbuf, cudaStream_t s) {
  const size_t kv_bytes = (size_t)d->L * d->d * sizeof(float);
  cudaError_t e = cudaMemsetAsync(dk, 0, kv_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_bytes, s);
  if (e != cudaSuccess) return cuda_status(e, "zeroing dk/dv");
  e = dsa::launch_attn_bwd_bf16(d->L, d->Hq, d->d, d->k, d->scale, q, k, v, idx, lse, dout, o_acc, dbuf, dq, dk,
                                dv, s);
  return cuda_status(e, "sparse_attn_bwd launch");
}

}  // namespace

namespace dsa {
// Lets entry points defined in other files of the library report a detail
// through dsa_last_error_message.
void set_last_error_message(const char* msg) { snprintf(g_msg, sizeof(g_msg), "%s", msg); }

// The checks dsa_layer_fwd makes on its dims and tensor pointers (everything
// but the workspace and o_acc), for entry points in other files that must
// reject bad arguments before they enqueue anything.
dsa_status check_layer_fwd_args(const dsa_dims* dims, const void* q, const void* k, const void* v,
                                const void* q_idx, const void* k_idx, const float* w, const void* o,
                                const float* lse, const int32_t* idx, const void* kpool) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, false);
  if (st) return st;
  REQUIRE_PTR(q);
  REQUIRE_PTR(k);
  REQUIRE_PTR(v);
  REQUIRE_PTR(q_idx);
  REQUIRE_PTR(k_idx);
  REQUIRE_PTR(w);
  REQUIRE_PTR(o);
  REQUIRE_PTR(lse);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(kpool);
  return DSA_OK;
}
}  // namespace dsa

extern "C" {

const char* dsa_status_string(dsa_status st) {
  switch (st) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case DSA_ERR_WORKSPACE: return "workspace missing or too small";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_TIMEOUT: return "device-side wait timed out";
    case DSA_ERR_BAD_INDEX: return "idx named a pool outside the query's causal range";
  }
  return "unknown status";
}

const char* dsa_last_error_message(void) { return g_msg; }

dsa_status dsa_validate_dims(const dsa_dims* dims, int32_t with_backward) {
  g_msg[0] = 0;
  return check_dims(dims, with_backward != 0);
}

size_t dsa_workspace_bytes(const dsa_dims* dims) {
  if (check_dims(dims, false) != DSA_OK) return 0;
  const int64_t C = dims->q_chunk < dims->L ? dims->q_chunk : dims->L;
  return indexer_topk_ws_bytes(dims, C);
}

size_t dsa_indexer_topk_workspace_bytes(const dsa_dims* dims, int64_t q_count) {
  if (check_dims(dims, false) != DSA_OK || q_count < 1 || q_count > dims->L) return 0;
  return indexer_topk_ws_bytes(dims, q_count);
}

dsa_status dsa_indexer_topk(const dsa_dims* dims, const void* q_idx, const void* kpool, const float* w,
                            int64_t q_begin, int64_t q_count, int32_t* idx, void* ws, size_t ws_bytes,
                            dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, false);
  if (st) return st;
  if ((st = check_range(dims, q_begin, q_count))) return st;
  REQUIRE_PTR(q_idx);
  REQUIRE_PTR(kpool);
  REQUIRE_PTR(w);
  REQUIRE_PTR(idx);
  const size_t need = indexer_topk_ws_bytes(dims, q_count);
  if (ws == nullptr || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", ws_bytes, need);
  if (!aligned16(ws)) return fail(DSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  return do_indexer_topk(dims, q_idx, kpool, w, q_begin, q_count, idx, ws, (cudaStream_t)stream);
}

dsa_status dsa_pool_keys(const dsa_dims* dims, const void* k_idx, void* kpool, dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, false);
  if (st) return st;
  REQUIRE_PTR(k_idx);
  REQUIRE_PTR(kpool);
  return do_pool(dims, k_idx, kpool, (cudaStream_t)stream);
}

dsa_status dsa_pool_keys_gated(const dsa_dims* dims, const void* k_idx, const float* gate, void* kpool,
                               dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, false);
  if (st) return st;
  REQUIRE_PTR(k_idx);
  REQUIRE_PTR(gate);
  REQUIRE_PTR(kpool);
  return do_pool(dims, k_idx, kpool, (cudaStream_t)stream, gate);
}

dsa_status dsa_indexer_score(const dsa_dims* dims, const void* q_idx, const void* kpool, const float* w,
                             int64_t q_begin, int64_t q_count, float* scores, dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, false);
  if (st) return st;
  if ((st = check_range(dims, q_begin, q_count))) return st;
  REQUIRE_PTR(q_idx);
  REQUIRE_PTR(kpool);
  REQUIRE_PTR(w);
  REQUIRE_PTR(scores);
  return do_score(dims, q_idx, kpool, w, q_begin, q_count, scores, (cudaStream_t)stream);
}

dsa_status dsa_topk(const dsa_dims* dims, const float* scores, int64_t q_begin, int64_t q_count, int32_t* idx,
                    dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, false);
  if (st) return st;
  if ((st = check_range(dims, q_begin, q_count))) return st;
  REQUIRE_PTR(scores);
  REQUIRE_PTR(idx);
  return do_topk(dims, scores, q_begin, q_count, idx, (cudaStream_t)stream);
}

dsa_status dsa_sparse_attn_fwd(const dsa_dims* dims, const void* q, const void* k, const void* v,
                               const int32_t* idx, void* o, float* lse, float* o_acc, dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, false);
  if (st) return st;
  REQUIRE_PTR(q);
  REQUIRE_PTR(k);
  REQUIRE_PTR(v);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(o);
  REQUIRE_PTR(lse);
  if (o_acc != nullptr && !aligned16(o_acc)) return fail(DSA_ERR_INVALID_ARG, "o_acc is not 16-byte aligned");
  return do_fwd(dims, q, k, v, idx, o, lse, o_acc, (cudaStream_t)stream);
}

size_t dsa_bwd_workspace_bytes(const dsa_dims* dims) {
  if (check_dims(dims, true) != DSA_OK) return 0;
  return bwd_ws_bytes(dims);
}

dsa_status dsa_sparse_attn_bwd(const dsa_dims* dims, const void* q, const void* k, const void* v,
                               const int32_t* idx, const void* o, const float* lse, const float* o_acc,
                               const void* dout, float* dq, float* dk, float* dv, void* ws, size_t ws_bytes,
                               dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, true);
  if (st) return st;
  REQUIRE_PTR(q);
  REQUIRE_PTR(k);
  REQUIRE_PTR(v);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(o);
  REQUIRE_PTR(lse);
  REQUIRE_PTR(dout);
  REQUIRE_PTR(dq);
  REQUIRE_PTR(dk);
  REQUIRE_PTR(dv);
  if (dk == dv) return fail(DSA_ERR_INVALID_ARG, "dk and dv must not alias");
  if (o_acc != nullptr) {
    if (!aligned16(o_acc)) return fail(DSA_ERR_INVALID_ARG, "o_acc is not 16-byte aligned");
    return do_bwd(dims, q, k, v, idx, lse, o_acc, dout, dq, dk, dv, nullptr, (cudaStream_t)stream);
  }
  const size_t need = bwd_ws_bytes(dims);
  if (ws == nullptr || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "backward workspace of %zu bytes given, %zu needed", ws_bytes, need);
  if (!aligned16(ws)) return fail(DSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  return do_bwd(dims, q, k, v, idx, lse, nullptr, dout, dq, dk, dv, static_cast<float*>(ws), (cudaStream_t)stream);
}

size_t dsa_bwd_det_workspace_bytes(const dsa_dims* dims) {
  if (check_dims(dims, true) != DSA_OK) return 0;
  if ((int64_t)dims->L * (dims->k + 1) >= ((int64_t)1 << 31)) return 0;
  return dsa::det_bwd_ws_bytes(dims->L, dims->Hq, dims->d, dims->k);
}

dsa_status dsa_sparse_attn_bwd_det(const dsa_dims* dims, const void* q, const void* k, const void* v,
                                   const int32_t* idx, const void* o, const float* lse, const float* o_acc,
                                   const void* dout, float* dq, float* dk, float* dv, void* ws, size_t ws_bytes,
                                   dsa_stream_t stream) {
  g_msg[0] = 0;
  dsa_status st = check_dims(dims, true);
  if (st) return st;
  if ((int64_t)dims->L * (dims->k + 1) >= ((int64_t)1 << 31))
    return fail(DSA_ERR_UNSUPPORTED, "the deterministic backward needs L * (k + 1) < 2^31");
  REQUIRE_PTR(q);
  REQUIRE_PTR(k);
  REQUIRE_PTR(v);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(o);
  REQUIRE_PTR(lse);
  REQUIRE_PTR(dout);
  REQUIRE_PTR(dq);
  REQUIRE_PTR(dk);
  REQUIRE_PTR(dv);
  if (dk == dv) return fail(DSA_ERR_INVALID_ARG, "dk and dv must not alias");
  if (o_acc != nullptr && !aligned16(o_acc)) return fail(DSA_ERR_INVALID_ARG, "o_acc is not 16-byte aligned");
  const size_t need = dsa::det_bwd_ws_bytes(dims->L, dims->Hq, dims->d, dims->k);
  if (ws == nullptr || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", ws_bytes, need);
  if (!aligned16(ws)) return fail(DSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  return cuda_status(dsa::launch_attn_bwd_det_bf16(dims->L, dims->Hq, dims->d, dims->k, dims->scale, q, k, v, idx,
                                                    lse, dout, o_acc, dq, dk, dv, ws, (cudaStream_t)stream),
                     "sparse_attn_bwd_det launch");
}

dsa_status dsa_layer_fwd(const dsa_dims* dims, const void* q, const void* k, const void* v, const void* q_idx,
                         const void* k_idx, const float* w, void* o, float* lse, float* o_acc, int32_t* idx,
                         void* kpool, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  dsa_status st = dsa::check_layer_fwd_args(dims, q, k, v, q_idx, k_idx, w, o, lse, idx, kpool);
  if (st) return st;
  if (o_acc != nullptr && !aligned16(o_acc)) return fail(DSA_ERR_INVALID_ARG, "o_acc is not 16-byte aligned");
  const size_t need = dsa_workspace_bytes(dims);
  if (ws == nullptr || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", ws_bytes, need);
  if (!aligned16(ws)) return fail(DSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  if ((st = do_pool(dims, k_idx, kpool, s))) return st;
  const int64_t C = dims->q_chunk;
  for (int64_t q0 = 0; q0 < dims->L; q0 += C) {
    const int64_t n = dims->L - q0 < C ? dims->L - q0 : C;
    if ((st = do_indexer_topk(dims, q_idx, kpool, w, q0, n, idx, ws, s))) return st;
  }
  return do_fwd(dims, q, k, v, idx, o, lse, o_acc, s);
}

dsa_status dsa_layer_bwd(const dsa_dims* dims, const void* q, const void* k, const void* v, const int32_t* idx,
                         const void* o, const float* lse, const float* o_acc, const void* dout, float* dq,
                         float* dk, float* dv, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  return dsa_sparse_attn_bwd(dims, q, k, v, idx, o, lse, o_acc, dout, dq, dk, dv, ws, ws_bytes, stream);
}

dsa_status dsa_check_device_error(dsa_stream_t stream) {
  g_msg[0] = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "stream synchronize");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, dsa::g_dev_error, sizeof(word));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(dsa::g_dev_error, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_status(e, "reading the device error word");
  if (word & dsa::DSA_DEV_ERR_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "a bounded device wait gave up (word 0x%x)", word);
  if (word & dsa::DSA_DEV_ERR_BAD_INDEX) return fail(DSA_ERR_BAD_INDEX, "idx held a pool outside elig(t) (word 0x%x)", word);
  return DSA_OK;
}

dsa_status dsa_selftest_bounded_wait(uint32_t spins, dsa_stream_t stream) {
  g_msg[0] = 0;
  if (spins == 0 || spins > (1u << 24)) return fail(DSA_ERR_INVALID_ARG, "spins must be in 1..2^24");
  dsa::selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(spins);
  return cuda_status(cudaGetLastError(), "selftest launch");
}

dsa_status dsa_set_indexer_topk_route(int32_t route) {
  g_msg[0] = 0;
  if (route != 0 && route != 1) return fail(DSA_ERR_INVALID_ARG, "route must be 0 or 1");
  g_indexer_topk_route = route;
  return DSA_OK;
}

dsa_status dsa_set_attn_fwd_route(int32_t route) {
  g_msg[0] = 0;
  if (route != 0 && route != 1) return fail(DSA_ERR_INVALID_ARG, "route must be 0 or 1");
  g_attn_fwd_route = route;
  return DSA_OK;
}

void dsa_set_wait_limit(uint32_t spins) {
  if (spins == 0) spins = 1;
  cudaMemcpyToSymbol(dsa::c_wait_limit, &spins, sizeof(spins));
}

}  // extern "C"
