// gca_retrieve_topk_noalloc: the retrieval entry point for callers that cannot hand the
// library a workspace.  The scratch it needs (the per-split candidate lists that the
// merge kernel combines, plus an error word) lives in one fixed array in device memory
// that every GPU loading this library holds until the process exits.
//
// Host code must never pass `g_noalloc_scratch` itself to a kernel: on the host that
// name is only a stand-in for the device array.  The device address is looked up once
// per device with cudaGetSymbolAddress and cached.
#include <cstdio>
#include <mutex>

#include "../../include/gca.h"
#include "common.cuh"
#include "internal.h"

namespace gca {
namespace {

constexpr size_t kNoAllocPartBytes = size_t(4) << 20;  // 4 MiB of split candidates
constexpr size_t kNoAllocBytes = kErrBytes + kNoAllocPartBytes;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_na_mu;
void* g_na_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on first use).
cudaError_t scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_na_ptr[dev] = p;
  }
  *out = g_na_ptr[dev];
  return cudaSuccess;
}

gca_status set_error(gca_status s, const char* msg) {
  set_error_detail(msg);
  return s;
}

}  // namespace
}  // namespace gca

using namespace gca;

extern "C" size_t gca_retrieve_noalloc_max_scratch(void) { return kNoAllocPartBytes; }

extern "C" gca_status gca_retrieve_topk_noalloc(const void* q_lmk, int64_t q_row_stride,
                                                int64_t q_batch_stride, const void* k_lmk,
                                                int64_t k_batch_stride, gca_dtype dtype, int B, int nQ,
                                                int nC, int D, int topk, int causal_offset, int use_gumbel,
                                                uint64_t seed, int group, int32_t* idx, float* scores,
                                                gca_stream_t stream) {
  // Every argument is checked before anything is queued on the stream, so a rejected call
  // leaves the array (and an error word that a previous call set) as it was.
  gca_status st = check_retrieve_args(q_lmk, q_row_stride, q_batch_stride, k_lmk, k_batch_stride, dtype, B, nQ,
                                      nC, D, topk, causal_offset, use_gumbel, group, idx, scores);
  if (st != GCA_OK) return st;
  // Size the scratch that the workspace-taking entry point would need and refuse a
  // problem that does not fit the fixed array.
  const size_t need = gca_retrieve_workspace_size(B, nQ, nC, topk, causal_offset);
  if (need > kNoAllocBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "gca_retrieve_topk_noalloc: this problem needs %zu bytes of candidate scratch, more than the "
             "fixed %zu; use gca_retrieve_topk with a workspace",
             need - kErrBytes, kNoAllocPartBytes);
    return set_error(GCA_ERR_UNSUPPORTED, msg);
  }
  void* ws = nullptr;
  cudaError_t e = scratch_ptr(&ws);
  if (e != cudaSuccess) return set_error(GCA_ERR_CUDA, cudaGetErrorString(e));
  // Only the error word must start at zero; every candidate list is written before it
  // is read.
  e = cudaMemsetAsync(ws, 0, kErrBytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(GCA_ERR_CUDA, cudaGetErrorString(e));
  return gca_retrieve_topk(q_lmk, q_row_stride, q_batch_stride, k_lmk, k_batch_stride, dtype, B, nQ, nC, D,
                           topk, causal_offset, use_gumbel, seed, group, idx, scores, ws, kNoAllocBytes, stream);
}

extern "C" gca_status gca_retrieve_noalloc_check_error(gca_stream_t stream, int* bad_value) {
  void* ws = nullptr;
  cudaError_t e = scratch_ptr(&ws);
  if (e != cudaSuccess) return set_error(GCA_ERR_CUDA, cudaGetErrorString(e));
  return gca_check_error(ws, stream, bad_value);
}

extern "C" gca_status gca_retrieve_noalloc_selftest_timeout(uint32_t spins, gca_stream_t stream) {
  void* ws = nullptr;
  cudaError_t e = scratch_ptr(&ws);
  if (e != cudaSuccess) return set_error(GCA_ERR_CUDA, cudaGetErrorString(e));
  return gca_selftest_timeout(ws, kErrBytes, spins, stream);
}
