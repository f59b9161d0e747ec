// C ABI entry points of the GCA library: argument validation, workspace carving, kernel
// launches, the device error word and launch instrumentation.  The operations
// themselves are documented in include/gca.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/gca.h"
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gca {
namespace {

thread_local std::string t_detail;

gca_status fail(gca_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
gca_status fail(gca_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_detail = buf;
  return s;
}

gca_status cuda_fail(cudaError_t e, const char* where) {
  return fail(GCA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---------------------------------------------------------------- instrumentation
std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;
bool g_prof = false;
struct Rec {
  const char* name;
  cudaEvent_t a, b;
};
std::vector<Rec> g_open;      // recorded, not yet collected
std::vector<cudaEvent_t> g_pool;
struct Row {
  std::string name;
  int launches;
  double ms;
};
std::vector<Row> g_table;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

void launch_begin(const char* name, cudaStream_t s) {
  if (!g_prof) return;
  std::lock_guard<std::mutex> lk(g_mu);
  Rec r{name, take_event(), take_event()};
  cudaEventRecord(r.a, s);
  g_open.push_back(r);
}

cudaError_t launch_end(const char* name, cudaStream_t s) {
  cudaError_t e = cudaGetLastError();
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_prof) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto it = g_open.rbegin(); it != g_open.rend(); ++it) {
      if (it->name == name) {
        cudaEventRecord(it->b, s);
        break;
      }
    }
  }
  return e;
}

int set_error_detail(const char* msg) {
  t_detail = msg;
  return 0;
}

cudaError_t allow_smem(const void* fn, int bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  struct Done {
    const void* fn;
    int dev, bytes;
  };
  static std::mutex mu;
  static std::vector<Done> done;  // largest limit set so far per (function, device)
  std::lock_guard<std::mutex> lk(mu);
  for (auto& d : done)
    if (d.fn == fn && d.dev == dev) {
      if (d.bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) d.bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.push_back(Done{fn, dev, bytes});
  return e;
}

}  // namespace gca

using namespace gca;

// ==================================================================== common
extern "C" const char* gca_status_string(gca_status s) {
  switch (s) {
    case GCA_OK: return "GCA_OK";
    case GCA_ERR_INVALID_ARG: return "GCA_ERR_INVALID_ARG";
    case GCA_ERR_UNSUPPORTED: return "GCA_ERR_UNSUPPORTED";
    case GCA_ERR_WORKSPACE: return "GCA_ERR_WORKSPACE";
    case GCA_ERR_CUDA: return "GCA_ERR_CUDA";
    case GCA_ERR_DEVICE_INDEX: return "GCA_ERR_DEVICE_INDEX";
    case GCA_ERR_TIMEOUT: return "GCA_ERR_TIMEOUT";
  }
  return "unknown gca_status";
}

extern "C" const char* gca_last_error_detail(void) { return t_detail.c_str(); }

static gca_status check_ws(void* ws, size_t have, size_t need) {
  if (ws == nullptr) return fail(GCA_ERR_WORKSPACE, "workspace pointer is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(GCA_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (have < need) return fail(GCA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
  return GCA_OK;
}

static gca_status check_landmarks(const void* q, int64_t q_rs, int64_t q_bs, const void* k, int64_t k_bs,
                                  gca_dtype dt, int B, int nQ, int nC, int D, int topk) {
  if (dt != GCA_F32 && dt != GCA_BF16) return fail(GCA_ERR_INVALID_ARG, "dtype must be GCA_F32 or GCA_BF16");
  if (!q || !k) return fail(GCA_ERR_INVALID_ARG, "landmark pointer is NULL");
  if (B < 1 || nQ < 1 || nC < 1) return fail(GCA_ERR_INVALID_ARG, "B, nQ and nC must be >= 1 (got %d, %d, %d)", B, nQ, nC);
  if (B > 65535) return fail(GCA_ERR_INVALID_ARG, "B must be <= 65535");
  if (topk < 1 || topk > GCA_MAX_TOPK) return fail(GCA_ERR_UNSUPPORTED, "topk must be in 1..16 (got %d)", topk);
  const int epv = dt == GCA_BF16 ? 8 : 4;
  if (dt == GCA_BF16 && (D < 64 || D > 1024 || D % 64))
    return fail(GCA_ERR_UNSUPPORTED, "bf16 landmark dim must be a multiple of 64 in 64..1024 (got %d)", D);
  if (dt == GCA_F32 && (D < 32 || D > 512 || D % 32))
    return fail(GCA_ERR_UNSUPPORTED, "f32 landmark dim must be a multiple of 32 in 32..512 (got %d)", D);
  if (!aligned16(q) || !aligned16(k)) return fail(GCA_ERR_INVALID_ARG, "landmark pointers must be 16-byte aligned");
  if (q_rs < D || q_rs % epv) return fail(GCA_ERR_INVALID_ARG, "q_row_stride must be >= D and a multiple of %d", epv);
  if (q_bs < 0 || q_bs % epv) return fail(GCA_ERR_INVALID_ARG, "q_batch_stride must be >= 0 and a multiple of %d", epv);
  if (B > 1 && q_bs < (int64_t)(nQ - 1) * q_rs + D)
    return fail(GCA_ERR_INVALID_ARG, "q_batch_stride too small for nQ rows");
  if (k_bs != 0 && (k_bs < (int64_t)nC * D || k_bs % epv))
    return fail(GCA_ERR_INVALID_ARG, "k_batch_stride must be 0 or >= nC*D and a multiple of %d", epv);
  return GCA_OK;
}

// ==================================================================== retrieval
extern "C" size_t gca_retrieve_workspace_size(int B, int nQ, int nC, int topk, int causal_offset) {
  if (B < 1 || nQ < 1 || nC < 1 || topk < 1 || causal_offset < 0) return kErrBytes;
  RetrievePlan p = retrieve_plan(B, nQ, nC, topk, causal_offset);
  return kErrBytes + align256(p.part_bytes);
}

gca_status gca::check_retrieve_args(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride,
                                    const void* k_lmk, int64_t k_batch_stride, gca_dtype dtype, int B, int nQ,
                                    int nC, int D, int topk, int causal_offset, int use_gumbel, int group,
                                    const int32_t* idx, const float* scores) {
  gca_status st = check_landmarks(q_lmk, q_row_stride, q_batch_stride, k_lmk, k_batch_stride, dtype, B, nQ,
                                  nC, D, topk);
  if (st != GCA_OK) return st;
  if (!idx || !scores) return fail(GCA_ERR_INVALID_ARG, "idx/scores pointer is NULL");
  if (causal_offset < 0) return fail(GCA_ERR_INVALID_ARG, "causal_offset must be >= 0");
  if (use_gumbel && (B > 256 || nQ > (1 << 24) || nC > (1 << 24) || group < 0 || group > 255))
    return fail(GCA_ERR_INVALID_ARG, "Gumbel noise needs B <= 256, nQ, nC <= 2^24, 0 <= group < 256");
  return GCA_OK;
}

static gca_status retrieve_topk_impl(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride,
                                     const void* k_lmk, int64_t k_batch_stride, gca_dtype dtype, int B, int nQ,
                                     int nC, int D, int topk, int causal_offset, int use_gumbel, uint64_t seed,
                                     const uint64_t* seed_dev, int group, int32_t* idx, float* scores, void* ws,
                                     size_t ws_bytes, gca_stream_t stream) {
  gca_status st = check_retrieve_args(q_lmk, q_row_stride, q_batch_stride, k_lmk, k_batch_stride, dtype, B, nQ,
                                      nC, D, topk, causal_offset, use_gumbel, group, idx, scores);
  if (st != GCA_OK) return st;
  if ((st = check_ws(ws, ws_bytes, gca_retrieve_workspace_size(B, nQ, nC, topk, causal_offset))) != GCA_OK)
    return st;
  RetrievePlan p = retrieve_plan(B, nQ, nC, topk, causal_offset);
  RetrieveArgs a{};
  a.q = q_lmk; a.q_rs = q_row_stride; a.q_bs = q_batch_stride;
  a.k = k_lmk; a.k_bs = k_batch_stride;
  a.bf16 = dtype == GCA_BF16;
  a.B = B; a.nQ = nQ; a.nC = nC; a.D = D; a.topk = topk; a.off = causal_offset;
  a.gumbel = use_gumbel ? 1 : 0; a.seed = seed; a.group = group; a.seed_dev = seed_dev;
  a.idx = idx; a.scores = scores;
  a.err = reinterpret_cast<ErrWord*>(ws);
  a.part = static_cast<unsigned char*>(ws) + kErrBytes;
  cudaError_t e = launch_retrieve(a, p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_retrieve_topk launch");
  return GCA_OK;
}

extern "C" gca_status gca_retrieve_topk(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride,
                                        const void* k_lmk, int64_t k_batch_stride, gca_dtype dtype, int B,
                                        int nQ, int nC, int D, int topk, int causal_offset, int use_gumbel,
                                        uint64_t seed, int group, int32_t* idx, float* scores, void* ws,
                                        size_t ws_bytes, gca_stream_t stream) {
  return retrieve_topk_impl(q_lmk, q_row_stride, q_batch_stride, k_lmk, k_batch_stride, dtype, B, nQ, nC, D, topk,
                            causal_offset, use_gumbel, seed, nullptr, group, idx, scores, ws, ws_bytes, stream);
}

extern "C" gca_status gca_retrieve_topk_dseed(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride,
                                              const void* k_lmk, int64_t k_batch_stride, gca_dtype dtype, int B,
                                              int nQ, int nC, int D, int topk, int causal_offset, int use_gumbel,
                                              const uint64_t* seed, int group, int32_t* idx, float* scores,
                                              void* ws, size_t ws_bytes, gca_stream_t stream) {
  if (!seed || (reinterpret_cast<uintptr_t>(seed) & 7))
    return fail(GCA_ERR_INVALID_ARG, "seed must be a non-NULL, 8-byte aligned device pointer");
  return retrieve_topk_impl(q_lmk, q_row_stride, q_batch_stride, k_lmk, k_batch_stride, dtype, B, nQ, nC, D, topk,
                            causal_offset, use_gumbel, 0, seed, group, idx, scores, ws, ws_bytes, stream);
}

// ==================================================================== GCA forward
static gca_status check_gca(const void* q, const void* k, const void* v, gca_dtype dt, int B, int nQ, int nC,
                            int H, int dh, const int32_t* idx, const float* scores, int topk, int shift,
                            bool need_scores = true) {
  if (dt != GCA_F32 && dt != GCA_BF16) return fail(GCA_ERR_INVALID_ARG, "dtype must be GCA_F32 or GCA_BF16");
  if (!q || !k || !v || !idx || (need_scores && !scores)) return fail(GCA_ERR_INVALID_ARG, "input pointer is NULL");
  if (B < 1 || nQ < 1 || nC < 1 || H < 1) return fail(GCA_ERR_INVALID_ARG, "B, nQ, nC, H must be >= 1");
  if (B > 65535 || H > 65535) return fail(GCA_ERR_INVALID_ARG, "B and H must be <= 65535");
  if ((int64_t)nQ * 64 > INT32_MAX || (int64_t)nC * 64 > INT32_MAX)
    return fail(GCA_ERR_INVALID_ARG, "sequence too long");
  if (dh != 32 && dh != 64) return fail(GCA_ERR_UNSUPPORTED, "head dim must be 32 or 64 (got %d)", dh);
  if (topk < 1 || topk > GCA_MAX_TOPK) return fail(GCA_ERR_UNSUPPORTED, "topk must be in 1..16 (got %d)", topk);
  if (shift != 0 && shift != 1) return fail(GCA_ERR_INVALID_ARG, "shift must be 0 or 1");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return fail(GCA_ERR_INVALID_ARG, "q/k/v must be 16-byte aligned");
  return GCA_OK;
}

extern "C" size_t gca_forward_workspace_size(void) { return kErrBytes; }

extern "C" gca_status gca_forward(const void* q, const void* k, const void* v, int64_t kv_batch_stride,
                                  gca_dtype dtype, int B, int nQ, int nC, int H, int dh, const int32_t* idx,
                                  const float* scores, int topk, int shift, void* o, float* lse, void* ws,
                                  size_t ws_bytes, gca_stream_t stream) {
  gca_status st = check_gca(q, k, v, dtype, B, nQ, nC, H, dh, idx, scores, topk, shift);
  if (st != GCA_OK) return st;
  if (!o || !lse) return fail(GCA_ERR_INVALID_ARG, "o/lse pointer is NULL");
  if (!aligned16(o) || !aligned16(lse)) return fail(GCA_ERR_INVALID_ARG, "o/lse must be 16-byte aligned");
  const int64_t per_seq = (int64_t)nC * 64 * H * dh;
  if (kv_batch_stride != 0 && (kv_batch_stride < per_seq || kv_batch_stride % 8))
    return fail(GCA_ERR_INVALID_ARG, "kv_batch_stride must be 0 or >= nC*64*H*dh and a multiple of 8");
  if ((st = check_ws(ws, ws_bytes, gca_forward_workspace_size())) != GCA_OK) return st;
  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.kv_bs = kv_batch_stride;
  a.bf16 = dtype == GCA_BF16; a.B = B; a.nQ = nQ; a.nC = nC; a.H = H; a.dh = dh;
  a.idx = idx; a.scores = scores; a.topk = topk; a.shift = shift;
  a.o = o; a.lse = lse; a.err = reinterpret_cast<ErrWord*>(ws);
  cudaError_t e = launch_forward(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_forward launch");
  return GCA_OK;
}

// ==================================================================== window attention and CCA
extern "C" gca_status gca_window_forward(const void* q, const void* k, const void* v, gca_dtype dtype, int B,
                                         int L, int H, int dh, int window, void* o, float* lse, int accumulate,
                                         void* ws, size_t ws_bytes, gca_stream_t stream) {
  if (dtype != GCA_F32 && dtype != GCA_BF16) return fail(GCA_ERR_INVALID_ARG, "dtype must be GCA_F32 or GCA_BF16");
  if (B < 1 || H < 1 || L < 64 || L % 64) return fail(GCA_ERR_INVALID_ARG, "B, H >= 1 and L a positive multiple of 64");
  if (dh != 32 && dh != 64) return fail(GCA_ERR_UNSUPPORTED, "dh must be 32 or 64");
  if (window < 64 || window % 64 || window > 63 * 64)
    return fail(GCA_ERR_UNSUPPORTED, "window must be a multiple of 64 in 64..4032");
  if (L / 64 > 65535 || B > 65535 || H > 65535) return fail(GCA_ERR_UNSUPPORTED, "L/64, B and H must be <= 65535");
  if (!q || !k || !v || !o || !lse) return fail(GCA_ERR_INVALID_ARG, "a pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(GCA_ERR_INVALID_ARG, "q, k, v, o, lse must be 16-byte aligned");
  gca_status st;
  if ((st = check_ws(ws, ws_bytes, gca_forward_workspace_size())) != GCA_OK) return st;
  BlockAttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.kv_bs = (int64_t)L * H * dh;
  a.bf16 = dtype == GCA_BF16; a.B = B; a.nQ = L / 64; a.nC = L / 64; a.H = H; a.dh = dh;
  a.mode = 0; a.window = window; a.o = o; a.lse = lse; a.accumulate = accumulate ? 1 : 0;
  a.err = reinterpret_cast<ErrWord*>(ws);
  cudaError_t e = launch_block_attn(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_window_forward launch");
  return GCA_OK;
}

extern "C" size_t gca_window_backward_workspace_size(int B, int L, int H) {
  if (B < 1 || L < 64 || H < 1) return kErrBytes;
  return kErrBytes + align256((size_t)B * (L / 64) * H * 64 * 4);
}

extern "C" gca_status gca_window_backward(const void* q, const void* k, const void* v, const void* o,
                                          const void* dout, const float* lse, gca_dtype dtype, int B, int L, int H,
                                          int dh, int window, void* dq, void* dk, void* dv, int accumulate,
                                          void* ws, size_t ws_bytes, gca_stream_t stream) {
  if (dtype != GCA_F32 && dtype != GCA_BF16) return fail(GCA_ERR_INVALID_ARG, "dtype must be GCA_F32 or GCA_BF16");
  if (B < 1 || H < 1 || L < 64 || L % 64) return fail(GCA_ERR_INVALID_ARG, "B, H >= 1 and L a positive multiple of 64");
  if (dh != 32 && dh != 64) return fail(GCA_ERR_UNSUPPORTED, "dh must be 32 or 64");
  if (window < 64 || window % 64 || window > 63 * 64)
    return fail(GCA_ERR_UNSUPPORTED, "window must be a multiple of 64 in 64..4032");
  if (L / 64 > 65535 || B > 65535 || H > 65535) return fail(GCA_ERR_UNSUPPORTED, "L/64, B and H must be <= 65535");
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return fail(GCA_ERR_INVALID_ARG, "a pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(GCA_ERR_INVALID_ARG, "all tensors must be 16-byte aligned");
  gca_status st;
  if ((st = check_ws(ws, ws_bytes, gca_window_backward_workspace_size(B, L, H))) != GCA_OK) return st;
  WindowBwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dout; a.lse = lse;
  a.Dbuf = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kErrBytes);
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.bf16 = dtype == GCA_BF16; a.B = B; a.nQ = L / 64; a.H = H; a.dh = dh; a.window = window;
  a.mode = 0; a.nC = a.nQ;
  a.accumulate = accumulate ? 1 : 0;
  a.err = reinterpret_cast<ErrWord*>(ws);
  cudaError_t e = launch_window_backward(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_window_backward launch");
  return GCA_OK;
}

extern "C" gca_status gca_cca_forward(const void* q, const void* k, const void* v, int64_t kv_batch_stride,
                                      gca_dtype dtype, int B, int nQ, int nC, int H, int dh, const int32_t* idx,
                                      int topk, int shift, void* o, float* lse, int accumulate, void* ws,
                                      size_t ws_bytes, gca_stream_t stream) {
  gca_status st = check_gca(q, k, v, dtype, B, nQ, nC, H, dh, idx, nullptr, topk, shift, false);
  if (st != GCA_OK) return st;
  if (!o || !lse) return fail(GCA_ERR_INVALID_ARG, "o/lse pointer is NULL");
  if (!aligned16(o) || !aligned16(lse)) return fail(GCA_ERR_INVALID_ARG, "o/lse must be 16-byte aligned");
  const int64_t per_seq = (int64_t)nC * 64 * H * dh;
  if (kv_batch_stride != 0 && (kv_batch_stride < per_seq || kv_batch_stride % 8))
    return fail(GCA_ERR_INVALID_ARG, "kv_batch_stride must be 0 or >= nC*64*H*dh and a multiple of 8");
  if ((st = check_ws(ws, ws_bytes, gca_forward_workspace_size())) != GCA_OK) return st;
  BlockAttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.kv_bs = kv_batch_stride;
  a.bf16 = dtype == GCA_BF16; a.B = B; a.nQ = nQ; a.nC = nC; a.H = H; a.dh = dh;
  a.mode = 1; a.idx = idx; a.topk = topk; a.shift = shift;
  a.o = o; a.lse = lse; a.accumulate = accumulate ? 1 : 0;
  a.err = reinterpret_cast<ErrWord*>(ws);
  cudaError_t e = launch_block_attn(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_cca_forward launch");
  return GCA_OK;
}

// ==================================================================== CCA backward
extern "C" size_t gca_cca_backward_workspace_size(int B, int nQ, int nC, int H, int topk) {
  if (B < 1 || nQ < 1 || nC < 1 || H < 1 || topk < 1) return kErrBytes;
  return kErrBytes + align256((size_t)B * nQ * H * 64 * 4) + align256((size_t)B * (nC + 1) * 4) +
         align256((size_t)B * nQ * topk * 4) + align256((size_t)B * nC * 4);
}

extern "C" gca_status gca_cca_backward(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                       const float* lse, gca_dtype dtype, int B, int nQ, int nC, int H, int dh,
                                       const int32_t* idx, int topk, int shift, void* dq, void* dk, void* dv,
                                       int accumulate, void* ws, size_t ws_bytes, gca_stream_t stream) {
  gca_status st = check_gca(q, k, v, dtype, B, nQ, nC, H, dh, idx, nullptr, topk, shift, false);
  if (st != GCA_OK) return st;
  if (!o || !dout || !lse || !dq || !dk || !dv) return fail(GCA_ERR_INVALID_ARG, "a pointer is NULL");
  if (!aligned16(o) || !aligned16(dout) || !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(GCA_ERR_INVALID_ARG, "all tensors must be 16-byte aligned");
  if ((st = check_ws(ws, ws_bytes, gca_cca_backward_workspace_size(B, nQ, nC, H, topk))) != GCA_OK) return st;
  unsigned char* base = static_cast<unsigned char*>(ws) + kErrBytes;
  WindowBwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dout; a.lse = lse;
  a.Dbuf = reinterpret_cast<float*>(base);
  base += align256((size_t)B * nQ * H * 64 * 4);
  a.csr_off = reinterpret_cast<int32_t*>(base);
  base += align256((size_t)B * (nC + 1) * 4);
  a.csr_ent = reinterpret_cast<int32_t*>(base);
  base += align256((size_t)B * nQ * topk * 4);
  a.csr_cur = reinterpret_cast<int32_t*>(base);
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.bf16 = dtype == GCA_BF16; a.B = B; a.nQ = nQ; a.H = H; a.dh = dh; a.window = 64;
  a.mode = 1; a.nC = nC; a.idx = idx; a.topk = topk; a.shift = shift;
  a.accumulate = accumulate ? 1 : 0;
  a.err = reinterpret_cast<ErrWord*>(ws);
  cudaError_t e = launch_window_backward(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_cca_backward launch");
  return GCA_OK;
}

// ==================================================================== chunk encoder
extern "C" size_t gca_chunk_encoder_workspace_size(int B, int nC, int d) {
  if (B < 1 || nC < 1 || d < 1) return kErrBytes;
  const size_t M = (size_t)B * nC * 65;
  return kErrBytes + 2 * align256(M * d * 2) + align256(M * 4 * d * 2);
}

extern "C" gca_status gca_chunk_encoder_forward(const void* x, gca_dtype dtype, int B, int nC, int d, int H,
                                                const gca_encoder_weights* w, void* y, void* k, void* v,
                                                void* k_lmk, void* ws, size_t ws_bytes, gca_stream_t stream) {
  if (dtype != GCA_F32 && dtype != GCA_BF16) return fail(GCA_ERR_INVALID_ARG, "dtype must be GCA_F32 or GCA_BF16");
  if (dtype != GCA_BF16) return fail(GCA_ERR_UNSUPPORTED, "the encoder runs in bf16 only");
  if (B < 1 || nC < 1 || H < 1) return fail(GCA_ERR_INVALID_ARG, "B, nC, H must be >= 1");
  if (d % 128 || d < 128 || d > 1024) return fail(GCA_ERR_UNSUPPORTED, "d must be a multiple of 128 in 128..1024");
  if (d != 64 * H) return fail(GCA_ERR_UNSUPPORTED, "the encoder's head dim d / H must be 64");
  if ((int64_t)B * nC > (int64_t)INT32_MAX / 65) return fail(GCA_ERR_UNSUPPORTED, "B * nC * 65 must fit in int32");
  if (!w) return fail(GCA_ERR_INVALID_ARG, "weights pointer is NULL");
  const void* ptrs[] = {x, y, k, v, k_lmk, w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o,
                        w->ln2_g, w->ln2_b, w->w_1, w->b_1, w->w_2, w->b_2, w->w_kv};
  for (const void* p : ptrs) {
    if (!p) return fail(GCA_ERR_INVALID_ARG, "a pointer is NULL");
    if (!aligned16(p)) return fail(GCA_ERR_INVALID_ARG, "all tensors must be 16-byte aligned");
  }
  gca_status st;
  if ((st = check_ws(ws, ws_bytes, gca_chunk_encoder_workspace_size(B, nC, d))) != GCA_OK) return st;
  const size_t M = (size_t)B * nC * 65;
  unsigned char* base = static_cast<unsigned char*>(ws) + kErrBytes;
  EncoderArgs a{};
  a.x = x; a.B = B; a.nC = nC; a.d = d; a.H = H;
  a.ln1_g = w->ln1_g; a.ln1_b = w->ln1_b; a.b_qkv = w->b_qkv; a.b_o = w->b_o;
  a.ln2_g = w->ln2_g; a.ln2_b = w->ln2_b; a.b_1 = w->b_1; a.b_2 = w->b_2;
  a.w_qkv = w->w_qkv; a.w_o = w->w_o; a.w_1 = w->w_1; a.w_2 = w->w_2; a.w_kv = w->w_kv;
  a.y = y; a.k = k; a.v = v; a.k_lmk = k_lmk;
  a.bufA = base;
  a.bufU = base + align256(M * d * 2);
  a.bufF = base + 2 * align256(M * d * 2);
  a.err = reinterpret_cast<ErrWord*>(ws);
  cudaError_t e = launch_chunk_encoder(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_chunk_encoder_forward launch");
  return GCA_OK;
}

// ==================================================================== chunk gather
extern "C" size_t gca_gather_workspace_size(void) { return kErrBytes; }

extern "C" gca_status gca_gather_chunks(const void* k_src, const void* v_src, int64_t src_batch_stride,
                                        gca_dtype dtype, int B, int nQ, int nC, int H, int dh,
                                        const int32_t* idx, int topk, void* k_dst, void* v_dst,
                                        int32_t* idx_local, void* ws, size_t ws_bytes, gca_stream_t stream) {
  if (dtype != GCA_F32 && dtype != GCA_BF16) return fail(GCA_ERR_INVALID_ARG, "dtype must be GCA_F32 or GCA_BF16");
  if (B < 1 || nQ < 1 || nC < 1 || H < 1) return fail(GCA_ERR_INVALID_ARG, "B, nQ, nC, H must be >= 1");
  if (topk < 1 || topk > kMaxTopk) return fail(GCA_ERR_UNSUPPORTED, "topk must be in 1..%d", kMaxTopk);
  if (dh != 32 && dh != 64) return fail(GCA_ERR_UNSUPPORTED, "dh must be 32 or 64");
  if (!k_src || !v_src || !idx || !k_dst || !v_dst || !idx_local)
    return fail(GCA_ERR_INVALID_ARG, "a pointer is NULL");
  if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_dst) || !aligned16(v_dst))
    return fail(GCA_ERR_INVALID_ARG, "k/v source and destination must be 16-byte aligned");
  const int64_t per_seq = (int64_t)nC * 64 * H * dh;
  if (src_batch_stride != 0 && (src_batch_stride < per_seq || src_batch_stride % 8))
    return fail(GCA_ERR_INVALID_ARG, "src_batch_stride must be 0 or >= nC*64*H*dh and a multiple of 8");
  if ((int64_t)nQ * topk > 65535 || B > 65535) return fail(GCA_ERR_UNSUPPORTED, "nQ*topk and B must be <= 65535");
  gca_status st;
  if ((st = check_ws(ws, ws_bytes, gca_gather_workspace_size())) != GCA_OK) return st;
  GatherArgs a{};
  a.k_src = k_src; a.v_src = v_src; a.src_bs = src_batch_stride;
  a.esize = dtype == GCA_BF16 ? 2 : 4; a.B = B; a.nQ = nQ; a.nC = nC; a.H = H; a.dh = dh; a.topk = topk;
  a.idx = idx; a.k_dst = k_dst; a.v_dst = v_dst; a.idx_local = idx_local;
  a.err = reinterpret_cast<ErrWord*>(ws);
  cudaError_t e = launch_gather(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_gather_chunks launch");
  return GCA_OK;
}

// ==================================================================== GCA backward
namespace {
struct BwdLayout {
  size_t D, dwp, off, ent, cur, wrow, ctr, total;
};
BwdLayout bwd_layout(int B, int nQ, int nC, int H, int topk) {
  BwdLayout L{};
  size_t p = kErrBytes;
  L.D = p; p += align256((size_t)B * nQ * H * topk * 64 * 4);
  L.dwp = p; p += align256((size_t)B * nQ * H * topk * 4);
  L.off = p; p += align256((size_t)B * (nC + 1) * 4);
  L.ent = p; p += align256((size_t)B * nQ * topk * 4);
  L.cur = p; p += align256((size_t)B * nC * 4);
  L.wrow = p; p += align256((size_t)B * nQ * topk * 4);
  L.ctr = p; p += 256;
  L.total = p;
  return L;
}
}  // namespace

extern "C" size_t gca_backward_workspace_size(int B, int nQ, int nC, int H, int topk) {
  if (B < 1 || nQ < 1 || nC < 1 || H < 1 || topk < 1) return kErrBytes;
  return bwd_layout(B, nQ, nC, H, topk).total;
}

extern "C" gca_status gca_backward(const void* q, const void* k, const void* v, gca_dtype dtype, int B, int nQ,
                                   int nC, int H, int dh, const int32_t* idx, const float* scores, int topk,
                                   int shift, const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                   float* dscores, int accumulate_dkv, void* ws, size_t ws_bytes,
                                   gca_stream_t stream) {
  gca_status st = check_gca(q, k, v, dtype, B, nQ, nC, H, dh, idx, scores, topk, shift);
  if (st != GCA_OK) return st;
  if (!dout || !lse || !dq || !dk || !dv || !dscores) return fail(GCA_ERR_INVALID_ARG, "output/gradient pointer is NULL");
  if (!aligned16(dout) || !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(GCA_ERR_INVALID_ARG, "dout/lse/dq/dk/dv must be 16-byte aligned");
  if ((st = check_ws(ws, ws_bytes, gca_backward_workspace_size(B, nQ, nC, H, topk))) != GCA_OK) return st;
  BwdLayout L = bwd_layout(B, nQ, nC, H, topk);
  unsigned char* w = static_cast<unsigned char*>(ws);
  BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.bf16 = dtype == GCA_BF16;
  a.B = B; a.nQ = nQ; a.nC = nC; a.H = H; a.dh = dh;
  a.idx = idx; a.scores = scores; a.topk = topk; a.shift = shift;
  a.dout = dout; a.lse = lse; a.dq = dq; a.dk = dk; a.dv = dv; a.dscores = dscores;
  a.acc_dkv = accumulate_dkv ? 1 : 0;
  a.err = reinterpret_cast<ErrWord*>(ws);
  a.Dbuf = reinterpret_cast<float*>(w + L.D);
  a.dwp = reinterpret_cast<float*>(w + L.dwp);
  a.csr_off = reinterpret_cast<int32_t*>(w + L.off);
  a.csr_ent = reinterpret_cast<int32_t*>(w + L.ent);
  a.csr_cur = reinterpret_cast<int32_t*>(w + L.cur);
  a.wrow = reinterpret_cast<float*>(w + L.wrow);
  a.kv_ctr = reinterpret_cast<int32_t*>(w + L.ctr);
  cudaError_t e = launch_backward(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_backward launch");
  return GCA_OK;
}

// ==================================================================== landmark gradients
namespace {
struct SbLayout {
  size_t off, ent, cur, total;
};
SbLayout sb_layout(int B, int nQ, int nC, int topk) {
  SbLayout L{};
  size_t p = kErrBytes;
  L.off = p; p += align256((size_t)B * (nC + 1) * 4);
  L.ent = p; p += align256((size_t)B * nQ * topk * 4);
  L.cur = p; p += align256((size_t)B * nC * 4);
  L.total = p;
  return L;
}
}  // namespace

extern "C" size_t gca_scores_backward_workspace_size(int B, int nQ, int nC, int topk) {
  if (B < 1 || nQ < 1 || nC < 1 || topk < 1) return kErrBytes;
  return sb_layout(B, nQ, nC, topk).total;
}

extern "C" gca_status gca_scores_backward(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride,
                                          const void* k_lmk, int64_t k_batch_stride, gca_dtype dtype, int B,
                                          int nQ, int nC, int D, const int32_t* idx, const float* dscores,
                                          int topk, void* dq_lmk, gca_dtype dq_dtype, int64_t dq_row_stride,
                                          int64_t dq_batch_stride, int dq_accumulate, float* dk_lmk, void* ws,
                                          size_t ws_bytes, gca_stream_t stream) {
  gca_status st = check_landmarks(q_lmk, q_row_stride, q_batch_stride, k_lmk, k_batch_stride, dtype, B, nQ,
                                  nC, D, topk);
  if (st != GCA_OK) return st;
  if (k_batch_stride == 0 && B > 1) return fail(GCA_ERR_INVALID_ARG, "k_batch_stride may not be 0 here");
  if (!idx || !dscores || !dq_lmk || !dk_lmk) return fail(GCA_ERR_INVALID_ARG, "pointer is NULL");
  if (dq_dtype != GCA_F32 && dq_dtype != GCA_BF16) return fail(GCA_ERR_INVALID_ARG, "dq_dtype must be GCA_F32 or GCA_BF16");
  if (dq_row_stride < D || dq_batch_stride < 0) return fail(GCA_ERR_INVALID_ARG, "dq strides out of range");
  if ((st = check_ws(ws, ws_bytes, gca_scores_backward_workspace_size(B, nQ, nC, topk))) != GCA_OK) return st;
  SbLayout L = sb_layout(B, nQ, nC, topk);
  unsigned char* w = static_cast<unsigned char*>(ws);
  ScoresBwdArgs a{};
  a.q = q_lmk; a.q_rs = q_row_stride; a.q_bs = q_batch_stride;
  a.k = k_lmk; a.k_bs = k_batch_stride;
  a.bf16 = dtype == GCA_BF16; a.B = B; a.nQ = nQ; a.nC = nC; a.D = D;
  a.idx = idx; a.ds = dscores; a.topk = topk;
  a.dq = dq_lmk; a.dq_bf16 = dq_dtype == GCA_BF16; a.dq_rs = dq_row_stride; a.dq_bs = dq_batch_stride;
  a.dq_acc = dq_accumulate ? 1 : 0; a.dk = dk_lmk;
  a.err = reinterpret_cast<ErrWord*>(ws);
  a.csr_off = reinterpret_cast<int32_t*>(w + L.off);
  a.csr_ent = reinterpret_cast<int32_t*>(w + L.ent);
  a.csr_cur = reinterpret_cast<int32_t*>(w + L.cur);
  cudaError_t e = launch_scores_backward(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_scores_backward launch");
  return GCA_OK;
}

// ==================================================================== errors, instrumentation
extern "C" gca_status gca_check_error(void* ws, gca_stream_t stream, int* bad_value) {
  if (!ws) return fail(GCA_ERR_WORKSPACE, "workspace pointer is NULL");
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gca_check_error sync");
  ErrWord h{};
  e = cudaMemcpy(&h, ws, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "gca_check_error read");
  if (h.flags == 0) return GCA_OK;
  const ErrWord zero{};
  e = cudaMemcpy(ws, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "gca_check_error clear");
  if (h.flags & kErrTimeout)
    return fail(GCA_ERR_TIMEOUT,
                "a bounded wait for tensor-core or copy completion ran out (wait sites 0x%x; first: site %d, "
                "CTA %d, tile %d, slot %d)",
                (unsigned)h.wait_sites, h.first[0] - 1, h.first[1], h.first[2], h.first[3]);
  if (bad_value) *bad_value = h.bad_value;
  return fail(GCA_ERR_DEVICE_INDEX, "a kernel met retrieved index %d outside [-1, nC)", h.bad_value);
}

// ==================================================================== wait self-test
namespace gca {
namespace {
constexpr int kSelftestSite = 30;

// One CTA waits on an mbarrier that nothing arrives at, with the same bounded wait the
// kernels use for tensor-core and copy completion: the wait runs out, every thread records
// the timeout in the error word, and the CTA exits normally.
__global__ void __launch_bounds__(32) selftest_timeout_kernel(ErrWord* err, uint32_t spins) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncwarp();
  if (!tc::mbar_wait(&bar, 0, spins)) flag_timeout(err, kSelftestSite, blockIdx.x, -1, threadIdx.x);
}
}  // namespace
}  // namespace gca

extern "C" gca_status gca_selftest_timeout(void* ws, size_t ws_bytes, uint32_t spins, gca_stream_t stream) {
  gca_status st;
  if ((st = check_ws(ws, ws_bytes, kErrBytes)) != GCA_OK) return st;
  if (spins < 1 || spins > (1u << 20)) return fail(GCA_ERR_INVALID_ARG, "spins must be in 1..2^20");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  launch_begin("selftest_timeout", s);
  gca::selftest_timeout_kernel<<<1, 32, 0, s>>>(reinterpret_cast<ErrWord*>(ws), spins);
  cudaError_t e = launch_end("selftest_timeout", s);
  if (e != cudaSuccess) return cuda_fail(e, "gca_selftest_timeout launch");
  return GCA_OK;
}

extern "C" uint64_t gca_launch_count(void) { return g_launches.load(); }

extern "C" gca_status gca_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof = true;
  return GCA_OK;
}

extern "C" int gca_profile_end(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof = false;
  g_table.clear();
  for (auto& r : g_open) {
    float ms = 0.f;
    cudaEventSynchronize(r.b);
    cudaEventElapsedTime(&ms, r.a, r.b);
    Row* row = nullptr;
    for (auto& t : g_table)
      if (t.name == r.name) row = &t;
    if (!row) {
      g_table.push_back(Row{r.name, 0, 0.0});
      row = &g_table.back();
    }
    row->launches += 1;
    row->ms += ms;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_open.clear();
  return (int)g_table.size();
}

extern "C" gca_status gca_profile_row(int i, const char** name, int* launches, double* total_ms) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (i < 0 || i >= (int)g_table.size()) return fail(GCA_ERR_INVALID_ARG, "profile row out of range");
  if (name) *name = g_table[i].name.c_str();
  if (launches) *launches = g_table[i].launches;
  if (total_ms) *total_ms = g_table[i].ms;
  return GCA_OK;
}
