// Gradient of the retrieval scores s_im = <q_lmk_i, k_lmk_j> / sqrt(D), j = idx[i,m], into
// both landmark sets.  The scores get their gradient from the fusion weights (Paper-Notes
// page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", 关键设计 / key design, "Grouped Cross-Attention");
// the Gumbel noise only chose the slots and has no gradient.
//
// One launch, lmk_grad_kernel: CTAs 0 .. nQ-1 (per sequence) each take a query row, the
// sum over its k slots of ds * k_lmk[j]; CTAs nQ .. nQ+nC-1 each take a key chunk, the sum
// over the rows that retrieved it (from the stable CSR, so in a fixed order) of
// ds * q_lmk[i].  The two halves are independent; sharing the launch fills the GPU with
// both at once.
#include "common.cuh"
#include "internal.h"

namespace gca {
namespace {

template <typename T, typename TO>
__device__ __forceinline__ void dq_lmk_row(const ScoresBwdArgs& a, int i, int b) {
  __shared__ int j_s[kMaxTopk];
  __shared__ float ds_s[kMaxTopk];
  if (threadIdx.x < a.topk) {
    const int64_t o = ((int64_t)b * a.nQ + i) * a.topk + threadIdx.x;
    int j = a.idx[o];
    if (j < -1 || j >= a.nC) {
      flag_bad_index(a.err, j);
      j = -1;
    }
    j_s[threadIdx.x] = j;
    ds_s[threadIdx.x] = a.ds[o];
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf((float)a.D);
  const T* kb = reinterpret_cast<const T*>(a.k) + (int64_t)b * a.k_bs;
  TO* out = reinterpret_cast<TO*>(a.dq) + (int64_t)b * a.dq_bs + (int64_t)i * a.dq_rs;
  for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
    float acc = 0.f;
    for (int m = 0; m < a.topk; ++m) {
      const int j = j_s[m];
      if (j >= 0) acc = fmaf(ds_s[m], Elem<T>::ld(kb + (int64_t)j * a.D + d), acc);
    }
    acc *= inv;
    if (a.dq_acc) acc += Elem<TO>::ld(out + d);
    Elem<TO>::st(out + d, acc);
  }
}

template <typename T>
__device__ __forceinline__ void dk_lmk_chunk(const ScoresBwdArgs& a, int j, int b) {
  __shared__ int row_s[256];
  __shared__ float ds_s[256];
  const int e0 = a.csr_off[(int64_t)b * (a.nC + 1) + j];
  const int e1 = a.csr_off[(int64_t)b * (a.nC + 1) + j + 1];
  const int32_t* ent = a.csr_ent + (int64_t)b * a.nQ * a.topk;
  const float inv = 1.0f / sqrtf((float)a.D);
  const T* qb = reinterpret_cast<const T*>(a.q) + (int64_t)b * a.q_bs;
  float* out = a.dk + ((int64_t)b * a.nC + j) * a.D;
  constexpr int kMaxD = 4;  // D <= 1024 in registers; larger D loops below
  float acc[kMaxD] = {0.f, 0.f, 0.f, 0.f};
  // The chunk's consumers (query row, score gradient) go to shared memory 256 at a time,
  // in CSR order, so the sum below has a fixed order and independent loads.
  for (int c0 = e0; c0 < e1; c0 += 256) {
    const int nc = min(256, e1 - c0);
    __syncthreads();
    if (threadIdx.x < nc) {
      const int e = ent[c0 + threadIdx.x];
      row_s[threadIdx.x] = e / a.topk;
      ds_s[threadIdx.x] = a.ds[(int64_t)b * a.nQ * a.topk + e];
    }
    __syncthreads();
    if (a.D <= kMaxD * 256) {
#pragma unroll
      for (int u = 0; u < kMaxD; ++u) {
        const int d = threadIdx.x + 256 * u;
        if (d < a.D)
          for (int c = 0; c < nc; ++c)
            acc[u] = fmaf(ds_s[c], Elem<T>::ld(qb + (int64_t)row_s[c] * a.q_rs + d), acc[u]);
      }
    } else {
      for (int d = threadIdx.x; d < a.D; d += 256) {
        float x = c0 == e0 ? 0.f : out[d];
        for (int c = 0; c < nc; ++c) x = fmaf(ds_s[c], Elem<T>::ld(qb + (int64_t)row_s[c] * a.q_rs + d), x);
        out[d] = x;
      }
    }
  }
  if (a.D <= kMaxD * 256) {
#pragma unroll
    for (int u = 0; u < kMaxD; ++u) {
      const int d = threadIdx.x + 256 * u;
      if (d < a.D) out[d] = acc[u] * inv;
    }
  } else {
    __syncthreads();
    for (int d = threadIdx.x; d < a.D; d += 256) out[d] = e1 > e0 ? out[d] * inv : 0.f;
  }
}

template <typename T, typename TO>
__global__ void __launch_bounds__(256) lmk_grad_kernel(ScoresBwdArgs a) {
  const int x = blockIdx.x, b = blockIdx.y;
  if (x < a.nQ) dq_lmk_row<T, TO>(a, x, b);
  else dk_lmk_chunk<T>(a, x - a.nQ, b);
}

}  // namespace

cudaError_t launch_scores_backward(const ScoresBwdArgs& a, cudaStream_t s) {
  cudaError_t e = launch_csr(a.idx, a.B, a.nQ, a.nQ, a.topk, a.nC, a.csr_off, a.csr_ent, a.csr_cur, a.err, s);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nQ + a.nC, a.B);
  launch_begin("lmk_grads", s);
  if (a.bf16) {
    if (a.dq_bf16) lmk_grad_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, s>>>(a);
    else lmk_grad_kernel<__nv_bfloat16, float><<<grid, 256, 0, s>>>(a);
  } else {
    if (a.dq_bf16) lmk_grad_kernel<float, __nv_bfloat16><<<grid, 256, 0, s>>>(a);
    else lmk_grad_kernel<float, float><<<grid, 256, 0, s>>>(a);
  }
  return launch_end("lmk_grads", s);
}

}  // namespace gca
