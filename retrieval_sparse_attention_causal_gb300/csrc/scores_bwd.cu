// Gradient of the retrieval scores s_im = <q_lmk_i, k_lmk_j> / sqrt(D), j = idx[i,m], into
// both landmark sets.  The scores get their gradient from the fusion weights (Paper-Notes
// page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", 关键设计 / key design, "Grouped Cross-Attention");
// the Gumbel noise only chose the slots and has no gradient.
//
// One launch, lmk_grad_kernel: CTAs 0 .. nQ-1 (per sequence) each take a query row, the
// sum over its k slots of ds * k_lmk[j]; CTAs nQ .. nQ+nC-1 each take a key chunk, the sum
// over the entries (i, m) with idx = j, in increasing entry order, of ds * q_lmk[i].  The
// two halves are independent; sharing the launch fills the GPU with both at once.
//
// A key chunk finds its entries by scanning the sequence's whole index array itself when
// that has at most kScanMax entries: thread t holds entries t + 256 r (r < 8), and per
// round a ballot, per-warp counts and one prefix place the matches in entry order.
// Longer arrays go through the stable CSR, built by a launch before.  Both give the same
// entries in the same order, so the same sums.  Rows go as 16-byte vectors when the
// pointers and strides allow it; the order of every sum is the same either way.
#include "common.cuh"
#include "internal.h"

namespace gca {
namespace {

constexpr int kScanMax = 2048;  // index entries per sequence up to which a key chunk scans

// Output-row vectors of V consecutive elements (V = 16 / sizeof(input element)).
template <int V> __device__ __forceinline__ void ld_out(const float* p, float* x) {
#pragma unroll
  for (int t = 0; t < V; t += 4) {
    const float4 f = *reinterpret_cast<const float4*>(p + t);
    x[t] = f.x; x[t + 1] = f.y; x[t + 2] = f.z; x[t + 3] = f.w;
  }
}
template <int V> __device__ __forceinline__ void ld_out(const __nv_bfloat16* p, float* x) {
  uint32_t w[V / 2];
  if constexpr (V == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    w[0] = u.x; w[1] = u.y;
  }
#pragma unroll
  for (int t = 0; t < V / 2; ++t) {
    x[2 * t] = __uint_as_float(w[t] << 16);
    x[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
  }
}
template <int V> __device__ __forceinline__ void st_out(float* p, const float* x) {
#pragma unroll
  for (int t = 0; t < V; t += 4) *reinterpret_cast<float4*>(p + t) = make_float4(x[t], x[t + 1], x[t + 2], x[t + 3]);
}
template <int V> __device__ __forceinline__ void st_out(__nv_bfloat16* p, const float* x) {
  uint32_t w[V / 2];
#pragma unroll
  for (int t = 0; t < V / 2; ++t) w[t] = pack_bf16(x[2 * t], x[2 * t + 1]);
  if constexpr (V == 8) *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  else *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
}

template <typename T, typename TO, bool VEC>
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
  if constexpr (VEC) {
    constexpr int V = Elem<T>::kVec;
    for (int d = threadIdx.x * V; d < a.D; d += blockDim.x * V) {
      float acc[V];
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = 0.f;
      for (int m0 = 0; m0 < a.topk; m0 += 8) {  // eight slots' rows in flight at once
        uint4 raw[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int m = m0 + u, j = m < a.topk ? j_s[m] : -1;
          if (j >= 0) raw[u] = *reinterpret_cast<const uint4*>(kb + (int64_t)j * a.D + d);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int m = m0 + u;
          if (m < a.topk && j_s[m] >= 0) {
            float x[V];
            unpack16(raw[u], x, (const T*)nullptr);
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = fmaf(ds_s[m], x[e], acc[e]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] *= inv;
      if (a.dq_acc) {
        float o[V];
        ld_out<V>(out + d, o);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] += o[e];
      }
      st_out<V>(out + d, acc);
    }
  } else {
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
}

// Entries (row, score gradient) of key chunk j, in increasing entry order, from a scan of
// the sequence's index array (n <= kScanMax entries); returns how many.
__device__ __forceinline__ int scan_consumers(const ScoresBwdArgs& a, int j, int b, int* row_s, float* ds_s) {
  __shared__ int off_s[kScanMax / 32];  // per (round, warp): entries before it
  __shared__ int total_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.nQ * a.topk, nw = blockDim.x >> 5, rounds = (n + blockDim.x - 1) / blockDim.x;
  const int32_t* ib = a.idx + (int64_t)b * n;
  const float* db = a.ds + (int64_t)b * n;
  constexpr int R = kScanMax / 256;  // rounds of a 256-thread CTA
  int jr[R];
  float dr[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {  // entry e = tid + 256 r: the rounds in order, lanes in order
    const int e = tid + r * blockDim.x;
    const bool in = r < rounds && e < n;
    jr[r] = in ? ib[e] : -1;
    dr[r] = in ? db[e] : 0.f;
  }
  unsigned bal[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    bal[r] = __ballot_sync(0xffffffffu, jr[r] == j);
    if (lane == 0) off_s[r * nw + warp] = __popc(bal[r]);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix over (round, warp) in that order
    const int slots = R * nw;
    int run = 0;
    for (int base = 0; base < slots; base += 32) {
      const int v = base + lane < slots ? off_s[base + lane] : 0;
      int incl = v;
#pragma unroll
      for (int k = 1; k < 32; k <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, k);
        if (lane >= k) incl += u;
      }
      if (base + lane < slots) off_s[base + lane] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) total_s = run;
  }
  __syncthreads();
  const unsigned below = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (jr[r] == j) {
      const int pos = off_s[r * nw + warp] + __popc(bal[r] & below);
      row_s[pos] = (tid + r * blockDim.x) / a.topk;
      ds_s[pos] = dr[r];
    }
  }
  __syncthreads();
  return total_s;
}

// dk_lmk[j] over consumers [0, nc) held in shared memory, added onto acc (vector path: the
// thread's columns d .. d + V - 1).
template <typename T, int V>
__device__ __forceinline__ void dk_accumulate(const T* qb, int64_t q_rs, int d, const int* row_s, const float* ds_s,
                                              int nc, float* acc) {
  int c = 0;
  for (; c + 4 <= nc; c += 4) {  // four rows in flight
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) raw[u] = *reinterpret_cast<const uint4*>(qb + (int64_t)row_s[c + u] * q_rs + d);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float x[V];
      unpack16(raw[u], x, (const T*)nullptr);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = fmaf(ds_s[c + u], x[e], acc[e]);
    }
  }
  for (; c < nc; ++c) {
    float x[V];
    unpack16(*reinterpret_cast<const uint4*>(qb + (int64_t)row_s[c] * q_rs + d), x, (const T*)nullptr);
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = fmaf(ds_s[c], x[e], acc[e]);
  }
}

template <typename T, bool VEC>
__device__ __forceinline__ void dk_lmk_chunk(const ScoresBwdArgs& a, int j, int b) {
  __shared__ int row_s[kScanMax];
  __shared__ float ds_s[kScanMax];
  const float inv = 1.0f / sqrtf((float)a.D);
  const T* qb = reinterpret_cast<const T*>(a.q) + (int64_t)b * a.q_bs;
  float* out = a.dk + ((int64_t)b * a.nC + j) * a.D;
  if (a.scan) {  // the whole consumer list at once
    const int nc = scan_consumers(a, j, b, row_s, ds_s);
    if constexpr (VEC) {
      constexpr int V = Elem<T>::kVec;
      for (int d = threadIdx.x * V; d < a.D; d += blockDim.x * V) {
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        dk_accumulate<T, V>(qb, a.q_rs, d, row_s, ds_s, nc, acc);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] *= inv;
        st_out<V>(out + d, acc);
      }
    } else {
      for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
        float acc = 0.f;
        for (int c = 0; c < nc; ++c) acc = fmaf(ds_s[c], Elem<T>::ld(qb + (int64_t)row_s[c] * a.q_rs + d), acc);
        out[d] = acc * inv;
      }
    }
    return;
  }
  // From the CSR, 256 consumers at a time; the partial sums wait in the output row.
  const int e0 = a.csr_off[(int64_t)b * (a.nC + 1) + j];
  const int e1 = a.csr_off[(int64_t)b * (a.nC + 1) + j + 1];
  const int32_t* ent = a.csr_ent + (int64_t)b * a.nQ * a.topk;
  for (int c0 = e0; c0 < e1; c0 += 256) {
    const int nc = min(256, e1 - c0);
    __syncthreads();
    if (threadIdx.x < nc) {
      const int e = ent[c0 + threadIdx.x];
      row_s[threadIdx.x] = e / a.topk;
      ds_s[threadIdx.x] = a.ds[(int64_t)b * a.nQ * a.topk + e];
    }
    __syncthreads();
    if constexpr (VEC) {
      constexpr int V = Elem<T>::kVec;
      for (int d = threadIdx.x * V; d < a.D; d += blockDim.x * V) {
        float acc[V];
        if (c0 == e0) {
#pragma unroll
          for (int e = 0; e < V; ++e) acc[e] = 0.f;
        } else {
          ld_out<V>(out + d, acc);
        }
        dk_accumulate<T, V>(qb, a.q_rs, d, row_s, ds_s, nc, acc);
        st_out<V>(out + d, acc);
      }
    } else {
      for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
        float x = c0 == e0 ? 0.f : out[d];
        for (int c = 0; c < nc; ++c) x = fmaf(ds_s[c], Elem<T>::ld(qb + (int64_t)row_s[c] * a.q_rs + d), x);
        out[d] = x;
      }
    }
  }
  __syncthreads();
  for (int d = threadIdx.x; d < a.D; d += blockDim.x) out[d] = e1 > e0 ? out[d] * inv : 0.f;
}

template <typename T, typename TO, bool VEC>
__global__ void __launch_bounds__(256) lmk_grad_kernel(ScoresBwdArgs a) {
  const int x = blockIdx.x, b = blockIdx.y;
  if (x < a.nQ) dq_lmk_row<T, TO, VEC>(a, x, b);
  else dk_lmk_chunk<T, VEC>(a, x - a.nQ, b);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename T, typename TO>
void launch_lmk(const ScoresBwdArgs& a, bool vec, dim3 grid, cudaStream_t s) {
  if (vec) lmk_grad_kernel<T, TO, true><<<grid, 256, 0, s>>>(a);
  else lmk_grad_kernel<T, TO, false><<<grid, 256, 0, s>>>(a);
}

}  // namespace

cudaError_t launch_scores_backward(const ScoresBwdArgs& a_in, cudaStream_t s) {
  ScoresBwdArgs a = a_in;
  a.scan = (int64_t)a.nQ * a.topk <= kScanMax ? 1 : 0;
  if (!a.scan) {
    cudaError_t e = launch_csr(a.idx, a.B, a.nQ, a.nQ, a.topk, a.nC, a.csr_off, a.csr_ent, a.csr_cur, a.err, s);
    if (e != cudaSuccess) return e;
  }
  // Vector path: every row of q, k, dq and dk starts on a 16-byte boundary.
  const int es = a.bf16 ? 2 : 4, eo = a.dq_bf16 ? 2 : 4;
  const bool vec = (a.D * es) % 16 == 0 && aligned16(a.q) && aligned16(a.k) && aligned16(a.dq) && aligned16(a.dk) &&
                   (a.q_rs * es) % 16 == 0 && (a.q_bs * es) % 16 == 0 && (a.k_bs * es) % 16 == 0 &&
                   (a.dq_rs * eo) % 16 == 0 && (a.dq_bs * eo) % 16 == 0 && a.D % 4 == 0;
  dim3 grid(a.nQ + a.nC, a.B);
  launch_begin("lmk_grads", s);
  if (a.bf16) {
    if (a.dq_bf16) launch_lmk<__nv_bfloat16, __nv_bfloat16>(a, vec, grid, s);
    else launch_lmk<__nv_bfloat16, float>(a, vec, grid, s);
  } else {
    if (a.dq_bf16) launch_lmk<float, __nv_bfloat16>(a, vec, grid, s);
    else launch_lmk<float, float>(a, vec, grid, s);
  }
  return launch_end("lmk_grads", s);
}

}  // namespace gca
