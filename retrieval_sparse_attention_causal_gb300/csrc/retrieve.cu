// Causal landmark scoring fused with per-row top-k selection.
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", section 关键设计 / key design: the current chunk's
// landmark scores the landmarks of earlier chunks and the top-k are kept; in training,
// Gumbel noise is added to the scores before the top-k.  The score is the scaled dot
// product <q_i, k_j> / sqrt(D).
//
// Two stage-1 kernels feed one merge kernel:
//   retrieve_rows_kernel  few query rows, very many candidates (decode at 16M context):
//                         each CTA streams a contiguous slice of one row's candidate
//                         landmarks with 16-byte loads straight from HBM, one warp per
//                         candidate row group; an HBM-bound dot-product sweep.
//   retrieve_tile_kernel  many query rows (training, prefill): 64 query rows stay in
//                         shared memory while 64-candidate tiles stream through a
//                         double-buffered cp.async pipeline; the 64x64 score tile is a
//                         bf16 tensor-core product (fp32 SIMT for f32 inputs).
//   retrieve_merge_kernel merges the per-split candidate lists of a row.
// Every stage keeps candidates under one total order (key descending, then index
// ascending), so the result does not depend on how the candidates were split.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gca {

namespace {

constexpr int kRowsThreads = 256;
constexpr int kTileThreads = 256;
constexpr int kTargetCtas = 152 * 4;  // four resident CTAs on each of GB300's 152 SMs

__device__ __forceinline__ int n_cand_row(int i, int off, int nC) {
  long long n = (long long)i + off;
  if (n < 0) n = 0;
  if (n > nC) n = nC;
  return (int)n;
}

__device__ __forceinline__ void write_row(const RetrieveArgs& a, int b, int i, const Cand* sel) {
  int32_t* idx = a.idx + ((int64_t)b * a.nQ + i) * a.topk;
  float* sc = a.scores + ((int64_t)b * a.nQ + i) * a.topk;
  for (int r = 0; r < a.topk; ++r) {
    const bool ok = sel[r].j != 0x7fffffff;
    idx[r] = ok ? sel[r].j : -1;
    sc[r] = ok ? sel[r].score : -CUDART_INF_F;
  }
}

__device__ __forceinline__ void write_part(const RetrieveArgs& a, int nsplit, int b, int i,
                                           int split, const Cand* sel) {
  Cand* p = reinterpret_cast<Cand*>(a.part) +
            (((int64_t)b * a.nQ + i) * nsplit + split) * a.topk;
  for (int r = 0; r < a.topk; ++r) p[r] = sel[r];
}

// ------------------------------------------------------------------ rows kernel
template <typename T, int NVMAX, int KC>
__global__ void __launch_bounds__(kRowsThreads)
retrieve_rows_kernel(RetrieveArgs a, int nsplit, int seg) {
  constexpr int EPV = 16 / sizeof(T);
  __shared__ Cand red[kRowsThreads / 32];
  __shared__ Cand sel[kMaxTopk];
  const int split = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = kRowsThreads / 32;
  const int n_i = n_cand_row(i, a.off, a.nC);
  const int j0 = split * seg;
  const int j1 = min(n_i, j0 + seg);
  const T* q = reinterpret_cast<const T*>(a.q) + (int64_t)b * a.q_bs + (int64_t)i * a.q_rs;
  const T* kb = reinterpret_cast<const T*>(a.k) + (int64_t)b * a.k_bs;
  const int nvec = a.D / EPV;
  const float inv = 1.0f / sqrtf((float)a.D);

  float qf[NVMAX][EPV];
#pragma unroll
  for (int t = 0; t < NVMAX; ++t) {
    const int vi = lane + 32 * t;
    if (vi < nvec) {
      const uint4 u = *reinterpret_cast<const uint4*>(q + vi * EPV);
      unpack16(u, qf[t], (const T*)nullptr);
    } else {
#pragma unroll
      for (int e = 0; e < EPV; ++e) qf[t][e] = 0.f;
    }
  }

  Cand L[KC];
  list_init(L);
  constexpr int R = 4;  // candidate rows in flight per warp
  for (int jb = j0 + warp * R; jb < j1; jb += nwarp * R) {
    uint4 raw[R][NVMAX];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j = jb + r;
#pragma unroll
      for (int t = 0; t < NVMAX; ++t) {
        const int vi = lane + 32 * t;
        if (j < j1 && vi < nvec)
          raw[r][t] = ldg_stream(kb + (int64_t)j * a.D + vi * EPV);
        else
          raw[r][t] = make_uint4(0, 0, 0, 0);
      }
    }
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float s = 0.f;
#pragma unroll
      for (int t = 0; t < NVMAX; ++t) {
        float f[EPV];
        unpack16(raw[r][t], f, (const T*)nullptr);
#pragma unroll
        for (int e = 0; e < EPV; ++e) s = fmaf(qf[t][e], f[e], s);
      }
      acc[r] = s;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], m);
    }
    if (lane < R) {
      const int j = jb + lane;
      float mine = acc[0];
#pragma unroll
      for (int r = 1; r < R; ++r) mine = (lane == r) ? acc[r] : mine;
      if (j < j1) {
        Cand c;
        c.score = mine * inv;
        c.key = a.gumbel ? c.score + gumbel_noise(a.seed, a.group, b, i, j) : c.score;
        c.j = j;
        list_insert(L, c);
      }
    }
  }
  block_select(L, a.topk, sel, red);
  if (threadIdx.x == 0) {
    if (nsplit == 1) write_row(a, b, i, sel);
    else write_part(a, nsplit, b, i, split, sel);
  }
}

// ------------------------------------------------------------------ merge kernel
template <int KC>
__global__ void __launch_bounds__(128) retrieve_merge_kernel(RetrieveArgs a, int nsplit) {
  __shared__ Cand red[4];
  __shared__ Cand sel[kMaxTopk];
  const int i = blockIdx.x, b = blockIdx.y;
  const Cand* p = reinterpret_cast<const Cand*>(a.part) + ((int64_t)b * a.nQ + i) * nsplit * a.topk;
  Cand L[KC];
  list_init(L);
  const int n = nsplit * a.topk;
  for (int c = threadIdx.x; c < n; c += blockDim.x) {
    const Cand x = p[c];
    if (x.j != 0x7fffffff) list_insert(L, x);
  }
  block_select(L, a.topk, sel, red);
  if (threadIdx.x == 0) write_row(a, b, i, sel);
}

// ------------------------------------------------------------------ tile kernel
// Shared memory: Q block (64 rows x D), two candidate chunk buffers, score tile.
struct TileSmem {
  static constexpr int kSt = 65;  // padded score-tile row (floats)
  static size_t bytes(int D, bool bf16) {
    if (bf16) return (size_t)64 * D * 2 + 2 * 64 * 128 + 64 * kSt * 4 + 1024;
    return (size_t)64 * (D + 1) * 4 + 64 * 33 * 4 + 64 * kSt * 4 + 1024;
  }
};

// Top-k phase over one 64x64 score tile held in shared memory.  Thread t owns row t/4
// and the 16 candidates of quarter t%4.
template <int KC>
__device__ __forceinline__ void tile_topk(const RetrieveArgs& a, const float* St, int b,
                                          int row0, int tile0, int j1, float inv, Cand (&L)[KC]) {
  const int rl = threadIdx.x >> 2, quarter = threadIdx.x & 3;
  const int i = row0 + rl;
  if (i >= a.nQ) return;
  const int lim = min(j1, n_cand_row(i, a.off, a.nC));
#pragma unroll 4
  for (int cc = 0; cc < 16; ++cc) {
    const int jl = quarter * 16 + cc;
    const int j = tile0 + jl;
    if (j < lim) {
      Cand c;
      c.score = St[rl * TileSmem::kSt + jl] * inv;
      c.key = a.gumbel ? c.score + gumbel_noise(a.seed, a.group, b, i, j) : c.score;
      c.j = j;
      list_insert(L, c);
    }
  }
}

// Merge the four quarter lists of each row (lanes 4r..4r+3) and write the result.
template <int KC>
__device__ __forceinline__ void tile_finish(const RetrieveArgs& a, int nsplit, int b, int row0,
                                            int split, Cand (&L)[KC]) {
  const int rl = threadIdx.x >> 2, quarter = threadIdx.x & 3;
  const int i = row0 + rl;
  Cand out[kMaxTopk];
  for (int r = 0; r < a.topk; ++r) {
    Cand best = L[0];
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      Cand o = shfl_xor_cand(best, m);
      if (better(o, best)) best = o;
    }
    if (best.j != 0x7fffffff && L[0].j == best.j) list_pop(L);
    if (r < kMaxTopk) out[r] = best;
  }
  if (quarter == 0 && i < a.nQ) {
    if (nsplit == 1) write_row(a, b, i, out);
    else write_part(a, nsplit, b, i, split, out);
  }
}

template <typename T, int KC>
__global__ void __launch_bounds__(kTileThreads)
retrieve_tile_kernel(RetrieveArgs a, int nsplit, int seg) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int split = blockIdx.x;
  const int rb = gridDim.y - 1 - blockIdx.y;  // largest row blocks first
  const int b = blockIdx.z;
  const int row0 = rb * 64;
  const int last_row = min(a.nQ - 1, row0 + 63);
  const int ncand = n_cand_row(last_row, a.off, a.nC);
  const int j0 = split * seg;
  const int j1 = min(ncand, j0 + seg);
  const float inv = 1.0f / sqrtf((float)a.D);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  Cand L[KC];
  list_init(L);

  if (j0 < j1) {
    const T* qb = reinterpret_cast<const T*>(a.q) + (int64_t)b * a.q_bs;
    const T* kb = reinterpret_cast<const T*>(a.k) + (int64_t)b * a.k_bs;
    const int ntiles = (j1 - j0 + 63) / 64;
    if constexpr (sizeof(T) == 2) {
      // ---------------- bf16: tensor-core score tiles
      const int nkc = a.D / 64;
      unsigned char* Qs = smem;                        // [nkc][64][128B] swizzled
      unsigned char* Ks = smem + (size_t)64 * a.D * 2;  // [2][64][128B]
      float* St = reinterpret_cast<float*>(Ks + 2 * 64 * 128);
      // Q block, all chunks.
      for (int u = tid; u < 64 * a.D / 8; u += kTileThreads) {
        const int r = u / (a.D / 8), cu = u % (a.D / 8);
        const int kc = cu >> 3, w = cu & 7;
        const int i = row0 + r;
        unsigned char* dst = Qs + (size_t)kc * 8192 + swz<128>(r, w);
        if (i < a.nQ) cp_async16(dst, qb + (int64_t)i * a.q_rs + cu * 8);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
      auto load_chunk = [&](int step, int stage) {
        const int t = step / nkc, kc = step % nkc;
        const int jt = j0 + t * 64;
        for (int u = tid; u < 64 * 8; u += kTileThreads) {
          const int r = u >> 3, w = u & 7;
          const int j = jt + r;
          unsigned char* dst = Ks + stage * 8192 + swz<128>(r, w);
          if (j < j1) cp_async16(dst, kb + (int64_t)j * a.D + kc * 64 + w * 8);
          else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
      };
      const int nsteps = ntiles * nkc;
      load_chunk(0, 0);
      cp_async_commit();
      const int rw = 16 * (warp & 3), cw = 32 * (warp >> 2);
      float acc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
      for (int step = 0; step < nsteps; ++step) {
        const int stage = step & 1;
        if (step + 1 < nsteps) load_chunk(step + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int kc = step % nkc;
        const uint32_t qbase = smem_u32(Qs + (size_t)kc * 8192);
        const uint32_t kbase = smem_u32(Ks + stage * 8192);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t af[4];
          ldsm_x4(af[0], af[1], af[2], af[3],
                  qbase + swz<128>(rw + (lane & 15), 2 * ks + (lane >> 4)));
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3,
                    kbase + swz<128>(cw + 16 * p + (lane & 7) + ((lane >> 4) << 3),
                                     2 * ks + ((lane >> 3) & 1)));
            mma_bf16(acc[2 * p], af, b0, b1);
            mma_bf16(acc[2 * p + 1], af, b2, b3);
          }
        }
        if (kc == nkc - 1) {
          const int g = lane >> 2, c = lane & 3;
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            const int col = cw + 8 * n + 2 * c;
            St[(rw + g) * TileSmem::kSt + col] = acc[n][0];
            St[(rw + g) * TileSmem::kSt + col + 1] = acc[n][1];
            St[(rw + g + 8) * TileSmem::kSt + col] = acc[n][2];
            St[(rw + g + 8) * TileSmem::kSt + col + 1] = acc[n][3];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
          }
          __syncthreads();
          tile_topk(a, St, b, row0, j0 + (step / nkc) * 64, j1, inv, L);
        }
        __syncthreads();
      }
    } else {
      // ---------------- f32: SIMT score tiles (exact fp32 products)
      const int ldq = a.D + 1;
      float* Qs = reinterpret_cast<float*>(smem);  // [64][D+1]
      float* Ks = Qs + 64 * ldq;                   // [64][33]
      float* St = Ks + 64 * 33;                    // [64][65]
      for (int u = tid; u < 64 * a.D; u += kTileThreads) {
        const int r = u / a.D, d = u % a.D;
        const int i = row0 + r;
        Qs[r * ldq + d] = (i < a.nQ) ? reinterpret_cast<const float*>(qb)[(int64_t)i * a.q_rs + d] : 0.f;
      }
      const int r0 = 4 * (tid >> 4), c0 = 4 * (tid & 15);
      for (int t = 0; t < ntiles; ++t) {
        const int jt = j0 + t * 64;
        float acc[4][4] = {};
        for (int d0 = 0; d0 < a.D; d0 += 32) {
          __syncthreads();
          for (int u = tid; u < 64 * 32; u += kTileThreads) {
            const int r = u >> 5, d = u & 31;
            const int j = jt + r;
            Ks[r * 33 + d] = (j < j1) ? reinterpret_cast<const float*>(kb)[(int64_t)j * a.D + d0 + d] : 0.f;
          }
          __syncthreads();
#pragma unroll 8
          for (int d = 0; d < 32; ++d) {
            float qv[4], kv[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              qv[x] = Qs[(r0 + x) * ldq + d0 + d];
              kv[x] = Ks[(c0 + x) * 33 + d];
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
              for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(qv[x], kv[y], acc[x][y]);
          }
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) St[(r0 + x) * TileSmem::kSt + c0 + y] = acc[x][y];
        __syncthreads();
        tile_topk(a, St, b, row0, jt, j1, inv, L);
      }
    }
  }
  tile_finish(a, nsplit, b, row0, split, L);
}

template <typename F>
cudaError_t with_kc(int topk, F&& f) {
  if (topk <= 4) return f(std::integral_constant<int, 4>{});
  if (topk <= 8) return f(std::integral_constant<int, 8>{});
  return f(std::integral_constant<int, 16>{});
}

}  // namespace

RetrievePlan retrieve_plan(int B, int nQ, int nC, int topk, int off) {
  RetrievePlan p{};
  long long ncand_max = (long long)(nQ - 1) + off;
  if (ncand_max > nC) ncand_max = nC;
  if (ncand_max < 0) ncand_max = 0;
  if (nQ <= 8) {
    p.rowwise = 1;
    long long rows = (long long)B * nQ;
    long long ns = (kTargetCtas + rows - 1) / rows;
    long long ns_max = (ncand_max + 255) / 256;  // at least 256 candidates per split
    if (ns > ns_max) ns = ns_max;
    if (ns < 1) ns = 1;
    long long seg = (ncand_max + ns - 1) / ns;
    seg = (seg + 31) / 32 * 32;
    if (seg < 32) seg = 32;
    ns = (ncand_max + seg - 1) / seg;
    if (ns < 1) ns = 1;
    p.nsplit = (int)ns;
    p.seg = (int)seg;
  } else {
    p.rowwise = 0;
    // Spread the (triangular) candidate work over about 8 CTAs per SM.
    const int nrb = (nQ + 63) / 64;
    long long work = 0;
    for (int rb = 0; rb < nrb; ++rb) {
      long long last = (long long)rb * 64 + 63;
      if (last > nQ - 1) last = nQ - 1;
      long long n = last + off;
      if (n > nC) n = nC;
      if (n < 0) n = 0;
      work += n;
    }
    work *= B;
    long long seg = work / (152 * 8);
    seg = (seg + 63) / 64 * 64;
    if (seg < 64) seg = 64;
    long long ns = (ncand_max + seg - 1) / seg;
    if (ns < 1) ns = 1;
    p.nsplit = (int)ns;
    p.seg = (int)seg;
  }
  p.part_bytes = p.nsplit > 1 ? (size_t)B * nQ * p.nsplit * topk * sizeof(Cand) : 0;
  return p;
}

cudaError_t launch_retrieve(const RetrieveArgs& a, const RetrievePlan& p, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (p.rowwise) {
    dim3 grid(p.nsplit, a.nQ, a.B);
    e = with_kc(a.topk, [&](auto kc) -> cudaError_t {
      constexpr int KC = decltype(kc)::value;
      const int epv = a.bf16 ? 8 : 4;
      const int nv = (a.D / epv + 31) / 32;  // 16-byte vectors per lane per row (1..4)
      launch_begin("retrieve_rows", s);
      auto go = [&](auto nvc) {
        constexpr int NV = decltype(nvc)::value;
        if (a.bf16) retrieve_rows_kernel<__nv_bfloat16, NV, KC><<<grid, kRowsThreads, 0, s>>>(a, p.nsplit, p.seg);
        else retrieve_rows_kernel<float, NV, KC><<<grid, kRowsThreads, 0, s>>>(a, p.nsplit, p.seg);
      };
      if (nv <= 1) go(std::integral_constant<int, 1>{});
      else if (nv == 2) go(std::integral_constant<int, 2>{});
      else if (nv == 3) go(std::integral_constant<int, 3>{});
      else go(std::integral_constant<int, 4>{});
      return launch_end("retrieve_rows", s);
    });
  } else {
    dim3 grid(p.nsplit, (a.nQ + 63) / 64, a.B);
    const int smem = (int)TileSmem::bytes(a.D, a.bf16 != 0);
    e = with_kc(a.topk, [&](auto kc) -> cudaError_t {
      constexpr int KC = decltype(kc)::value;
      const void* fn = a.bf16 ? (const void*)retrieve_tile_kernel<__nv_bfloat16, KC>
                              : (const void*)retrieve_tile_kernel<float, KC>;
      cudaError_t e2 = allow_smem(fn, smem);
      if (e2 != cudaSuccess) return e2;
      launch_begin("retrieve_tile", s);
      if (a.bf16) retrieve_tile_kernel<__nv_bfloat16, KC><<<grid, kTileThreads, smem, s>>>(a, p.nsplit, p.seg);
      else retrieve_tile_kernel<float, KC><<<grid, kTileThreads, smem, s>>>(a, p.nsplit, p.seg);
      return launch_end("retrieve_tile", s);
    });
  }
  if (e != cudaSuccess || p.nsplit == 1) return e;
  dim3 mg(a.nQ, a.B);
  return with_kc(a.topk, [&](auto kc) -> cudaError_t {
    constexpr int KC = decltype(kc)::value;
    launch_begin("retrieve_merge", s);
    retrieve_merge_kernel<KC><<<mg, 128, 0, s>>>(a, p.nsplit);
    return launch_end("retrieve_merge", s);
  });
}

}  // namespace gca
