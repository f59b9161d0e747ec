// Device helpers shared by the kernels of the GCA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

namespace gca {

constexpr int kChunk = 64;    // tokens per chunk
constexpr int kMaxTopk = 16;  // largest supported top-k

// Device error word: the first 256 bytes of every workspace.
struct ErrWord {
  int flags;      // bit 0: an index outside [-1, nC) was met; bit 1: a bounded wait ran out
  int bad_value;  // last offending index
  int wait_sites; // bit s % 32: the wait at site s ran out (sites are numbered per kernel)
  int first[4];   // the first wait that ran out: site + 1, CTA, tile, slot (0 until then)
};
constexpr int kErrIndex = 1;
constexpr int kErrTimeout = 2;
constexpr size_t kErrBytes = 256;

__device__ __forceinline__ void flag_bad_index(ErrWord* e, int v) {
  if (e) {
    atomicOr(&e->flags, kErrIndex);
    atomicExch(&e->bad_value, v);
  }
}

// A bounded wait on an mbarrier ran out (the kernel carried on instead of hanging).
__device__ __forceinline__ void flag_timeout(ErrWord* e, int site = 0, int cta = -1, int tile = -1, int slot = -1) {
  if (e) {
    atomicOr(&e->flags, kErrTimeout);
    atomicOr(&e->wait_sites, 1 << (site & 31));
    if (atomicCAS(&e->first[0], 0, site + 1) == 0) {
      e->first[1] = cta;
      e->first[2] = tile;
      e->first[3] = slot;
    }
  }
}

// ---------------------------------------------------------------- element access
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float ld(const float* p) { return *p; }
  static __device__ __forceinline__ void st(float* p, float v) { *p = v; }
  static constexpr int kVec = 4;  // elements per 16-byte vector
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
  static constexpr int kVec = 8;
};

// 16-byte vector -> floats
__device__ __forceinline__ void unpack16(const uint4& u, float* f, const float*) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4& u, float* f, const __nv_bfloat16*) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    f[2 * t] = __uint_as_float(w[t] << 16);
    f[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------- query-tile order
// Tile t in [0, nQ * H * B) of the persistent forward and query-side kernels, as (query
// chunk c, head h, sequence b).  The chunks c >= L of every sequence-head come first,
// head-major with c fastest (the CTAs in flight share that sequence-head's K/V in L2);
// the first L chunks of each follow.  Under causal retrieval those rows have fewer valid
// slots (L = min(nQ, shift + topk)), so the tiles that start last are the light ones and
// the kernels' tails are short.  Any order gives the same results.
__device__ __forceinline__ void query_tile(int nQ, int H, int B, int L, int t, int& c, int& h, int& b) {
  const int F = nQ - L, nfull = F * H * B;
  int hb;
  if (t < nfull) {
    hb = t / F;
    c = L + (t - hb * F);
  } else {
    const int u = t - nfull;
    hb = u / L;
    c = u - hb * L;
  }
  h = hb % H;
  b = hb / H;
}

// ---------------------------------------------------------------- splitmix64 noise
// splitmix64 (Steele, Lea & Flood, 2014): output number n from state `seed`.
__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t n) {
  uint64_t z = seed + n * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Gumbel(0,1) sample for candidate pair (group, b, i, j).
__device__ __forceinline__ float gumbel_noise(uint64_t seed, int group, int b, int i, int j) {
  const uint64_t ctr = ((uint64_t)(uint32_t)group << 56) | ((uint64_t)(uint32_t)b << 48) |
                       ((uint64_t)(uint32_t)i << 24) | (uint64_t)(uint32_t)j;
  const uint64_t h = splitmix64(seed, ctr + 1);
  const float u = ((float)(uint32_t)(h >> 41) + 0.5f) * (1.0f / 8388608.0f);
  return -logf(-logf(u));
}

// ---------------------------------------------------------------- top-k candidates
struct Cand {
  float key;    // selection key (score + noise)
  float score;  // clean score
  int j;        // candidate chunk
};
__device__ __forceinline__ Cand empty_cand() { return Cand{-CUDART_INF_F, -CUDART_INF_F, 0x7fffffff}; }
// Total order: larger key first, equal keys -> lower index first.
__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
  return a.key > b.key || (a.key == b.key && a.j < b.j);
}

// Sorted register list of the KC best candidates seen so far (L[0] best).
template <int KC>
__device__ __forceinline__ void list_insert(Cand (&L)[KC], const Cand& c) {
  if (!better(c, L[KC - 1])) return;
  bool placed = false;
#pragma unroll
  for (int t = KC - 1; t > 0; --t) {
    const bool mv = better(c, L[t - 1]);
    Cand nt = placed ? L[t] : (mv ? L[t - 1] : c);
    placed = placed || !mv;
    L[t] = nt;
  }
  if (!placed) L[0] = c;
}
template <int KC>
__device__ __forceinline__ void list_init(Cand (&L)[KC]) {
#pragma unroll
  for (int t = 0; t < KC; ++t) L[t] = empty_cand();
}
template <int KC>
__device__ __forceinline__ void list_pop(Cand (&L)[KC]) {
#pragma unroll
  for (int t = 0; t < KC - 1; ++t) L[t] = L[t + 1];
  L[KC - 1] = empty_cand();
}

__device__ __forceinline__ Cand shfl_cand(const Cand& c, int src, int width = 32) {
  Cand r;
  r.key = __shfl_sync(0xffffffffu, c.key, src, width);
  r.score = __shfl_sync(0xffffffffu, c.score, src, width);
  r.j = __shfl_sync(0xffffffffu, c.j, src, width);
  return r;
}
__device__ __forceinline__ Cand shfl_xor_cand(const Cand& c, int m, int width = 32) {
  Cand r;
  r.key = __shfl_xor_sync(0xffffffffu, c.key, m, width);
  r.score = __shfl_xor_sync(0xffffffffu, c.score, m, width);
  r.j = __shfl_xor_sync(0xffffffffu, c.j, m, width);
  return r;
}

// Block-wide selection of the `k` best candidates from the threads' sorted lists.
// Requires candidate indices to be distinct across threads.  Every thread of the
// block must call it; out[0..k) is written by thread 0 into shared memory `out`.
// `red` must hold blockDim.x/32 Cand.
template <int KC>
__device__ void block_select(Cand (&L)[KC], int k, Cand* out, Cand* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int r = 0; r < k; ++r) {
    Cand best = L[0];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      Cand o = shfl_xor_cand(best, m);
      if (better(o, best)) best = o;
    }
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (warp == 0) {
      Cand b2 = lane < nw ? red[lane] : empty_cand();
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        Cand o = shfl_xor_cand(b2, m);
        if (better(o, b2)) b2 = o;
      }
      if (lane == 0) red[0] = b2;
    }
    __syncthreads();
    const Cand win = red[0];
    if (threadIdx.x == 0) out[r] = win;
    if (win.j != 0x7fffffff && L[0].j == win.j && L[0].key == win.key) list_pop(L);
    __syncthreads();
  }
}

// ---------------------------------------------------------------- retrieval weights
// w = softmax over valid slots (idx >= 0) of the scores of one row; computed by one
// warp into shared memory.  Indices outside [-1, nC) are flagged and treated as empty.
// Writes w[m] (0 for invalid slots) and jidx[m] (-1 for invalid); returns nothing.
__device__ __forceinline__ void row_weights_warp(const int32_t* idx_row, const float* sc_row,
                                                 int topk, int nC, float* w, int* jidx,
                                                 ErrWord* err) {
  const int lane = threadIdx.x & 31;
  int j = -1;
  float s = -CUDART_INF_F;
  if (lane < topk) {
    j = idx_row[lane];   // both loads in flight at once (the score of an empty slot is
    s = sc_row[lane];    // read and discarded)
    if (j < -1 || j >= nC) {
      flag_bad_index(err, j);
      j = -1;
    }
    if (j < 0) s = -CUDART_INF_F;
  }
  float mx = s;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  float e = (j >= 0) ? expf(s - mx) : 0.f;
  float sum = e;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
  if (lane < topk) {
    w[lane] = (j >= 0) ? e / sum : 0.f;
    jidx[lane] = j;
  }
}

// ---------------------------------------------------------------- mma.sync helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D (f32)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte unit `u` of row `r` in a swizzled tile with ROWB bytes per row
// (ROWB = 128: xor with r & 7; ROWB = 64: xor with (r >> 1) & 3), so that the eight
// row addresses of one ldmatrix phase hit eight different bank groups.
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int r, int u) {
  if constexpr (ROWB == 128) return r * 128 + ((u ^ (r & 7)) << 4);
  else return r * 64 + ((u ^ ((r >> 1) & 3)) << 4);
}

}  // namespace gca
