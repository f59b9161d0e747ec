// Causal landmark scoring with the per-row top-k in the epilogue, on tcgen05 (bf16).
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", 关键设计 / key design (causal retrieval; Gumbel top-k):
// query landmark i scores every earlier chunk's landmark with <q_i, k_j> / sqrt(D) and keeps
// the best k; in training the selection key carries Gumbel noise, the returned score does
// not.
//
// For many query rows (prefill-sized problems) the scores are a dense product: S = Q K^T with
// Q [128 rows][D] and K [256 candidates][D] per tile, D in steps of 64 through a 3-stage
// TMA ring, tcgen05.mma M = 128, N = 256 into one of two TMEM accumulators (so that a
// tile's selection overlaps the next tile's products).  A CTA takes one 128-row block and
// one segment of its candidate tiles; tiles past the block's last candidate (causal) are
// never made.  Warps 2-9 read a row's scores a thread per row over half of a tile's
// columns, scale by D^-1/2, drop candidates j >= i + offset, add the noise of
// (seed, group, b, i, j) for the key, and keep the row's best k in registers under the
// total order of the other retrieval kernels (key descending, then index ascending)
// across the segment's tiles.  Per 32 candidates a bitmask marks those at or above the
// list's last key (and the row's other half-list's), and only those go through the
// sorted insertion.  Each (row, segment, half) list goes to the partial buffer, which the
// merge kernels reduce to the row's result, so the outcome does not depend on the split.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tc_rows.cuh"

namespace gca {
namespace {

constexpr int kBM = 128, kBN = 256, kStages = 3, kThreads = 320;
constexpr uint32_t kABytes = kBM * 128, kStage = (kBM + kBN) * 128;
constexpr int kRowF = 33;  // floats per selection thread's staging row (32 values + 1: no bank conflicts)
constexpr int kKeyRow = 8 * 32 * kRowF;  // the keys' rows follow the 256 threads' score rows
constexpr int kSmem = kStages * kStage + 2 * kKeyRow * 4 + 1024;
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ int n_cand(int i, int off, int nC) {
  long long n = (long long)i + off;
  return (int)(n < 0 ? 0 : (n > nC ? nC : n));
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag, ErrWord* err, int site,
                                              int tile) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (tc::mbar_try(bar, parity)) return true;
    if ((it & 15) == 15 && *reinterpret_cast<volatile int*>(abort_flag)) return false;
  }
  flag_timeout(err, site, blockIdx.x, tile);
  atomicExch(abort_flag, 1);
  return false;
}

// Selection-list entries: with noise a candidate carries its key and its clean score;
// without, the key is the score and the entry is one float lighter to move.
struct KeyJ {
  float key;
  int j;
};
template <bool kNoise>
struct EntryOf {
  using T = Cand;
};
template <>
struct EntryOf<false> {
  using T = KeyJ;
};
__device__ __forceinline__ Cand as_cand(const Cand& c) { return c; }
__device__ __forceinline__ Cand as_cand(const KeyJ& c) { return Cand{c.key, c.key, c.j}; }
__device__ __forceinline__ void set_empty(Cand& c) { c = empty_cand(); }
__device__ __forceinline__ void set_empty(KeyJ& c) { c = KeyJ{-CUDART_INF_F, 0x7fffffff}; }

// The same sorted insertion and total order as the other retrieval kernels' lists.
template <class T>
__device__ __forceinline__ bool ahead(const T& x, const T& y) {
  return x.key > y.key || (x.key == y.key && x.j < y.j);
}
// The entries ahead of c form a prefix of the sorted list, so all KC comparisons are
// independent: entry t keeps its value inside the prefix, takes c just past it and its
// predecessor's value beyond.
template <class T, int KC>
__device__ __forceinline__ void insert_sorted(T (&L)[KC], const T& c) {
  if (!ahead(c, L[KC - 1])) return;
  bool in[KC];
#pragma unroll
  for (int t = 0; t < KC; ++t) in[t] = ahead(L[t], c);
#pragma unroll
  for (int t = KC - 1; t > 0; --t) L[t] = in[t] ? L[t] : (in[t - 1] ? c : L[t - 1]);
  if (!in[0]) L[0] = c;
}

// Writes one (row, segment, half) list to the partial buffer.  The register list is kept
// sorted by better() with its empty entries at the tail, and the merge of the heads of the
// lists (retrieve.cu) relies on that order.
template <class T, int KC>
__device__ __forceinline__ void put_list(const RetrieveArgs& a, int nsplit, int b, int i, int split,
                                         const T (&L)[KC]) {
  Cand* p = reinterpret_cast<Cand*>(a.part) + (((int64_t)b * a.nQ + i) * nsplit + split) * a.topk;
#pragma unroll
  for (int r = 0; r < KC; ++r)
    if (r < a.topk) p[r] = as_cand(L[r]);
}

template <int KC, bool kNoise>
__global__ void __launch_bounds__(kThreads, 1)
retrieve_tc_kernel(RetrieveArgs a, int ns, int sl, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK) {
  if (a.seed_dev) a.seed = *a.seed_dev;
  constexpr int NST = kStages;
  constexpr uint32_t kId = tc::idesc_bf16(kBM, kBN, false);
  const int seg = blockIdx.x, mb = gridDim.y - 1 - blockIdx.y, b = blockIdx.z;  // largest row blocks first
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = mb * kBM;
  const int cand = n_cand(min(a.nQ - 1, m0 + kBM - 1), a.off, a.nC);  // the block's last row has the most
  const int t0 = seg * sl, t1 = min((cand + kBN - 1) / kBN, t0 + sl);
  const int nt = t1 > t0 ? t1 - t0 : 0;
  const int nsplit = 2 * ns;
  const int qz = a.q_bs == 0 ? 0 : b, kz = a.k_bs == 0 ? 0 : b;
  // epilogue rows: warp w >= 2 reads TMEM lane quarter w % 4, column half (w - 2) / 4
  const int row = m0 + 32 * (warp & 3) + lane, half = (warp - 2) >> 2;

  if (nt == 0) {  // nothing in this segment: its lists are empty
    if (warp >= 2 && row < a.nQ) {
      Cand L[KC];
      list_init(L);
      put_list(a, nsplit, b, row, 2 * seg + half, L);
    }
    return;
  }
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[NST], empty[NST], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  // Last key of each (half, row) list, published after every chunk (see the selection).
  __shared__ float thr_s[2][kBM];
  const int kt = a.D / 64;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < NST; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&acc_full[x], 1);
      tc::mbar_init(&acc_empty[x], 8);
    }
    tc::mbar_init(&drain, 1);
    tc::fence_mbar_init();
    abort_s = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, 2 * kBN);
  for (int t = threadIdx.x; t < 2 * kBM; t += blockDim.x) (&thr_s[0][0])[t] = -CUDART_INF_F;
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = t0; ok && t < t1; ++t) {
        for (int kb = 0; kb < kt; ++kb) {
          const int s = it % NST;
          if (it >= NST && !wait_or_abort(&empty[s], (uint32_t)(it / NST - 1) & 1, &abort_s, a.err, 20, t)) {
            ok = false;
            break;
          }
          unsigned char* st = sm + s * kStage;
          tc::mbar_expect_tx(&full[s], kStage);
          tc::tma_load_3d(st, &tmQ, kb * 64, m0, qz, &full[s]);
          tc::tma_load_3d(st + kABytes, &tmK, kb * 64, t * kBN, kz, &full[s]);
          ++it;
        }
      }
      if (*reinterpret_cast<volatile int*>(&abort_s))  // let the copies already issued land
        for (int j = std::max(0, it - NST); j < it; ++j) tc::mbar_wait(&full[j % NST], (uint32_t)(j / NST) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    int it = 0;
    bool issued = false, ok = true;
    for (int i = 0; ok && i < nt; ++i) {
      const int buf = i & 1;
      if (i >= 2 && !wait_or_abort(&acc_empty[buf], (uint32_t)((i >> 1) - 1) & 1, &abort_s, a.err, 21, t0 + i)) break;
      tc::fence_after();
      const uint32_t d = tmem + buf * kBN;
      for (int kb = 0; kb < kt; ++kb, ++it) {
        const int s = it % NST;
        if (!wait_or_abort(&full[s], (uint32_t)(it / NST) & 1, &abort_s, a.err, 22, t0 + i)) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint32_t sa = tc::su32(sm + s * kStage);
        const uint64_t da = tc::desc_km(sa), db = tc::desc_km(sa + kABytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_warp(d, da + kk * tc::kKStepKm, db + kk * tc::kKStepKm, kId, (kb | kk) != 0 ? 1u : 0u);
        tc::commit_warp(&empty[s]);
        issued = true;
      }
      if (ok) tc::commit_warp(&acc_full[buf]);
    }
    if (issued) {  // no product may still run when TMEM is released
      tc::commit_warp(&drain);
      if (!tc::mbar_wait(&drain, 0) && lane == 0) flag_timeout(a.err, 23, blockIdx.x);
    }
  } else {
    // ------------------------------------------------------------ selection warps
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int lim = row < a.nQ ? n_cand(row, a.off, a.nC) : 0;
    // The thread's 32 scores and keys of a chunk go through its own shared-memory rows, so
    // that the selection loop indexes them without spilling the register array.
    float* mine = reinterpret_cast<float*>(sm + NST * kStage) + ((warp - 2) * 32 + lane) * kRowF;
    const float inv = 1.0f / sqrtf((float)a.D);
    // The row's other half-list publishes its last key: a candidate below it has KC >= k
    // better candidates of the same row there, so it cannot be among the row's best k and
    // is not inserted (a stale value is an older, lower last key: still a valid bound).
    volatile float* thr_own = &thr_s[half][32 * (warp & 3) + lane];
    const volatile float* thr_other = &thr_s[half ^ 1][32 * (warp & 3) + lane];
    using T = typename EntryOf<kNoise>::T;
    T L[KC];
#pragma unroll
    for (int r = 0; r < KC; ++r) set_empty(L[r]);
    for (int i = 0; i < nt; ++i) {
      const int buf = i & 1;
      if (!wait_or_abort(&acc_full[buf], (uint32_t)(i >> 1) & 1, &abort_s, a.err, 24, t0 + i)) break;
      tc::fence_after();
      const int j0 = (t0 + i) * kBN + 128 * half;
      const uint32_t tcol = tmem + lane_base + buf * kBN + 128 * half;
      float v[2][32];
      tc::ld32x32b_x32(tcol, v[0]);
      tc::ld_wait_row(v[0]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c + 1 < 4) tc::ld32x32b_x32(tcol + 32 * (c + 1), v[(c + 1) & 1]);
        const float(&cur)[32] = v[c & 1];
        const int jc = j0 + 32 * c;
        if (jc < lim) {
          // Bit e of `pass` marks the chunk's candidates whose key is at least that of the
          // list's last entry as it stands before the chunk (and at least the other half's).
          // That entry only improves, so an unmarked candidate cannot enter; the marked ones
          // go through the insertion in index order, which checks each against the list as
          // it is then (ties included).
          const float last = fmaxf(L[KC - 1].key, *thr_other);
          uint32_t pass = 0;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float sc = cur[e] * inv;
            const float key = kNoise ? sc + gumbel_noise(a.seed, a.group, b, row, jc + e) : sc;
            mine[e] = sc;
            if (kNoise) mine[kKeyRow + e] = key;
            if (key >= last && jc + e < lim) pass |= 1u << e;
          }
          while (pass) {
            const int e = __ffs(pass) - 1;
            pass &= pass - 1;
            T cd;
            if constexpr (kNoise) {
              cd.score = mine[e];
              cd.key = mine[kKeyRow + e];
            } else {
              cd.key = mine[e];
            }
            cd.j = jc + e;
            insert_sorted(L, cd);
          }
          *thr_own = L[KC - 1].key;
        }
        if (c + 1 < 4) tc::ld_wait_row(v[(c + 1) & 1]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
    }
    if (row < a.nQ) put_list(a, nsplit, b, row, 2 * seg + half, L);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 2 * kBN);
  }
}

}  // namespace

bool retrieve_tc_eligible(const RetrieveArgs& a) {
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  // Only where there are enough 128 x 256 tiles to fill the GPU (prefill-sized problems);
  // small ones (a training step's 256 rows) keep the 64-row tile kernel's finer split.
  const long long cand = std::min<long long>((long long)a.nQ - 1 + a.off, a.nC);
  const long long tiles = (long long)a.B * ((a.nQ + kBM - 1) / kBM) * ((cand + kBN - 1) / kBN) / 2;
  return a.bf16 && a.D >= 64 && a.D % 64 == 0 && a.q_rs % 8 == 0 && a.q_bs % 8 == 0 && a.k_bs % 8 == 0 &&
         a16(a.q) && a16(a.k) && tiles >= 4 * 152;
}

cudaError_t launch_retrieve_tc(const RetrieveArgs& a, const RetrievePlan& p, cudaStream_t s) {
  CUtensorMap tq, tk;
  cudaError_t e = make_lmk_tmap(&tq, a.q, a.D, a.nQ, a.B, a.q_rs, a.q_bs, kBM);
  if (e == cudaSuccess) e = make_lmk_tmap(&tk, a.k, a.D, a.nC, a.B, a.D, a.k_bs, kBN);
  if (e != cudaSuccess) return e;
  const int g = a.gumbel ? 1 : 0;
  const dim3 grid(p.tc_ns[g], (a.nQ + kBM - 1) / kBM, a.B);
  auto go = [&](auto kernel) -> cudaError_t {
    cudaError_t e2 = allow_smem((const void*)kernel, kSmem);
    if (e2 != cudaSuccess) return e2;
    launch_begin("retrieve_tc", s);
    kernel<<<grid, kThreads, kSmem, s>>>(a, p.tc_ns[g], p.tc_sl[g], tq, tk);
    return launch_end("retrieve_tc", s);
  };
  if (a.gumbel) {
    if (a.topk <= 4) return go(retrieve_tc_kernel<4, true>);
    if (a.topk <= 8) return go(retrieve_tc_kernel<8, true>);
    return go(retrieve_tc_kernel<16, true>);
  }
  if (a.topk <= 4) return go(retrieve_tc_kernel<4, false>);
  if (a.topk <= 8) return go(retrieve_tc_kernel<8, false>);
  return go(retrieve_tc_kernel<16, false>);
}

}  // namespace gca
