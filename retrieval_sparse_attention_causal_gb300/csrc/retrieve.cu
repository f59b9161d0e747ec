// Causal landmark scoring fused with per-row top-k selection.
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", section 关键设计 / key design: the current chunk's
// landmark scores the landmarks of earlier chunks and the top-k are kept; in training,
// Gumbel noise is added to the scores before the top-k.  The score is the scaled dot
// product <q_i, k_j> / sqrt(D).
//
// Two stage-1 kernels feed one merge kernel:
//   retrieve_stream_kernel few query rows, very many candidates (decode at 16M context):
//                         each CTA streams a contiguous slice of one row's candidate
//                         landmarks through a 4-stage shared-memory ring filled by 1-D
//                         bulk copies (TMA) from a producer warp; eight consumer warps
//                         take the dot products out of shared memory.  One CTA per SM,
//                         one wave; an HBM-bound sweep.
//   retrieve_tile_kernel  many query rows (training, prefill): 64 query rows stay in
//                         shared memory while 64-candidate tiles stream through a
//                         double-buffered cp.async pipeline; the 64x64 score tile is a
//                         bf16 tensor-core product (fp32 SIMT for f32 inputs).
//   retrieve_tc_kernel    (retrieve_tc.cu) the same for bf16 landmarks in TMA-compatible
//                         layouts: 128-row x 256-candidate score tiles on tcgen05 with
//                         the selection in the epilogue; the row-block path then takes it
//                         instead of retrieve_tile_kernel.
//   retrieve_merge_kernel / retrieve_merge_warp_kernel / retrieve_merge_heads_kernel
//                         merge the per-split candidate lists of a row (a block per row
//                         for few rows; a warp per row for many, walking the sorted lists'
//                         heads when they are few and short).  The bf16 tile kernel with
//                         2 to 8 splits needs none of them: its split CTAs form a thread-
//                         block cluster and merge each other's lists through distributed
//                         shared memory.
// Every stage keeps candidates under one total order (key descending, then index
// ascending), so the result does not depend on how the candidates were split.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gca {

namespace {

constexpr int kTileThreads = 256;
constexpr long long kWarpMergeRows = 256;  // from this many rows on, the merge takes a warp per row

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

// Partial lists: every producer (write_part here, put_list in retrieve_tc.cu) writes
// each (row, split) list in the order of better(): best first, ties by the lower index,
// empty entries (j = 0x7fffffff) only at the tail.  retrieve_merge_heads_kernel relies on
// it: it only ever looks at the head of each list.  The other merges re-insert every
// entry and do not need it.
__device__ __forceinline__ void write_part(const RetrieveArgs& a, int nsplit, int b, int i,
                                           int split, const Cand* sel) {
  Cand* p = reinterpret_cast<Cand*>(a.part) +
            (((int64_t)b * a.nQ + i) * nsplit + split) * a.topk;
  for (int r = 0; r < a.topk; ++r) p[r] = sel[r];
}

// ------------------------------------------------------------------ stream kernel
constexpr int kStreamStages = 4;
constexpr int kStreamConsumers = 8;
constexpr int kStreamThreads = 32 * (kStreamConsumers + 1);
constexpr int kStreamStageBytes = 48 * 1024;

// Candidate rows per stage: a multiple of 8 (one row per consumer warp per step), at
// most 32, within one 48 KB stage.
__host__ __device__ inline int stream_rows(int D, int elem) {
  int r = kStreamStageBytes / (D * elem);
  r = r > 32 ? 32 : r;
  return r / 8 * 8;
}

template <typename T, int NV, int KC>
__global__ void __launch_bounds__(kStreamThreads, 1)
retrieve_stream_kernel(RetrieveArgs a, int nsplit, int seg) {
  if (a.seed_dev) a.seed = *a.seed_dev;
  constexpr int EPV = 16 / sizeof(T), NST = kStreamStages, NCW = kStreamConsumers;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ Cand red[kStreamThreads / 32];
  __shared__ Cand sel[kMaxTopk];
  __shared__ __align__(8) uint64_t full[NST], empty[NST];
  const int split = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_i = n_cand_row(i, a.off, a.nC);
  const int j0 = split * seg;
  const int j1 = min(n_i, j0 + seg);
  const int rows = stream_rows(a.D, sizeof(T));
  const int nchunks = j1 > j0 ? (j1 - j0 + rows - 1) / rows : 0;
  const size_t row_bytes = (size_t)a.D * sizeof(T);
  const T* kb = reinterpret_cast<const T*>(a.k) + (int64_t)b * a.k_bs;
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      tc::mbar_init(&full[st], 1);
      tc::mbar_init(&empty[st], NCW);
    }
    tc::fence_mbar_init();
  }
  __syncthreads();
  Cand L[KC];
  list_init(L);
  bool ok = true;
  if (warp == NCW) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      for (int c = 0; c < nchunks; ++c) {
        const int st = c % NST;
        if (c >= NST) ok = tc::mbar_wait(&empty[st], (c / NST - 1) & 1) && ok;
        const int r0 = j0 + c * rows;
        const int nr = min(rows, j1 - r0);
        const uint32_t bytes = (uint32_t)(nr * row_bytes);
        tc::mbar_expect_tx(&full[st], bytes);
        tc::bulk_load(ring + (size_t)st * kStreamStageBytes, kb + (int64_t)r0 * a.D, bytes, &full[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ consumer warps
    const T* q = reinterpret_cast<const T*>(a.q) + (int64_t)b * a.q_bs + (int64_t)i * a.q_rs;
    const int nvec = a.D / EPV;
    const float inv = 1.0f / sqrtf((float)a.D);
    float qf[NV][EPV];
#pragma unroll
    for (int t = 0; t < NV; ++t) {
      const int vi = lane + 32 * t;
      if (vi < nvec) {
        const uint4 u = *reinterpret_cast<const uint4*>(q + vi * EPV);
        unpack16(u, qf[t], (const T*)nullptr);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) qf[t][e] = 0.f;
      }
    }
    for (int c = 0; c < nchunks; ++c) {
      const int st = c % NST;
      ok = tc::mbar_wait(&full[st], (c / NST) & 1) && ok;
      const int r0 = j0 + c * rows;
      const int nr = min(rows, j1 - r0);
      const unsigned char* stage = ring + (size_t)st * kStreamStageBytes;
      float acc[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {  // this warp's rows: warp, warp + 8, ...
        const int rr = warp + NCW * t;
        float sum = 0.f;
        if (rr < nr) {
          const T* row = reinterpret_cast<const T*>(stage + (size_t)rr * row_bytes);
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            const int vi = lane + 32 * v;
            if (vi < nvec) {
              float f[EPV];
              unpack16(*reinterpret_cast<const uint4*>(row + vi * EPV), f, (const T*)nullptr);
#pragma unroll
              for (int e = 0; e < EPV; ++e) sum = fmaf(qf[v][e], f[e], sum);
            }
          }
        }
        acc[t] = sum;
      }
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], m);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[st]);
      if (lane < 4) {
        const int rr = warp + NCW * lane;
        float mine = acc[0];
#pragma unroll
        for (int t = 1; t < 4; ++t) mine = (lane == t) ? acc[t] : mine;
        if (rr < nr) {
          const int j = r0 + rr;
          Cand cnd;
          cnd.score = mine * inv;
          cnd.key = a.gumbel ? cnd.score + gumbel_noise(a.seed, a.group, b, i, j) : cnd.score;
          cnd.j = j;
          list_insert(L, cnd);
        }
      }
    }
  }
  if (!ok) flag_timeout(a.err);
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

// One warp per row, for problems with many rows (training, prefill): the lanes take the
// row's candidates in turn into register lists, then k rounds of a butterfly maximum under
// the total order pick the winners, the owning lane dropping each from its list.
template <int KC>
__global__ void __launch_bounds__(256) retrieve_merge_warp_kernel(RetrieveArgs a, int nsplit, int rows) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);  // row b * nQ + i
  if (r >= rows) return;
  const Cand* p = reinterpret_cast<const Cand*>(a.part) + (int64_t)r * nsplit * a.topk;
  Cand L[KC];
  list_init(L);
  const int n = nsplit * a.topk;
  for (int c = lane; c < n; c += 32) {
    const Cand x = p[c];
    if (x.j != 0x7fffffff) list_insert(L, x);
  }
  Cand mine = empty_cand();  // lane q keeps the q-th winner
  for (int q = 0; q < a.topk; ++q) {
    Cand best = L[0];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      const Cand o = shfl_xor_cand(best, m);
      if (better(o, best)) best = o;
    }
    if (lane == q) mine = best;
    if (best.j != 0x7fffffff && L[0].j == best.j && L[0].key == best.key) list_pop(L);
  }
  if (lane < a.topk) {
    const bool ok = mine.j != 0x7fffffff;
    a.idx[(int64_t)r * a.topk + lane] = ok ? mine.j : -1;
    a.scores[(int64_t)r * a.topk + lane] = ok ? mine.score : -CUDART_INF_F;
  }
}

// One warp per row when the row's lists are few and short (up to 32 lists, kHeadsMax
// candidates): the lists are sorted already, so they are staged in shared memory, lane l
// holds the head of list l, and each of k rounds takes the best head (a butterfly over
// the lists' lanes on (key, index)) and moves the winning lane to its list's next entry.
constexpr int kHeadsMax = 128;
__global__ void __launch_bounds__(256) retrieve_merge_heads_kernel(RetrieveArgs a, int nsplit, int rows) {
  __shared__ Cand st[8][kHeadsMax];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int r = blockIdx.x * 8 + w;  // row b * nQ + i
  if (r >= rows) return;
  const int n = nsplit * a.topk;
  const Cand* p = reinterpret_cast<const Cand*>(a.part) + (int64_t)r * n;
  for (int c = lane; c < n; c += 32) st[w][c] = p[c];
  __syncwarp();
  int width = 1;
  while (width < nsplit) width <<= 1;
  int pos = 0;
  Cand head = lane < nsplit ? st[w][lane * a.topk] : empty_cand();
  int32_t* idx = a.idx + (int64_t)r * a.topk;
  float* sc = a.scores + (int64_t)r * a.topk;
  for (int q = 0; q < a.topk; ++q) {
    float bk = head.key;
    int bj = head.j;
    for (int m = width >> 1; m >= 1; m >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, m);
      const int oj = __shfl_xor_sync(0xffffffffu, bj, m);
      if (ok > bk || (ok == bk && oj < bj)) {
        bk = ok;
        bj = oj;
      }
    }
    bj = __shfl_sync(0xffffffffu, bj, 0);  // lanes 0 .. width-1 hold the lists' best
    if (bj == 0x7fffffff) {                // every list is spent: pad the rest
      if (lane == 0)
        for (int t = q; t < a.topk; ++t) {
          idx[t] = -1;
          sc[t] = -CUDART_INF_F;
        }
      break;
    }
    if (lane < nsplit && head.j == bj) {  // indices are unique across the lists
      idx[q] = bj;
      sc[q] = head.score;
      ++pos;
      head = pos < a.topk ? st[w][lane * a.topk + pos] : empty_cand();
    }
  }
}

// ------------------------------------------------------------------ tile kernel
// Shared memory: Q block (64 rows x D), a ring of candidate chunk buffers (bf16; two for
// f32), score tile.
constexpr int kTileStages = 6;  // 64-candidate x 64-dim chunks in flight (bf16)
struct TileSmem {
  static constexpr int kSt = 65;  // padded score-tile row (floats)
  static size_t bytes(int D, bool bf16, int rows = 64) {
    if (bf16) return (size_t)rows * D * 2 + kTileStages * 64 * 128 + rows * kSt * 4 + 1024;
    return (size_t)64 * (D + 1) * 4 + 64 * 33 * 4 + 64 * kSt * 4 + 1024;
  }
};

// Top-k phase over one ROWS x 64 score tile held in shared memory.  Thread t owns row
// t / TPR and the 64 / TPR candidates of part t % TPR (TPR = 256 / ROWS threads a row).
template <int KC, int ROWS>
__device__ __forceinline__ void tile_topk(const RetrieveArgs& a, const float* St, int b,
                                          int row0, int tile0, int j1, float inv, Cand (&L)[KC]) {
  constexpr int TPR = kTileThreads / ROWS, CPT = 64 / TPR;
  const int rl = threadIdx.x / TPR, quarter = threadIdx.x % TPR;
  const int i = row0 + rl;
  if (i >= a.nQ) return;
  const int lim = min(j1, n_cand_row(i, a.off, a.nC));
#pragma unroll 4
  for (int cc = 0; cc < CPT; ++cc) {
    const int jl = quarter * CPT + cc;
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

// Merge the TPR part lists of each row (lanes TPR r .. TPR r + TPR - 1) and write the result:
// the row's output, the split's part list in global memory, or (lists != nullptr) the
// split's list in this CTA's shared memory for the cluster merge.
template <int KC, int ROWS>
__device__ __forceinline__ void tile_finish(const RetrieveArgs& a, int nsplit, int b, int row0,
                                            int split, Cand (&L)[KC], Cand* lists) {
  constexpr int TPR = kTileThreads / ROWS;
  const int rl = threadIdx.x / TPR, quarter = threadIdx.x % TPR;
  const int i = row0 + rl;
  Cand out[kMaxTopk];
  for (int r = 0; r < a.topk; ++r) {
    Cand best = L[0];
#pragma unroll
    for (int m = 1; m < TPR; m <<= 1) {
      Cand o = shfl_xor_cand(best, m);
      if (better(o, best)) best = o;
    }
    if (best.j != 0x7fffffff && L[0].j == best.j) list_pop(L);
    if (r < kMaxTopk) out[r] = best;
  }
  if (quarter == 0 && i < a.nQ) {
    if (lists) {
      for (int r = 0; r < a.topk; ++r) lists[rl * kMaxTopk + r] = out[r];
    } else if (nsplit == 1) {
      write_row(a, b, i, out);
    } else {
      write_part(a, nsplit, b, i, split, out);
    }
  }
}

// ---- thread-block cluster: the nsplit CTAs of one row block (cluster rank = split)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; shared-memory writes before it are visible to
// the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The Cand at this CTA's shared-memory address p, in CTA `rank` of the cluster.
__device__ __forceinline__ Cand ld_cand_cluster(const Cand* p, uint32_t rank) {
  uint32_t ad, k, sc, j;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ad) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(k) : "r"(ad) : "memory");
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sc) : "r"(ad + 4) : "memory");
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(j) : "r"(ad + 8) : "memory");
  return Cand{__uint_as_float(k), __uint_as_float(sc), (int)j};
}

// After tile_finish wrote every split's lists: CTA s merges rows s, s + nsplit, ... of the
// row block, a warp per row.  Lane l < nsplit copies list l (sorted, best first) from CTA l
// into registers; each of k rounds takes the best head over the lanes (key descending,
// index ascending, as everywhere) and the lane that held it moves to its next entry.  The
// splits' candidate ranges are disjoint, so exactly one lane holds the winning index.
template <int KC, int ROWS>
__device__ __forceinline__ void cluster_merge(const RetrieveArgs& a, int nsplit, int b, int row0, const Cand* lists) {
  cluster_sync();  // every split's lists are in place
  const uint32_t me = cluster_rank();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int width = 1;
  while (width < nsplit) width <<= 1;
  for (int rl = (int)me + nsplit * warp; rl < ROWS; rl += nsplit * (kTileThreads / 32)) {
    const int i = row0 + rl;
    if (i >= a.nQ) break;
    Cand H[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k)
      H[k] = (lane < nsplit && k < a.topk) ? ld_cand_cluster(lists + rl * kMaxTopk + k, (uint32_t)lane) : empty_cand();
    int32_t* idx = a.idx + ((int64_t)b * a.nQ + i) * a.topk;
    float* sc = a.scores + ((int64_t)b * a.nQ + i) * a.topk;
    for (int q = 0; q < a.topk; ++q) {
      float bk = H[0].key;
      int bj = H[0].j;
      for (int m = width >> 1; m >= 1; m >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, m);
        const int oj = __shfl_xor_sync(0xffffffffu, bj, m);
        if (ok > bk || (ok == bk && oj < bj)) {
          bk = ok;
          bj = oj;
        }
      }
      bj = __shfl_sync(0xffffffffu, bj, 0);
      if (bj == 0x7fffffff) {  // every list is spent: pad the rest
        if (lane == 0)
          for (int t = q; t < a.topk; ++t) {
            idx[t] = -1;
            sc[t] = -CUDART_INF_F;
          }
        break;
      }
      if (lane < nsplit && H[0].j == bj) {
        idx[q] = bj;
        sc[q] = H[0].score;
        list_pop(H);
      }
    }
  }
  cluster_sync();  // no CTA exits while another still reads its lists
}

// ROWS query rows per CTA: 64, or 32 (bf16 only) when the problem has too few 64-row
// blocks to occupy the GPU.
// cl = 1: launched as clusters of nsplit CTAs along x (bf16 only); the splits merge in the
// cluster instead of through the part lists.
template <typename T, int KC, int ROWS>
__global__ void __launch_bounds__(kTileThreads)
retrieve_tile_kernel(RetrieveArgs a, int nsplit, int seg, int cl) {
  if (a.seed_dev) a.seed = *a.seed_dev;
  static_assert(ROWS == 64 || (ROWS == 32 && sizeof(T) == 2), "32-row blocks are bf16 only");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int split = blockIdx.x;
  const int rb = gridDim.y - 1 - blockIdx.y;  // largest row blocks first
  const int b = blockIdx.z;
  const int row0 = rb * ROWS;
  const int last_row = min(a.nQ - 1, row0 + ROWS - 1);
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
      unsigned char* Qs = smem;                          // [nkc][ROWS][128B] swizzled
      unsigned char* Ks = smem + (size_t)ROWS * a.D * 2;  // [kTileStages][64][128B]
      float* St = reinterpret_cast<float*>(Ks + kTileStages * 64 * 128);
      // Q block, all chunks.
      for (int u = tid; u < ROWS * a.D / 8; u += kTileThreads) {
        const int r = u / (a.D / 8), cu = u % (a.D / 8);
        const int kc = cu >> 3, w = cu & 7;
        const int i = row0 + r;
        unsigned char* dst = Qs + (size_t)kc * (ROWS * 128) + swz<128>(r, w);
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
      // A ring of kTileStages chunks: kTileStages - 1 loads stay in flight ahead of the
      // products (one commit group per step, empty ones past the end, so that the group
      // count stays uniform; the Q block rides in the first group).
      const int nsteps = ntiles * nkc;
      for (int st = 0; st < kTileStages - 1; ++st) {
        if (st < nsteps) load_chunk(st, st);
        cp_async_commit();
      }
      // Warp tiles of 16 rows x (32 or 16) candidates: NP pairs of 8-candidate MMA tiles.
      constexpr int NP = ROWS == 64 ? 2 : 1;
      const int rw = ROWS == 64 ? 16 * (warp & 3) : 16 * (warp & 1);
      const int cw = ROWS == 64 ? 32 * (warp >> 2) : 16 * (warp >> 1);
      float acc[2 * NP][4];
#pragma unroll
      for (int n = 0; n < 2 * NP; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
      for (int step = 0; step < nsteps; ++step) {
        const int stage = step % kTileStages;
        cp_async_wait<kTileStages - 2>();
        __syncthreads();  // chunk `step` is in; the stage of step - 1 is free
        if (step + kTileStages - 1 < nsteps) load_chunk(step + kTileStages - 1, (step + kTileStages - 1) % kTileStages);
        cp_async_commit();
        const int kc = step % nkc;
        const uint32_t qbase = smem_u32(Qs + (size_t)kc * (ROWS * 128));
        const uint32_t kbase = smem_u32(Ks + stage * 8192);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t af[4];
          ldsm_x4(af[0], af[1], af[2], af[3],
                  qbase + swz<128>(rw + (lane & 15), 2 * ks + (lane >> 4)));
#pragma unroll
          for (int p = 0; p < NP; ++p) {
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
          for (int n = 0; n < 2 * NP; ++n) {
            const int col = cw + 8 * n + 2 * c;
            St[(rw + g) * TileSmem::kSt + col] = acc[n][0];
            St[(rw + g) * TileSmem::kSt + col + 1] = acc[n][1];
            St[(rw + g + 8) * TileSmem::kSt + col] = acc[n][2];
            St[(rw + g + 8) * TileSmem::kSt + col + 1] = acc[n][3];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
          }
          __syncthreads();
          tile_topk<KC, ROWS>(a, St, b, row0, j0 + (step / nkc) * 64, j1, inv, L);
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
        tile_topk<KC, ROWS>(a, St, b, row0, jt, j1, inv, L);
      }
    }
  }
  // The ring is idle here: every step's loads were waited for, and the loop ended on a
  // barrier after the last reads; the lists reuse its first bytes.
  Cand* lists = (cl && sizeof(T) == 2) ? reinterpret_cast<Cand*>(smem + (size_t)ROWS * a.D * 2) : nullptr;
  if (lists) cp_async_wait<0>();
  tile_finish<KC, ROWS>(a, nsplit, b, row0, split, L, lists);
  if (lists) cluster_merge<KC, ROWS>(a, nsplit, b, row0, lists);
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
    // Streaming kernel, one CTA per SM: at launch the candidates of each row are split
    // so that all CTAs form one wave.  The workspace holds the largest split count the
    // launch can choose (sized for up to 1216 SMs' worth of CTAs, at least 256
    // candidates per split).
    p.rowwise = 1;
    long long rows = (long long)B * nQ;
    long long ns = (1216 + rows - 1) / rows;
    long long ns_max = (ncand_max + 255) / 256;
    if (ns > ns_max) ns = ns_max;
    if (ns < 1) ns = 1;
    p.nsplit = (int)ns;
    p.seg = 0;
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
    // tcgen05 path: 128-row blocks, 256-candidate tiles; the last block has the most tiles.
    // Segments of tc_sl tiles per block.  Every segment's lists start empty and fill at a
    // cost, so without noise (cheap candidates) about two CTAs per SM over the grid; with
    // noise each candidate costs more and the balance counts for more: about four.
    const long long nmb = (nQ + 127) / 128;
    const long long nt_max = ncand_max > 0 ? (ncand_max + 255) / 256 : 1;
    for (int g = 0; g < 2; ++g) {
      const long long target = (g ? 4 : 2) * 152;
      long long tns = (target + B * nmb - 1) / (B * nmb);
      if (tns > nt_max) tns = nt_max;
      if (tns < 1) tns = 1;
      const long long tsl = (nt_max + tns - 1) / tns;
      p.tc_sl[g] = (int)tsl;
      p.tc_ns[g] = (int)((nt_max + tsl - 1) / tsl);
    }
  }
  p.part_bytes = p.nsplit > 1 ? (size_t)B * nQ * p.nsplit * topk * sizeof(Cand) : 0;
  if (!p.rowwise)
    p.part_bytes = std::max(p.part_bytes, (size_t)B * nQ * 2 * std::max(p.tc_ns[0], p.tc_ns[1]) * topk * sizeof(Cand));
  return p;
}

cudaError_t launch_retrieve(const RetrieveArgs& a, const RetrievePlan& p, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  int nsplit = p.nsplit;
  if (p.rowwise) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long rows = (long long)a.B * a.nQ;
    long long ns = sms / rows;
    if (ns < 1) ns = 1;
    if (ns > p.nsplit) ns = p.nsplit;
    long long ncand_max = (long long)(a.nQ - 1) + a.off;
    if (ncand_max > a.nC) ncand_max = a.nC;
    if (ncand_max < 1) ncand_max = 1;
    const int seg = (int)((ncand_max + ns - 1) / ns);
    nsplit = (int)ns;
    dim3 grid(nsplit, a.nQ, a.B);
    const int elem = a.bf16 ? 2 : 4;
    const int smem = kStreamStages * kStreamStageBytes;
    e = with_kc(a.topk, [&](auto kc) -> cudaError_t {
      constexpr int KC = decltype(kc)::value;
      const int nv = (a.D / (16 / elem) + 31) / 32;  // 16-byte vectors per lane per row (1..4)
      auto go = [&](auto nvc) -> cudaError_t {
        constexpr int NV = decltype(nvc)::value;
        const void* fn = a.bf16 ? (const void*)retrieve_stream_kernel<__nv_bfloat16, NV, KC>
                                : (const void*)retrieve_stream_kernel<float, NV, KC>;
        cudaError_t e2 = allow_smem(fn, smem);
        if (e2 != cudaSuccess) return e2;
        launch_begin("retrieve_stream", s);
        if (a.bf16) retrieve_stream_kernel<__nv_bfloat16, NV, KC><<<grid, kStreamThreads, smem, s>>>(a, nsplit, seg);
        else retrieve_stream_kernel<float, NV, KC><<<grid, kStreamThreads, smem, s>>>(a, nsplit, seg);
        return launch_end("retrieve_stream", s);
      };
      if (nv <= 1) return go(std::integral_constant<int, 1>{});
      if (nv == 2) return go(std::integral_constant<int, 2>{});
      if (nv == 3) return go(std::integral_constant<int, 3>{});
      return go(std::integral_constant<int, 4>{});
    });
  } else if (retrieve_tc_eligible(a)) {
    e = launch_retrieve_tc(a, p, s);
    nsplit = 2 * p.tc_ns[a.gumbel ? 1 : 0];
  } else {
    // bf16 problems with fewer 64-row CTAs than two per SM take 32-row blocks (twice the
    // CTAs, half the selection work per thread).
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const bool r32 = a.bf16 && (long long)p.nsplit * ((a.nQ + 63) / 64) * a.B < 2LL * sms;
    const int rows = r32 ? 32 : 64;
    dim3 grid(p.nsplit, (a.nQ + rows - 1) / rows, a.B);
    const int smem = (int)TileSmem::bytes(a.D, a.bf16 != 0, rows);
    // bf16 with 2 to 8 splits (the portable cluster size): the splits of a row block
    // merge in their cluster, and no merge launch follows.
    bool cl = a.bf16 && p.nsplit >= 2 && p.nsplit <= 8;
    e = with_kc(a.topk, [&](auto kc) -> cudaError_t {
      constexpr int KC = decltype(kc)::value;
      const void* fn = a.bf16 ? (r32 ? (const void*)retrieve_tile_kernel<__nv_bfloat16, KC, 32>
                                     : (const void*)retrieve_tile_kernel<__nv_bfloat16, KC, 64>)
                              : (const void*)retrieve_tile_kernel<float, KC, 64>;
      cudaError_t e2 = allow_smem(fn, smem);
      if (e2 != cudaSuccess) return e2;
      launch_begin("retrieve_tile", s);
      if (cl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kTileThreads);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)p.nsplit;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (r32) e2 = cudaLaunchKernelEx(&cfg, retrieve_tile_kernel<__nv_bfloat16, KC, 32>, a, p.nsplit, p.seg, 1);
        else e2 = cudaLaunchKernelEx(&cfg, retrieve_tile_kernel<__nv_bfloat16, KC, 64>, a, p.nsplit, p.seg, 1);
        if (e2 == cudaSuccess) return launch_end("retrieve_tile", s);
        // A cluster launch the device cannot place is refused before anything runs: take
        // the plain launch and the merge launch instead.
        (void)cudaGetLastError();
        cl = false;
      }
      if (a.bf16 && r32) {
        retrieve_tile_kernel<__nv_bfloat16, KC, 32><<<grid, kTileThreads, smem, s>>>(a, p.nsplit, p.seg, 0);
      } else if (a.bf16) {
        retrieve_tile_kernel<__nv_bfloat16, KC, 64><<<grid, kTileThreads, smem, s>>>(a, p.nsplit, p.seg, 0);
      } else {
        retrieve_tile_kernel<float, KC, 64><<<grid, kTileThreads, smem, s>>>(a, p.nsplit, p.seg, 0);
      }
      return launch_end("retrieve_tile", s);
    });
    if (cl) nsplit = 1;  // merged already
  }
  if (e != cudaSuccess || nsplit == 1) return e;
  const long long rows = (long long)a.B * a.nQ;
  return with_kc(a.topk, [&](auto kc) -> cudaError_t {
    constexpr int KC = decltype(kc)::value;
    // Each variant has its own launch name, so that the profile table and the tests can
    // tell which one ran.
    const char* name;
    if (rows >= kWarpMergeRows && nsplit <= 32 && (long long)nsplit * a.topk <= kHeadsMax) {
      name = "retrieve_merge_heads";
      launch_begin(name, s);
      retrieve_merge_heads_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a, nsplit, (int)rows);
    } else if (rows >= kWarpMergeRows) {  // a warp per row, lists into registers
      name = "retrieve_merge_warp";
      launch_begin(name, s);
      retrieve_merge_warp_kernel<KC><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a, nsplit, (int)rows);
    } else {  // a block per row: few rows, long lists (decode)
      name = "retrieve_merge_block";
      launch_begin(name, s);
      retrieve_merge_kernel<KC><<<dim3(a.nQ, a.B), 128, 0, s>>>(a, nsplit);
    }
    return launch_end(name, s);
  });
}

}  // namespace gca
