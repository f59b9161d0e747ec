// GCA forward: per retrieved chunk cross-attention with its own softmax, fused with the
// softmax(retrieval score) weighting of the k results.
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", section 关键设计 / key design, item "Grouped
// Cross-Attention": every token of the current chunk attends to each retrieved chunk
// separately, and the outputs are combined with the softmax-normalised retrieval
// scores (unlike chunked cross-attention, which concatenates the chunks under one
// softmax).  Query chunk c uses retrieval row c - shift (the next-chunk rule).
//
// One CTA per (query chunk, head, sequence), launched head-major so that the CTAs in
// flight share one sequence-head's K/V (4 MB at L = 16K) in L2.  Per valid slot: a
// 64 x 64 x dh tile S = Q K^T, a row softmax in registers, and O += (w_m / l) P V.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "waits.cuh"

namespace gca {
namespace {

using bf16 = __nv_bfloat16;
constexpr int UPR_FWD = 8;  // 16-byte units per 64-element bf16 row

// ------------------------------------------------------------------ bf16 tensor-core path
template <int DH>
__global__ void __launch_bounds__(128) gca_fwd_mma_kernel(FwdArgs a) {
  constexpr int ROWB = DH * 2;     // bytes per 64-element tile row
  constexpr int TILE = 64 * ROWB;  // bytes per tile
  constexpr int UPR = ROWB / 16;   // 16-byte units per row
  __shared__ __align__(1024) unsigned char sm[TILE * 5];  // Q, 2 x (K, V)
  __shared__ float w_s[kMaxTopk];
  __shared__ int j_s[kMaxTopk];
  __shared__ int slot_s[kMaxTopk];
  __shared__ int nslot_s;
  unsigned char* Qs = sm;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;  // elements between consecutive tokens
  const bf16* qg = reinterpret_cast<const bf16*>(a.q) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  bf16* og = reinterpret_cast<bf16*>(a.o) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  float* lse = a.lse + (((int64_t)b * a.nQ + c) * a.H + h) * a.topk * 64;
  const int r = c - a.shift;

  if (warp == 0) {
    if (r >= 0) {
      row_weights_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk, a.scores + ((int64_t)b * a.nQ + r) * a.topk,
                       a.topk, a.nC, w_s, j_s, a.err);
    } else if (lane < a.topk) {
      w_s[lane] = 0.f;
      j_s[lane] = -1;
    }
    __syncwarp();
    if (lane == 0) {
      int n = 0;
      for (int m = 0; m < a.topk; ++m)
        if (j_s[m] >= 0) slot_s[n++] = m;
      nslot_s = n;
    }
  }
  __syncthreads();
  const int ns = nslot_s;
  for (int x = tid; x < a.topk * 64; x += 128)
    if (j_s[x >> 6] < 0) lse[x] = -CUDART_INF_F;
  if (ns == 0) {
    for (int u = tid; u < 64 * UPR; u += 128) {
      const int row = u / UPR, w = u % UPR;
      *reinterpret_cast<uint4*>(og + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  const bf16* kbase = reinterpret_cast<const bf16*>(a.k) + (int64_t)b * a.kv_bs + h * DH;
  const bf16* vbase = reinterpret_cast<const bf16*>(a.v) + (int64_t)b * a.kv_bs + h * DH;
  for (int u = tid; u < 64 * UPR; u += 128) {
    const int row = u / UPR, w = u % UPR;
    cp_async16(Qs + swz<ROWB>(row, w), qg + row * ts + w * 8);
  }
  auto load_kv = [&](int si, int stage) {
    const int64_t j = j_s[slot_s[si]];
    unsigned char* Ks = sm + TILE * (1 + 2 * stage);
    unsigned char* Vs = Ks + TILE;
    const bf16* kg = kbase + j * 64 * ts;
    const bf16* vg = vbase + j * 64 * ts;
    for (int u = tid; u < 64 * UPR; u += 128) {
      const int row = u / UPR, w = u % UPR;
      cp_async16(Ks + swz<ROWB>(row, w), kg + row * ts + w * 8);
      cp_async16(Vs + swz<ROWB>(row, w), vg + row * ts + w * 8);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  const float scale = 1.0f / sqrtf((float)DH);
  const float sl2 = scale * 1.4426950408889634f;
  float o[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
  uint32_t qf[DH / 16][4];
  const int g = lane >> 2;

  for (int si = 0; si < ns; ++si) {
    const int stage = si & 1;
    if (si + 1 < ns) load_kv(si + 1, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (si == 0) {
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks)
        ldsm_x4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3],
                smem_u32(Qs) + swz<ROWB>(16 * warp + (lane & 15), 2 * ks + (lane >> 4)));
    }
    const uint32_t ksm = smem_u32(sm + TILE * (1 + 2 * stage));
    const uint32_t vsm = ksm + TILE;
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, ksm + swz<ROWB>(16 * p + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)));
        mma_bf16(s[2 * p], qf[ks], b0, b1);
        mma_bf16(s[2 * p + 1], qf[ks], b2, b3);
      }
    }
    // Row softmax: this thread holds rows g and g+8 of the warp's 16 rows.
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
      mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
    }
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      s[n][0] = exp2f((s[n][0] - mx0) * sl2);
      s[n][1] = exp2f((s[n][1] - mx0) * sl2);
      s[n][2] = exp2f((s[n][2] - mx1) * sl2);
      s[n][3] = exp2f((s[n][3] - mx1) * sl2);
      l0 += s[n][0] + s[n][1];
      l1 += s[n][2] + s[n][3];
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, m);
      l1 += __shfl_xor_sync(0xffffffffu, l1, m);
    }
    const int mslot = slot_s[si];
    const float wm = w_s[mslot];
    if ((lane & 3) == 0) {
      lse[mslot * 64 + 16 * warp + g] = mx0 * scale + logf(l0);
      lse[mslot * 64 + 16 * warp + g + 8] = mx1 * scale + logf(l1);
    }
    const float c0 = wm / l0, c1 = wm / l1;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0] * c0, s[2 * kk][1] * c0);
      pa[1] = pack_bf16(s[2 * kk][2] * c1, s[2 * kk][3] * c1);
      pa[2] = pack_bf16(s[2 * kk + 1][0] * c0, s[2 * kk + 1][1] * c0);
      pa[3] = pack_bf16(s[2 * kk + 1][2] * c1, s[2 * kk + 1][3] * c1);
#pragma unroll
      for (int dp = 0; dp < DH / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, vsm + swz<ROWB>(16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dp + (lane >> 4)));
        mma_bf16(o[2 * dp], pa, b0, b1);
        mma_bf16(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  // Epilogue: stage O through shared memory (the Q tile is no longer needed) and write
  // 16-byte rows.
  const int cq = lane & 3;
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) {
    const int r0 = 16 * warp + g;
    *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0, n) + cq * 4) = pack_bf16(o[n][0], o[n][1]);
    *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0 + 8, n) + cq * 4) = pack_bf16(o[n][2], o[n][3]);
  }
  __syncthreads();
  for (int u = tid; u < 64 * UPR; u += 128) {
    const int row = u / UPR, w = u % UPR;
    *reinterpret_cast<uint4*>(og + row * ts + w * 8) = *reinterpret_cast<const uint4*>(Qs + swz<ROWB>(row, w));
  }
}


// ------------------------------------------------------------------ bf16 tcgen05 path (dh = 64)
// Same decomposition on the 5th-generation tensor cores, warp-specialised and persistent:
// four CTAs per SM, each walking the tiles (query chunk, head, sequence) blockIdx.x,
// blockIdx.x + gridDim.x, ... in head-major order (the CTAs in flight share one
// sequence-head's K/V in L2), the light first chunks of every sequence-head last
// (query_tile).  Roles:
//   * warp 6 (metadata): each tile's retrieval row (valid slots, chunks, fusion weights)
//     into a ring of records, a few tiles ahead;
//   * warp 5 (producer, lane 0): Q of each tile into one of two buffers, and the K and V
//     tiles of its slots into a 2-stage ring that runs on across tiles;
//   * warp 4 (MMA): per slot S = Q K^T into TMEM columns 0-63, then, once the softmax warps
//     have stored P~, O += P~ V into columns 64-127 (M = 64, N = 64, K steps of 16); the
//     next slot's S goes into the same columns after the PV product (the tensor pipe runs
//     this warp's products in issue order), across tile boundaries too;
//   * warps 0-3 (softmax): read S with tcgen05.ld, do the row softmax in registers (packed
//     f32x2 arithmetic on pairs of columns), write the slot's LSE row and store
//     P~ = (w_m / l) P as bf16 pairs into TMEM columns 0-31, the A operand of O += P~ V
//     (V MN-major from shared memory).  After a tile's last slot
//     they read O, release the accumulator and write O out as bf16 from registers.
// A tile's only start-up cost is then reading O out: the next tile's metadata, Q and first
// K/V tiles are loaded while the current tile runs.
constexpr int kFwdStages = 2;
constexpr int kFwdMetaRecs = 4;
constexpr int kFwdThreads = 224;
constexpr int kFwdMma = 4, kFwdProd = 5, kFwdMeta = 6;
constexpr int kFwdTcSmem = 2 * 8192 + kFwdStages * 2 * 8192 + 1024;  // Q x 2, ring of (K, V)

struct FwdMeta {
  int c, h, b, ns, end;
  int slot[kMaxTopk];
  int j[kMaxTopk];
  float w[kMaxTopk];
};

__global__ void __launch_bounds__(kFwdThreads, 4)
gca_fwd_tc_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  constexpr int DH = 64, TILE = 8192, NST = kFwdStages, MR = kFwdMetaRecs;
  constexpr uint32_t kIdS = tc::idesc_bf16(64, 64, false);
  constexpr uint32_t kIdPV = tc::idesc_bf16(64, DH, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* qbuf = sm;             // buffer x at qbuf + x TILE
  unsigned char* ring = sm + 2 * TILE;  // stage st: K at ring + 2 st TILE, V after it
  __shared__ FwdMeta meta[MR];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  __shared__ __align__(8) uint64_t meta_full[MR], meta_empty[MR], bar_q[2], qfree[2], bar_kv[NST], ring_empty[NST],
      bar_s, pready, o_full, o_free, drain;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int ntiles = a.nQ * a.H * a.B;
  if (warp == kFwdProd && lane == 0) {
    for (int x = 0; x < MR; ++x) {
      tc::mbar_init(&meta_full[x], 1);
      tc::mbar_init(&meta_empty[x], 6);  // softmax warps, MMA warp, producer
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&bar_q[x], 1);
      tc::mbar_init(&qfree[x], 1);
    }
    for (int st = 0; st < NST; ++st) {
      tc::mbar_init(&bar_kv[st], 1);
      tc::mbar_init(&ring_empty[st], 1);
    }
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&pready, 4);
    tc::mbar_init(&o_full, 1);
    tc::mbar_init(&o_free, 4);
    tc::mbar_init(&drain, 1);
    tc::fence_mbar_init();
    abort_s = 0;
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 128);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tS = tmem_slot, tO = tmem_slot + 64;
  // Every role parks while it waits (try_wait with a suspend hint), so that a waiting warp
  // leaves its SM sub-partition's issue slots to the warps that work.
  auto P = [&](uint64_t* bar, uint32_t parity, int site, int tile, int slot) {
    return park_or_abort(bar, parity, &abort_s, a.err, site, tile, slot);
  };


  if (warp == kFwdMeta) {
    // ------------------------------------------------------------ metadata warp
    int k = 0;
    for (int t = blockIdx.x;; t += gridDim.x, ++k) {
      const int mb = k % MR;
      if (k >= MR && !P(&meta_empty[mb], ((k / MR) - 1) & 1, 40, k, -1)) break;
      FwdMeta& M = meta[mb];
      if (t >= ntiles) {
        if (lane == 0) {
          M.end = 1;
          tc::mbar_arrive(&meta_full[mb]);
        }
        break;
      }
      int c, h, b;
      query_tile(a.nQ, a.H, a.B, min(a.nQ, a.shift + a.topk), t, c, h, b);
      const int r = c - a.shift;
      if (r >= 0) {
        row_weights_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk, a.scores + ((int64_t)b * a.nQ + r) * a.topk,
                         a.topk, a.nC, M.w, M.j, a.err);
      } else if (lane < a.topk) {
        M.w[lane] = 0.f;
        M.j[lane] = -1;
      }
      __syncwarp();
      if (lane == 0) {
        int n = 0;
        for (int m = 0; m < a.topk; ++m)
          if (M.j[m] >= 0) M.slot[n++] = m;
        M.ns = n;
        M.c = c;
        M.h = h;
        M.b = b;
        M.end = 0;
        tc::mbar_arrive(&meta_full[mb]);
      }
      __syncwarp();
    }
  } else if (warp == kFwdProd) {
    // ------------------------------------------------------------ producer warp (lane 0)
    if (lane == 0) {
      int gs = 0, tq = 0, nq[2] = {0, 0}, nkv[NST];
      for (int st = 0; st < NST; ++st) nkv[st] = 0;
      for (int k = 0;; ++k) {
        const int mb = k % MR;
        if (!P(&meta_full[mb], (k / MR) & 1, 41, k, -1)) break;
        const FwdMeta& M = meta[mb];
        if (M.end) break;
        const int ns = M.ns, c = M.c, h = M.h, b = M.b;
        const int bkv = a.kv_bs == 0 ? 0 : b;
        bool ok = true;
        if (ns > 0) {
          const int qb = tq & 1;
          if (tq >= 2 && !P(&qfree[qb], ((tq >> 1) - 1) & 1, 42, k, -1)) break;
          tc::mbar_expect_tx(&bar_q[qb], TILE);
          tc::tma_load_4d(qbuf + qb * TILE, &tmQ, 0, h, c * 64, b, &bar_q[qb]);
          ++nq[qb];
          for (int x = 0; x < ns; ++x, ++gs) {
            const int st = gs % NST;
            if (gs >= NST && !P(&ring_empty[st], ((gs / NST) - 1) & 1, 43, k, gs)) {
              ok = false;
              break;
            }
            const int j = M.j[M.slot[x]];
            unsigned char* Ks = ring + 2 * st * TILE;
            tc::mbar_expect_tx(&bar_kv[st], 2 * TILE);
            tc::tma_load_4d(Ks, &tmK, 0, h, j * 64, bkv, &bar_kv[st]);
            tc::tma_load_4d(Ks + TILE, &tmV, 0, h, j * 64, bkv, &bar_kv[st]);
            ++nkv[st];
          }
          ++tq;
        }
        tc::mbar_arrive(&meta_empty[mb]);
        if (!ok) break;
      }
      // After an abort, let the copies already issued land before the CTA exits.
      if (*reinterpret_cast<volatile int*>(&abort_s)) {
        for (int x = 0; x < 2; ++x)
          if (nq[x] > 0) tc::mbar_wait(&bar_q[x], (nq[x] - 1) & 1);
        for (int st = 0; st < NST; ++st)
          if (nkv[st] > 0) tc::mbar_wait(&bar_kv[st], (nkv[st] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kFwdMma) {
    // ------------------------------------------------------------ MMA warp
    const uint64_t dQ0 = tc::desc_km(tc::su32(qbuf));
    const uint64_t dRingKm = tc::desc_km(tc::su32(ring)), dRingMn = tc::desc_mn(tc::su32(ring));
    constexpr uint64_t kTileStep = TILE >> 4, kStage = (2 * TILE) >> 4;
    bool issued = false;
    int gs = 0, tq = 0;
    // S of global slot g (tile with Q buffer qb).
    auto issue_s = [&](int g, int qb) -> bool {
      if (!P(&bar_kv[g % NST], (g / NST) & 1, 44, -1, g)) return false;
      const uint64_t dq = dQ0 + qb * kTileStep, dk = dRingKm + (g % NST) * kStage;
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tS, dq, dk, kIdS, 0u);
      tc::commit_warp(&bar_s);
      issued = true;
      return true;
    };
    bool alive = true;
    bool pending_s = false;  // S of the current tile's first slot was issued at the end of the last tile
    for (int k = 0; alive; ++k) {
      const int mb = k % MR;
      if (!P(&meta_full[mb], (k / MR) & 1, 45, k, -1)) break;
      const int ns = meta[mb].ns, end = meta[mb].end;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&meta_empty[mb]);
      if (end) break;
      if (ns == 0) continue;
      const int qb = tq & 1;
      if (!pending_s) {
        if (!P(&bar_q[qb], (tq >> 1) & 1, 46, k, -1)) break;
        if (!issue_s(gs, qb)) break;
      }
      pending_s = false;
      for (int si = 0; si < ns; ++si, ++gs) {
        if (!P(&pready, gs & 1, 47, k, gs)) {  // P~(gs) is in TMEM columns 0-31
          alive = false;
          break;
        }
        tc::fence_after();
        if (si == 0 && tq >= 1 && !P(&o_free, (tq - 1) & 1, 48, k, gs)) {  // the last tile's O is read
          alive = false;
          break;
        }
        const uint64_t dv = dRingMn + (gs % NST) * kStage + kTileStep;
        tc::mma4_ts<8, 16, 24, tc::kKStepMn>(tO, tS, dv, kIdPV, si > 0 ? 1u : 0u);
        tc::commit_warp(&ring_empty[gs % NST]);
        if (si + 1 < ns) {
          if (!issue_s(gs + 1, qb)) {
            alive = false;
            break;
          }
        } else {
          tc::commit_warp(&qfree[qb]);
          tc::commit_warp(&o_full);
          // The next tile's first S right away, if its metadata and Q are in.
          const int nb = (k + 1) % MR;
          if (tc::mbar_test(&meta_full[nb], ((k + 1) / MR) & 1)) {
            const FwdMeta& N = meta[nb];
            if (!N.end && N.ns > 0 && P(&bar_q[(tq + 1) & 1], ((tq + 1) >> 1) & 1, 46, k + 1, -1)) {
              if (!issue_s(gs + 1, (tq + 1) & 1)) {
                alive = false;
                break;
              }
              pending_s = true;
            }
          }
        }
      }
      ++tq;
    }
    // No product may still be running when TMEM is released (after an abort in particular).
    if (issued) {
      tc::commit_warp(&drain);
      if (!tc::mbar_wait(&drain, 0) && lane == 0) flag_timeout(a.err, 49, blockIdx.x, -1, gs);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int g = lane >> 2, cq = lane & 3;
    const int row0 = 16 * warp + g;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * 1.4426950408889634f;
    int gs = 0, tq = 0;
    for (int k = 0;; ++k) {
      const int mb = k % MR;
      if (!P(&meta_full[mb], (k / MR) & 1, 50, k, -1)) break;
      const FwdMeta& M = meta[mb];
      if (M.end) break;
      const int ns = M.ns, c = M.c, h = M.h, b = M.b;
      float* lse = a.lse + (((int64_t)b * a.nQ + c) * a.H + h) * a.topk * 64;
      bf16* og = reinterpret_cast<bf16*>(a.o) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
      // LSE rows of the slots that retrieved nothing.
      for (int x = tid; x < a.topk * 64; x += 128)
        if (M.j[x >> 6] < 0) lse[x] = -CUDART_INF_F;
      if (ns == 0) {  // nothing retrieved: O is zero
        for (int u = tid; u < 64 * UPR_FWD; u += 128) {
          const int row = u / UPR_FWD, w = u % UPR_FWD;
          *reinterpret_cast<uint4*>(og + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&meta_empty[mb]);
        continue;
      }
      bool alive = true;
      for (int si = 0; si < ns; ++si, ++gs) {
        // S(gs) from the MMA-completion barrier (the next S is issued only after every
        // softmax warp has handed over P~(gs), so the phase cannot run ahead).
        if (!P(&bar_s, gs & 1, 51, k, gs)) {
          alive = false;
          break;
        }
        float s[8][4];
        tc::ld16x256_x8(tS + lane_base, s);
        tc::ld_wait(s);
        float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          mx0 = tc::max3(mx0, s[n][0], s[n][1]);
          mx1 = tc::max3(mx1, s[n][2], s[n][3]);
        }
#pragma unroll
        for (int m = 1; m <= 2; m <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
        }
        const uint64_t sl2x2 = tc::f2(sl2, sl2);
        const uint64_t o0 = tc::f2(-mx0 * sl2, -mx0 * sl2), o1 = tc::f2(-mx1 * sl2, -mx1 * sl2);
        uint64_t l0x2 = tc::f2(0.f, 0.f), l1x2 = l0x2;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          float x0, x1, x2, x3;
          tc::uf2(tc::fma2(tc::f2(s[n][0], s[n][1]), sl2x2, o0), x0, x1);
          tc::uf2(tc::fma2(tc::f2(s[n][2], s[n][3]), sl2x2, o1), x2, x3);
          s[n][0] = tc::ex2(x0);
          s[n][1] = tc::ex2(x1);
          s[n][2] = tc::ex2(x2);
          s[n][3] = tc::ex2(x3);
          l0x2 = tc::add2(l0x2, tc::f2(s[n][0], s[n][1]));
          l1x2 = tc::add2(l1x2, tc::f2(s[n][2], s[n][3]));
        }
        float l0, l1;
        {
          float u0, u1;
          tc::uf2(l0x2, u0, u1);
          l0 = u0 + u1;
          tc::uf2(l1x2, u0, u1);
          l1 = u0 + u1;
        }
#pragma unroll
        for (int m = 1; m <= 2; m <<= 1) {
          l0 += __shfl_xor_sync(0xffffffffu, l0, m);
          l1 += __shfl_xor_sync(0xffffffffu, l1, m);
        }
        const int mslot = M.slot[si];
        const float wm = M.w[mslot];
        if (cq == 0) {
          lse[mslot * 64 + row0] = mx0 * scale + __logf(l0);
          lse[mslot * 64 + row0 + 8] = mx1 * scale + __logf(l1);
        }
        const float c0 = __fdividef(wm, l0), c1 = __fdividef(wm, l1);
        const uint64_t c0x2 = tc::f2(c0, c0), c1x2 = tc::f2(c1, c1);
        // P~ as the TMEM A operand: the pair of keys (8n + 2cq, +1) of rows g and g + 8
        // goes to column 4n + cq (two 16-column stores).
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pv[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a0, a1, b0, b1;
            tc::uf2(tc::mul2(tc::f2(s[4 * half + i][0], s[4 * half + i][1]), c0x2), a0, a1);
            tc::uf2(tc::mul2(tc::f2(s[4 * half + i][2], s[4 * half + i][3]), c1x2), b0, b1);
            pv[2 * i] = pack_bf16(a0, a1);
            pv[2 * i + 1] = pack_bf16(b0, b1);
          }
          tc::st16x128_x4(tS + lane_base + 16 * half, pv);
        }
        tc::st_wait();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&pready);
      }
      if (!alive) break;
      // The tile's O: from TMEM (once the last O += P~ V is done), then straight to global
      // memory from registers.
      if (!P(&o_full, tq & 1, 52, k, gs)) break;
      tc::fence_after();
      float o[8][4];
      tc::ld16x256_x8(tO + lane_base, o);
      tc::ld_wait(o);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&o_free);
        tc::mbar_arrive(&meta_empty[mb]);
      }
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int col = 8 * n + 2 * cq;
        *reinterpret_cast<uint32_t*>(og + (int64_t)row0 * ts + col) = pack_bf16(o[n][0], o[n][1]);
        *reinterpret_cast<uint32_t*>(og + (int64_t)(row0 + 8) * ts + col) = pack_bf16(o[n][2], o[n][3]);
      }
      ++tq;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tmem_slot, 128);
  }
}

// ------------------------------------------------------------------ f32 SIMT path
// One thread per query token; exact fp32 products and expf, for the f32 configuration.
template <int DH>
__global__ void __launch_bounds__(64) gca_fwd_f32_kernel(FwdArgs a) {
  __shared__ float Ks[64][DH + 1];
  __shared__ float Vs[64][DH + 1];
  __shared__ float w_s[kMaxTopk];
  __shared__ int j_s[kMaxTopk];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x;
  const int64_t ts = (int64_t)a.H * DH;
  const float* qg = reinterpret_cast<const float*>(a.q) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  float* og = reinterpret_cast<float*>(a.o) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  float* lse = a.lse + (((int64_t)b * a.nQ + c) * a.H + h) * a.topk * 64;
  const int r = c - a.shift;
  if (t < 32) {
    if (r >= 0) {
      row_weights_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk, a.scores + ((int64_t)b * a.nQ + r) * a.topk,
                       a.topk, a.nC, w_s, j_s, a.err);
    } else if (t < a.topk) {
      w_s[t] = 0.f;
      j_s[t] = -1;
    }
  }
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)DH);
  float qv[DH], o[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    qv[d] = qg[t * ts + d];
    o[d] = 0.f;
  }
  for (int m = 0; m < a.topk; ++m) {
    const int64_t j = j_s[m];
    if (j < 0) {
      lse[m * 64 + t] = -CUDART_INF_F;
      continue;
    }
    __syncthreads();
    const float* kg = reinterpret_cast<const float*>(a.k) + (int64_t)b * a.kv_bs + j * 64 * ts + h * DH;
    const float* vg = reinterpret_cast<const float*>(a.v) + (int64_t)b * a.kv_bs + j * 64 * ts + h * DH;
    for (int x = t; x < 64 * DH; x += 64) {
      const int row = x / DH, d = x % DH;
      Ks[row][d] = kg[row * ts + d];
      Vs[row][d] = vg[row * ts + d];
    }
    __syncthreads();
    float sc[64];
    float mx = -CUDART_INF_F;
#pragma unroll 4
    for (int key = 0; key < 64; ++key) {
      float acc = 0.f;
#pragma unroll
      for (int d = 0; d < DH; ++d) acc = fmaf(qv[d], Ks[key][d], acc);
      sc[key] = acc * scale;
      mx = fmaxf(mx, sc[key]);
    }
    float l = 0.f;
#pragma unroll 4
    for (int key = 0; key < 64; ++key) {
      sc[key] = expf(sc[key] - mx);
      l += sc[key];
    }
    lse[m * 64 + t] = mx + logf(l);
    const float coef = w_s[m] / l;
#pragma unroll 4
    for (int key = 0; key < 64; ++key) {
      const float p = sc[key] * coef;
#pragma unroll
      for (int d = 0; d < DH; ++d) o[d] = fmaf(p, Vs[key][d], o[d]);
    }
  }
#pragma unroll
  for (int d = 0; d < DH; ++d) og[t * ts + d] = o[d];
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s) {
  dim3 grid(a.nQ, a.H, a.B);
  if (a.bf16 && a.dh == 64) {
    CUtensorMap tq, tk, tv;
    cudaError_t e = make_head_tmap(&tq, a.q, 64, a.H, (int64_t)a.nQ * 64, a.B, (int64_t)a.nQ * 64 * a.H * 64);
    if (e == cudaSuccess) e = make_head_tmap(&tk, a.k, 64, a.H, (int64_t)a.nC * 64, a.B, a.kv_bs);
    if (e == cudaSuccess) e = make_head_tmap(&tv, a.v, 64, a.H, (int64_t)a.nC * 64, a.B, a.kv_bs);
    if (e == cudaSuccess) e = allow_smem((const void*)gca_fwd_tc_kernel, kFwdTcSmem);
    int dev = 0, sms = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long ntiles = (long long)a.nQ * a.H * a.B;
    const int g1 = (int)std::min<long long>(ntiles, 4LL * sms);  // four CTAs per SM (TMEM: 128 columns each)
    launch_begin("gca_fwd", s);
    gca_fwd_tc_kernel<<<g1, kFwdThreads, kFwdTcSmem, s>>>(a, tq, tk, tv);
    return launch_end("gca_fwd", s);
  }
  if (a.bf16) {
    launch_begin("gca_fwd_mma", s);
    gca_fwd_mma_kernel<32><<<grid, 128, 0, s>>>(a);
    return launch_end("gca_fwd_mma", s);
  }
  launch_begin("gca_fwd_f32", s);
  if (a.dh == 64) gca_fwd_f32_kernel<64><<<grid, 64, 0, s>>>(a);
  else gca_fwd_f32_kernel<32><<<grid, 64, 0, s>>>(a);
  return launch_end("gca_fwd_f32", s);
}

}  // namespace gca
