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
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gca {
namespace {

using bf16 = __nv_bfloat16;

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
// Same decomposition on the 5th-generation tensor cores, warp-specialised.
//   * Warp 4 (control): lane 0 issues the TMA tile loads (Q once; K and V of each
//     retrieved chunk into a 2-stage ring); the whole warp waits on the mbarriers and
//     issues tcgen05.mma through an elected lane (M = 64 query rows, N = 64, K steps of
//     16).  S = Q K^T goes to TMEM columns 0-63; the fused output O, accumulated over
//     all slots, to columns 64-127.
//   * Warps 0-3 (softmax): read S with tcgen05.ld, do the row softmax in registers and
//     store P~ = (w_m / l) P as bf16 pairs into TMEM columns 0-31 (over the S they have
//     read), where it is the A operand of O += P~ V (V from shared memory, MN-major).
// Per slot: the softmax warps take S(m) from the MMA-completion mbarrier and hand P~(m)
// back through a named barrier; the control warp then issues O += P~(m) V(m) followed by
// S(m+1) = Q K(m+1)^T.  The tensor pipe runs one CTA's MMAs in issue order, so S(m+1)
// overwrites columns 0-63 only after the PV product has read P~(m); and S(m+1) complete
// implies PV(m) complete, so P~(m+1) may be stored once S(m+1) has been read.  128 TMEM
// columns per CTA let four CTAs share an SM and overlap one another's softmax and MMAs.
constexpr int kFwdStages = 2;  // the descriptor selection below assumes two stages
// Q and the ring of (K, V) take 41 KB; the request is padded to 46 KB so that at most
// four CTAs share an SM: a fifth would find all 512 TMEM columns taken.
constexpr int kFwdTcSmem = 46 * 1024 + 1024;
constexpr int kFwdThreads = 160;
enum { kBarPReady = 2 };

__global__ void __launch_bounds__(kFwdThreads, 4)
gca_fwd_tc_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  constexpr int DH = 64, ROWB = 128, TILE = 8192, UPR = 8, NST = kFwdStages, NT = kFwdThreads;
  constexpr uint32_t kIdS = tc::idesc_bf16(64, 64, false);
  constexpr uint32_t kIdPV = tc::idesc_bf16(64, DH, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* Qs = sm;
  unsigned char* ring = sm + TILE;  // stage st: K at ring + 2*st*TILE, V after it
  __shared__ float w_s[kMaxTopk];
  __shared__ int j_s[kMaxTopk];
  __shared__ int slot_s[kMaxTopk];
  __shared__ int nslot_s;
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar_q, bar_kv[NST], bar_s, bar_o;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  bf16* og = reinterpret_cast<bf16*>(a.o) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  float* lse = a.lse + (((int64_t)b * a.nQ + c) * a.H + h) * a.topk * 64;
  const int r = c - a.shift;
  const int bkv = a.kv_bs == 0 ? 0 : b;

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
      tc::mbar_init(&bar_q, 1);
      for (int st = 0; st < NST; ++st) tc::mbar_init(&bar_kv[st], 1);
      tc::mbar_init(&bar_s, 1);
      tc::mbar_init(&bar_o, 1);
      tc::fence_mbar_init();
    }
  }
  __syncthreads();
  const int ns = nslot_s;
  for (int x = tid; x < a.topk * 64; x += NT)
    if (j_s[x >> 6] < 0) lse[x] = -CUDART_INF_F;
  if (ns == 0) {
    for (int u = tid; u < 64 * UPR; u += NT) {
      const int row = u / UPR, w = u % UPR;
      *reinterpret_cast<uint4*>(og + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 128);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tS = tmem_slot, tO = tmem_slot + 64;

  if (warp == 4) {
    // ------------------------------------------------------------ control warp
    bool ok = true;
    auto load_slot = [&](int x) {  // K, V tiles of slot x into stage x % NST (lane 0)
      const int st = x % NST;
      const int j = j_s[slot_s[x]];
      unsigned char* Ks = ring + 2 * st * TILE;
      tc::mbar_expect_tx(&bar_kv[st], 2 * TILE);
      tc::tma_load_4d(Ks, &tmK, 0, h, j * 64, bkv, &bar_kv[st]);
      tc::tma_load_4d(Ks + TILE, &tmV, 0, h, j * 64, bkv, &bar_kv[st]);
    };
    // Operand descriptors, built once: Q and the K / V tile of every ring stage.
    const uint64_t dQ = tc::desc_km(tc::su32(Qs));
    uint64_t dK[NST], dV[NST];
#pragma unroll
    for (int st = 0; st < NST; ++st) {
      dK[st] = tc::desc_km(tc::su32(ring + 2 * st * TILE));
      dV[st] = tc::desc_mn(tc::su32(ring + (2 * st + 1) * TILE));
    }
    auto issue_s = [&](int x) {  // whole warp
      const uint64_t dk = x % NST == 0 ? dK[0] : dK[1];
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks)
        tc::mma_warp(tS, dQ + ks * tc::kKStepKm, dk + ks * tc::kKStepKm, kIdS, ks > 0 ? 1u : 0u);
      tc::commit_warp(&bar_s);
    };
    if (lane == 0) {
      tc::mbar_expect_tx(&bar_q, TILE);
      tc::tma_load_4d(Qs, &tmQ, 0, h, c * 64, b, &bar_q);
      for (int x = 0; x < NST && x < ns; ++x) load_slot(x);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bar_q, 0) && ok;
    ok = tc::mbar_wait(&bar_kv[0], 0) && ok;
    issue_s(0);
    for (int si = 0; si < ns; ++si) {
      tc::named_sync(kBarPReady, NT);  // P~(si) is in TMEM columns 0-31
      tc::fence_after();
      const uint64_t dv = si % NST == 0 ? dV[0] : dV[1];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_ts_warp(tO, tS + 8 * kk, dv + kk * tc::kKStepMn, kIdPV, (si > 0 || kk > 0) ? 1u : 0u);
      tc::commit_warp(&bar_o);
      if (si + 1 < ns) {
        ok = tc::mbar_wait(&bar_kv[(si + 1) % NST], ((si + 1) / NST) & 1) && ok;
        issue_s(si + 1);
      }
      ok = tc::mbar_wait(&bar_o, si & 1) && ok;  // ring stage si % NST is free
      if (lane == 0) {
        if (si + NST < ns) load_slot(si + NST);
        if (!ok) flag_timeout(a.err);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int g = lane >> 2, cq = lane & 3;
    const int row0 = 16 * warp + g;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * 1.4426950408889634f;
    for (int si = 0; si < ns; ++si) {
      // Acquire S(si) straight from the MMA-completion barrier (S(si+1) is only issued
      // after every softmax thread has handed over P~(si), so the phase cannot run ahead).
      if (!tc::mbar_wait(&bar_s, si & 1)) flag_timeout(a.err);
      float s[8][4];
#pragma unroll
      for (int cb = 0; cb < 8; ++cb) tc::ld16x256(tS + lane_base + cb * 8, s[cb]);
      tc::ld_wait(s);
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
      const float o0 = -mx0 * sl2, o1 = -mx1 * sl2;
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        s[n][0] = tc::ex2(fmaf(s[n][0], sl2, o0));
        s[n][1] = tc::ex2(fmaf(s[n][1], sl2, o0));
        s[n][2] = tc::ex2(fmaf(s[n][2], sl2, o1));
        s[n][3] = tc::ex2(fmaf(s[n][3], sl2, o1));
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
      if (cq == 0) {
        lse[mslot * 64 + row0] = mx0 * scale + __logf(l0);
        lse[mslot * 64 + row0 + 8] = mx1 * scale + __logf(l1);
      }
      const float c0 = __fdividef(wm, l0), c1 = __fdividef(wm, l1);
      // P~ as the TMEM A operand: the pair of keys (8n + 2cq, +1) of rows g and g + 8
      // goes to column 4n + cq (two 16-column stores).
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pv[2 * i] = pack_bf16(s[4 * half + i][0] * c0, s[4 * half + i][1] * c0);
          pv[2 * i + 1] = pack_bf16(s[4 * half + i][2] * c1, s[4 * half + i][3] * c1);
        }
        tc::st16x128_x4(tS + lane_base + 16 * half, pv);
      }
      tc::st_wait();
      tc::fence_before();
      tc::named_arrive(kBarPReady, NT);
    }
  }
  // Every O += P~ V has completed (the control warp waited for the last one).
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp < 4) {
    const int g = lane >> 2, cq = lane & 3;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    float o[8][4];
#pragma unroll
    for (int cb = 0; cb < 8; ++cb) tc::ld16x256(tO + lane_base + cb * 8, o[cb]);
    tc::ld_wait(o);
    // Stage O through the Q tile (its last reader, the final S = Q K^T, is done).
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      const int r0 = 16 * warp + g;
      *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0, n) + cq * 4) = pack_bf16(o[n][0], o[n][1]);
      *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0 + 8, n) + cq * 4) = pack_bf16(o[n][2], o[n][3]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tmem_slot, 128);
  }
  for (int u = tid; u < 64 * UPR; u += NT) {
    const int row = u / UPR, w = u % UPR;
    *reinterpret_cast<uint4*>(og + row * ts + w * 8) = *reinterpret_cast<const uint4*>(Qs + swz<ROWB>(row, w));
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
    if (e != cudaSuccess) return e;
    launch_begin("gca_fwd", s);
    gca_fwd_tc_kernel<<<grid, kFwdThreads, kFwdTcSmem, s>>>(a, tq, tk, tv);
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
