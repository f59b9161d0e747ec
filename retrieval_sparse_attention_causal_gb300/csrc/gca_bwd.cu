// GCA backward: dQ, dK, dV and the gradient into the retrieval scores.
//
// The scores enter the output only through the fusion weights w = softmax(scores); this
// is what lets the retriever learn from the language-model loss (Paper-Notes page on
// "Efficient Length-Generalizable Attention via Causal Retrieval for Long-Context
// Language Modeling", sections 研究背景与动机 / motivation, 关键设计 / key design, item
// "Grouped Cross-Attention", and 亮点与洞察 / insights).
//
// Kernels, in launch order:
//   gca_bwd_q   one CTA per (query chunk, head, sequence).  Recomputes P from the saved
//               LSE, forms dPo = dO V^T, D = rowsum(P * dPo) (= <dO, A_m>), dQ and the
//               per-head partial dw_m = sum_t D_m[t].  Saves D for the key-side pass.
//   gca_dscores one warp per retrieval row: dw_m = sum over heads, then
//               dscores = w * (dw - <w, dw>).
//   gca_csr     per sequence: counting sort of the (row, slot) entries by retrieved chunk,
//               stable, so every key chunk gets its consumers in a fixed order.
//   gca_bwd_kv  one CTA per (key chunk, head, sequence): loops over the chunk's
//               consumers and accumulates dK, dV in registers.  No atomics anywhere, so
//               the result is bitwise reproducible.
#include "common.cuh"
#include "internal.h"

namespace gca {
namespace {

using bf16 = __nv_bfloat16;
constexpr float kLog2e = 1.4426950408889634f;

// Weight of slot m of one retrieval row, evaluated by a full warp (all lanes return it).
__device__ __forceinline__ float slot_weight_warp(const int32_t* idx_row, const float* sc_row,
                                                  int topk, int nC, int m, ErrWord* err) {
  const int lane = threadIdx.x & 31;
  int j = -1;
  float s = -CUDART_INF_F;
  if (lane < topk) {
    j = idx_row[lane];
    if (j < -1 || j >= nC) {
      flag_bad_index(err, j);
      j = -1;
    }
    if (j >= 0) s = sc_row[lane];
  }
  float mx = s;
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
  float e = (j >= 0) ? expf(s - mx) : 0.f;
  float sum = e;
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, k);
  const float wl = (j >= 0) ? e / sum : 0.f;
  return __shfl_sync(0xffffffffu, wl, m);
}

// ------------------------------------------------------------------ gca_bwd_q (bf16)
template <int DH>
__global__ void __launch_bounds__(128) gca_bwd_q_mma_kernel(BwdArgs a) {
  constexpr int ROWB = DH * 2, TILE = 64 * ROWB, UPR = ROWB / 16;
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* Qs = sm;
  unsigned char* dOs = sm + TILE;
  __shared__ float w_s[kMaxTopk];
  __shared__ int j_s[kMaxTopk];
  __shared__ int slot_s[kMaxTopk];
  __shared__ int nslot_s;
  __shared__ float dwred[4][kMaxTopk];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2;
  const int64_t ts = (int64_t)a.H * DH;
  const int64_t tok0 = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  const bf16* qg = reinterpret_cast<const bf16*>(a.q) + tok0;
  const bf16* dog = reinterpret_cast<const bf16*>(a.dout) + tok0;
  bf16* dqg = reinterpret_cast<bf16*>(a.dq) + tok0;
  const int64_t rowbase = ((int64_t)b * a.nQ + c) * a.H + h;
  const float* lse = a.lse + rowbase * a.topk * 64;
  float* Dg = a.Dbuf + rowbase * a.topk * 64;
  float* dwp = a.dwp + rowbase * a.topk;
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
  if (tid < 4 * kMaxTopk) dwred[tid / kMaxTopk][tid % kMaxTopk] = 0.f;
  __syncthreads();
  const int ns = nslot_s;
  if (ns == 0) {
    for (int u = tid; u < 64 * UPR; u += 128) {
      const int row = u / UPR, w = u % UPR;
      *reinterpret_cast<uint4*>(dqg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
    }
    if (tid < a.topk) dwp[tid] = 0.f;
    return;
  }
  const bf16* kbase = reinterpret_cast<const bf16*>(a.k) + (int64_t)b * a.nC * 64 * ts + h * DH;
  const bf16* vbase = reinterpret_cast<const bf16*>(a.v) + (int64_t)b * a.nC * 64 * ts + h * DH;
  for (int u = tid; u < 64 * UPR; u += 128) {
    const int row = u / UPR, w = u % UPR;
    cp_async16(Qs + swz<ROWB>(row, w), qg + row * ts + w * 8);
    cp_async16(dOs + swz<ROWB>(row, w), dog + row * ts + w * 8);
  }
  auto load_kv = [&](int si, int stage) {
    const int64_t j = j_s[slot_s[si]];
    unsigned char* Ks = sm + TILE * (2 + 2 * stage);
    unsigned char* Vs = Ks + TILE;
    for (int u = tid; u < 64 * UPR; u += 128) {
      const int row = u / UPR, w = u % UPR;
      cp_async16(Ks + swz<ROWB>(row, w), kbase + (j * 64 + row) * ts + w * 8);
      cp_async16(Vs + swz<ROWB>(row, w), vbase + (j * 64 + row) * ts + w * 8);
    }
  };
  load_kv(0, 0);
  cp_async_commit();
  const float scale = 1.0f / sqrtf((float)DH);
  const float sl2 = scale * kLog2e;
  float dq[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dq[n][e] = 0.f;
  uint32_t qf[DH / 16][4], df[DH / 16][4];
  for (int si = 0; si < ns; ++si) {
    const int stage = si & 1;
    if (si + 1 < ns) load_kv(si + 1, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (si == 0) {
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
        const uint32_t off = swz<ROWB>(16 * warp + (lane & 15), 2 * ks + (lane >> 4));
        ldsm_x4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], smem_u32(Qs) + off);
        ldsm_x4(df[ks][0], df[ks][1], df[ks][2], df[ks][3], smem_u32(dOs) + off);
      }
    }
    const int m = slot_s[si];
    const float wm = w_s[m];
    const int row0 = 16 * warp + g;
    const float lse0 = lse[m * 64 + row0] * kLog2e, lse1 = lse[m * 64 + row0 + 8] * kLog2e;
    const uint32_t ksm = smem_u32(sm + TILE * (2 + 2 * stage));
    const uint32_t vsm = ksm + TILE;
    float s[8][4], dp[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = dp[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t off = swz<ROWB>(16 * p + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1));
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, ksm + off);
        mma_bf16(s[2 * p], qf[ks], b0, b1);
        mma_bf16(s[2 * p + 1], qf[ks], b2, b3);
        ldsm_x4(b0, b1, b2, b3, vsm + off);
        mma_bf16(dp[2 * p], df[ks], b0, b1);
        mma_bf16(dp[2 * p + 1], df[ks], b2, b3);
      }
    }
    float D0 = 0.f, D1 = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      s[n][0] = exp2f(s[n][0] * sl2 - lse0);
      s[n][1] = exp2f(s[n][1] * sl2 - lse0);
      s[n][2] = exp2f(s[n][2] * sl2 - lse1);
      s[n][3] = exp2f(s[n][3] * sl2 - lse1);
      D0 = fmaf(s[n][0], dp[n][0], fmaf(s[n][1], dp[n][1], D0));
      D1 = fmaf(s[n][2], dp[n][2], fmaf(s[n][3], dp[n][3], D1));
    }
#pragma unroll
    for (int k = 1; k <= 2; k <<= 1) {
      D0 += __shfl_xor_sync(0xffffffffu, D0, k);
      D1 += __shfl_xor_sync(0xffffffffu, D1, k);
    }
    float part = 0.f;
    if ((lane & 3) == 0) {
      Dg[m * 64 + row0] = D0;
      Dg[m * 64 + row0 + 8] = D1;
      part = D0 + D1;
    }
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) part += __shfl_xor_sync(0xffffffffu, part, k);
    if (lane == 0) dwred[warp][m] = part;
    const float cs = wm * scale;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0] * (dp[2 * kk][0] - D0) * cs, s[2 * kk][1] * (dp[2 * kk][1] - D0) * cs);
      pa[1] = pack_bf16(s[2 * kk][2] * (dp[2 * kk][2] - D1) * cs, s[2 * kk][3] * (dp[2 * kk][3] - D1) * cs);
      pa[2] = pack_bf16(s[2 * kk + 1][0] * (dp[2 * kk + 1][0] - D0) * cs, s[2 * kk + 1][1] * (dp[2 * kk + 1][1] - D0) * cs);
      pa[3] = pack_bf16(s[2 * kk + 1][2] * (dp[2 * kk + 1][2] - D1) * cs, s[2 * kk + 1][3] * (dp[2 * kk + 1][3] - D1) * cs);
#pragma unroll
      for (int dpi = 0; dpi < DH / 16; ++dpi) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, ksm + swz<ROWB>(16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dpi + (lane >> 4)));
        mma_bf16(dq[2 * dpi], pa, b0, b1);
        mma_bf16(dq[2 * dpi + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  if (tid < a.topk) dwp[tid] = ((dwred[0][tid] + dwred[1][tid]) + dwred[2][tid]) + dwred[3][tid];
  const int cq = lane & 3;
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) {
    const int r0 = 16 * warp + g;
    *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0, n) + cq * 4) = pack_bf16(dq[n][0], dq[n][1]);
    *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0 + 8, n) + cq * 4) = pack_bf16(dq[n][2], dq[n][3]);
  }
  __syncthreads();
  for (int u = tid; u < 64 * UPR; u += 128) {
    const int row = u / UPR, w = u % UPR;
    *reinterpret_cast<uint4*>(dqg + row * ts + w * 8) = *reinterpret_cast<const uint4*>(Qs + swz<ROWB>(row, w));
  }
}

// ------------------------------------------------------------------ gca_bwd_kv (bf16)
template <int DH>
__global__ void __launch_bounds__(128) gca_bwd_kv_mma_kernel(BwdArgs a) {
  constexpr int ROWB = DH * 2, TILE = 64 * ROWB, UPR = ROWB / 16;
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* Ks = sm;
  unsigned char* Vs = sm + TILE;
  __shared__ __align__(16) float lse_s[2][64];
  __shared__ __align__(16) float D_s[2][64];
  __shared__ float cw_s[2];
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, cq = lane & 3;
  const int64_t ts = (int64_t)a.H * DH;
  const int64_t ktok0 = ((int64_t)b * a.nC * 64 + (int64_t)j * 64) * ts + h * DH;
  const int e0 = a.csr_off[(int64_t)b * (a.nC + 1) + j];
  const int e1 = a.csr_off[(int64_t)b * (a.nC + 1) + j + 1];
  const int32_t* ent = a.csr_ent + (int64_t)b * a.nQ * a.topk;
  bf16* dkg = reinterpret_cast<bf16*>(a.dk) + ktok0;
  bf16* dvg = reinterpret_cast<bf16*>(a.dv) + ktok0;
  const int ncons = e1 - e0;
  if (ncons == 0) {
    if (!a.acc_dkv) {
      for (int u = tid; u < 64 * UPR; u += 128) {
        const int row = u / UPR, w = u % UPR;
        *reinterpret_cast<uint4*>(dkg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(dvg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }
  const bf16* kg = reinterpret_cast<const bf16*>(a.k) + ktok0;
  const bf16* vg = reinterpret_cast<const bf16*>(a.v) + ktok0;
  for (int u = tid; u < 64 * UPR; u += 128) {
    const int row = u / UPR, w = u % UPR;
    cp_async16(Ks + swz<ROWB>(row, w), kg + row * ts + w * 8);
    cp_async16(Vs + swz<ROWB>(row, w), vg + row * ts + w * 8);
  }
  auto load_cons = [&](int ci, int stage) {
    const int e = ent[e0 + ci];
    const int r = e / a.topk, m = e % a.topk;
    const int c = r + a.shift;
    const int64_t tok0 = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
    const bf16* qg = reinterpret_cast<const bf16*>(a.q) + tok0;
    const bf16* dog = reinterpret_cast<const bf16*>(a.dout) + tok0;
    unsigned char* Qs = sm + TILE * (2 + 2 * stage);
    unsigned char* dOs = Qs + TILE;
    for (int u = tid; u < 64 * UPR; u += 128) {
      const int row = u / UPR, w = u % UPR;
      cp_async16(Qs + swz<ROWB>(row, w), qg + row * ts + w * 8);
      cp_async16(dOs + swz<ROWB>(row, w), dog + row * ts + w * 8);
    }
    const int64_t rb = ((((int64_t)b * a.nQ + c) * a.H + h) * a.topk + m) * 64;
    if (tid < 16) cp_async16(&lse_s[stage][tid * 4], a.lse + rb + tid * 4);
    else if (tid < 32) cp_async16(&D_s[stage][(tid - 16) * 4], a.Dbuf + rb + (tid - 16) * 4);
    if (warp == 1) {
      const float wv = slot_weight_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk,
                                        a.scores + ((int64_t)b * a.nQ + r) * a.topk, a.topk, a.nC, m, a.err);
      if (lane == 0) cw_s[stage] = wv;
    }
  };
  load_cons(0, 0);
  cp_async_commit();
  const float scale = 1.0f / sqrtf((float)DH);
  const float sl2 = scale * kLog2e;
  float dk[DH / 8][4], dv[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[n][e] = dv[n][e] = 0.f;
  for (int ci = 0; ci < ncons; ++ci) {
    const int stage = ci & 1;
    if (ci + 1 < ncons) load_cons(ci + 1, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t qsm = smem_u32(sm + TILE * (2 + 2 * stage));
    const uint32_t dsm_ = qsm + TILE;
    const float w = cw_s[stage];
    float st[8][4], dpt[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[n][e] = dpt[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      uint32_t kf[4], vf[4];
      const uint32_t aoff = swz<ROWB>(16 * warp + (lane & 15), 2 * ks + (lane >> 4));
      ldsm_x4(kf[0], kf[1], kf[2], kf[3], smem_u32(Ks) + aoff);
      ldsm_x4(vf[0], vf[1], vf[2], vf[3], smem_u32(Vs) + aoff);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t off = swz<ROWB>(16 * p + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1));
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, qsm + off);
        mma_bf16(st[2 * p], kf, b0, b1);
        mma_bf16(st[2 * p + 1], kf, b2, b3);
        ldsm_x4(b0, b1, b2, b3, dsm_ + off);
        mma_bf16(dpt[2 * p], vf, b0, b1);
        mma_bf16(dpt[2 * p + 1], vf, b2, b3);
      }
    }
    // Columns of this thread: queries 8n + 2cq + {0, 1}.
    const float cs = w * scale;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int q0 = 8 * n + 2 * cq;
      const float l0 = lse_s[stage][q0] * kLog2e, l1 = lse_s[stage][q0 + 1] * kLog2e;
      const float d0 = D_s[stage][q0], d1 = D_s[stage][q0 + 1];
      const float p0 = exp2f(st[n][0] * sl2 - l0), p1 = exp2f(st[n][1] * sl2 - l1);
      const float p2 = exp2f(st[n][2] * sl2 - l0), p3 = exp2f(st[n][3] * sl2 - l1);
      dpt[n][0] = p0 * (dpt[n][0] - d0) * cs;
      dpt[n][1] = p1 * (dpt[n][1] - d1) * cs;
      dpt[n][2] = p2 * (dpt[n][2] - d0) * cs;
      dpt[n][3] = p3 * (dpt[n][3] - d1) * cs;
      st[n][0] = p0 * w;
      st[n][1] = p1 * w;
      st[n][2] = p2 * w;
      st[n][3] = p3 * w;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4], sa[4];
      pa[0] = pack_bf16(st[2 * kk][0], st[2 * kk][1]);
      pa[1] = pack_bf16(st[2 * kk][2], st[2 * kk][3]);
      pa[2] = pack_bf16(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      pa[3] = pack_bf16(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      sa[0] = pack_bf16(dpt[2 * kk][0], dpt[2 * kk][1]);
      sa[1] = pack_bf16(dpt[2 * kk][2], dpt[2 * kk][3]);
      sa[2] = pack_bf16(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      sa[3] = pack_bf16(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
      for (int dpi = 0; dpi < DH / 16; ++dpi) {
        const uint32_t off = swz<ROWB>(16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dpi + (lane >> 4));
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, dsm_ + off);
        mma_bf16(dv[2 * dpi], pa, b0, b1);
        mma_bf16(dv[2 * dpi + 1], pa, b2, b3);
        ldsm_x4_t(b0, b1, b2, b3, qsm + off);
        mma_bf16(dk[2 * dpi], sa, b0, b1);
        mma_bf16(dk[2 * dpi + 1], sa, b2, b3);
      }
    }
    __syncthreads();
  }
  // Epilogue: stage dK in the K tile and dV in the V tile, then write 16-byte rows.
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) {
    const int r0 = 16 * warp + g;
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(sm + TILE * 2) + (r0 * DH + 8 * n + 2 * cq)) = make_float2(dk[n][0], dk[n][1]);
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(sm + TILE * 2) + ((r0 + 8) * DH + 8 * n + 2 * cq)) = make_float2(dk[n][2], dk[n][3]);
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(sm + TILE * 4) + (r0 * DH + 8 * n + 2 * cq)) = make_float2(dv[n][0], dv[n][1]);
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(sm + TILE * 4) + ((r0 + 8) * DH + 8 * n + 2 * cq)) = make_float2(dv[n][2], dv[n][3]);
  }
  __syncthreads();
  const float* dkf = reinterpret_cast<const float*>(sm + TILE * 2);
  const float* dvf = reinterpret_cast<const float*>(sm + TILE * 4);
  for (int u = tid; u < 64 * UPR; u += 128) {
    const int row = u / UPR, w = u % UPR;
    float vk[8], vv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      vk[e] = dkf[row * DH + w * 8 + e];
      vv[e] = dvf[row * DH + w * 8 + e];
    }
    if (a.acc_dkv) {
      const uint4 ok = *reinterpret_cast<const uint4*>(dkg + row * ts + w * 8);
      const uint4 ov = *reinterpret_cast<const uint4*>(dvg + row * ts + w * 8);
      float fk[8], fv[8];
      unpack16(ok, fk, (const bf16*)nullptr);
      unpack16(ov, fv, (const bf16*)nullptr);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        vk[e] += fk[e];
        vv[e] += fv[e];
      }
    }
    uint4 outk, outv;
    outk.x = pack_bf16(vk[0], vk[1]); outk.y = pack_bf16(vk[2], vk[3]);
    outk.z = pack_bf16(vk[4], vk[5]); outk.w = pack_bf16(vk[6], vk[7]);
    outv.x = pack_bf16(vv[0], vv[1]); outv.y = pack_bf16(vv[2], vv[3]);
    outv.z = pack_bf16(vv[4], vv[5]); outv.w = pack_bf16(vv[6], vv[7]);
    *reinterpret_cast<uint4*>(dkg + row * ts + w * 8) = outk;
    *reinterpret_cast<uint4*>(dvg + row * ts + w * 8) = outv;
  }
}

// ------------------------------------------------------------------ f32 SIMT variants
template <int DH>
__global__ void __launch_bounds__(64) gca_bwd_q_f32_kernel(BwdArgs a) {
  __shared__ float Ks[64][DH + 1];
  __shared__ float Vs[64][DH + 1];
  __shared__ float w_s[kMaxTopk];
  __shared__ int j_s[kMaxTopk];
  __shared__ float red[2];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int64_t tok0 = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  const int64_t rowbase = ((int64_t)b * a.nQ + c) * a.H + h;
  const float* lse = a.lse + rowbase * a.topk * 64;
  float* Dg = a.Dbuf + rowbase * a.topk * 64;
  float* dwp = a.dwp + rowbase * a.topk;
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
  const float* qg = reinterpret_cast<const float*>(a.q) + tok0;
  const float* dog = reinterpret_cast<const float*>(a.dout) + tok0;
  float qv[DH], dov[DH], dq[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    qv[d] = qg[t * ts + d];
    dov[d] = dog[t * ts + d];
    dq[d] = 0.f;
  }
  for (int m = 0; m < a.topk; ++m) {
    const int64_t j = j_s[m];
    if (j < 0) {
      if (t == 0) dwp[m] = 0.f;
      continue;
    }
    __syncthreads();
    const float* kg = reinterpret_cast<const float*>(a.k) + ((int64_t)b * a.nC * 64 + j * 64) * ts + h * DH;
    const float* vg = reinterpret_cast<const float*>(a.v) + ((int64_t)b * a.nC * 64 + j * 64) * ts + h * DH;
    for (int x = t; x < 64 * DH; x += 64) {
      const int row = x / DH, d = x % DH;
      Ks[row][d] = kg[row * ts + d];
      Vs[row][d] = vg[row * ts + d];
    }
    __syncthreads();
    const float l = lse[m * 64 + t];
    float p[64], dp[64];
    float Dm = 0.f;
    for (int key = 0; key < 64; ++key) {
      float sdot = 0.f, pdot = 0.f;
#pragma unroll
      for (int d = 0; d < DH; ++d) {
        sdot = fmaf(qv[d], Ks[key][d], sdot);
        pdot = fmaf(dov[d], Vs[key][d], pdot);
      }
      p[key] = expf(sdot * scale - l);
      dp[key] = pdot;
      Dm = fmaf(p[key], pdot, Dm);
    }
    Dg[m * 64 + t] = Dm;
    const float cs = w_s[m] * scale;
    for (int key = 0; key < 64; ++key) {
      const float ds = p[key] * (dp[key] - Dm) * cs;
#pragma unroll
      for (int d = 0; d < DH; ++d) dq[d] = fmaf(ds, Ks[key][d], dq[d]);
    }
    float part = Dm;
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) part += __shfl_xor_sync(0xffffffffu, part, k);
    if (lane == 0) red[warp] = part;
    __syncthreads();
    if (t == 0) dwp[m] = red[0] + red[1];
  }
  float* dqg = reinterpret_cast<float*>(a.dq) + tok0;
#pragma unroll
  for (int d = 0; d < DH; ++d) dqg[t * ts + d] = dq[d];
}

template <int DH>
__global__ void __launch_bounds__(64) gca_bwd_kv_f32_kernel(BwdArgs a) {
  __shared__ float Qs[64][DH + 1];
  __shared__ float dOs[64][DH + 1];
  __shared__ float lse_s[64], D_s[64];
  __shared__ float w_s;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x;
  const int64_t ts = (int64_t)a.H * DH;
  const int64_t ktok0 = ((int64_t)b * a.nC * 64 + (int64_t)j * 64) * ts + h * DH;
  const int e0 = a.csr_off[(int64_t)b * (a.nC + 1) + j];
  const int e1 = a.csr_off[(int64_t)b * (a.nC + 1) + j + 1];
  const int32_t* ent = a.csr_ent + (int64_t)b * a.nQ * a.topk;
  const float scale = 1.0f / sqrtf((float)DH);
  float kv[DH], vv[DH], dk[DH], dv[DH];
  const float* kg = reinterpret_cast<const float*>(a.k) + ktok0;
  const float* vg = reinterpret_cast<const float*>(a.v) + ktok0;
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    kv[d] = kg[t * ts + d];
    vv[d] = vg[t * ts + d];
    dk[d] = dv[d] = 0.f;
  }
  for (int ci = e0; ci < e1; ++ci) {
    const int e = ent[ci];
    const int r = e / a.topk, m = e % a.topk;
    const int c = r + a.shift;
    __syncthreads();
    const int64_t tok0 = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
    const float* qg = reinterpret_cast<const float*>(a.q) + tok0;
    const float* dog = reinterpret_cast<const float*>(a.dout) + tok0;
    for (int x = t; x < 64 * DH; x += 64) {
      const int row = x / DH, d = x % DH;
      Qs[row][d] = qg[row * ts + d];
      dOs[row][d] = dog[row * ts + d];
    }
    const int64_t rb = ((((int64_t)b * a.nQ + c) * a.H + h) * a.topk + m) * 64;
    lse_s[t] = a.lse[rb + t];
    D_s[t] = a.Dbuf[rb + t];
    if (t < 32) {
      const float wv = slot_weight_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk,
                                        a.scores + ((int64_t)b * a.nQ + r) * a.topk, a.topk, a.nC, m, a.err);
      if (t == 0) w_s = wv;
    }
    __syncthreads();
    const float w = w_s;
    for (int q = 0; q < 64; ++q) {
      float sdot = 0.f, pdot = 0.f;
#pragma unroll
      for (int d = 0; d < DH; ++d) {
        sdot = fmaf(Qs[q][d], kv[d], sdot);
        pdot = fmaf(dOs[q][d], vv[d], pdot);
      }
      const float p = expf(sdot * scale - lse_s[q]);
      const float ds = w * p * (pdot - D_s[q]) * scale;
      const float wp = w * p;
#pragma unroll
      for (int d = 0; d < DH; ++d) {
        dv[d] = fmaf(wp, dOs[q][d], dv[d]);
        dk[d] = fmaf(ds, Qs[q][d], dk[d]);
      }
    }
  }
  float* dkg = reinterpret_cast<float*>(a.dk) + ktok0;
  float* dvg = reinterpret_cast<float*>(a.dv) + ktok0;
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    if (a.acc_dkv) {
      dkg[t * ts + d] += dk[d];
      dvg[t * ts + d] += dv[d];
    } else {
      dkg[t * ts + d] = dk[d];
      dvg[t * ts + d] = dv[d];
    }
  }
}

// ------------------------------------------------------------------ dscores
__global__ void __launch_bounds__(256) gca_dscores_kernel(BwdArgs a) {
  // One CTA per retrieval row r (query chunk c = r + shift).  dw_m, the gradient of the
  // fused output with respect to fusion weight m, is the sum of the D rows of slot m over
  // heads and query rows (D = rowsum(P * dO V^T) = dO . O_m per row); then
  // ds_m = w_m (dw_m - sum_n w_n dw_n), the softmax backward.  Fixed summation order.
  const int r = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = r + a.shift;
  float* out = a.dscores + ((int64_t)b * a.nQ + r) * a.topk;
  // The persistent key-side kernel that runs after this one claims its tiles from this
  // counter.
  if (r == 0 && b == 0 && tid == 0 && a.kv_ctr) *a.kv_ctr = 0;
  if (c >= a.nQ) {
    if (tid < a.topk) out[tid] = 0.f;
    return;
  }
  __shared__ float w_s[kMaxTopk];
  __shared__ int j_s[kMaxTopk];
  __shared__ float dw_s[kMaxTopk];
  if (warp == 0)
    row_weights_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk, a.scores + ((int64_t)b * a.nQ + r) * a.topk,
                     a.topk, a.nC, w_s, j_s, nullptr);
  __syncthreads();
  const float* Dc = a.Dbuf + ((int64_t)b * a.nQ + c) * a.H * a.topk * 64;
  for (int m = warp; m < a.topk; m += 8) {
    float acc = 0.f;
    if (j_s[m] >= 0) {
      // Four heads' loads in flight together, the sum in head order.
      int h = 0;
      for (; h + 4 <= a.H; h += 4) {
        float x[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float* p = Dc + ((int64_t)(h + v) * a.topk + m) * 64;
          x[v] = p[lane] + p[lane + 32];
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) acc += x[v];
      }
      for (; h < a.H; ++h) {
        const float* p = Dc + ((int64_t)h * a.topk + m) * 64;
        acc += p[lane] + p[lane + 32];
      }
    }
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
    if (lane == 0) dw_s[m] = acc;
  }
  __syncthreads();
  if (warp == 0) {
    float w = 0.f, dw = 0.f;
    bool valid = false;
    if (lane < a.topk) {
      w = w_s[lane];
      valid = j_s[lane] >= 0;
      dw = valid ? dw_s[lane] : 0.f;
    }
    float sum = w * dw;
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, k);
    if (lane < a.topk) out[lane] = valid ? w * (dw - sum) : 0.f;
  }
}

// ------------------------------------------------------------------ CSR of consumers
// One CTA per sequence: per-chunk counts, an exclusive scan into the offsets, then a fill
// by one warp, 32 entries at a time in entry order (ranks inside a step from
// __match_any_sync), so that every chunk's list is in increasing entry order.  kSmem keeps
// the counters and fill cursors in shared memory (nC <= kCsrSmemChunks), so that the
// fill's step-to-step dependence goes through shared memory; the entries of the next step
// are loaded while the current one is placed.
constexpr int kCsrSmemChunks = 16384;
constexpr int kCsrParChunks = 8192, kCsrParEntries = 8192;  // the parallel fill's shared-memory limits

// The same CSR with a parallel fill (nC <= kCsrParChunks, entries <= kCsrParEntries):
// counts and cursors in shared memory; every entry takes a slot of its chunk's segment by
// a shared atomic (in any order), then one warp per chunk writes each of the segment's
// entries at its rank, the number of smaller entry indices in the segment, which is the
// entry-order position.
__device__ __forceinline__ void csr_par_body(const int32_t* idx, int ld_rows, int nrows, int topk, int nC,
                                             int32_t* off, int32_t* ent, ErrWord* err, int b) {
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;         // [nC]: counts, then offsets, then fill cursors
  int32_t* beg = sh + nC;    // [nC + 1]: offsets
  int32_t* tmp = beg + nC + 1;  // [n]: entries, unordered within each segment
  __shared__ int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* ib = idx + (int64_t)b * ld_rows * topk;
  int32_t* ob = off + (int64_t)b * (nC + 1);
  int32_t* eb = ent + (int64_t)b * ld_rows * topk;
  const int n = nrows * topk;
  for (int j = tid; j < nC; j += 1024) cnt[j] = 0;
  __syncthreads();
  for (int e = tid; e < n; e += 1024) {
    const int j = ib[e];
    if (j >= 0 && j < nC) atomicAdd(&cnt[j], 1);
    else if (j != -1) flag_bad_index(err, j);
  }
  __syncthreads();
  const int per = (nC + 1023) / 1024;
  const int lo = min(nC, tid * per), hi = min(nC, lo + per);
  int mine = 0;
  for (int j = lo; j < hi; ++j) mine += cnt[j];
  int incl = mine;
#pragma unroll
  for (int k = 1; k < 32; k <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, k);
    if (lane >= k) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, k);
      if (lane >= k) v += u;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  int run = incl - mine + (warp > 0 ? wsum[warp - 1] : 0);
  for (int j = lo; j < hi; ++j) {
    const int cj = cnt[j];
    beg[j] = run;
    ob[j] = run;
    cnt[j] = run;
    run += cj;
  }
  if (tid == 1023) {
    beg[nC] = wsum[31];
    ob[nC] = wsum[31];
  }
  __syncthreads();
  for (int e = tid; e < n; e += 1024) {
    const int j = ib[e];
    if (j >= 0 && j < nC) tmp[atomicAdd(&cnt[j], 1)] = e;
  }
  __syncthreads();
  for (int j = warp; j < nC; j += 32) {
    const int s0 = beg[j], len = beg[j + 1] - s0;
    for (int x = lane; x < len; x += 32) {
      const int v = tmp[s0 + x];
      int rank = 0;
      for (int y = 0; y < len; ++y) rank += tmp[s0 + y] < v;
      eb[s0 + rank] = v;
    }
  }
}

__global__ void __launch_bounds__(1024) csr_par_kernel(const int32_t* idx, int ld_rows, int nrows, int topk, int nC,
                                                       int32_t* off, int32_t* ent, ErrWord* err) {
  csr_par_body(idx, ld_rows, nrows, topk, nC, off, ent, err, blockIdx.x);
}

// The score gradient of four retrieval rows per 1024-thread CTA (eight warps per row; the
// same sums, in the same order, as gca_dscores_kernel), for the launch shared with the CSR.
__device__ __forceinline__ void dscores_rows4(const BwdArgs& a, int rb, int b) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, grp = warp >> 3, gw = warp & 7;
  const int r = 4 * rb + grp, c = r + a.shift;
  __shared__ float w_s[4][kMaxTopk];
  __shared__ int j_s[4][kMaxTopk];
  __shared__ float dw_s[4][kMaxTopk];
  if (rb == 0 && b == 0 && tid == 0 && a.kv_ctr) *a.kv_ctr = 0;  // the key side's tile counter
  const bool row_ok = r < a.nQ, act = row_ok && c < a.nQ;
  float* out = a.dscores + ((int64_t)b * a.nQ + r) * a.topk;
  if (row_ok && !act && gw == 0 && lane < a.topk) out[lane] = 0.f;
  if (act && gw == 0)
    row_weights_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk, a.scores + ((int64_t)b * a.nQ + r) * a.topk,
                     a.topk, a.nC, w_s[grp], j_s[grp], nullptr);
  __syncthreads();
  if (act) {
    const float* Dc = a.Dbuf + ((int64_t)b * a.nQ + c) * a.H * a.topk * 64;
    for (int m = gw; m < a.topk; m += 8) {
      float acc = 0.f;
      if (j_s[grp][m] >= 0) {
        int h = 0;
        for (; h + 4 <= a.H; h += 4) {
          float x[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float* p = Dc + ((int64_t)(h + v) * a.topk + m) * 64;
            x[v] = p[lane] + p[lane + 32];
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) acc += x[v];
        }
        for (; h < a.H; ++h) {
          const float* p = Dc + ((int64_t)h * a.topk + m) * 64;
          acc += p[lane] + p[lane + 32];
        }
      }
#pragma unroll
      for (int k = 16; k >= 1; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
      if (lane == 0) dw_s[grp][m] = acc;
    }
  }
  __syncthreads();
  if (act && gw == 0) {
    float w = 0.f, dw = 0.f;
    bool valid = false;
    if (lane < a.topk) {
      w = w_s[grp][lane];
      valid = j_s[grp][lane] >= 0;
      dw = valid ? dw_s[grp][lane] : 0.f;
    }
    float sum = w * dw;
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, k);
    if (lane < a.topk) out[lane] = valid ? w * (dw - sum) : 0.f;
  }
}

// One launch for two independent passes of the backward: CTAs 0 .. B-1 build the CSR of
// consumers of sequence blockIdx.x (the parallel fill), the rest take the score
// gradient, four retrieval rows each.
__global__ void __launch_bounds__(1024) dscores_csr_kernel(BwdArgs a, int nrows) {
  if ((int)blockIdx.x < a.B) {
    csr_par_body(a.idx, a.nQ, nrows, a.topk, a.nC, a.csr_off, a.csr_ent, a.err, blockIdx.x);
    return;
  }
  const int x = blockIdx.x - a.B, nrb = (a.nQ + 3) / 4;
  dscores_rows4(a, x % nrb, x / nrb);
}

template <bool kSmem>
__global__ void __launch_bounds__(1024) csr_kernel(const int32_t* idx, int ld_rows, int nrows, int topk,
                                                    int nC, int32_t* off, int32_t* ent, int32_t* cur,
                                                    ErrWord* err) {
  extern __shared__ int32_t cnt_s[];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* ib = idx + (int64_t)b * ld_rows * topk;
  int32_t* cnt = kSmem ? cnt_s : cur + (int64_t)b * nC;
  int32_t* ob = off + (int64_t)b * (nC + 1);
  int32_t* eb = ent + (int64_t)b * ld_rows * topk;
  const int n = nrows * topk;
  for (int j = tid; j < nC; j += 1024) cnt[j] = 0;
  __syncthreads();
  for (int e = tid; e < n; e += 1024) {
    const int j = ib[e];
    if (j >= 0 && j < nC) atomicAdd(&cnt[j], 1);
    else if (j != -1) flag_bad_index(err, j);
  }
  __syncthreads();
  // Exclusive scan: thread t owns the contiguous range [t*per, (t+1)*per).
  __shared__ int wsum[32];
  const int per = (nC + 1023) / 1024;
  const int lo = min(nC, tid * per), hi = min(nC, lo + per);
  int mine = 0;
  for (int j = lo; j < hi; ++j) mine += cnt[j];
  int incl = mine;
#pragma unroll
  for (int k = 1; k < 32; k <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, k);
    if (lane >= k) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, k);
      if (lane >= k) v += u;
    }
    wsum[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  int run = incl - mine + (warp > 0 ? wsum[warp - 1] : 0);
  for (int j = lo; j < hi; ++j) {
    const int cj = cnt[j];
    ob[j] = run;
    cnt[j] = run;  // becomes the fill cursor
    run += cj;
  }
  if (tid == 1023) ob[nC] = wsum[31];
  __syncthreads();
  // Stable fill by one warp, 32 entries at a time, in entry order.
  if (warp == 0) {
    int jn = lane < n ? ib[lane] : -1;
    for (int base = 0; base < n; base += 32) {
      const int e = base + lane;
      int j = jn;
      jn = (e + 32 < n) ? ib[e + 32] : -1;  // next step's entry, in flight meanwhile
      const bool valid = e < n && j >= 0 && j < nC;
      if (!valid) j = -1;
      const unsigned grp = __match_any_sync(0xffffffffu, j);
      const int rank = __popc(grp & ((1u << lane) - 1));
      int pos = 0;
      if (valid) pos = cnt[j] + rank;
      __syncwarp();
      if (valid) {
        eb[pos] = e;
        if (rank == 0) cnt[j] += __popc(grp);
      }
      __syncwarp();
    }
  }
}

size_t bwd_q_smem(int dh) { return (size_t)64 * dh * 2 * 6 + 1024; }
size_t bwd_kv_smem(int dh) { return (size_t)64 * dh * 2 * 6 + 1024; }

}  // namespace

cudaError_t launch_csr(const int32_t* idx, int B, int ld_rows, int nrows, int topk, int nC,
                       int32_t* off, int32_t* ent, int32_t* cur, ErrWord* err, cudaStream_t s) {
  const int n = nrows * topk;
  if (nC <= kCsrParChunks && n <= kCsrParEntries) {
    const int sm = (2 * nC + 1 + n) * (int)sizeof(int32_t);
    cudaError_t e = allow_smem((const void*)csr_par_kernel, sm);
    if (e != cudaSuccess) return e;
    launch_begin("gca_csr", s);
    csr_par_kernel<<<B, 1024, sm, s>>>(idx, ld_rows, nrows, topk, nC, off, ent, err);
    return launch_end("gca_csr", s);
  }
  if (nC <= kCsrSmemChunks) {
    const int sm = nC * (int)sizeof(int32_t);
    cudaError_t e = allow_smem((const void*)csr_kernel<true>, sm);
    if (e != cudaSuccess) return e;
    launch_begin("gca_csr", s);
    csr_kernel<true><<<B, 1024, sm, s>>>(idx, ld_rows, nrows, topk, nC, off, ent, cur, err);
    return launch_end("gca_csr", s);
  }
  launch_begin("gca_csr", s);
  csr_kernel<false><<<B, 1024, 0, s>>>(idx, ld_rows, nrows, topk, nC, off, ent, cur, err);
  return launch_end("gca_csr", s);
}

cudaError_t launch_backward(const BwdArgs& a, cudaStream_t s) {
  cudaError_t e;
  dim3 gq(a.nQ, a.H, a.B), gk(a.nC, a.H, a.B);
  const bool tc = a.bf16 && a.dh == 64;
  if (tc) {
    if ((e = launch_bwd_q_tc(a, s)) != cudaSuccess) return e;
  } else if (a.bf16) {
    const int sq = (int)bwd_q_smem(a.dh);
    const void* fq = (const void*)gca_bwd_q_mma_kernel<32>;
    if ((e = allow_smem(fq, sq)) != cudaSuccess) return e;
    launch_begin("gca_bwd_q_mma", s);
    gca_bwd_q_mma_kernel<32><<<gq, 128, sq, s>>>(a);
    if ((e = launch_end("gca_bwd_q_mma", s)) != cudaSuccess) return e;
  } else {
    launch_begin("gca_bwd_q_f32", s);
    if (a.dh == 64) gca_bwd_q_f32_kernel<64><<<gq, 64, 0, s>>>(a);
    else gca_bwd_q_f32_kernel<32><<<gq, 64, 0, s>>>(a);
    if ((e = launch_end("gca_bwd_q_f32", s)) != cudaSuccess) return e;
  }
  const int nrows = a.nQ - a.shift > 0 ? a.nQ - a.shift : 0;
  if (a.nC <= kCsrParChunks && nrows * a.topk <= kCsrParEntries) {
    // The score gradient and the CSR share one launch.
    const int sm = (2 * a.nC + 1 + nrows * a.topk) * (int)sizeof(int32_t);
    if ((e = allow_smem((const void*)dscores_csr_kernel, sm)) != cudaSuccess) return e;
    launch_begin("gca_dscores_csr", s);
    dscores_csr_kernel<<<a.B + a.B * ((a.nQ + 3) / 4), 1024, sm, s>>>(a, nrows);
    if ((e = launch_end("gca_dscores_csr", s)) != cudaSuccess) return e;
  } else {
    launch_begin("gca_dscores", s);
    gca_dscores_kernel<<<dim3(a.nQ, a.B), 256, 0, s>>>(a);
    if ((e = launch_end("gca_dscores", s)) != cudaSuccess) return e;
    if ((e = launch_csr(a.idx, a.B, a.nQ, nrows, a.topk, a.nC, a.csr_off, a.csr_ent, a.csr_cur, a.err, s)) !=
        cudaSuccess)
      return e;
  }
  if (tc) return launch_bwd_kv_tc(a, s);
  if (a.bf16) {
    const int sk = (int)bwd_kv_smem(a.dh);
    if ((e = allow_smem((const void*)gca_bwd_kv_mma_kernel<32>, sk)) != cudaSuccess) return e;
    launch_begin("gca_bwd_kv_mma", s);
    gca_bwd_kv_mma_kernel<32><<<gk, 128, sk, s>>>(a);
    return launch_end("gca_bwd_kv_mma", s);
  }
  launch_begin("gca_bwd_kv_f32", s);
  if (a.dh == 64) gca_bwd_kv_f32_kernel<64><<<gk, 64, 0, s>>>(a);
  else gca_bwd_kv_f32_kernel<32><<<gk, 64, 0, s>>>(a);
  return launch_end("gca_bwd_kv_f32", s);
}

}  // namespace gca
