// Chunk / landmark encoder: one pre-LN bidirectional Transformer layer over each chunk's
// 65 rows (its 64 tokens and its LMK token), then the K/V transform shared by the upper
// layers.
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", 整体框架 (framework): the lower layers' output, with an
// LMK token closing every chunk, passes a bidirectional Transformer encoder that yields
// the chunk representations and the landmark representations shared by every upper
// layer; 关键设计 / GCA (key design): the K/V transform is shared across layers.  The
// layer's form (pre-LN, d -> 4d -> d MLP with the erf GELU, LayerNorm eps 1e-5,
// bias-free K/V transform) is a reading: the pages give none.
//
// Rows stay in sequence order with the LMK rows in place, row m = (b nC + c) 65 + t, so
// every step is a row-wise pass or a GEMM and a chunk's rows are contiguous:
//   LN1(x) -> A;  A W_qkv^T + b -> F (as [M][3d]);  attention per (chunk, head) -> A;
//   x + A W_o^T + b -> U;  LN2(U) -> A;  GELU(A W_1^T + b) -> F;
//   U + F W_2^T + b -> y (LMK rows also -> k_lmk);  y W_kv^T -> K, V (token rows only).
// The GEMMs share one persistent tcgen05 kernel with the step's epilogue fused.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tc_rows.cuh"

namespace gca {
namespace {

using bf16 = __nv_bfloat16;
constexpr int kRows = 65;  // rows per chunk: 64 tokens, then the LMK token
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // lo in the low half
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ LayerNorm
// One warp per RPW rows, held in registers as packed bf16 (every load issued before the
// first reduction, so that a warp keeps RPW rows in flight with few registers): mean, then
// the population variance of the centred values, y = (x - mean) / sqrt(var + 1e-5) * g + b.
// NV 16-byte vectors per lane cover d <= 256 NV.
template <int NV, int RPW>
__global__ void __launch_bounds__(256) enc_layernorm_kernel(const bf16* __restrict__ x, const float* __restrict__ g,
                                                            const float* __restrict__ b, bf16* __restrict__ y,
                                                            int64_t M, int d) {
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW;
  const int lane = threadIdx.x & 31;
  const int nv = d / 8;
  uint4 raw[RPW][NV];
#pragma unroll
  for (int r = 0; r < RPW; ++r)
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = lane + 32 * i;
      raw[r][i] = (row0 + r < M && v < nv) ? __ldg(reinterpret_cast<const uint4*>(x + (row0 + r) * d) + v)
                                           : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    if (row0 + r >= M) break;  // uniform across the warp
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float f[8];
      unpack16(raw[r][i], f, static_cast<const bf16*>(nullptr));
#pragma unroll
      for (int e = 0; e < 8; ++e) s += f[e];
    }
    const float mean = warp_sum(s) / (float)d;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (lane + 32 * i < nv) {
        float f[8];
        unpack16(raw[r][i], f, static_cast<const bf16*>(nullptr));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float t = f[e] - mean;
          q += t * t;
        }
      }
    const float rstd = rsqrtf(warp_sum(q) / (float)d + 1e-5f);
    uint4* yr = reinterpret_cast<uint4*>(y + (row0 + r) * d);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = lane + 32 * i;
      if (v < nv) {
        float f[8];
        unpack16(raw[r][i], f, static_cast<const bf16*>(nullptr));
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(g) + 2 * v);
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(g) + 2 * v + 1);
        const float4 b0 = __ldg(reinterpret_cast<const float4*>(b) + 2 * v);
        const float4 b1 = __ldg(reinterpret_cast<const float4*>(b) + 2 * v + 1);
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (f[e] - mean) * rstd * gg[e] + bb[e];
        yr[v] = make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
      }
    }
  }
}

// ------------------------------------------------------------------ GEMM with fused epilogue
// C[M][N] = A[M][K] W[N][K]^T in bf16 with fp32 accumulation: 128 x BN tiles, K in steps of
// 64 through a 4-stage TMA ring, tcgen05.mma M = 128, N = BN, K = 16 into one of two TMEM
// accumulators, so that the epilogue of a tile overlaps the products of the next.  One
// CTA per SM, persistent over the tiles; consecutive tiles share their rows of A.
// Warp 0 loads, warp 1 issues the products, warps 2-9 run the epilogue: warp w reads
// TMEM lane quarter w % 4 (a row per thread) over half of the tile's columns, one 32-column
// chunk at a time with the next chunk's load in flight, applies the step's epilogue and
// writes the chunk (32 rows x 64 bytes) through its own swizzled staging buffer with a TMA
// store, so that global writes go out as whole lines.
enum Epi { kEpiBias = 0, kEpiGelu = 1, kEpiResid = 2, kEpiKV = 3 };

struct GemmArgs {
  int M, N, K;
  const float* bias;  // [N]
  const bf16* resid;  // [M][N] (kEpiResid)
  bf16* out;          // [M][N]; kEpiKV: K [M][d] (M counts token rows there)
  bf16* out2;         // kEpiResid: the LMK rows [M / 65][N] (or null); kEpiKV: V
  int d;              // kEpiKV: columns of K and of V
  ErrWord* err;
};

constexpr int kGemmStages = 4, kGemmEpiWarps = 8, kGemmThreads = 32 * (2 + kGemmEpiWarps);
constexpr int kStageBufBytes = 2 * 32 * 64;  // per epilogue warp: two 32 x 32 bf16 chunks
template <int BN>
constexpr int gemm_smem() {
  return kGemmStages * (128 + BN) * 128 + kGemmEpiWarps * kStageBufBytes + 1024;
}

// Bounded wait for phase `parity` of `bar` that gives up early once the CTA's abort flag
// is raised; on running out it records `site` and raises the flag.
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

// GELU(x) = x Phi(x) = x (1 + erf(x / sqrt 2)) / 2, with erf from Abramowitz & Stegun,
// Handbook of Mathematical Functions, 7.1.26 (Hastings' rational approximation, absolute
// error <= 1.5e-7): for z = |x| / sqrt 2 and t = 1 / (1 + p z),
//     q = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2) = 1 - erf(z),
// so 1 + erf(x / sqrt 2) is 2 - q for x >= 0 and q for x < 0 (no cancellation for x < 0).
// Branch-free: one reciprocal and one exp2 on the special-function unit; the error of the
// result stays near 2e-7 max(1, |GELU(x)|), far below the bf16 output's rounding.
__device__ __forceinline__ float gelu(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  float t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, z, 1.0f)));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f), 0.254829592f);
  const float q = poly * tc::ex2(-(z * z) * kLog2e);
  return 0.5f * x * (x >= 0.f ? 2.0f - q : q);
}

// 32 consecutive columns as bf16: four 16-byte stores.
__device__ __forceinline__ void store32(bf16* dst, const float (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d4[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}

// Math of the step's epilogue on a 32-column chunk (everything but the store).
template <int EPI>
__device__ __forceinline__ void epilogue_math(const GemmArgs& a, int col, const uint4 (&res)[4], float (&v)[32]) {
  if (EPI != kEpiKV) {
    const float4* b4 = reinterpret_cast<const float4*>(a.bias + col);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 bb = __ldg(b4 + q);
      v[4 * q] += bb.x;
      v[4 * q + 1] += bb.y;
      v[4 * q + 2] += bb.z;
      v[4 * q + 3] += bb.w;
    }
  }
  if (EPI == kEpiGelu) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = gelu(v[j]);
  }
  if (EPI == kEpiResid) {  // the residual's 32 values, loaded before the accumulator was ready
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
      unpack16(res[q], f, static_cast<const bf16*>(nullptr));
#pragma unroll
      for (int e = 0; e < 8; ++e) v[8 * q + e] += f[e];
    }
  }
}

// Row `lane` of a 32 x 32 bf16 chunk into the 64-byte-swizzled staging buffer.
__device__ __forceinline__ void stage_row(unsigned char* buf, int lane, const float (&v)[32]) {
  uint4* row = reinterpret_cast<uint4*>(buf + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    row[u ^ sw] = make_uint4(pack_bf16(v[8 * u], v[8 * u + 1]), pack_bf16(v[8 * u + 2], v[8 * u + 3]),
                             pack_bf16(v[8 * u + 4], v[8 * u + 5]), pack_bf16(v[8 * u + 6], v[8 * u + 7]));
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
enc_gemm_kernel(GemmArgs a, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2) {
  constexpr int NST = kGemmStages;
  constexpr uint32_t kABytes = 128 * 128, kStage = (128 + BN) * 128;
  constexpr uint32_t kId = tc::idesc_bf16(128, BN, false);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  // full / empty per use of a ring stage; acc_full / acc_empty per use of an accumulator.
  __shared__ __align__(8) uint64_t full[NST], empty[NST], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = a.N / BN, ntiles = ((a.M + 127) / 128) * nt, kt = a.K / 64;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < NST; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], kGemmEpiWarps);
    }
    tc::mbar_init(&drain, 1);
    tc::fence_mbar_init();
    abort_s = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC)) : "memory");
    if (EPI == kEpiKV) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC2)) : "memory");
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, 2 * BN);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;  // loads issued
      bool ok = true;
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        const int m0 = (t / nt) * 128, n0 = (t % nt) * BN;
        for (int kb = 0; kb < kt; ++kb) {
          const int s = it % NST;
          if (it >= NST && !wait_or_abort(&empty[s], (uint32_t)(it / NST - 1) & 1, &abort_s, a.err, 20, t)) {
            ok = false;
            break;
          }
          unsigned char* st = sm + s * kStage;
          tc::mbar_expect_tx(&full[s], kStage);
          if (EPI == kEpiKV) tc::tma_load_3d(st, &tmA, kb * 64, 0, m0 / 64, &full[s]);  // two chunks' token rows
          else tc::tma_load_2d(st, &tmA, kb * 64, m0, &full[s]);
          tc::tma_load_2d(st + kABytes, &tmB, kb * 64, n0, &full[s]);
          ++it;
        }
      }
      // After an abort, let the copies already issued land before the CTA exits.
      if (*reinterpret_cast<volatile int*>(&abort_s))
        for (int j = std::max(0, it - NST); j < it; ++j) tc::mbar_wait(&full[j % NST], (uint32_t)(j / NST) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    int it = 0, i = 0;
    bool issued = false, ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      if (i >= 2 && !wait_or_abort(&acc_empty[buf], (uint32_t)((i >> 1) - 1) & 1, &abort_s, a.err, 21, t)) break;
      tc::fence_after();
      const uint32_t d = tmem + buf * BN;
      for (int kb = 0; kb < kt; ++kb, ++it) {
        const int s = it % NST;
        if (!wait_or_abort(&full[s], (uint32_t)(it / NST) & 1, &abort_s, a.err, 22, t)) {
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
    // No product may still be running when TMEM is released.
    if (issued) {
      tc::commit_warp(&drain);
      if (!tc::mbar_wait(&drain, 0) && lane == 0) flag_timeout(a.err, 23, blockIdx.x);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    constexpr int HALF = BN / 2, NCH = HALF / 32;
    const int ew = warp - 2, q = warp & 3, hf = ew >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    unsigned char* stg = sm + NST * kStage + ew * kStageBufBytes;
    int sb = 0;  // staging buffer to fill next
    int i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      const int row0 = (t / nt) * 128 + 32 * q, row = row0 + lane;
      const int col0 = (t % nt) * BN + hf * HALF;
      // The residual does not depend on the products: fetch the warp's part of the tile
      // (its row, HALF columns) now, so that the loads overlap the wait below.
      uint4 res[NCH][4];
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          res[c][u] = (EPI == kEpiResid && row < a.M)
                          ? __ldg(reinterpret_cast<const uint4*>(a.resid + (size_t)row * a.N + col0 + 32 * c) + u)
                          : make_uint4(0u, 0u, 0u, 0u);
      if (!wait_or_abort(&acc_full[buf], (uint32_t)(i >> 1) & 1, &abort_s, a.err, 24, t)) break;
      tc::fence_after();
      const uint32_t tcol = tmem + lane_base + buf * BN + hf * HALF;
      float v[2][32];
      tc::ld32x32b_x32(tcol, v[0]);
      tc::ld_wait_row(v[0]);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        if (c + 1 < NCH) tc::ld32x32b_x32(tcol + 32 * (c + 1), v[(c + 1) & 1]);
        float(&cur)[32] = v[c & 1];
        const int col = col0 + 32 * c;
        epilogue_math<EPI>(a, col, res[c], cur);
        {
          unsigned char* sbuf = stg + sb * (kStageBufBytes / 2);
          if (lane == 0) tc::bulk_wait_read<1>();  // this buffer's previous store has read it
          __syncwarp();
          stage_row(sbuf, lane, cur);
          tc::fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            // K/V transform: rows are token rows; columns below d go to K, the rest to V.
            if (EPI == kEpiKV && col >= a.d) tc::tma_store_2d(&tmC2, col - a.d, row0, sbuf);
            else tc::tma_store_2d(&tmC, col, row0, sbuf);
            tc::bulk_commit();
          }
          sb ^= 1;
          if (EPI == kEpiResid && a.out2 != nullptr && row < a.M && row % kRows == kRows - 1)
            store32(a.out2 + (size_t)(row / kRows) * a.N + col, cur);
        }
        if (c + 1 < NCH) tc::ld_wait_row(v[(c + 1) & 1]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
    }
    if (lane == 0) tc::bulk_wait_all();
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 2 * BN);
  }
}

// ------------------------------------------------------------------ attention inside a chunk
// One CTA per (chunk, group of kAttnHpc heads), the heads in turn with the next head's
// operands loading meanwhile (two stages).  The chunk's 65 rows of Q, K and V (head dim
// 64) arrive by TMA as 80-row boxes (the MMA's N granularity is 16; keys 65..79 are
// masked, rows past the end of the tensor read as zeros).  Per head: S = Q K^T (M = 128,
// N = 80; A rows 80..127 read the neighbouring tile and are never used) into TMEM columns
// 0-79; thread r owns row r: the softmax over the 65 keys, the bf16 P over the first 40
// columns as the A operand of O = P V (M = 128, N = 64, K = 80, into columns 64-127),
// then O's row scaled by 1 / sum.
constexpr int kAttnThreads = 128, kAttnKeys = 80, kAttnHpc = 4;
constexpr uint32_t kAttnBox = kAttnKeys * 128;  // 10 KB: one operand of one head
constexpr uint32_t kAttnStage = 3 * kAttnBox;    // Q, K, V
constexpr int kAttnSmem = 2 * kAttnStage + 1024;  // 61 KB: three CTAs per SM (TMEM: 128 columns each)

__global__ void __launch_bounds__(kAttnThreads) enc_attn_tc_kernel(int M, int d, int H,
                                                                   const __grid_constant__ CUtensorMap tm,
                                                                   bf16* __restrict__ out, ErrWord* err) {
  constexpr uint32_t kIdS = tc::idesc_bf16(128, kAttnKeys, false);
  constexpr uint32_t kIdO = tc::idesc_bf16(128, 64, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  // bar_ld[st] per load into stage st; bar_mma twice per head (S, then O); drain at exit.
  __shared__ __align__(8) uint64_t bar_ld[2], bar_mma, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = threadIdx.x;
  const int bc = blockIdx.x, h0 = blockIdx.y * kAttnHpc, nh = min(kAttnHpc, H - h0);
  const int row0 = bc * kRows;
  int nld[2] = {0, 0};  // loads issued per stage (thread 0)
  auto issue_load = [&](int i) {
    const int st = i & 1, h = h0 + i;
    unsigned char* b = sm + st * kAttnStage;
    tc::mbar_expect_tx(&bar_ld[st], kAttnStage);
    tc::tma_load_2d(b, &tm, h * 64, row0, &bar_ld[st]);
    tc::tma_load_2d(b + kAttnBox, &tm, d + h * 64, row0, &bar_ld[st]);
    tc::tma_load_2d(b + 2 * kAttnBox, &tm, 2 * d + h * 64, row0, &bar_ld[st]);
    ++nld[st];
  };
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar_ld[0], 1);
    tc::mbar_init(&bar_ld[1], 1);
    tc::mbar_init(&bar_mma, 1);
    tc::mbar_init(&drain, 1);
    tc::fence_mbar_init();
    abort_s = 0;
    issue_load(0);
    if (nh > 1) issue_load(1);
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 128);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tS = tmem_slot, tO = tmem_slot + 64;
  const uint32_t lb = (uint32_t)(32 * warp) << 16;
  const bool live = r < kRows && row0 + r < M;
  const float sl2 = 0.125f * kLog2e;  // dh^-1/2 with dh = 64, in base 2
  bool issued = false;

  for (int i = 0; i < nh; ++i) {
    const int st = i & 1, h = h0 + i;
    unsigned char* b = sm + st * kAttnStage;
    if (warp == 0) {
      if (wait_or_abort(&bar_ld[st], (uint32_t)(i >> 1) & 1, &abort_s, err, 25, bc)) {
        tc::fence_after();
        const uint64_t dq = tc::desc_km(tc::su32(b)), dk = tc::desc_km(tc::su32(b + kAttnBox));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_warp(tS, dq + kk * tc::kKStepKm, dk + kk * tc::kKStepKm, kIdS, kk > 0);
        tc::commit_warp(&bar_mma);
        issued = true;
      }
    }
    wait_or_abort(&bar_mma, 0, &abort_s, err, 26, bc);
    tc::fence_after();
    float s0[32], s1[32], s2[16];
    tc::ld32x32b_x32(tS + lb, s0);
    tc::ld32x32b_x32(tS + lb + 32, s1);
    tc::ld32x32b_x16(tS + lb + 64, s2);
    tc::ld_wait_row(s0);
    tc::ld_wait_row(s1);
    tc::ld_wait_row(s2);
    float mx = s2[0];  // key 64, the LMK token
#pragma unroll
    for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fmaxf(s0[j], s1[j]));
    float sum = 0.f;
    uint32_t p[40];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float a0 = tc::ex2((s0[2 * j] - mx) * sl2), a1 = tc::ex2((s0[2 * j + 1] - mx) * sl2);
      const float b0 = tc::ex2((s1[2 * j] - mx) * sl2), b1 = tc::ex2((s1[2 * j + 1] - mx) * sl2);
      sum += (a0 + a1) + (b0 + b1);
      p[j] = live ? pack_bf16(a0, a1) : 0u;
      p[16 + j] = live ? pack_bf16(b0, b1) : 0u;
    }
    const float c64 = tc::ex2((s2[0] - mx) * sl2);
    sum += c64;
    p[32] = live ? pack_bf16(c64, 0.f) : 0u;  // keys 65..79 are masked
#pragma unroll
    for (int j = 33; j < 40; ++j) p[j] = 0u;
#pragma unroll
    for (int c = 0; c < 5; ++c) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = p[8 * c + e];
      tc::st32x32b_x8(tS + lb + 8 * c, w);
    }
    tc::st_wait();
    tc::fence_before();
    __syncthreads();  // every row's P is in TMEM
    if (*reinterpret_cast<volatile int*>(&abort_s)) break;
    if (warp == 0) {
      tc::fence_after();
      const uint64_t dv = tc::desc_mn(tc::su32(b + 2 * kAttnBox));
#pragma unroll
      for (int kk = 0; kk < 5; ++kk) tc::mma_ts_warp(tO, tS + 8 * kk, dv + kk * tc::kKStepMn, kIdO, kk > 0);
      tc::commit_warp(&bar_mma);
    }
    wait_or_abort(&bar_mma, 1, &abort_s, err, 27, bc);
    tc::fence_after();
    float o0[32], o1[32];
    tc::ld32x32b_x32(tO + lb, o0);
    tc::ld32x32b_x32(tO + lb + 32, o1);
    tc::ld_wait_row(o0);
    tc::ld_wait_row(o1);
    tc::fence_before();
    __syncthreads();  // O read by every row (the next S overwrites columns 64-79); stage st is free
    if (*reinterpret_cast<volatile int*>(&abort_s)) break;
    if (threadIdx.x == 0 && i + 2 < nh) issue_load(i + 2);
    if (live) {
      const float inv = 1.0f / sum;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        o0[j] *= inv;
        o1[j] *= inv;
      }
      bf16* dst = out + (size_t)(row0 + r) * d + h * 64;
      store32(dst, o0);
      store32(dst + 32, o1);
    }
  }
  // After an abort: no product may still run when TMEM is released, and no copy may
  // still land in shared memory when the CTA exits.
  if (warp == 0 && issued) {
    tc::commit_warp(&drain);
    if (!tc::mbar_wait(&drain, 0) && lane == 0) flag_timeout(err, 28, bc);
  }
  if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&abort_s))
    for (int st = 0; st < 2; ++st)
      if (nld[st] > 0) tc::mbar_wait(&bar_ld[st], (uint32_t)(nld[st] - 1) & 1);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tS, 128);
  }
}

// ------------------------------------------------------------------ host side
template <int BN, int EPI>
cudaError_t run_gemm(const GemmArgs& g, const void* A, const void* W, int sms, cudaStream_t s, const char* name) {
  // kEpiKV: g.M counts token rows; A is [M / 64][65][K] (the LMK rows are skipped by the
  // load) and the outputs are K and V, [M][d] each.
  CUtensorMap ta, tb, tc_, tc2;
  cudaError_t e = EPI == kEpiKV ? make_chunk_token_tmap(&ta, A, g.K, g.M / 64) : make_rows_tmap(&ta, A, g.K, g.M, 128);
  if (e == cudaSuccess) e = make_rows_tmap(&tb, W, g.K, g.N, BN);
  if (e == cudaSuccess) e = make_store_tmap(&tc_, g.out, EPI == kEpiKV ? g.d : g.N, g.M);
  if (e == cudaSuccess) e = make_store_tmap(&tc2, EPI == kEpiKV ? g.out2 : g.out, EPI == kEpiKV ? g.d : g.N, g.M);
  if (e == cudaSuccess) e = allow_smem((const void*)enc_gemm_kernel<BN, EPI>, gemm_smem<BN>());
  if (e != cudaSuccess) return e;
  const int tiles = ((g.M + 127) / 128) * (g.N / BN);
  launch_begin(name, s);
  enc_gemm_kernel<BN, EPI><<<std::min(tiles, sms), kGemmThreads, gemm_smem<BN>(), s>>>(g, ta, tb, tc_, tc2);
  return launch_end(name, s);
}

cudaError_t run_layernorm(const bf16* x, const float* g, const float* b, bf16* y, int64_t M, int d, cudaStream_t s,
                          const char* name) {
  constexpr int RPW = 2;
  const unsigned grid = (unsigned)((M + 8 * RPW - 1) / (8 * RPW));
  launch_begin(name, s);
  if (d <= 256) enc_layernorm_kernel<1, RPW><<<grid, 256, 0, s>>>(x, g, b, y, M, d);
  else if (d <= 512) enc_layernorm_kernel<2, RPW><<<grid, 256, 0, s>>>(x, g, b, y, M, d);
  else if (d <= 768) enc_layernorm_kernel<3, RPW><<<grid, 256, 0, s>>>(x, g, b, y, M, d);
  else enc_layernorm_kernel<4, RPW><<<grid, 256, 0, s>>>(x, g, b, y, M, d);
  return launch_end(name, s);
}

template <int BN>
cudaError_t run_encoder(const EncoderArgs& a, int sms, cudaStream_t s) {
  const int d = a.d, M = a.B * a.nC * kRows;
  const bf16* x = static_cast<const bf16*>(a.x);
  bf16 *A = static_cast<bf16*>(a.bufA), *U = static_cast<bf16*>(a.bufU), *F = static_cast<bf16*>(a.bufF);
  cudaError_t e = run_layernorm(x, a.ln1_g, a.ln1_b, A, M, d, s, "enc_ln1");
  GemmArgs g{};
  g.M = M;
  g.err = a.err;
  if (e == cudaSuccess) {
    g.N = 3 * d; g.K = d; g.bias = a.b_qkv; g.out = F;
    e = run_gemm<BN, kEpiBias>(g, A, a.w_qkv, sms, s, "enc_qkv");
  }
  if (e == cudaSuccess) {
    CUtensorMap tm;
    e = make_rows_tmap(&tm, F, 3 * d, M, kAttnKeys);
    if (e == cudaSuccess) e = allow_smem((const void*)enc_attn_tc_kernel, kAttnSmem);
    if (e != cudaSuccess) return e;
    launch_begin("enc_attn", s);
    enc_attn_tc_kernel<<<dim3(a.B * a.nC, (a.H + kAttnHpc - 1) / kAttnHpc), kAttnThreads, kAttnSmem, s>>>(M, d, a.H, tm,
                                                                                                       A, a.err);
    e = launch_end("enc_attn", s);
  }
  if (e == cudaSuccess) {
    g.N = d; g.K = d; g.bias = a.b_o; g.resid = x; g.out = U; g.out2 = nullptr;
    e = run_gemm<BN, kEpiResid>(g, A, a.w_o, sms, s, "enc_out");
  }
  if (e == cudaSuccess) e = run_layernorm(U, a.ln2_g, a.ln2_b, A, M, d, s, "enc_ln2");
  if (e == cudaSuccess) {
    g.N = 4 * d; g.K = d; g.bias = a.b_1; g.out = F;
    e = run_gemm<BN, kEpiGelu>(g, A, a.w_1, sms, s, "enc_mlp1");
  }
  if (e == cudaSuccess) {
    g.N = d; g.K = 4 * d; g.bias = a.b_2; g.resid = U; g.out = static_cast<bf16*>(a.y);
    g.out2 = static_cast<bf16*>(a.k_lmk);
    e = run_gemm<BN, kEpiResid>(g, F, a.w_2, sms, s, "enc_mlp2");
  }
  if (e == cudaSuccess) {
    g.M = a.B * a.nC * 64; g.N = 2 * d; g.K = d; g.bias = nullptr; g.resid = nullptr; g.d = d;
    g.out = static_cast<bf16*>(a.k); g.out2 = static_cast<bf16*>(a.v);
    e = run_gemm<BN, kEpiKV>(g, a.y, a.w_kv, sms, s, "enc_kv");
  }
  return e;
}

}  // namespace

cudaError_t launch_chunk_encoder(const EncoderArgs& a, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  return a.d % 256 == 0 ? run_encoder<256>(a, sms, s) : run_encoder<128>(a, sms, s);
}

}  // namespace gca
