// Attention with one softmax over a list of 64-key blocks: the sliding-window causal
// self-attention that sits beside GCA in the attention block, and chunked cross-attention
// (CCA), the variant GCA is contrasted with.
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling": 损失函数/训练策略 (training strategy: sliding-window
// self-attention, W = 512, beside the top-k retrieval) and 关键设计 / key design, item
// "Grouped Cross-Attention" (CCA concatenates the retrieved chunks under one softmax and
// the retrieval scores take no part).
//
// Per (query chunk c, head h, sequence b) the key blocks are
//   window: blocks c - W/64 .. c of the same sequence (clipped at 0); block c - W/64 keeps
//           keys j > i of query row i (its first W-token window starts inside it), block c
//           keeps j <= i (causal), the others are whole;
//   CCA:    the valid retrieved chunks idx[b, c - shift, m], whole.
// The softmax runs online across the blocks: a running row maximum and sum, with the
// output accumulator rescaled when the maximum grows.  O and LSE = log sum exp of the
// scaled logits (natural log) per query row; `accumulate` adds O into the output buffer
// (the attention block's sum of this sublayer and GCA).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gca {
namespace {

using bf16 = __nv_bfloat16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxBlocks = 64;
enum { kMaskNone = 0, kMaskTail = 1, kMaskCausal = 2 };

// Block list of CTA (c, b): key chunk and mask type of each block, in order; returns the count.
__device__ int block_list(const BlockAttnArgs& a, int b, int c, int* js, int* ms) {
  int n = 0;
  if (a.mode == 0) {
    const int wb = a.window / 64;
    const int j0 = c - wb;
    for (int j = j0 < 0 ? 0 : j0; j <= c; ++j) {
      js[n] = j;
      ms[n] = j == c ? kMaskCausal : (j == j0 ? kMaskTail : kMaskNone);
      ++n;
    }
  } else {
    const int r = c - a.shift;
    if (r >= 0) {
      const int32_t* row = a.idx + ((int64_t)b * a.nQ + r) * a.topk;
      for (int m = 0; m < a.topk; ++m) {
        const int j = row[m];
        if (j >= 0 && j < a.nC) {
          js[n] = j;
          ms[n] = kMaskNone;
          ++n;
        } else if (j != -1) {
          flag_bad_index(a.err, j);
        }
      }
    }
  }
  return n;
}

// ------------------------------------------------------------------ bf16 tcgen05 path (dh = 64)
//   * warp 4 (control): TMA loads (Q once; K, V of each block into a 2-stage ring) and
//     tcgen05.mma through an elected lane: S = Q K^T into TMEM columns 0-63, O += P V into
//     columns 64-127 (the first block overwrites).
//   * warps 0-3 (softmax, full rows): mask, running maximum, rescale O in TMEM when the
//     maximum of one of the warp's rows grew, P = exp(S - max) as bf16 into columns 0-31
//     (the A operand of O += P V), running sum.  S(n+1) follows PV(n) in the tensor pipe's
//     order, so it overwrites P(n) only after the product has read it, and S(n+1) complete
//     implies PV(n) complete: O is final for the rescale of block n+1.
constexpr int kBaThreads = 160;
constexpr int kBaSmem = 46 * 1024 + 1024;  // Q + 2 x (K, V) = 40 KB, padded so that at most 4 CTAs share an SM
enum { kBarPReady = 2 };

__global__ void __launch_bounds__(kBaThreads, 4)
block_attn_tc_kernel(BlockAttnArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  constexpr int DH = 64, ROWB = 128, TILE = 8192, UPR = 8, NST = 2, NT = kBaThreads;
  constexpr uint32_t kIdS = tc::idesc_bf16(64, 64, false);
  constexpr uint32_t kIdPV = tc::idesc_bf16(64, DH, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* Qs = sm;
  unsigned char* ring = sm + TILE;  // stage st: K at ring + 2 st TILE, V after it
  __shared__ int js[kMaxBlocks], ms[kMaxBlocks];
  __shared__ int nb_s;
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar_q, bar_kv[NST], bar_s, bar_o;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  bf16* og = reinterpret_cast<bf16*>(a.o) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  float* lse = a.lse + (((int64_t)b * a.nQ + c) * a.H + h) * 64;
  const int bkv = a.kv_bs == 0 ? 0 : b;

  if (tid == 0) {
    nb_s = block_list(a, b, c, js, ms);
    tc::mbar_init(&bar_q, 1);
    for (int st = 0; st < NST; ++st) tc::mbar_init(&bar_kv[st], 1);
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_o, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  const int nb = nb_s;
  if (nb == 0) {  // nothing to attend to: O = 0 (or unchanged when accumulating), LSE = -inf
    if (!a.accumulate)
      for (int u = tid; u < 64 * UPR; u += NT) {
        const int row = u / UPR, w = u % UPR;
        *reinterpret_cast<uint4*>(og + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
      }
    if (tid < 64) lse[tid] = -CUDART_INF_F;
    return;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 128);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tS = tmem_slot, tO = tmem_slot + 64;
  float inv0 = 0.f, inv1 = 0.f;  // 1 / row sums (softmax warps), for the epilogue

  if (warp == 4) {
    // ------------------------------------------------------------ control warp
    bool ok = true;
    auto load_block = [&](int x) {  // lane 0
      const int st = x % NST;
      unsigned char* Ks = ring + 2 * st * TILE;
      tc::mbar_expect_tx(&bar_kv[st], 2 * TILE);
      tc::tma_load_4d(Ks, &tmK, 0, h, js[x] * 64, bkv, &bar_kv[st]);
      tc::tma_load_4d(Ks + TILE, &tmV, 0, h, js[x] * 64, bkv, &bar_kv[st]);
    };
    const uint64_t dQ = tc::desc_km(tc::su32(Qs));
    uint64_t dK[NST], dV[NST];
#pragma unroll
    for (int st = 0; st < NST; ++st) {
      dK[st] = tc::desc_km(tc::su32(ring + 2 * st * TILE));
      dV[st] = tc::desc_mn(tc::su32(ring + (2 * st + 1) * TILE));
    }
    auto issue_s = [&](int x) {  // whole warp
      const uint64_t dk = x % NST == 0 ? dK[0] : dK[1];
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tS, dQ, dk, kIdS, 0u);
      tc::commit_warp(&bar_s);
    };
    if (lane == 0) {
      tc::mbar_expect_tx(&bar_q, TILE);
      tc::tma_load_4d(Qs, &tmQ, 0, h, c * 64, b, &bar_q);
      for (int x = 0; x < NST && x < nb; ++x) load_block(x);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bar_q, 0) && ok;
    ok = tc::mbar_wait(&bar_kv[0], 0) && ok;
    issue_s(0);
    for (int n = 0; n < nb; ++n) {
      tc::named_sync(kBarPReady, NT);  // P(n) in TMEM columns 0-31 and O rescaled
      tc::fence_after();
      const uint64_t dv = n % NST == 0 ? dV[0] : dV[1];
      tc::mma4_ts<8, 16, 24, tc::kKStepMn>(tO, tS, dv, kIdPV, n > 0 ? 1u : 0u);
      tc::commit_warp(&bar_o);
      if (n + 1 < nb) {
        ok = tc::mbar_wait(&bar_kv[(n + 1) % NST], ((n + 1) / NST) & 1) && ok;
        issue_s(n + 1);
      }
      ok = tc::mbar_wait(&bar_o, n & 1) && ok;  // ring stage n % NST is free
      if (lane == 0) {
        if (n + NST < nb) load_block(n + NST);
        if (!ok) flag_timeout(a.err);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int g = lane >> 2, cq = lane & 3;
    const int row0 = 16 * warp + g;  // rows row0 and row0 + 8 of the chunk
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * kLog2e;
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;  // running maxima of the raw logits
    float l0 = 0.f, l1 = 0.f;                        // running sums
    for (int n = 0; n < nb; ++n) {
      if (!tc::mbar_wait(&bar_s, n & 1)) flag_timeout(a.err);  // S(n); PV(n-1) is done as well
      float s[8][4];
#pragma unroll
      for (int cb = 0; cb < 8; ++cb) tc::ld16x256(tS + lane_base + cb * 8, s[cb]);
      tc::ld_wait(s);
      const int mk = ms[n];
      if (mk != kMaskNone) {
#pragma unroll
        for (int cb = 0; cb < 8; ++cb)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = 8 * cb + 2 * cq + (e & 1), row = row0 + 8 * (e >> 1);
            const bool drop = mk == kMaskCausal ? col > row : col <= row;
            if (drop) s[cb][e] = -CUDART_INF_F;
          }
      }
      float b0 = -CUDART_INF_F, b1 = -CUDART_INF_F;
#pragma unroll
      for (int cb = 0; cb < 8; ++cb) {
        b0 = fmaxf(b0, fmaxf(s[cb][0], s[cb][1]));
        b1 = fmaxf(b1, fmaxf(s[cb][2], s[cb][3]));
      }
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, m));
        b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, m));
      }
      const float n0 = fmaxf(mx0, b0), n1 = fmaxf(mx1, b1);
      // Rescale factors of the accumulated output and sum (1 while a row has seen nothing).
      const float a0 = n0 == -CUDART_INF_F ? 1.f : tc::ex2((mx0 - n0) * sl2);
      const float a1 = n1 == -CUDART_INF_F ? 1.f : tc::ex2((mx1 - n1) * sl2);
      mx0 = n0;
      mx1 = n1;
      const float o0 = n0 == -CUDART_INF_F ? 0.f : -n0 * sl2, o1 = n1 == -CUDART_INF_F ? 0.f : -n1 * sl2;
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int cb = 0; cb < 8; ++cb) {
        s[cb][0] = tc::ex2(fmaf(s[cb][0], sl2, o0));
        s[cb][1] = tc::ex2(fmaf(s[cb][1], sl2, o0));
        s[cb][2] = tc::ex2(fmaf(s[cb][2], sl2, o1));
        s[cb][3] = tc::ex2(fmaf(s[cb][3], sl2, o1));
        p0 += s[cb][0] + s[cb][1];
        p1 += s[cb][2] + s[cb][3];
      }
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        p0 += __shfl_xor_sync(0xffffffffu, p0, m);
        p1 += __shfl_xor_sync(0xffffffffu, p1, m);
      }
      l0 = l0 * a0 + p0;
      l1 = l1 * a1 + p1;
      // O holds the sum over blocks < n (PV(n-1) is complete); rescale it if needed.
      if (n > 0 && !__all_sync(0xffffffffu, a0 == 1.f && a1 == 1.f)) {
        float ov[8][4];
#pragma unroll
        for (int cb = 0; cb < 8; ++cb) tc::ld16x256(tO + lane_base + cb * 8, ov[cb]);
        tc::ld_wait(ov);
#pragma unroll
        for (int cb = 0; cb < 8; ++cb) {
          ov[cb][0] *= a0;
          ov[cb][1] *= a0;
          ov[cb][2] *= a1;
          ov[cb][3] *= a1;
          tc::st16x256(tO + lane_base + cb * 8, ov[cb]);
        }
      }
      // P (unnormalised) as the TMEM A operand: keys (8n + 2cq, +1) of rows g and g + 8
      // go to column 4n + cq.
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pv[2 * i] = pack_bf16(s[4 * half + i][0], s[4 * half + i][1]);
          pv[2 * i + 1] = pack_bf16(s[4 * half + i][2], s[4 * half + i][3]);
        }
        tc::st16x128_x4(tS + lane_base + 16 * half, pv);
      }
      tc::st_wait();
      tc::fence_before();
      tc::named_arrive(kBarPReady, NT);
    }
    if (cq == 0) {
      lse[row0] = l0 > 0.f ? mx0 * scale + __logf(l0) : -CUDART_INF_F;
      lse[row0 + 8] = l1 > 0.f ? mx1 * scale + __logf(l1) : -CUDART_INF_F;
    }
    inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
    inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  }
  // Every PV has completed (the control warp waited for the last one): O / l, staged
  // through the Q tile (its last reader, the final S = Q K^T, is done).
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp < 4) {
    const int g = lane >> 2, cq = lane & 3;
    const int row0 = 16 * warp + g;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    float o[8][4];
#pragma unroll
    for (int cb = 0; cb < 8; ++cb) tc::ld16x256(tO + lane_base + cb * 8, o[cb]);
    tc::ld_wait(o);
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(row0, n) + cq * 4) = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
      *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(row0 + 8, n) + cq * 4) = pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
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
    uint4 val = *reinterpret_cast<const uint4*>(Qs + swz<ROWB>(row, w));
    if (a.accumulate) {
      const uint4 old = *reinterpret_cast<const uint4*>(og + row * ts + w * 8);
      float fo[8], fn[8];
      unpack16(old, fo, (const bf16*)nullptr);
      unpack16(val, fn, (const bf16*)nullptr);
      val.x = pack_bf16(fo[0] + fn[0], fo[1] + fn[1]);
      val.y = pack_bf16(fo[2] + fn[2], fo[3] + fn[3]);
      val.z = pack_bf16(fo[4] + fn[4], fo[5] + fn[5]);
      val.w = pack_bf16(fo[6] + fn[6], fo[7] + fn[7]);
    }
    *reinterpret_cast<uint4*>(og + row * ts + w * 8) = val;
  }
}

// ------------------------------------------------------------------ SIMT path (f32, or dh = 32)
// One thread per query row, exact two-pass softmax per block list (expf), for the small
// configurations.
template <typename T, int DH>
__global__ void __launch_bounds__(64) block_attn_simt_kernel(BlockAttnArgs a) {
  __shared__ float Ks[64][DH + 1];
  __shared__ float Vs[64][DH + 1];
  __shared__ int js[kMaxBlocks], ms[kMaxBlocks];
  __shared__ int nb_s;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x;
  const int64_t ts = (int64_t)a.H * DH;
  const T* qg = reinterpret_cast<const T*>(a.q) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  T* og = reinterpret_cast<T*>(a.o) + ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  float* lse = a.lse + (((int64_t)b * a.nQ + c) * a.H + h) * 64;
  if (t == 0) nb_s = block_list(a, b, c, js, ms);
  __syncthreads();
  const int nb = nb_s;
  const float scale = 1.0f / sqrtf((float)DH);
  float qv[DH], o[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    qv[d] = Elem<T>::ld(qg + t * ts + d);
    o[d] = 0.f;
  }
  float mx = -CUDART_INF_F, l = 0.f;
  for (int pass = 0; pass < 2; ++pass) {  // pass 0: row maximum and sum; pass 1: output
    for (int n = 0; n < nb; ++n) {
      __syncthreads();
      const int64_t kb = (int64_t)b * a.kv_bs + (int64_t)js[n] * 64 * ts + h * DH;
      for (int x = t; x < 64 * DH; x += 64) {
        const int row = x / DH, d = x % DH;
        Ks[row][d] = Elem<T>::ld(reinterpret_cast<const T*>(a.k) + kb + row * ts + d);
        Vs[row][d] = Elem<T>::ld(reinterpret_cast<const T*>(a.v) + kb + row * ts + d);
      }
      __syncthreads();
      for (int key = 0; key < 64; ++key) {
        if (ms[n] == kMaskCausal && key > t) continue;
        if (ms[n] == kMaskTail && key <= t) continue;
        float acc = 0.f;
#pragma unroll
        for (int d = 0; d < DH; ++d) acc = fmaf(qv[d], Ks[key][d], acc);
        const float sv = acc * scale;
        if (pass == 0) {
          if (sv > mx) {
            l = l * expf(mx - sv) + 1.f;
            mx = sv;
          } else {
            l += expf(sv - mx);
          }
        } else {
          const float p = expf(sv - mx) / l;
#pragma unroll
          for (int d = 0; d < DH; ++d) o[d] = fmaf(p, Vs[key][d], o[d]);
        }
      }
    }
  }
  lse[t] = l > 0.f ? mx + logf(l) : -CUDART_INF_F;
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    float v = o[d];
    if (a.accumulate) v += Elem<T>::ld(og + t * ts + d);
    Elem<T>::st(og + t * ts + d, v);
  }
}

}  // namespace

cudaError_t launch_block_attn(const BlockAttnArgs& a, cudaStream_t s) {
  dim3 grid(a.nQ, a.H, a.B);
  const char* name = a.mode == 0 ? "window_attn" : "cca";
  if (a.bf16 && a.dh == 64) {
    CUtensorMap tq, tk, tv;
    cudaError_t e = make_head_tmap(&tq, a.q, 64, a.H, (int64_t)a.nQ * 64, a.B, (int64_t)a.nQ * 64 * a.H * 64);
    if (e == cudaSuccess) e = make_head_tmap(&tk, a.k, 64, a.H, (int64_t)a.nC * 64, a.B, a.kv_bs);
    if (e == cudaSuccess) e = make_head_tmap(&tv, a.v, 64, a.H, (int64_t)a.nC * 64, a.B, a.kv_bs);
    if (e == cudaSuccess) e = allow_smem((const void*)block_attn_tc_kernel, kBaSmem);
    if (e != cudaSuccess) return e;
    launch_begin(name, s);
    block_attn_tc_kernel<<<grid, kBaThreads, kBaSmem, s>>>(a, tq, tk, tv);
    return launch_end(name, s);
  }
  launch_begin(name, s);
  if (a.bf16) block_attn_simt_kernel<bf16, 32><<<grid, 64, 0, s>>>(a);
  else if (a.dh == 64) block_attn_simt_kernel<float, 64><<<grid, 64, 0, s>>>(a);
  else block_attn_simt_kernel<float, 32><<<grid, 64, 0, s>>>(a);
  return launch_end(name, s);
}

}  // namespace gca
