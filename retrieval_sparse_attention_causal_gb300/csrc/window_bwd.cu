// Backward of the sliding-window causal self-attention (block_attn.cu, window mode).
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", 损失函数/训练策略 (training strategy: sliding-window
// self-attention, W = 512, trained beside the top-k retrieval).  With P the masked row
// softmax (recomputed from the saved LSE), per sequence and head:
//     D = rowsum(dO * O),  dS = P * (dO V^T - D),
//     dQ = dS K / sqrt(dh),  dK = dS^T Q / sqrt(dh),  dV = P^T dO.
// Three kernels: D per row; a query-side pass (per query chunk over its window blocks,
// dQ); a key-side pass (per key chunk over the query chunks whose window covers it, dK and
// dV).  Neither needs atomics, so the result is deterministic.
//
// The same passes give the backward of CCA (block_attn.cu, CCA mode; Paper-Notes page,
// 关键设计 / Grouped Cross-Attention: one joint softmax over the concatenated retrieved
// chunks): the query side walks the valid retrieved chunks of row c - shift instead of
// the window blocks, the key side walks the query chunks whose row retrieved the chunk
// (the consumer lists of the GCA backward, in entry order), and no block is masked.  Both tensor-core passes
// follow the GCA backward's layout: a control warp issues TMA loads and tcgen05.mma, eight
// element warps (TMEM lane quarter w % 4, column half w / 4) do the arithmetic and store
// the bf16 A operand of the next product into TMEM over the columns they read.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gca {
namespace {

using bf16 = __nv_bfloat16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kEW = 8, kThreads = 32 * (kEW + 1), kCtl = kEW;
constexpr int TILE = 8192, ROWB = 128, UPR = 8, DH = 64;
enum { kBarOpReady = 2 };

// ------------------------------------------------------------------ D = rowsum(dO * O)
// LPR consecutive lanes per (token, head) row, one 16-byte vector of O and of dO each, so a
// warp reads 32 contiguous vectors; the partial dot products meet by shuffles.
// D [B][L/64][H][64] like the LSE.
template <typename T, int DHT>
__global__ void __launch_bounds__(256) window_d_kernel(WindowBwdArgs a) {
  constexpr int EPV = Elem<T>::kVec, LPR = DHT / EPV;
  static_assert(32 % LPR == 0, "a row's lanes stay inside one warp");
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = g / LPR;  // token * H + h
  const int part = (int)(g % LPR);
  const int64_t nrows = (int64_t)a.B * a.nQ * 64 * a.H;
  float acc = 0.f;
  if (row < nrows) {
    const uint4 ov = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.o) + row * DHT) + part);
    const uint4 dv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.dout) + row * DHT) + part);
    float of[EPV], df[EPV];
    unpack16(ov, of, static_cast<const T*>(nullptr));
    unpack16(dv, df, static_cast<const T*>(nullptr));
#pragma unroll
    for (int x = 0; x < EPV; ++x) acc = fmaf(of[x], df[x], acc);
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < nrows && part == 0) {
    const int64_t tok = row / a.H;
    const int h = (int)(row % a.H);
    a.Dbuf[((tok / 64) * a.H + h) * 64 + tok % 64] = acc;  // tok / 64 = b * nQ + c
  }
}

// CCA: the valid retrieved chunks of the row that query chunk c reads (slot order);
// indices outside [-1, nC) are flagged and skipped.  Returns their count.
__device__ __forceinline__ int cca_blocks(const WindowBwdArgs& a, int b, int c, int (&blk)[kMaxTopk]) {
  const int r = c - a.shift;
  int n = 0;
  if (r < 0) return 0;
  const int32_t* row = a.idx + ((int64_t)b * a.nQ + r) * a.topk;
  for (int m = 0; m < a.topk; ++m) {
    const int j = row[m];
    if (j >= 0 && j < a.nC) blk[n++] = j;
    else if (j != -1 && threadIdx.x == 0) flag_bad_index(a.err, j);
  }
  return n;
}

// Mask of key column kc against query row qr inside a block pair: kind 1 (tail block of
// the window) keeps kc > qr, kind 2 (diagonal block) keeps kc <= qr.
__device__ __forceinline__ bool dropped(int kind, int kc, int qr) {
  return kind == 1 ? kc <= qr : (kind == 2 ? kc > qr : false);
}

// ------------------------------------------------------------------ query side (bf16, dh = 64)
constexpr int kQStages = 4;
constexpr int kQSmem = TILE * (2 + 2 * kQStages) + 1024;  // Q, dO, ring of (K, V)

__global__ void __launch_bounds__(kThreads, 2)
window_bwd_q_tc_kernel(WindowBwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  constexpr int NST = kQStages, NT = kThreads;
  constexpr uint32_t kIdKm = tc::idesc_bf16(64, 64, false);
  constexpr uint32_t kIdMn = tc::idesc_bf16(64, 64, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* Qs = sm;
  unsigned char* dOs = sm + TILE;
  unsigned char* ring = sm + 2 * TILE;
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar_q, bar_kv[NST], bar_s, bar_o, sfree, dq_done[2];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int64_t tok0 = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
  bf16* dqg = reinterpret_cast<bf16*>(a.dq) + tok0;
  const int64_t rowbase = (((int64_t)b * a.nQ + c) * a.H + h) * 64;
  const int wb = a.window / 64;
  const int j0 = c - wb < 0 ? 0 : c - wb;  // window: key blocks j0 .. c
  int blk[kMaxTopk];                        // CCA: the row's valid retrieved chunks
  const int nb = a.mode == 0 ? c - j0 + 1 : cca_blocks(a, b, c, blk);
  auto block_of = [&](int n) { return a.mode == 0 ? j0 + n : blk[n]; };
  auto kind_of = [&](int n) {
    const int j = j0 + n;
    return a.mode != 0 ? 0 : (j == c ? 2 : (j == c - wb ? 1 : 0));
  };
  if (nb == 0) {  // CCA: no valid slot, dQ = 0
    if (!a.accumulate)
      for (int u = tid; u < 64 * UPR; u += kThreads)
        *reinterpret_cast<uint4*>(dqg + (u / UPR) * ts + (u % UPR) * 8) = make_uint4(0, 0, 0, 0);
    return;
  }

  if (tid == 0) {
    tc::mbar_init(&bar_q, 1);
    for (int st = 0; st < NST; ++st) tc::mbar_init(&bar_kv[st], 1);
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_o, 1);
    tc::mbar_init(&sfree, kEW);
    tc::mbar_init(&dq_done[0], 1);
    tc::mbar_init(&dq_done[1], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 256);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // TMEM: S, dPo, dQ, and two dS buffers (32 columns each): the next block's S, dPo go in
  // as soon as the element warps hold the current ones in registers.
  const uint32_t tS = tmem_slot, tP = tmem_slot + 64, tQ = tmem_slot + 128, tdS = tmem_slot + 192;

  if (warp == kCtl) {
    // ------------------------------------------------------------ control warp
    bool ok = true;
    auto load_block = [&](int x) {  // lane 0
      const int st = x % NST;
      unsigned char* Ks = ring + 2 * st * TILE;
      tc::mbar_expect_tx(&bar_kv[st], 2 * TILE);
      tc::tma_load_4d(Ks, &tmK, 0, h, block_of(x) * 64, b, &bar_kv[st]);
      tc::tma_load_4d(Ks + TILE, &tmV, 0, h, block_of(x) * 64, b, &bar_kv[st]);
    };
    const uint64_t dQd = tc::desc_km(tc::su32(Qs)), dOd = tc::desc_km(tc::su32(dOs));
    const uint64_t dRingKm = tc::desc_km(tc::su32(ring)), dRingMn = tc::desc_mn(tc::su32(ring));
    constexpr uint64_t kStage = (2 * TILE) >> 4, kTileStep = TILE >> 4;
    auto issue_s = [&](int x) {  // S = Q K^T and dPo = dO V^T of block x (whole warp)
      const uint64_t dk = dRingKm + (x % NST) * kStage, dv = dk + kTileStep;
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tS, dQd, dk, kIdKm, 0u);
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tP, dOd, dv, kIdKm, 0u);
      tc::commit_warp(&bar_s);
    };
    if (lane == 0) {
      tc::mbar_expect_tx(&bar_q, 2 * TILE);
      tc::tma_load_4d(Qs, &tmQ, 0, h, c * 64, b, &bar_q);
      tc::tma_load_4d(dOs, &tmdO, 0, h, c * 64, b, &bar_q);
      for (int x = 0; x < NST && x < nb; ++x) load_block(x);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bar_q, 0) && ok;
    ok = tc::mbar_wait(&bar_kv[0], 0) && ok;
    issue_s(0);
    for (int n = 0; n < nb; ++n) {
      // S(n), dPo(n) are in the element warps' registers: the next pair goes in now.
      ok = tc::mbar_wait(&sfree, n & 1) && ok;
      tc::fence_after();
      if (n + 1 < nb) {
        ok = tc::mbar_wait(&bar_kv[(n + 1) % NST], ((n + 1) / NST) & 1) && ok;
        issue_s(n + 1);
      }
      tc::named_sync(kBarOpReady, NT);  // dS(n) is in dS buffer n & 1
      tc::fence_after();
      const uint64_t dk = dRingMn + (n % NST) * kStage;
      // dQ += dS K  (K as the MN-major B operand)
      tc::mma4_ts<8, 16, 24, tc::kKStepMn>(tQ, tdS + 32 * (n & 1), dk, kIdMn, n > 0 ? 1u : 0u);
      tc::commit_warp(&bar_o);
      tc::commit_warp(&dq_done[n & 1]);
      ok = tc::mbar_wait(&bar_o, n & 1) && ok;  // ring stage n % NST is free
      if (lane == 0) {
        if (n + NST < nb) load_block(n + NST);
        if (!ok) flag_timeout(a.err);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ element-wise warps
    const int g = lane >> 2, cq = lane & 3, quarter = warp & 3, hc = warp >> 2;
    const int row0 = 16 * quarter + g;
    const uint32_t lane_q = (uint32_t)(32 * quarter) << 16;
    const uint32_t lane_base = lane_q + 32 * hc;
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * kLog2e;
    const float lse0 = a.lse[rowbase + row0] * kLog2e, lse1 = a.lse[rowbase + row0 + 8] * kLog2e;
    const float D0 = a.Dbuf[rowbase + row0], D1 = a.Dbuf[rowbase + row0 + 8];
    for (int n = 0; n < nb; ++n) {
      if (!tc::mbar_wait(&bar_s, n & 1)) flag_timeout(a.err);  // S(n), dPo(n)
      float s[4][4], dp[4][4];
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tS + lane_base + cb * 8, s[cb]);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tP + lane_base + cb * 8, dp[cb]);
      tc::ld_wait(s);
      tc::ld_wait(dp);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sfree);
      const int kind = kind_of(n);
      uint32_t dv[8];
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {  // key columns 32hc + 8cb + 2cq (+1)
        float ds[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kc = 32 * hc + 8 * cb + 2 * cq + (e & 1), qr = row0 + 8 * (e >> 1);
          const float l = e < 2 ? lse0 : lse1, dd = e < 2 ? D0 : D1;
          const float p = dropped(kind, kc, qr) ? 0.f : tc::ex2(fmaf(s[cb][e], sl2, -l));
          ds[e] = p * (dp[cb][e] - dd) * scale;
        }
        dv[2 * cb] = pack_bf16(ds[0], ds[1]);
        dv[2 * cb + 1] = pack_bf16(ds[2], ds[3]);
      }
      // dS buffer n & 1 is free once dQ(n - 2) has read it.
      if (n >= 2 && !tc::mbar_wait(&dq_done[n & 1], ((n >> 1) - 1) & 1)) flag_timeout(a.err);
      tc::st16x128_x4(tdS + 32 * (n & 1) + lane_q + 16 * hc, dv);
      tc::st_wait();
      tc::fence_before();
      tc::named_arrive(kBarOpReady, NT);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp < kEW) {  // dQ from TMEM, staged through the Q tile
    const int g = lane >> 2, cq = lane & 3, quarter = warp & 3, hc = warp >> 2;
    const uint32_t lane_base = ((uint32_t)(32 * quarter) << 16) + 32 * hc;
    float o[4][4];
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tQ + lane_base + cb * 8, o[cb]);
    tc::ld_wait(o);
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int r0 = 16 * quarter + g;
      *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0, 4 * hc + n) + cq * 4) = pack_bf16(o[n][0], o[n][1]);
      *reinterpret_cast<uint32_t*>(Qs + swz<ROWB>(r0 + 8, 4 * hc + n) + cq * 4) = pack_bf16(o[n][2], o[n][3]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tmem_slot, 256);
  }
  for (int u = tid; u < 64 * UPR; u += NT) {
    const int row = u / UPR, w = u % UPR;
    uint4 val = *reinterpret_cast<const uint4*>(Qs + swz<ROWB>(row, w));
    if (a.accumulate) {
      const uint4 old = *reinterpret_cast<const uint4*>(dqg + row * ts + w * 8);
      float fo[8], fn[8];
      unpack16(old, fo, (const bf16*)nullptr);
      unpack16(val, fn, (const bf16*)nullptr);
      val.x = pack_bf16(fo[0] + fn[0], fo[1] + fn[1]); val.y = pack_bf16(fo[2] + fn[2], fo[3] + fn[3]);
      val.z = pack_bf16(fo[4] + fn[4], fo[5] + fn[5]); val.w = pack_bf16(fo[6] + fn[6], fo[7] + fn[7]);
    }
    *reinterpret_cast<uint4*>(dqg + row * ts + w * 8) = val;
  }
}

// ------------------------------------------------------------------ key side (bf16, dh = 64)
constexpr int kKVStages = 4;
constexpr int kKVStageBytes = 2 * TILE + 1024;  // Q, dO tiles + LSE and D rows
constexpr int kKVSmem = TILE * 2 + kKVStages * kKVStageBytes + 1024;

__global__ void __launch_bounds__(kThreads, 2)
window_bwd_kv_tc_kernel(WindowBwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  constexpr int NST = kKVStages, NT = kThreads;
  constexpr uint32_t kIdKm = tc::idesc_bf16(64, 64, false);
  constexpr uint32_t kIdMn = tc::idesc_bf16(64, 64, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* Ks = sm;
  unsigned char* Vs = sm + TILE;
  unsigned char* ring = sm + 2 * TILE;  // stage st: Q, dO, lse[64], D[64]
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar_k, bar_c[NST], bar_s1, bar_s2, op_v, op_k, bar_o;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int64_t ktok0 = ((int64_t)b * a.nC * 64 + (int64_t)j * 64) * ts + h * DH;
  bf16* dkg = reinterpret_cast<bf16*>(a.dk) + ktok0;
  bf16* dvg = reinterpret_cast<bf16*>(a.dv) + ktok0;
  const int wb = a.window / 64;
  const int c1 = j + wb < a.nQ - 1 ? j + wb : a.nQ - 1;  // window: query chunks j .. c1 see key chunk j
  const int e0 = a.mode == 0 ? 0 : a.csr_off[(int64_t)b * (a.nC + 1) + j];
  const int ncons = a.mode == 0 ? c1 - j + 1 : a.csr_off[(int64_t)b * (a.nC + 1) + j + 1] - e0;
  const int32_t* ent = a.mode == 0 ? nullptr : a.csr_ent + (int64_t)b * a.nQ * a.topk + e0;
  // Window: consumer x is query chunk j + x, x = 0 the diagonal block (keep key <= query),
  // x = wb the block where the window starts (keep key > query).  CCA: the query chunk of
  // the x-th entry of the chunk's consumer list, unmasked.
  auto cons_of = [&](int x) { return a.mode == 0 ? j + x : ent[x] / a.topk + a.shift; };
  auto kind_of = [&](int x) { return a.mode != 0 ? 0 : (x == 0 ? 2 : (x == wb ? 1 : 0)); };
  if (ncons == 0) {  // CCA: never retrieved, dK = dV = 0
    if (!a.accumulate)
      for (int u = tid; u < 64 * UPR; u += kThreads) {
        *reinterpret_cast<uint4*>(dkg + (u / UPR) * ts + (u % UPR) * 8) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(dvg + (u / UPR) * ts + (u % UPR) * 8) = make_uint4(0, 0, 0, 0);
      }
    return;
  }

  if (warp == kCtl && lane == 0) {
    tc::mbar_init(&bar_k, 1);
    for (int st = 0; st < NST; ++st) tc::mbar_init(&bar_c[st], 1);
    tc::mbar_init(&bar_s1, 1);
    tc::mbar_init(&bar_s2, 1);
    tc::mbar_init(&op_v, kEW);
    tc::mbar_init(&op_k, kEW);
    tc::mbar_init(&bar_o, 1);
    tc::fence_mbar_init();
    tc::mbar_expect_tx(&bar_k, 2 * TILE);
    tc::tma_load_4d(Ks, &tmK, 0, h, j * 64, b, &bar_k);
    tc::tma_load_4d(Vs, &tmV, 0, h, j * 64, b, &bar_k);
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 256);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tS = tmem_slot, tP = tmem_slot + 64, tdV = tmem_slot + 128, tdK = tmem_slot + 192;

  if (warp == kCtl) {
    // ------------------------------------------------------------ control warp
    bool ok = true;
    auto load_cons = [&](int x) {  // lane 0: consumer x's Q, dO tiles, LSE and D rows
      const int st = x % NST;
      const int c = cons_of(x);
      unsigned char* base = ring + st * kKVStageBytes;
      const int64_t rb = (((int64_t)b * a.nQ + c) * a.H + h) * 64;
      tc::mbar_expect_tx(&bar_c[st], 2 * TILE + 512);
      tc::tma_load_4d(base, &tmQ, 0, h, c * 64, b, &bar_c[st]);
      tc::tma_load_4d(base + TILE, &tmdO, 0, h, c * 64, b, &bar_c[st]);
      tc::bulk_load(base + 2 * TILE, a.lse + rb, 256, &bar_c[st]);
      tc::bulk_load(base + 2 * TILE + 256, a.Dbuf + rb, 256, &bar_c[st]);
    };
    const uint64_t dKd = tc::desc_km(tc::su32(Ks)), dVd = tc::desc_km(tc::su32(Vs));
    const uint64_t dRingKm = tc::desc_km(tc::su32(ring)), dRingMn = tc::desc_mn(tc::su32(ring));
    constexpr uint64_t kStage = kKVStageBytes >> 4, kTileStep = TILE >> 4;
    // The products of consumer x go in the order dV(x), S^T(x + 1), dK(x), dPo^T(x + 1):
    // S^T(x + 1) overwrites P^T(x), which only dV(x) reads, and dPo^T(x + 1) overwrites
    // dS^T(x), which only dK(x) reads, so each product only follows the one it has to.
    auto issue_st = [&](int x) {  // S^T = K Q^T of consumer x (whole warp)
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tS, dKd, dRingKm + (x % NST) * kStage, kIdKm, 0u);
      tc::commit_warp(&bar_s1);
    };
    auto issue_dpt = [&](int x) {  // dPo^T = V dO^T of consumer x
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tP, dVd, dRingKm + (x % NST) * kStage + kTileStep, kIdKm, 0u);
      tc::commit_warp(&bar_s2);
    };
    if (lane == 0)
      for (int x = 0; x < NST && x < ncons; ++x) load_cons(x);
    __syncwarp();
    ok = tc::mbar_wait(&bar_k, 0) && ok;
    ok = tc::mbar_wait(&bar_c[0], 0) && ok;
    issue_st(0);
    issue_dpt(0);
    for (int ci = 0; ci < ncons; ++ci) {
      const uint64_t bq = dRingMn + (ci % NST) * kStage, bdo = bq + kTileStep;
      // dV += P^T dO once P^T is in (each element warp's query pairs over the first 16 of
      // its 32 columns: the K steps' A columns are 0, 8, 32, 40).
      ok = tc::mbar_wait(&op_v, ci & 1) && ok;
      tc::fence_after();
      tc::mma4_ts<8, 32, 40, tc::kKStepMn>(tdV, tS, bdo, kIdMn, ci > 0 ? 1u : 0u);
      const bool more = ci + 1 < ncons;
      if (more) {
        ok = tc::mbar_wait(&bar_c[(ci + 1) % NST], ((ci + 1) / NST) & 1) && ok;
        issue_st(ci + 1);
      }
      ok = tc::mbar_wait(&op_k, ci & 1) && ok;
      tc::fence_after();
      tc::mma4_ts<8, 32, 40, tc::kKStepMn>(tdK, tP, bq, kIdMn, ci > 0 ? 1u : 0u);
      tc::commit_warp(&bar_o);
      if (more) issue_dpt(ci + 1);
      ok = tc::mbar_wait(&bar_o, ci & 1) && ok;  // ring stage ci % NST is free
      if (lane == 0) {
        if (ci + NST < ncons) load_cons(ci + NST);
        if (!ok) flag_timeout(a.err);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ element-wise warps
    const int g = lane >> 2, cq = lane & 3, quarter = warp & 3, hc = warp >> 2;
    const int key0 = 16 * quarter + g;  // key rows key0, key0 + 8
    const uint32_t lane_q = (uint32_t)(32 * quarter) << 16;
    const uint32_t lane_base = lane_q + 32 * hc;
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * kLog2e;
    for (int ci = 0; ci < ncons; ++ci) {
      if (!tc::mbar_wait(&bar_s1, ci & 1)) flag_timeout(a.err);  // S^T(ci)
      const int st = ci % NST;
      tc::mbar_wait(&bar_c[st], (ci / NST) & 1);  // observe the rows' phase (complete)
      const float* lrow = reinterpret_cast<const float*>(ring + st * kKVStageBytes + 2 * TILE) + 32 * hc;
      const float* drow = lrow + 64;
      float s[4][4];
      tc::ld16x256_x4(tS + lane_base, s);
      tc::ld_wait(s);
      const int kind = kind_of(ci);
      // P^T, stored over the columns this warp has read: the pair of queries
      // (32hc + 8n + 2cq, +1) of key rows g and g + 8 goes to column 32hc + 4n + cq.
      uint32_t pv[8];
#pragma unroll
      for (int n = 0; n < 4; ++n) {  // query columns 32hc + 8n + 2cq (+1)
        const float2 l2 = *reinterpret_cast<const float2*>(lrow + 8 * n + 2 * cq);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qc = 32 * hc + 8 * n + 2 * cq + (e & 1), kr = key0 + 8 * (e >> 1);
          const float l = (e & 1) ? l2.y : l2.x;
          s[n][e] = dropped(kind, kr, qc) ? 0.f : tc::ex2(fmaf(s[n][e], sl2, -l * kLog2e));
        }
        pv[2 * n] = pack_bf16(s[n][0], s[n][1]);
        pv[2 * n + 1] = pack_bf16(s[n][2], s[n][3]);
      }
      tc::st16x128_x4(tS + lane_base, pv);
      tc::st_wait();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&op_v);
      // dS^T from dPo^T, over its own columns too.
      if (!tc::mbar_wait(&bar_s2, ci & 1)) flag_timeout(a.err);  // dPo^T(ci)
      tc::fence_after();
      float dp[4][4];
      tc::ld16x256_x4(tP + lane_base, dp);
      tc::ld_wait(dp);
      uint32_t dv[8];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const float2 d2 = *reinterpret_cast<const float2*>(drow + 8 * n + 2 * cq);
        dv[2 * n] = pack_bf16(s[n][0] * (dp[n][0] - d2.x) * scale, s[n][1] * (dp[n][1] - d2.y) * scale);
        dv[2 * n + 1] = pack_bf16(s[n][2] * (dp[n][2] - d2.x) * scale, s[n][3] * (dp[n][3] - d2.y) * scale);
      }
      tc::st16x128_x4(tP + lane_base, dv);
      tc::st_wait();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&op_k);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp < kEW) {  // dK (TMEM 192-255) into the K tile, dV (128-191) into the V tile
    const int g = lane >> 2, cq = lane & 3, quarter = warp & 3, hc = warp >> 2;
    const uint32_t lane_base = ((uint32_t)(32 * quarter) << 16) + 32 * hc;
    float o[4][4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      unsigned char* dst = half ? Vs : Ks;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::ld16x256((half ? tdV : tdK) + lane_base + cb * 8, o[cb]);
      tc::ld_wait(o);
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int r0 = 16 * quarter + g;
        *reinterpret_cast<uint32_t*>(dst + swz<ROWB>(r0, 4 * hc + n) + cq * 4) = pack_bf16(o[n][0], o[n][1]);
        *reinterpret_cast<uint32_t*>(dst + swz<ROWB>(r0 + 8, 4 * hc + n) + cq * 4) = pack_bf16(o[n][2], o[n][3]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tmem_slot, 256);
  }
  for (int u = tid; u < 64 * UPR; u += NT) {
    const int row = u / UPR, w = u % UPR;
    uint4 vk = *reinterpret_cast<const uint4*>(Ks + swz<ROWB>(row, w));
    uint4 vv = *reinterpret_cast<const uint4*>(Vs + swz<ROWB>(row, w));
    if (a.accumulate) {
      const uint4 ok = *reinterpret_cast<const uint4*>(dkg + row * ts + w * 8);
      const uint4 ov = *reinterpret_cast<const uint4*>(dvg + row * ts + w * 8);
      float fk[8], fv[8], nk[8], nv[8];
      unpack16(ok, fk, (const bf16*)nullptr);
      unpack16(ov, fv, (const bf16*)nullptr);
      unpack16(vk, nk, (const bf16*)nullptr);
      unpack16(vv, nv, (const bf16*)nullptr);
      vk.x = pack_bf16(nk[0] + fk[0], nk[1] + fk[1]); vk.y = pack_bf16(nk[2] + fk[2], nk[3] + fk[3]);
      vk.z = pack_bf16(nk[4] + fk[4], nk[5] + fk[5]); vk.w = pack_bf16(nk[6] + fk[6], nk[7] + fk[7]);
      vv.x = pack_bf16(nv[0] + fv[0], nv[1] + fv[1]); vv.y = pack_bf16(nv[2] + fv[2], nv[3] + fv[3]);
      vv.z = pack_bf16(nv[4] + fv[4], nv[5] + fv[5]); vv.w = pack_bf16(nv[6] + fv[6], nv[7] + fv[7]);
    }
    *reinterpret_cast<uint4*>(dkg + row * ts + w * 8) = vk;
    *reinterpret_cast<uint4*>(dvg + row * ts + w * 8) = vv;
  }
}

// ------------------------------------------------------------------ SIMT path (f32, or dh = 32)
// One thread per query row (dQ) and per key row (dK, dV), two passes over the blocks.
template <typename T, int DHT>
__global__ void __launch_bounds__(64) window_bwd_q_simt_kernel(WindowBwdArgs a) {
  __shared__ float Ks[64][DHT + 1], Vs[64][DHT + 1];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
  const int64_t ts = (int64_t)a.H * DHT;
  const int64_t tok = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64 + t) * ts + h * DHT;
  const int64_t rb = (((int64_t)b * a.nQ + c) * a.H + h) * 64 + t;
  const float scale = 1.0f / sqrtf((float)DHT), lse = a.lse[rb], D = a.Dbuf[rb];
  float qv[DHT], dov[DHT], dq[DHT];
  for (int d = 0; d < DHT; ++d) {
    qv[d] = Elem<T>::ld(reinterpret_cast<const T*>(a.q) + tok + d);
    dov[d] = Elem<T>::ld(reinterpret_cast<const T*>(a.dout) + tok + d);
    dq[d] = 0.f;
  }
  const int wb = a.window / 64, j0 = c - wb < 0 ? 0 : c - wb;
  int blk[kMaxTopk];
  const int nb = a.mode == 0 ? c - j0 + 1 : cca_blocks(a, b, c, blk);
  for (int n = 0; n < nb; ++n) {
    const int jb = a.mode == 0 ? j0 + n : blk[n];
    __syncthreads();
    const int64_t kb = ((int64_t)b * a.nC * 64 + (int64_t)jb * 64) * ts + h * DHT;
    for (int x = t; x < 64 * DHT; x += 64) {
      const int row = x / DHT, d = x % DHT;
      Ks[row][d] = Elem<T>::ld(reinterpret_cast<const T*>(a.k) + kb + row * ts + d);
      Vs[row][d] = Elem<T>::ld(reinterpret_cast<const T*>(a.v) + kb + row * ts + d);
    }
    __syncthreads();
    const int kind = a.mode != 0 ? 0 : (jb == c ? 2 : (jb == c - wb ? 1 : 0));
    for (int key = 0; key < 64; ++key) {
      if (dropped(kind, key, t)) continue;
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < DHT; ++d) {
        s = fmaf(qv[d], Ks[key][d], s);
        dp = fmaf(dov[d], Vs[key][d], dp);
      }
      const float ds = expf(s * scale - lse) * (dp - D) * scale;
      for (int d = 0; d < DHT; ++d) dq[d] = fmaf(ds, Ks[key][d], dq[d]);
    }
  }
  for (int d = 0; d < DHT; ++d) {
    T* p = reinterpret_cast<T*>(a.dq) + tok + d;
    Elem<T>::st(p, a.accumulate ? Elem<T>::ld(p) + dq[d] : dq[d]);
  }
}

template <typename T, int DHT>
__global__ void __launch_bounds__(64) window_bwd_kv_simt_kernel(WindowBwdArgs a) {
  __shared__ float Qs[64][DHT + 1], dOs[64][DHT + 1], ls[64], Ds[64];
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
  const int64_t ts = (int64_t)a.H * DHT;
  const int64_t tok = ((int64_t)b * a.nC * 64 + (int64_t)j * 64 + t) * ts + h * DHT;
  const float scale = 1.0f / sqrtf((float)DHT);
  float kv[DHT], vv[DHT], dk[DHT], dv[DHT];
  for (int d = 0; d < DHT; ++d) {
    kv[d] = Elem<T>::ld(reinterpret_cast<const T*>(a.k) + tok + d);
    vv[d] = Elem<T>::ld(reinterpret_cast<const T*>(a.v) + tok + d);
    dk[d] = dv[d] = 0.f;
  }
  const int wb = a.window / 64;
  const int c1 = j + wb < a.nQ - 1 ? j + wb : a.nQ - 1;
  const int e0 = a.mode == 0 ? 0 : a.csr_off[(int64_t)b * (a.nC + 1) + j];
  const int ncons = a.mode == 0 ? c1 - j + 1 : a.csr_off[(int64_t)b * (a.nC + 1) + j + 1] - e0;
  const int32_t* ent = a.mode == 0 ? nullptr : a.csr_ent + (int64_t)b * a.nQ * a.topk + e0;
  for (int x = 0; x < ncons; ++x) {
    const int c = a.mode == 0 ? j + x : ent[x] / a.topk + a.shift;
    __syncthreads();
    const int64_t qb = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DHT;
    for (int x = t; x < 64 * DHT; x += 64) {
      const int row = x / DHT, d = x % DHT;
      Qs[row][d] = Elem<T>::ld(reinterpret_cast<const T*>(a.q) + qb + row * ts + d);
      dOs[row][d] = Elem<T>::ld(reinterpret_cast<const T*>(a.dout) + qb + row * ts + d);
    }
    const int64_t rb = (((int64_t)b * a.nQ + c) * a.H + h) * 64;
    ls[t] = a.lse[rb + t];
    Ds[t] = a.Dbuf[rb + t];
    __syncthreads();
    const int kind = a.mode != 0 ? 0 : (c == j ? 2 : (c == j + wb ? 1 : 0));
    for (int qr = 0; qr < 64; ++qr) {
      if (dropped(kind, t, qr)) continue;  // this thread's key t against query row qr
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < DHT; ++d) {
        s = fmaf(Qs[qr][d], kv[d], s);
        dp = fmaf(dOs[qr][d], vv[d], dp);
      }
      const float p = expf(s * scale - ls[qr]);
      const float ds = p * (dp - Ds[qr]) * scale;
      for (int d = 0; d < DHT; ++d) {
        dv[d] = fmaf(p, dOs[qr][d], dv[d]);
        dk[d] = fmaf(ds, Qs[qr][d], dk[d]);
      }
    }
  }
  for (int d = 0; d < DHT; ++d) {
    T* pk = reinterpret_cast<T*>(a.dk) + tok + d;
    T* pv = reinterpret_cast<T*>(a.dv) + tok + d;
    Elem<T>::st(pk, a.accumulate ? Elem<T>::ld(pk) + dk[d] : dk[d]);
    Elem<T>::st(pv, a.accumulate ? Elem<T>::ld(pv) + dv[d] : dv[d]);
  }
}

}  // namespace

cudaError_t launch_window_backward(const WindowBwdArgs& a, cudaStream_t s) {
  const int64_t nrows = (int64_t)a.B * a.nQ * 64 * a.H;
  const int lpr = a.dh * (a.bf16 ? 2 : 4) / 16;  // lanes per row in window_d_kernel
  const unsigned dgrid = (unsigned)((nrows * lpr + 255) / 256);
  launch_begin("window_d", s);
  if (a.bf16) {
    if (a.dh == 64) window_d_kernel<bf16, 64><<<dgrid, 256, 0, s>>>(a);
    else window_d_kernel<bf16, 32><<<dgrid, 256, 0, s>>>(a);
  } else {
    if (a.dh == 64) window_d_kernel<float, 64><<<dgrid, 256, 0, s>>>(a);
    else window_d_kernel<float, 32><<<dgrid, 256, 0, s>>>(a);
  }
  cudaError_t e = launch_end("window_d", s);
  if (e != cudaSuccess) return e;
  const char* nq = a.mode == 0 ? "window_bwd_q" : "cca_bwd_q";
  const char* nkv = a.mode == 0 ? "window_bwd_kv" : "cca_bwd_kv";
  if (a.mode != 0) {  // the consumers of every key chunk, in entry order
    const int nrows = a.nQ - a.shift;
    e = launch_csr(a.idx, a.B, a.nQ, nrows > 0 ? nrows : 0, a.topk, a.nC, const_cast<int32_t*>(a.csr_off),
                   const_cast<int32_t*>(a.csr_ent), a.csr_cur, a.err, s);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(a.nQ, a.H, a.B), gridk(a.nC, a.H, a.B);
  if (a.bf16 && a.dh == 64) {
    CUtensorMap tq, tdo, tk, tv;
    const int64_t bs = (int64_t)a.nQ * 64 * a.H * 64, rows = (int64_t)a.nQ * 64;
    const int64_t kbs = (int64_t)a.nC * 64 * a.H * 64, krows = (int64_t)a.nC * 64;
    e = make_head_tmap(&tq, a.q, 64, a.H, rows, a.B, bs);
    if (e == cudaSuccess) e = make_head_tmap(&tdo, a.dout, 64, a.H, rows, a.B, bs);
    if (e == cudaSuccess) e = make_head_tmap(&tk, a.k, 64, a.H, krows, a.B, kbs);
    if (e == cudaSuccess) e = make_head_tmap(&tv, a.v, 64, a.H, krows, a.B, kbs);
    if (e == cudaSuccess) e = allow_smem((const void*)window_bwd_q_tc_kernel, kQSmem);
    if (e == cudaSuccess) e = allow_smem((const void*)window_bwd_kv_tc_kernel, kKVSmem);
    if (e != cudaSuccess) return e;
    launch_begin(nq, s);
    window_bwd_q_tc_kernel<<<grid, kThreads, kQSmem, s>>>(a, tq, tdo, tk, tv);
    if ((e = launch_end(nq, s)) != cudaSuccess) return e;
    launch_begin(nkv, s);
    window_bwd_kv_tc_kernel<<<gridk, kThreads, kKVSmem, s>>>(a, tq, tdo, tk, tv);
    return launch_end(nkv, s);
  }
  launch_begin(nq, s);
  if (a.bf16) window_bwd_q_simt_kernel<bf16, 32><<<grid, 64, 0, s>>>(a);
  else if (a.dh == 64) window_bwd_q_simt_kernel<float, 64><<<grid, 64, 0, s>>>(a);
  else window_bwd_q_simt_kernel<float, 32><<<grid, 64, 0, s>>>(a);
  if ((e = launch_end(nq, s)) != cudaSuccess) return e;
  launch_begin(nkv, s);
  if (a.bf16) window_bwd_kv_simt_kernel<bf16, 32><<<gridk, 64, 0, s>>>(a);
  else if (a.dh == 64) window_bwd_kv_simt_kernel<float, 64><<<gridk, 64, 0, s>>>(a);
  else window_bwd_kv_simt_kernel<float, 32><<<gridk, 64, 0, s>>>(a);
  return launch_end(nkv, s);
}

}  // namespace gca
