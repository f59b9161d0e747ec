// GCA backward on the 5th-generation tensor cores (bf16, dh = 64).
//
// The same two passes as the mma.sync kernels (query side: P, D = rowsum(P * dO V^T),
// dQ and per-head dw; key side: dK and dV over the consumers of each chunk), here
// warp-specialised like the forward: warp 8 is the control warp (lane 0 issues the TMA
// tile loads into a ring of stages; the whole warp waits on the mbarriers and issues
// tcgen05.mma through an elected lane, accumulators in TMEM); warps 0-7 read the
// products with tcgen05.ld, do the element-wise part in registers and store the bf16
// operand of the next product (dS, or w P^T and dS^T) into TMEM over the columns they
// have read, where the next MMA takes it as its A operand.  One 64 x 64 tile in shared
// memory serves as a K-major operand in one product and as an MN-major operand in
// another (K as the B of S = Q K^T and of dQ = dS K; Q and dO as the B of S^T and dPo^T
// and of dK, dV).
//
// Per slot (consumer) the control warp issues the products that read the element warps'
// operand, then the next S / dPo pair into the same columns: the tensor pipe runs one
// CTA's MMAs in issue order, so the overwrite follows the read, and the completion of
// the next pair (the element warps' mbarrier) implies that of the products before it.
//
// Source of the method: Paper-Notes page on "Efficient Length-Generalizable Attention via
// Causal Retrieval for Long-Context Language Modeling", 关键设计 / key design, item
// "Grouped Cross-Attention" (the retrieval scores are trained through the fusion weights).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gca {
namespace {

using bf16 = __nv_bfloat16;
constexpr float kLog2e = 1.4426950408889634f;
// Eight element-wise warps (warp w reads TMEM lane quarter w % 4, i.e. 16 rows, and
// column half w / 4) and one control warp.
constexpr int kEW = 8;
constexpr int kThreads = 32 * (kEW + 1);
constexpr int kCtl = kEW;  // control warp index
constexpr int TILE = 8192, ROWB = 128, UPR = 8, DH = 64;
enum { kBarOpReady = 2, kBarEW = 3 };

// ================================================================== query side
// Persistent: each CTA walks the tiles (query chunk, head, sequence) blockIdx.x,
// blockIdx.x + gridDim.x, ... (head-major, so the CTAs in flight share K/V in L2), with
// three warp roles:
//   * warp 9 (producer): reads each tile's retrieval row (slots and fusion weights) into
//     a ring of metadata records one tile ahead of its loads; lane 0 streams Q, dO and the
//     tile's LSE rows (double-buffered) and the K / V tiles of its slots through a ring of
//     stages that runs on across tile boundaries, so the next tile's loads overlap the
//     current tile;
//   * warp 8 (MMA): issues S = Q K^T and dPo = dO V^T one slot ahead of the element warps
//     (also across tile boundaries) and dQ += dS K once dS is in TMEM;
//   * warps 0-7 (element): P = exp(S - LSE), D = rowsum(P * dPo) (stored; the retrieval
//     score gradient sums it later), dS = w P (dPo - D) / sqrt(dh) into TMEM, and at the
//     end of a tile dQ from TMEM to global memory.
// TMEM (256 columns): S 0-63, dPo 64-127, dQ 128-191, two dS buffers (bf16 pairs, the A
// operand of dQ += dS K) 192-223 and 224-255.
//
// Every hand-over is an mbarrier with a bounded wait.  A wait that runs out records its
// site and raises a CTA-wide abort flag; every role then stops issuing work (the MMA
// warp drains its products, the producer its copies) and the CTA exits, so a protocol
// fault can neither hang the kernel nor let a role run on stale metadata.
constexpr int kQStages = 3;
constexpr int kQThreads = kThreads + 32;  // + producer warp
constexpr int kProd = kEW + 1;
constexpr int kQBuf = 2 * TILE + kMaxTopk * 64 * 4;  // Q, dO, LSE rows of every slot
constexpr int kQSmem = 2 * kQBuf + TILE * (2 * kQStages + 1) + 1024;  // 2 x (Q, dO, LSE), ring of (K, V), dQ staging
static_assert(kQBuf % 1024 == 0, "Q / dO tiles must stay 1024-byte aligned");
constexpr uint32_t kWaitLimit = 1u << 21;
// Metadata records in flight: the producer fills tile k+1's record while tile k's loads
// are issued, and that must not wait for a record still in use (tile k-1's is released
// only when its dQ is out, which needs tile k's first loads).
constexpr int kMetaBufs = 4;

struct QTileMeta {
  int ns;
  int slot[kMaxTopk];
  int j[kMaxTopk];
  float w[kMaxTopk];
};

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Bounded wait for phase `parity` of `bar` that gives up early once the CTA's abort flag
// is raised; on running out it records `site` (with CTA, tile, slot) and raises the flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag, ErrWord* err,
                                              int site, int tile, int slot) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (tc::mbar_try(bar, parity)) return true;
    if ((it & 15) == 15 && *reinterpret_cast<volatile int*>(abort_flag)) return false;
  }
  flag_timeout(err, site, blockIdx.x, tile, slot);
  atomicExch(abort_flag, 1);
  return false;
}

__global__ void __launch_bounds__(kQThreads, 2)
gca_bwd_q_tc_kernel(BwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  constexpr int NST = kQStages;
  constexpr uint32_t kIdKm = tc::idesc_bf16(64, 64, false);  // B K-major
  constexpr uint32_t kIdMn = tc::idesc_bf16(64, 64, true);   // B MN-major
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* qbuf = sm;                 // buffer x at qbuf + x kQBuf: Q, dO, LSE
  unsigned char* ring = sm + 2 * kQBuf;     // stage st: K at ring + 2 st TILE, V after it
  unsigned char* dqst = ring + 2 * NST * TILE;
  __shared__ QTileMeta meta[kMetaBufs];
  __shared__ float Dx[2][2][64];  // [slot parity][column half][row]: partial row sums of D
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  // Phases: meta_* and bar_q / qfree per use of a buffer; bar_kv / ring_empty per use of
  // a stage; bar_s per slot; sfree / opready alternate by slot parity (each waited once per
  // two slots, so no waiter can be lapped); ewb per element-warp exchange; dq_full per tile.
  __shared__ __align__(8) uint64_t meta_full[kMetaBufs], meta_empty[kMetaBufs], bar_q[2], qfree[2], bar_kv[NST],
      ring_empty[NST], bar_s, sfree[2], opready[2], ewb, dq_full, drain;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int ntiles = a.nQ * a.H * a.B;

  if (warp == kProd && lane == 0) {
    for (int x = 0; x < kMetaBufs; ++x) {
      tc::mbar_init(&meta_full[x], 1);
      tc::mbar_init(&meta_empty[x], kEW + 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&bar_q[x], 1);
      tc::mbar_init(&qfree[x], 1);
      tc::mbar_init(&sfree[x], kEW);
      tc::mbar_init(&opready[x], kEW);
    }
    for (int st = 0; st < NST; ++st) {
      tc::mbar_init(&bar_kv[st], 1);
      tc::mbar_init(&ring_empty[st], 1);
    }
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&ewb, kEW);
    tc::mbar_init(&dq_full, 1);
    tc::mbar_init(&drain, 1);
    tc::fence_mbar_init();
    abort_s = 0;
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmdO);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, 256);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tS = tmem_slot, tP = tmem_slot + 64, tQ = tmem_slot + 128, tdS = tmem_slot + 192;
  auto W = [&](uint64_t* bar, uint32_t parity, int site, int tile, int slot) {
    return wait_or_abort(bar, parity, &abort_s, a.err, site, tile, slot);
  };

  if (warp == kProd) {
    // ------------------------------------------------------------ producer warp
    int gs = 0, nq[2] = {0, 0}, nkv[NST];
#pragma unroll
    for (int st = 0; st < NST; ++st) nkv[st] = 0;
    // Metadata of tile k (whole warp): slots and fusion weights of its retrieval row.
    auto prepare_meta = [&](int k, int t) -> bool {
      const int mb = k % kMetaBufs;
      if (k >= kMetaBufs && !W(&meta_empty[mb], ((k / kMetaBufs) - 1) & 1, 1, k, -1)) return false;
      const int c = t % a.nQ, b = t / (a.nQ * a.H);
      const int r = c - a.shift;
      QTileMeta& M = meta[mb];
      if (r >= 0) {
        row_weights_warp(a.idx + ((int64_t)b * a.nQ + r) * a.topk, a.scores + ((int64_t)b * a.nQ + r) * a.topk,
                         a.topk, a.nC, M.w, M.j, a.err);
      } else if (lane < a.topk) {
        M.w[lane] = 0.f;
        M.j[lane] = -1;
      }
      __syncwarp();
      // The key side takes every consumer's fusion weight from this table (one head writes it).
      if (r >= 0 && (t / a.nQ) % a.H == 0 && lane < a.topk) a.wrow[((int64_t)b * a.nQ + r) * a.topk + lane] = M.w[lane];
      if (lane == 0) {
        int n = 0;
        for (int m = 0; m < a.topk; ++m)
          if (M.j[m] >= 0) M.slot[n++] = m;
        M.ns = n;
        tc::mbar_arrive(&meta_full[mb]);
      }
      __syncwarp();
      return true;
    };
    bool alive = prepare_meta(0, blockIdx.x);
    for (int k = 0, t = blockIdx.x; alive && t < ntiles; ++k, t += gridDim.x) {
      const int buf = k & 1;
      const int c = t % a.nQ, h = (t / a.nQ) % a.H, b = t / (a.nQ * a.H);
      if (lane == 0) {  // Q, dO and the LSE rows of tile k
        if (k >= 2 && !W(&qfree[buf], ((k - 2) >> 1) & 1, 2, k, -1)) {
          alive = false;
        } else {
          unsigned char* Qs = qbuf + buf * kQBuf;
          const uint32_t lse_bytes = (uint32_t)a.topk * 64 * 4;
          tc::mbar_expect_tx(&bar_q[buf], 2 * TILE + lse_bytes);
          tc::tma_load_4d(Qs, &tmQ, 0, h, c * 64, b, &bar_q[buf]);
          tc::tma_load_4d(Qs + TILE, &tmdO, 0, h, c * 64, b, &bar_q[buf]);
          tc::bulk_load(Qs + 2 * TILE, a.lse + (((int64_t)b * a.nQ + c) * a.H + h) * a.topk * 64, lse_bytes,
                        &bar_q[buf]);
          ++nq[buf];
        }
      }
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
      if (!alive) break;
      // The next tile's metadata, a tile ahead of its loads.
      if (t + (int)gridDim.x < ntiles && !prepare_meta(k + 1, t + gridDim.x)) break;
      if (lane == 0) {  // K / V tiles of tile k's slots
        const QTileMeta& M = meta[k % kMetaBufs];
        const int n = M.ns;
        for (int x = 0; x < n; ++x, ++gs) {
          const int st = gs % NST;
          if (gs >= NST && !W(&ring_empty[st], ((gs / NST) - 1) & 1, 3, k, gs)) {
            alive = false;
            break;
          }
          const int j = M.j[M.slot[x]];
          unsigned char* Ks = ring + 2 * st * TILE;
          tc::mbar_expect_tx(&bar_kv[st], 2 * TILE);
          tc::tma_load_4d(Ks, &tmK, 0, h, j * 64, b, &bar_kv[st]);
          tc::tma_load_4d(Ks + TILE, &tmV, 0, h, j * 64, b, &bar_kv[st]);
          ++nkv[st];
        }
      }
      gs = __shfl_sync(0xffffffffu, gs, 0);
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
    }
    // After an abort, let the copies already issued land before the CTA exits.
    if (lane == 0 && *reinterpret_cast<volatile int*>(&abort_s)) {
      for (int x = 0; x < 2; ++x)
        if (nq[x] > 0) tc::mbar_wait(&bar_q[x], (nq[x] - 1) & 1);
      for (int st = 0; st < NST; ++st)
        if (nkv[st] > 0) tc::mbar_wait(&bar_kv[st], (nkv[st] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == kCtl) {
    // ------------------------------------------------------------ MMA warp
    const uint64_t dQ0 = tc::desc_km(tc::su32(qbuf));  // + buffer offset
    const uint64_t dRingKm = tc::desc_km(tc::su32(ring)), dRingMn = tc::desc_mn(tc::su32(ring));
    constexpr uint64_t kStage = (2 * TILE) >> 4, kTileStep = TILE >> 4;
    bool issued = false;
    // Take tile (k, t): wait for its metadata and its Q / dO tiles, release the metadata
    // record (only ns is needed here) and, if it has no slots, its Q / dO buffer too.
    // Returns its slot count, -1 past the last tile, -2 on abort.
    auto take_tile = [&](int k, int t) -> int {
      if (t >= ntiles) return -1;
      const int buf = k & 1, mb = k % kMetaBufs;
      if (!W(&meta_full[mb], (k / kMetaBufs) & 1, 4, k, -1)) return -2;
      const int ns = meta[mb].ns;
      if (!W(&bar_q[buf], (k >> 1) & 1, 5, k, -1)) return -2;
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&meta_empty[mb]);
        if (ns == 0) tc::mbar_arrive(&qfree[buf]);
      }
      return ns;
    };
    auto issue_s = [&](int g, int buf, int k) -> bool {  // S, dPo of global slot g (whole warp)
      const uint64_t dq = dQ0 + buf * (kQBuf >> 4), ddo = dq + kTileStep;
      const uint64_t dk = dRingKm + (g % NST) * kStage, dv = dk + kTileStep;
      if (!W(&bar_kv[g % NST], (g / NST) & 1, 6, k, g)) return false;
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
        tc::mma_warp(tS, dq + ks * tc::kKStepKm, dk + ks * tc::kKStepKm, kIdKm, ks > 0 ? 1u : 0u);
        tc::mma_warp(tP, ddo + ks * tc::kKStepKm, dv + ks * tc::kKStepKm, kIdKm, ks > 0 ? 1u : 0u);
      }
      tc::commit_warp(&bar_s);
      issued = true;
      return true;
    };
    // Before the first tile nothing is in flight, so empty tiles can be skipped freely.
    int k = 0, t = blockIdx.x, si = 0, g = 0;
    int ns = take_tile(k, t);
    while (ns == 0) ns = take_tile(++k, t += gridDim.x);
    if (ns > 0 && !issue_s(0, k & 1, k)) ns = -2;
    while (ns > 0) {
      // S(g), dPo(g) are in the element warps' registers: the next pair may overwrite them.
      if (!W(&sfree[g & 1], (g >> 1) & 1, 10, k, g)) break;
      int nk = k, nt = t, nns = ns, nsi = si + 1;
      if (nsi == ns) {
        // Look one tile ahead only: the tile after an empty one cannot be prepared before
        // this tile's metadata is released, which waits for this tile's dQ.
        nk = k + 1;
        nt = t + gridDim.x;
        nsi = 0;
        nns = take_tile(nk, nt);
      }
      if (nns > 0 && !issue_s(g + 1, nk & 1, nk)) break;
      if (nns == -2) break;
      if (!W(&opready[g & 1], (g >> 1) & 1, 11, k, g)) break;  // dS(g) is in buffer g & 1
      tc::fence_after();
      const uint64_t dk = dRingMn + (g % NST) * kStage;
      const uint32_t ta = tdS + 32 * (g & 1);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // dQ += dS K  (K as the MN-major B operand)
        tc::mma_ts_warp(tQ, ta + 8 * kk, dk + kk * tc::kKStepMn, kIdMn, (si > 0 || kk > 0) ? 1u : 0u);
      tc::commit_warp(&ring_empty[g % NST]);
      if (si == ns - 1) {
        tc::commit_warp(&qfree[k & 1]);
        tc::commit_warp(&dq_full);
      }
      if (nns == 0) {  // the next tile was empty: with this tile finished, skip ahead
        while (nns == 0) nns = take_tile(++nk, nt += gridDim.x);
        if (nns > 0 && !issue_s(g + 1, nk & 1, nk)) break;
      }
      k = nk;
      t = nt;
      ns = nns;
      si = nsi;
      ++g;
    }
    // No product may still be running when TMEM is released (after an abort in particular).
    if (issued) {
      tc::commit_warp(&drain);
      if (!tc::mbar_wait(&drain, 0) && lane == 0) flag_timeout(a.err, 13, blockIdx.x, k, g);
    }
  } else {
    // ------------------------------------------------------------ element-wise warps
    const int g = lane >> 2, cq = lane & 3, quarter = warp & 3, hc = warp >> 2;
    const int row0 = 16 * quarter + g;
    const int etid = tid;  // 0..255
    const uint32_t lane_q = (uint32_t)(32 * quarter) << 16;
    const uint32_t lane_base = lane_q + 32 * hc;
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * kLog2e;
    int gs = 0, kq = 0, ewc = 0;
    bool alive = true;
    for (int k = 0, t = blockIdx.x; alive && t < ntiles; ++k, t += gridDim.x) {
      const int buf = k & 1;
      const int c = t % a.nQ, h = (t / a.nQ) % a.H, b = t / (a.nQ * a.H);
      const int64_t tok0 = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
      bf16* dqg = reinterpret_cast<bf16*>(a.dq) + tok0;
      const int64_t rowbase = ((int64_t)b * a.nQ + c) * a.H + h;
      float* Dg = a.Dbuf + rowbase * a.topk * 64;
      const int mb = k % kMetaBufs;
      if (!W(&meta_full[mb], (k / kMetaBufs) & 1, 7, k, -1)) break;
      const QTileMeta& M = meta[mb];
      const int ns = M.ns;
      if (ns == 0) {  // nothing retrieved: dQ is zero
        for (int u = etid; u < 64 * UPR; u += 32 * kEW) {
          const int row = u / UPR, w = u % UPR;
          *reinterpret_cast<uint4*>(dqg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&meta_empty[mb]);
        continue;
      }
      // The tile's LSE rows came with its Q and dO (observe that phase; the MMA warp has
      // waited for it before issuing the tile's first product).
      if (!W(&bar_q[buf], (k >> 1) & 1, 14, k, -1)) break;
      const float* lse_s = reinterpret_cast<const float*>(qbuf + buf * kQBuf + 2 * TILE);
      for (int si = 0; si < ns; ++si, ++gs) {
        const int m = M.slot[si];
        const float lse0 = lse_s[m * 64 + row0] * kLog2e, lse1 = lse_s[m * 64 + row0 + 8] * kLog2e;
        // S(gs) complete; it was issued after dQ(gs - 2), so dS buffer gs & 1 is free too.
        if (!W(&bar_s, gs & 1, 8, k, gs)) {
          alive = false;
          break;
        }
        float s[4][4], dp[4][4];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tS + lane_base + cb * 8, s[cb]);
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tP + lane_base + cb * 8, dp[cb]);
        tc::ld_wait(s);
        tc::ld_wait(dp);
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sfree[gs & 1]);
        float D0 = 0.f, D1 = 0.f;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          s[n][0] = tc::ex2(fmaf(s[n][0], sl2, -lse0));
          s[n][1] = tc::ex2(fmaf(s[n][1], sl2, -lse0));
          s[n][2] = tc::ex2(fmaf(s[n][2], sl2, -lse1));
          s[n][3] = tc::ex2(fmaf(s[n][3], sl2, -lse1));
          D0 = fmaf(s[n][0], dp[n][0], fmaf(s[n][1], dp[n][1], D0));
          D1 = fmaf(s[n][2], dp[n][2], fmaf(s[n][3], dp[n][3], D1));
        }
#pragma unroll
        for (int kx = 1; kx <= 2; kx <<= 1) {
          D0 += __shfl_xor_sync(0xffffffffu, D0, kx);
          D1 += __shfl_xor_sync(0xffffffffu, D1, kx);
        }
        // Combine the two column halves in a fixed order (deterministic).
        if (cq == 0) {
          Dx[gs & 1][hc][row0] = D0;
          Dx[gs & 1][hc][row0 + 8] = D1;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&ewb);
        if (!W(&ewb, ewc & 1, 12, k, gs)) {
          alive = false;
          break;
        }
        ++ewc;
        D0 = Dx[gs & 1][0][row0] + Dx[gs & 1][1][row0];
        D1 = Dx[gs & 1][0][row0 + 8] + Dx[gs & 1][1][row0 + 8];
        const float cs = M.w[m] * scale;
        // dS as the TMEM A operand of dQ += dS K: keys (32hc + 8n + 2cq, +1) of rows g and
        // g + 8 go to column 16hc + 4n + cq of buffer gs & 1.
        uint32_t dv[8];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          dv[2 * n] = pack_bf16(s[n][0] * (dp[n][0] - D0) * cs, s[n][1] * (dp[n][1] - D0) * cs);
          dv[2 * n + 1] = pack_bf16(s[n][2] * (dp[n][2] - D1) * cs, s[n][3] * (dp[n][3] - D1) * cs);
        }
        tc::st16x128_x4(tdS + 32 * (gs & 1) + lane_q + 16 * hc, dv);
        tc::st_wait();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&opready[gs & 1]);
        if (hc == 0 && cq == 0) {  // D rows (after the hand-over)
          Dg[m * 64 + row0] = D0;
          Dg[m * 64 + row0 + 8] = D1;
        }
      }
      if (!alive) break;
      // Tile epilogue: dQ from TMEM through the staging tile to global memory, and dw.
      if (!W(&dq_full, kq & 1, 9, k, gs)) break;
      ++kq;
      float o[4][4];
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tQ + lane_base + cb * 8, o[cb]);
      tc::ld_wait(o);
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        *reinterpret_cast<uint32_t*>(dqst + swz<ROWB>(row0, 4 * hc + n) + cq * 4) = pack_bf16(o[n][0], o[n][1]);
        *reinterpret_cast<uint32_t*>(dqst + swz<ROWB>(row0 + 8, 4 * hc + n) + cq * 4) = pack_bf16(o[n][2], o[n][3]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ewb);
      if (!W(&ewb, ewc & 1, 12, k, gs)) break;
      ++ewc;
      for (int u = etid; u < 64 * UPR; u += 32 * kEW) {
        const int row = u / UPR, w = u % UPR;
        *reinterpret_cast<uint4*>(dqg + row * ts + w * 8) = *reinterpret_cast<const uint4*>(dqst + swz<ROWB>(row, w));
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&meta_empty[mb]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem_slot, 256);
  }
}

// ================================================================== key side
constexpr int kKVStages = 4;
constexpr int kKVStageBytes = 2 * TILE + 1024;  // Q, dO tiles + LSE and D rows (1 KB keeps tiles aligned)
constexpr int kKVSmem = TILE * 2 + kKVStages * kKVStageBytes + 1024;  // K, V, ring
constexpr int kConsTab = 256;

__global__ void __launch_bounds__(kThreads, 2)
gca_bwd_kv_tc_kernel(BwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  constexpr int NST = kKVStages, NT = kThreads;
  constexpr uint32_t kIdKm = tc::idesc_bf16(64, 64, false);
  constexpr uint32_t kIdMn = tc::idesc_bf16(64, 64, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* Ks = sm;
  unsigned char* Vs = sm + TILE;
  unsigned char* ring = sm + 2 * TILE;  // stage st at ring + st * kKVStageBytes: Q, dO, lse[64], D[64]
  __shared__ float w_st[NST];
  __shared__ float wtab[kConsTab];  // weight of each consumer (first kConsTab consumers)
  __shared__ int etab[kConsTab];    // its (row, slot) entry
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar_k, bar_c[NST], bar_s, bar_o;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int64_t ktok0 = ((int64_t)b * a.nC * 64 + (int64_t)j * 64) * ts + h * DH;
  const int e0 = a.csr_off[(int64_t)b * (a.nC + 1) + j];
  const int e1 = a.csr_off[(int64_t)b * (a.nC + 1) + j + 1];
  const int32_t* ent = a.csr_ent + (int64_t)b * a.nQ * a.topk;
  const float* wrow = a.wrow + (int64_t)b * a.nQ * a.topk;
  bf16* dkg = reinterpret_cast<bf16*>(a.dk) + ktok0;
  bf16* dvg = reinterpret_cast<bf16*>(a.dv) + ktok0;
  const int ncons = e1 - e0;
  if (ncons == 0) {
    if (!a.acc_dkv) {
      for (int u = tid; u < 64 * UPR; u += NT) {
        const int row = u / UPR, w = u % UPR;
        *reinterpret_cast<uint4*>(dkg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(dvg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }
  if (warp == kCtl && lane == 0) {
    tc::mbar_init(&bar_k, 1);
    for (int st = 0; st < NST; ++st) tc::mbar_init(&bar_c[st], 1);
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_o, 1);
    tc::fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmdO);
    // K and V of this chunk first: they do not depend on the consumer table.
    tc::mbar_expect_tx(&bar_k, 2 * TILE);
    tc::tma_load_4d(Ks, &tmK, 0, h, j * 64, b, &bar_k);
    tc::tma_load_4d(Vs, &tmV, 0, h, j * 64, b, &bar_k);
  }
  if (warp == kCtl) {  // consumer table: entries and fusion weights (from the query side)
    for (int x = lane; x < ncons && x < kConsTab; x += 32) {
      const int e = ent[e0 + x];
      etab[x] = e;
      wtab[x] = wrow[e];
    }
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
      const int e = x < kConsTab ? etab[x] : ent[e0 + x];
      const int r = e / a.topk, m = e % a.topk;
      const int c = r + a.shift;
      w_st[st] = x < kConsTab ? wtab[x] : wrow[e];
      unsigned char* base = ring + st * kKVStageBytes;
      const int64_t rb = ((((int64_t)b * a.nQ + c) * a.H + h) * a.topk + m) * 64;
      tc::mbar_expect_tx(&bar_c[st], 2 * TILE + 512);
      tc::tma_load_4d(base, &tmQ, 0, h, c * 64, b, &bar_c[st]);
      tc::tma_load_4d(base + TILE, &tmdO, 0, h, c * 64, b, &bar_c[st]);
      tc::bulk_load(base + 2 * TILE, a.lse + rb, 256, &bar_c[st]);
      tc::bulk_load(base + 2 * TILE + 256, a.Dbuf + rb, 256, &bar_c[st]);
    };
    // Operand descriptors, built once (ring stages: base + stage offset).
    const uint64_t dKd = tc::desc_km(tc::su32(Ks)), dVd = tc::desc_km(tc::su32(Vs));
    const uint64_t dRingKm = tc::desc_km(tc::su32(ring)), dRingMn = tc::desc_mn(tc::su32(ring));
    constexpr uint64_t kStage = kKVStageBytes >> 4, kTileStep = TILE >> 4;
    auto issue_s = [&](int x) {  // S^T = K Q^T and dPo^T = V dO^T of consumer x (whole warp)
      const uint64_t dq = dRingKm + (x % NST) * kStage, ddo = dq + kTileStep;
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
        tc::mma_warp(tS, dKd + ks * tc::kKStepKm, dq + ks * tc::kKStepKm, kIdKm, ks > 0 ? 1u : 0u);
        tc::mma_warp(tP, dVd + ks * tc::kKStepKm, ddo + ks * tc::kKStepKm, kIdKm, ks > 0 ? 1u : 0u);
      }
      tc::commit_warp(&bar_s);
    };
    if (lane == 0)
      for (int x = 0; x < NST && x < ncons; ++x) load_cons(x);
    __syncwarp();
    ok = tc::mbar_wait(&bar_k, 0) && ok;
    ok = tc::mbar_wait(&bar_c[0], 0) && ok;
    issue_s(0);
    for (int ci = 0; ci < ncons; ++ci) {
      tc::named_sync(kBarOpReady, NT);  // w P^T and dS^T are in TMEM columns 0-31, 64-95
      tc::fence_after();
      const uint64_t bq = dRingMn + (ci % NST) * kStage, bdo = bq + kTileStep;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t acc = (ci > 0 || kk > 0) ? 1u : 0u;
        tc::mma_ts_warp(tdV, tS + 8 * kk, bdo + kk * tc::kKStepMn, kIdMn, acc);
        tc::mma_ts_warp(tdK, tP + 8 * kk, bq + kk * tc::kKStepMn, kIdMn, acc);
      }
      tc::commit_warp(&bar_o);
      if (ci + 1 < ncons) {
        ok = tc::mbar_wait(&bar_c[(ci + 1) % NST], ((ci + 1) / NST) & 1) && ok;
        issue_s(ci + 1);
      }
      ok = tc::mbar_wait(&bar_o, ci & 1) && ok;  // ring stage ci % NST is free
      if (lane == 0) {
        if (ci + NST < ncons) load_cons(ci + NST);
        if (!ok) flag_timeout(a.err);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ element-wise warps
    const int cq = lane & 3, quarter = warp & 3, hc = warp >> 2;
    const uint32_t lane_q = (uint32_t)(32 * quarter) << 16;
    const uint32_t lane_base = lane_q + 32 * hc;
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * kLog2e;
    for (int ci = 0; ci < ncons; ++ci) {
      if (!tc::mbar_wait(&bar_s, ci & 1)) flag_timeout(a.err);  // acquire S^T(ci), dPo^T(ci)
      const int st = ci % NST;
      // The rows came in by bulk copy: observe their mbarrier phase (already complete).
      tc::mbar_wait(&bar_c[st], (ci / NST) & 1);
      const float* lrow = reinterpret_cast<const float*>(ring + st * kKVStageBytes + 2 * TILE) + 32 * hc;
      const float* drow = lrow + 64;
      const float w = w_st[st];
      float s[4][4], dp[4][4];
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tS + lane_base + cb * 8, s[cb]);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tc::ld16x256(tP + lane_base + cb * 8, dp[cb]);
      tc::ld_wait(s);
      tc::ld_wait(dp);
      const float cs = w * scale;
#pragma unroll
      for (int n = 0; n < 4; ++n) {  // columns are queries 32hc + 8n + 2cq (+1)
        const float2 l2 = *reinterpret_cast<const float2*>(lrow + 8 * n + 2 * cq);
        const float2 d2 = *reinterpret_cast<const float2*>(drow + 8 * n + 2 * cq);
        const float la = l2.x * kLog2e, lb = l2.y * kLog2e;
        const float p0 = tc::ex2(fmaf(s[n][0], sl2, -la)), p1 = tc::ex2(fmaf(s[n][1], sl2, -lb));
        const float p2 = tc::ex2(fmaf(s[n][2], sl2, -la)), p3 = tc::ex2(fmaf(s[n][3], sl2, -lb));
        dp[n][0] = p0 * (dp[n][0] - d2.x) * cs;
        dp[n][1] = p1 * (dp[n][1] - d2.y) * cs;
        dp[n][2] = p2 * (dp[n][2] - d2.x) * cs;
        dp[n][3] = p3 * (dp[n][3] - d2.y) * cs;
        s[n][0] = p0 * w;
        s[n][1] = p1 * w;
        s[n][2] = p2 * w;
        s[n][3] = p3 * w;
      }
      // w P^T and dS^T as TMEM A operands (keys are rows): queries (32hc + 8n + 2cq, +1)
      // of key rows g and g + 8 go to column 16hc + 4n + cq of S^T's and dPo^T's columns.
      // Both column halves must have read S^T and dPo^T before either half stores.
      uint32_t pv[8], dv[8];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        pv[2 * n] = pack_bf16(s[n][0], s[n][1]);
        pv[2 * n + 1] = pack_bf16(s[n][2], s[n][3]);
        dv[2 * n] = pack_bf16(dp[n][0], dp[n][1]);
        dv[2 * n + 1] = pack_bf16(dp[n][2], dp[n][3]);
      }
      tc::named_sync(kBarEW, 32 * kEW);
      tc::st16x128_x4(tS + lane_q + 16 * hc, pv);
      tc::st16x128_x4(tP + lane_q + 16 * hc, dv);
      tc::st_wait();
      tc::fence_before();
      tc::named_arrive(kBarOpReady, NT);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // Epilogue: dK from TMEM columns 192-255 into the K tile, dV (128-191) into the V tile
  // (fp32 values staged as bf16 in the same swizzled layout), then 16-byte rows.
  if (warp < kEW) {
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
    if (a.acc_dkv) {
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

}  // namespace

// Launch the tensor-core query-side and key-side kernels (bf16, dh = 64).
cudaError_t launch_bwd_q_tc(const BwdArgs& a, cudaStream_t s) {
  CUtensorMap tq, tdo, tk, tv;
  const int64_t qb = (int64_t)a.nQ * 64 * a.H * 64, kb = (int64_t)a.nC * 64 * a.H * 64;
  cudaError_t e = make_head_tmap(&tq, a.q, 64, a.H, (int64_t)a.nQ * 64, a.B, qb);
  if (e == cudaSuccess) e = make_head_tmap(&tdo, a.dout, 64, a.H, (int64_t)a.nQ * 64, a.B, qb);
  if (e == cudaSuccess) e = make_head_tmap(&tk, a.k, 64, a.H, (int64_t)a.nC * 64, a.B, kb);
  if (e == cudaSuccess) e = make_head_tmap(&tv, a.v, 64, a.H, (int64_t)a.nC * 64, a.B, kb);
  if (e == cudaSuccess) e = allow_smem((const void*)gca_bwd_q_tc_kernel, kQSmem);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long ntiles = (long long)a.nQ * a.H * a.B;
  const int grid = (int)std::min<long long>(ntiles, 2LL * sms);  // two CTAs per SM (TMEM: 256 columns each)
  launch_begin("gca_bwd_q", s);
  gca_bwd_q_tc_kernel<<<grid, kQThreads, kQSmem, s>>>(a, tq, tdo, tk, tv);
  return launch_end("gca_bwd_q", s);
}

cudaError_t launch_bwd_kv_tc(const BwdArgs& a, cudaStream_t s) {
  CUtensorMap tq, tdo, tk, tv;
  const int64_t qb = (int64_t)a.nQ * 64 * a.H * 64, kb = (int64_t)a.nC * 64 * a.H * 64;
  cudaError_t e = make_head_tmap(&tq, a.q, 64, a.H, (int64_t)a.nQ * 64, a.B, qb);
  if (e == cudaSuccess) e = make_head_tmap(&tdo, a.dout, 64, a.H, (int64_t)a.nQ * 64, a.B, qb);
  if (e == cudaSuccess) e = make_head_tmap(&tk, a.k, 64, a.H, (int64_t)a.nC * 64, a.B, kb);
  if (e == cudaSuccess) e = make_head_tmap(&tv, a.v, 64, a.H, (int64_t)a.nC * 64, a.B, kb);
  if (e == cudaSuccess) e = allow_smem((const void*)gca_bwd_kv_tc_kernel, kKVSmem);
  if (e != cudaSuccess) return e;
  launch_begin("gca_bwd_kv", s);
  gca_bwd_kv_tc_kernel<<<dim3(a.nC, a.H, a.B), kThreads, kKVSmem, s>>>(a, tq, tdo, tk, tv);
  return launch_end("gca_bwd_kv", s);
}

}  // namespace gca
