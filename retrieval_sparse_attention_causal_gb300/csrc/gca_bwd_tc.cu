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
#include "waits.cuh"

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
// blockIdx.x + gridDim.x, ... (head-major, so the CTAs in flight share K/V in L2; the
// light first chunks of every sequence-head last, query_tile), with three warp roles:
//   * warp 9 (producer): reads each tile's retrieval row (slots and fusion weights) into
//     a ring of metadata records one tile ahead of its loads; lane 0 streams Q, dO and the
//     tile's LSE rows (double-buffered) and the K / V tiles of its slots through a ring of
//     stages that runs on across tile boundaries, so the next tile's loads overlap the
//     current tile;
//   * warp 8 (MMA): issues S = Q K^T and dPo = dO V^T one slot ahead of the element warps
//     (also across tile boundaries) and dQ += dS K once dS is in TMEM;
//   * warps 0-7 (element): w P = exp(S - LSE + log w) (the weight in the exponent),
//     D = rowsum(w P * dPo) / w (stored; the retrieval score gradient sums it later),
//     w P (dPo - D) into TMEM, and at the end of a tile dQ from TMEM to global memory,
//     where it takes the 1/sqrt(dh) of the logits once.
// TMEM (256 columns): S 0-63, dPo 64-127, dQ 128-191, two dS buffers (bf16 pairs, the A
// operand of dQ += dS K) 192-223 and 224-255.
//
// Every hand-over is an mbarrier with a bounded wait.  A wait that runs out records its
// site and raises a CTA-wide abort flag; every role then stops issuing work (the MMA
// warp drains its products, the producer its copies) and the CTA exits, so a protocol
// fault can neither hang the kernel nor let a role run on stale metadata.
constexpr int kQStages = 4;
constexpr int kQThreads = kThreads + 32;  // + producer warp
constexpr int kProd = kEW + 1;
constexpr int kQBuf = 2 * TILE + kMaxTopk * 64 * 4;  // Q, dO, LSE rows of every slot
constexpr int kQSmem = 2 * kQBuf + TILE * 2 * kQStages + 1024;  // 2 x (Q, dO, LSE), ring of (K, V)
static_assert(kQBuf % 1024 == 0, "Q / dO tiles must stay 1024-byte aligned");
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
  __shared__ QTileMeta meta[kMetaBufs];
  __shared__ float Dx[2][2][64];  // [slot parity][column half][row]: partial row sums of D
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  // Phases: meta_* and bar_q / qfree per use of a buffer; bar_kv / ring_empty per use of
  // a stage; bar_s per slot; sfree / opready alternate by slot parity (each waited once per
  // two slots, so no waiter can be lapped); ewb[q] per exchange between the two element
  // warps of row quarter q; dq_full per tile.
  __shared__ __align__(8) uint64_t meta_full[kMetaBufs], meta_empty[kMetaBufs], bar_q[2], qfree[2], bar_kv[NST],
      ring_empty[NST], bar_s, sfree[2], opready[2], ewb[4], dq_full, drain;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int ntiles = a.nQ * a.H * a.B;
  const int qL = min(a.nQ, a.shift + a.topk);  // light chunks per sequence-head (query_tile)

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
    for (int x = 0; x < 4; ++x) tc::mbar_init(&ewb[x], 2);
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
  // Waits park (try_wait with a suspend hint), so that a waiting warp takes no issue slots
  // from the warps that work; only the short exchange between the two element warps of a
  // row quarter spins (W).
  auto P = [&](uint64_t* bar, uint32_t parity, int site, int tile, int slot) {
    return park_or_abort(bar, parity, &abort_s, a.err, site, tile, slot);
  };
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
      if (k >= kMetaBufs && !P(&meta_empty[mb], ((k / kMetaBufs) - 1) & 1, 1, k, -1)) return false;
      int c, h, b;
      query_tile(a.nQ, a.H, a.B, qL, t, c, h, b);
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
      if (r >= 0 && h == 0 && lane < a.topk) a.wrow[((int64_t)b * a.nQ + r) * a.topk + lane] = M.w[lane];
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
      int c, h, b;
      query_tile(a.nQ, a.H, a.B, qL, t, c, h, b);
      if (lane == 0) {  // Q, dO and the LSE rows of tile k
        if (k >= 2 && !P(&qfree[buf], ((k - 2) >> 1) & 1, 2, k, -1)) {
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
          if (gs >= NST && !P(&ring_empty[st], ((gs / NST) - 1) & 1, 3, k, gs)) {
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
      if (!P(&meta_full[mb], (k / kMetaBufs) & 1, 4, k, -1)) return -2;
      const int ns = meta[mb].ns;
      if (!P(&bar_q[buf], (k >> 1) & 1, 5, k, -1)) return -2;
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
      if (!P(&bar_kv[g % NST], (g / NST) & 1, 6, k, g)) return false;
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tS, dq, dk, kIdKm, 0u);
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tP, ddo, dv, kIdKm, 0u);
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
      if (!P(&sfree[g & 1], (g >> 1) & 1, 10, k, g)) break;
      int nk = k, nt = t, nns = ns, nsi = si + 1;
      const bool last = nsi == ns;
      // Inside a tile the next slot's S, dPo go first, to overlap this slot's dS.  After a
      // tile's last slot its dQ goes first: the next tile's first K / V tiles may still be
      // on their way, and the tile's write-out should not wait for them.
      if (!last && !issue_s(g + 1, k & 1, k)) break;
      if (!P(&opready[g & 1], (g >> 1) & 1, 11, k, g)) break;  // dS(g) is in buffer g & 1
      tc::fence_after();
      const uint64_t dk = dRingMn + (g % NST) * kStage;
      const uint32_t ta = tdS + 32 * (g & 1);
      // dQ += dS K  (K as the MN-major B operand)
      tc::mma4_ts<8, 16, 24, tc::kKStepMn>(tQ, ta, dk, kIdMn, si > 0 ? 1u : 0u);
      tc::commit_warp(&ring_empty[g % NST]);
      if (last) {
        tc::commit_warp(&qfree[k & 1]);
        tc::commit_warp(&dq_full);
        // The next tile with slots (the one after is prepared only once this tile's
        // metadata is released, which the take releases).
        nk = k + 1;
        nt = t + gridDim.x;
        nsi = 0;
        nns = take_tile(nk, nt);
        while (nns == 0) nns = take_tile(++nk, nt += gridDim.x);
        if (nns == -2) break;
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
      int c, h, b;
      query_tile(a.nQ, a.H, a.B, qL, t, c, h, b);
      const int64_t tok0 = ((int64_t)b * a.nQ * 64 + (int64_t)c * 64) * ts + h * DH;
      bf16* dqg = reinterpret_cast<bf16*>(a.dq) + tok0;
      const int64_t rowbase = ((int64_t)b * a.nQ + c) * a.H + h;
      float* Dg = a.Dbuf + rowbase * a.topk * 64;
      const int mb = k % kMetaBufs;
      if (!P(&meta_full[mb], (k / kMetaBufs) & 1, 7, k, -1)) break;
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
      if (!P(&bar_q[buf], (k >> 1) & 1, 14, k, -1)) break;
      const float* lse_s = reinterpret_cast<const float*>(qbuf + buf * kQBuf + 2 * TILE);
      for (int si = 0; si < ns; ++si, ++gs) {
        const int m = M.slot[si];
        // w P = exp2(S sl2 - LSE log2 e + log2 w): the fusion weight rides in the exponent,
        // so D comes out as w D and dS as dS / sqrt(dh) (the 1/sqrt(dh) goes onto dQ once
        // per tile).
        const float wm = M.w[m], lw = __log2f(wm);
        const float lse0 = fmaf(-lse_s[m * 64 + row0], kLog2e, lw), lse1 = fmaf(-lse_s[m * 64 + row0 + 8], kLog2e, lw);
        // S(gs) complete; it was issued after dQ(gs - 2), so dS buffer gs & 1 is free too.
        if (!P(&bar_s, gs & 1, 8, k, gs)) {
          alive = false;
          break;
        }
        float s[4][4], dp[4][4];
        tc::ld16x256_x4(tS + lane_base, s);
        tc::ld16x256_x4(tP + lane_base, dp);
        tc::ld_wait(s);
        tc::ld_wait(dp);
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sfree[gs & 1]);
        const uint64_t sl2x2 = tc::f2(sl2, sl2), o0 = tc::f2(lse0, lse0), o1 = tc::f2(lse1, lse1);
        uint64_t D0x2 = tc::f2(0.f, 0.f), D1x2 = D0x2;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          float x0, x1, x2, x3;
          tc::uf2(tc::fma2(tc::f2(s[n][0], s[n][1]), sl2x2, o0), x0, x1);
          tc::uf2(tc::fma2(tc::f2(s[n][2], s[n][3]), sl2x2, o1), x2, x3);
          s[n][0] = tc::ex2(x0);
          s[n][1] = tc::ex2(x1);
          s[n][2] = tc::ex2(x2);
          s[n][3] = tc::ex2(x3);
          D0x2 = tc::fma2(tc::f2(s[n][0], s[n][1]), tc::f2(dp[n][0], dp[n][1]), D0x2);
          D1x2 = tc::fma2(tc::f2(s[n][2], s[n][3]), tc::f2(dp[n][2], dp[n][3]), D1x2);
        }
        float D0, D1;
        {
          float u0, u1;
          tc::uf2(D0x2, u0, u1);
          D0 = u0 + u1;
          tc::uf2(D1x2, u0, u1);
          D1 = u0 + u1;
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
        if (lane == 0) tc::mbar_arrive(&ewb[quarter]);
        if (!W(&ewb[quarter], ewc & 1, 12, k, gs)) {
          alive = false;
          break;
        }
        ++ewc;
        // D = (w D) / w.  A slot whose weight is 0 or subnormal (its 1/w would overflow) has
        // w P = 0 and dS = 0, and its D rows are weighted by that w wherever they are used,
        // so they are set to 0.
        const float rw = wm >= 1.17549435e-38f ? __frcp_rn(wm) : 0.f;
        D0 = (Dx[gs & 1][0][row0] + Dx[gs & 1][1][row0]) * rw;
        D1 = (Dx[gs & 1][0][row0 + 8] + Dx[gs & 1][1][row0 + 8]) * rw;
        // dS as the TMEM A operand of dQ += dS K: keys (32hc + 8n + 2cq, +1) of rows g and
        // g + 8 go to column 16hc + 4n + cq of buffer gs & 1.
        uint32_t dv[8];
        const uint64_t nD0 = tc::f2(-D0, -D0), nD1 = tc::f2(-D1, -D1);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          float a0, a1, b0, b1;
          tc::uf2(tc::mul2(tc::f2(s[n][0], s[n][1]), tc::add2(tc::f2(dp[n][0], dp[n][1]), nD0)), a0, a1);
          tc::uf2(tc::mul2(tc::f2(s[n][2], s[n][3]), tc::add2(tc::f2(dp[n][2], dp[n][3]), nD1)), b0, b1);
          dv[2 * n] = pack_bf16(a0, a1);
          dv[2 * n + 1] = pack_bf16(b0, b1);
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
      // Tile epilogue: dQ from TMEM straight to global memory (each warp its 16 rows and
      // 32 columns; no staging, so the K / V ring can hold one more stage).
      if (!P(&dq_full, kq & 1, 9, k, gs)) break;
      ++kq;
      float o[4][4];
      tc::ld16x256_x4(tQ + lane_base, o);
      tc::ld_wait(o);
      tc::fence_before();
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int col = 32 * hc + 8 * n + 2 * cq;
        *reinterpret_cast<uint32_t*>(dqg + (int64_t)row0 * ts + col) = pack_bf16(o[n][0] * scale, o[n][1] * scale);
        *reinterpret_cast<uint32_t*>(dqg + (int64_t)(row0 + 8) * ts + col) =
            pack_bf16(o[n][2] * scale, o[n][3] * scale);
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
// Persistent, two CTAs per SM.  The tiles (key chunk j, head h, sequence b) are claimed
// from a counter in the workspace (zeroed by the dscores kernel that runs before), in
// blocks of a few heads of one sequence whose Q, dO, K and V fit in L2 together (8 MB per
// head at L = 16K; a.kv_hb heads per block), chunk-major inside a block: the CTAs in
// flight share those operands in L2, and inside a block the chunks with the most
// consumers (the early ones) start first, so the last tiles of the kernel are light.  A
// tile's consumers are taken in CSR (entry) order, so every dK, dV sum runs in a fixed
// order: the result does not depend on which CTA claimed the tile.
//
// The pipe takes an M = 64 product only about as fast as it runs it, and one issuing warp
// with its own waits keeps it busy only part of the time; two CTAs per SM give it two
// issuers whose waits overlap each other's products.
//
// Roles (11 warps):
//   * warp 10 (metadata): claims tiles two at a time, writes the zero gradients of the
//     chunks nobody retrieved, and for the others loads the consumer table (query chunk,
//     slot and fusion weight of each consumer, all lanes at once) into a ring of metadata
//     records a few tiles ahead of the producer;
//   * warp 9 (producer, lane 0): streams the tiles: K and V of each tile into one of two
//     buffers, and per consumer Q, dO, its LSE row and its D row into a ring of stages,
//     with a record (fusion weight, tile, first / last flags, buffer indices);
//   * warp 8 (MMA): per consumer x, S^T = K Q^T and dPo^T = V dO^T into TMEM (each with
//     its own commit); dV += (w P^T) dO as soon as the element warps have stored w P^T,
//     dK += dS^T Q once dS^T is in, then the next consumer's S^T, dPo^T over the same
//     columns (the tensor pipe runs this warp's products in issue order).  The barriers of the next batch
//     are tested (test_wait, which does not block) and the records read before the
//     current batch is issued, and looked at after it;
//   * warps 0-7 (element): w P^T = exp(S^T - LSE + log w) (the weight in the exponent),
//     dS^T = w P^T (dPo^T - D) (the 1/sqrt(dh) goes onto dK once per tile);
//     each warp stores its bf16 operands over the TMEM columns it has itself read (no
//     cross-warp barrier).  After the consumer that follows a tile's last one they read
//     the tile's dK and dV (each warp its 16 rows and 32 columns), release the
//     accumulators and write the rows out as bf16 (adding to dK, dV when accumulating),
//     straight from registers.
// TMEM (256 columns): S^T 0-63, dPo^T 64-127, dV 128-191, dK 192-255.
//
// Every wait is bounded: one that runs out records (site, CTA, tile, consumer) and raises
// a CTA-wide abort flag; the roles stop, the MMA warp drains its products and the producer
// its copies, and the CTA exits.
constexpr int kKVStages = 4;
constexpr int kKVStageBytes = 2 * TILE + 1024;  // Q, dO; LSE row, D row, consumer record
constexpr int kKVMma = kEW;                      // 8
constexpr int kKVProd = kKVMma + 1;              // 9
constexpr int kKVMetaW = kKVProd + 1;            // 10
constexpr int kKVThreads = 32 * (kKVMetaW + 1);  // 352
constexpr int kKVMetaRecs = 4, kKVMetaCons = 64, kKVBatch = 2;
constexpr int kKVSmem = 2 * 2 * TILE + kKVStages * kKVStageBytes + 1024;  // K/V x 2, ring

enum { kRecFirst = 1, kRecLast = 2, kRecEnd = 4 };
struct KVConsRec {
  float w;
  int flags;
  int kb;  // K/V buffer of the consumer's tile
  int tc;  // ordinal of the tile among this CTA's tiles with consumers
  int j, h, b;
};
// A tile's consumer table: query chunk c and slot m packed as (c << 4) | m, and the fusion
// weight, for its first kKVMetaCons consumers (the producer reads any further ones from
// the CSR itself).
struct KVMeta {
  int j, h, b, ncons, e0, end;
  int cm[kKVMetaCons];
  float w[kKVMetaCons];
};

// Tile t of the key side: blocks of a.kv_hb heads of one sequence (the last block of a
// sequence may have fewer), chunk-major inside a block.
__device__ __forceinline__ void kv_tile(const BwdArgs& a, int t, int& j, int& h, int& b) {
  const int per_seq = a.H * a.nC;
  b = t / per_seq;
  const int rem = t - b * per_seq;
  const int hb0 = rem / (a.kv_hb * a.nC) * a.kv_hb;
  const int hbn = min(a.kv_hb, a.H - hb0);
  const int r2 = rem - hb0 * a.nC;
  j = r2 / hbn;
  h = hb0 + r2 % hbn;
}

__global__ void __launch_bounds__(kKVThreads, 2)
gca_bwd_kv_tc_kernel(BwdArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  constexpr int NST = kKVStages, MR = kKVMetaRecs, MC = kKVMetaCons, NB = kKVBatch;
  constexpr uint32_t kIdKm = tc::idesc_bf16(64, 64, false);
  constexpr uint32_t kIdMn = tc::idesc_bf16(64, 64, true);
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  unsigned char* kvbuf = sm;            // buffer kb: K at kvbuf + 2 kb TILE, V after it
  unsigned char* ring = sm + 4 * TILE;  // stage st: Q, dO, lse[64], D[64], record
  __shared__ KVMeta meta[MR];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  __shared__ __align__(8) uint64_t bar_c[NST], ring_empty[NST], bar_kv[2], kv_empty[2], bar_s1, bar_s2, op_v, op_k,
      acc_full, acc_empty, meta_full[MR], meta_empty[MR], drain;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ts = (int64_t)a.H * DH;
  const int ntiles = a.nC * a.H * a.B;
  auto crec = [&](int x) -> KVConsRec* {
    return reinterpret_cast<KVConsRec*>(ring + (x % NST) * kKVStageBytes + 2 * TILE + 512);
  };

  if (warp == kKVProd && lane == 0) {
    for (int st = 0; st < NST; ++st) {
      tc::mbar_init(&bar_c[st], 1);
      tc::mbar_init(&ring_empty[st], 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&bar_kv[x], 1);
      tc::mbar_init(&kv_empty[x], 1);
    }
    tc::mbar_init(&bar_s1, 1);
    tc::mbar_init(&bar_s2, 1);
    tc::mbar_init(&op_v, kEW);
    tc::mbar_init(&op_k, kEW);
    tc::mbar_init(&acc_full, 1);
    tc::mbar_init(&acc_empty, kEW);
    for (int x = 0; x < MR; ++x) {
      tc::mbar_init(&meta_full[x], 1);
      tc::mbar_init(&meta_empty[x], 1);
    }
    tc::mbar_init(&drain, 1);
    tc::fence_mbar_init();
    abort_s = 0;
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmdO);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 256);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = tmem_slot;
  // Every role parks while it waits (try_wait with a suspend hint), so that a waiting warp
  // takes no issue slots from the warps that work.
  auto W = [&](uint64_t* bar, uint32_t parity, int site, int tile, int slot) {
    return park_or_abort(bar, parity, &abort_s, a.err, site, tile, slot);
  };

  if (warp == kKVMetaW) {
    // ------------------------------------------------------------ metadata warp
    int k = 0;  // metadata records written
    bool alive = true;
    while (alive) {
      int t0 = 0;
      if (lane == 0) t0 = atomicAdd(a.kv_ctr, NB);
      t0 = __shfl_sync(0xffffffffu, t0, 0);
      if (t0 >= ntiles) break;
      // CSR bounds of the batch's tiles: lane l < NB reads the start of tile t0 + l, lane
      // NB + l its end.
      int v = 0;
      if (lane < 2 * NB && t0 + lane % NB < ntiles) {
        int jj, hh, bb;
        kv_tile(a, t0 + lane % NB, jj, hh, bb);
        v = a.csr_off[(int64_t)bb * (a.nC + 1) + jj + (lane >= NB ? 1 : 0)];
      }
      int e0s[NB], ns[NB], rk[NB];
#pragma unroll
      for (int l = 0; l < NB; ++l) {
        e0s[l] = __shfl_sync(0xffffffffu, v, l);
        const int e1 = __shfl_sync(0xffffffffu, v, NB + l);
        ns[l] = t0 + l < ntiles ? e1 - e0s[l] : 0;
      }
#pragma unroll
      for (int l = 0; l < NB; ++l) {
        rk[l] = -1;
        const int tt = t0 + l;
        if (tt >= ntiles) continue;
        int j, h, b;
        kv_tile(a, tt, j, h, b);
        if (ns[l] == 0) {  // nobody retrieved the chunk: zero gradients
          if (!a.acc_dkv) {
            const int64_t ktok0 = ((int64_t)b * a.nC * 64 + (int64_t)j * 64) * ts + h * DH;
            bf16* dkg = reinterpret_cast<bf16*>(a.dk) + ktok0;
            bf16* dvg = reinterpret_cast<bf16*>(a.dv) + ktok0;
            for (int u = lane; u < 64 * UPR; u += 32) {
              const int row = u / UPR, w = u % UPR;
              *reinterpret_cast<uint4*>(dkg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(dvg + row * ts + w * 8) = make_uint4(0, 0, 0, 0);
            }
          }
          continue;
        }
        rk[l] = k++;
        if (rk[l] >= MR && lane == 0 && !W(&meta_empty[rk[l] % MR], ((rk[l] / MR) - 1) & 1, 18, rk[l], -1))
          alive = false;
        alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
        if (!alive) break;
        if (lane == 0) {
          KVMeta& M = meta[rk[l] % MR];
          M.j = j; M.h = h; M.b = b; M.ncons = ns[l]; M.e0 = e0s[l]; M.end = 0;
        }
      }
      if (!alive) break;
      // The consumer tables of the batch, every lane at once: entry x of tile l is taken
      // by lane x % 32 in step 2 l + x / 32 (entries, then their fusion weights).
      int ev[2 * NB];
#pragma unroll
      for (int i = 0; i < 2 * NB; ++i) {
        const int l = i >> 1, x = lane + 32 * (i & 1);
        ev[i] = -1;
        if (rk[l] >= 0 && x < ns[l]) {
          const int b = (t0 + l) / (a.nC * a.H);  // the sequence of tile t0 + l
          ev[i] = a.csr_ent[(int64_t)b * a.nQ * a.topk + e0s[l] + x];
        }
      }
#pragma unroll
      for (int i = 0; i < 2 * NB; ++i) {
        const int l = i >> 1, x = lane + 32 * (i & 1);
        if (ev[i] >= 0) {
          const int b = (t0 + l) / (a.nC * a.H);
          KVMeta& M = meta[rk[l] % MR];
          M.w[x] = a.wrow[(int64_t)b * a.nQ * a.topk + ev[i]];
          M.cm[x] = ((ev[i] / a.topk + a.shift) << 4) | (ev[i] % a.topk);
        }
      }
      __syncwarp();
      if (lane == 0)
#pragma unroll
        for (int l = 0; l < NB; ++l)
          if (rk[l] >= 0) tc::mbar_arrive(&meta_full[rk[l] % MR]);
      __syncwarp();
    }
    if (lane == 0 && alive && (k < MR || W(&meta_empty[k % MR], ((k / MR) - 1) & 1, 18, k, -1))) {
      meta[k % MR].end = 1;
      tc::mbar_arrive(&meta_full[k % MR]);
    }
    __syncwarp();
  } else if (warp == kKVProd) {
    // ------------------------------------------------------------ producer warp (lane 0)
    if (lane == 0) {
      int gx = 0, tcn = 0, nkv[2] = {0, 0}, nc[NST];
      for (int st = 0; st < NST; ++st) nc[st] = 0;
      bool alive = true;
      // Stage for consumer record gx (waits until the stage's last consumer is finished).
      auto take_stage = [&](int site) -> bool {
        return gx < NST || W(&ring_empty[gx % NST], ((gx / NST) - 1) & 1, site, tcn, gx);
      };
      for (int k = 0; alive; ++k) {
        if (!W(&meta_full[k % MR], (k / MR) & 1, 19, k, -1)) {
          alive = false;
          break;
        }
        const KVMeta& M = meta[k % MR];
        if (M.end) break;
        const int j = M.j, h = M.h, b = M.b, ncons = M.ncons, e0 = M.e0;
        const int kb = tcn & 1;
        if (tcn >= 2 && !W(&kv_empty[kb], ((tcn >> 1) - 1) & 1, 21, tcn, -1)) {
          alive = false;
          break;
        }
        tc::mbar_expect_tx(&bar_kv[kb], 2 * TILE);
        tc::tma_load_4d(kvbuf + 2 * kb * TILE, &tmK, 0, h, j * 64, b, &bar_kv[kb]);
        tc::tma_load_4d(kvbuf + (2 * kb + 1) * TILE, &tmV, 0, h, j * 64, b, &bar_kv[kb]);
        ++nkv[kb];
        for (int x = 0; x < ncons; ++x, ++gx) {
          if (!take_stage(22)) {
            alive = false;
            break;
          }
          int c, m;
          float w;
          if (x < MC) {
            c = M.cm[x] >> 4;
            m = M.cm[x] & 15;
            w = M.w[x];
          } else {  // beyond the table: straight from the CSR
            const int e = a.csr_ent[(int64_t)b * a.nQ * a.topk + e0 + x];
            c = e / a.topk + a.shift;
            m = e % a.topk;
            w = a.wrow[(int64_t)b * a.nQ * a.topk + e];
          }
          const int st = gx % NST;
          KVConsRec* rec = crec(gx);
          rec->w = w;
          rec->flags = (x == 0 ? kRecFirst : 0) | (x == ncons - 1 ? kRecLast : 0);
          rec->kb = kb;
          rec->tc = tcn;
          rec->j = j;
          rec->h = h;
          rec->b = b;
          unsigned char* base = ring + st * kKVStageBytes;
          const int64_t rb = ((((int64_t)b * a.nQ + c) * a.H + h) * a.topk + m) * 64;
          tc::mbar_expect_tx(&bar_c[st], 2 * TILE + 512);
          tc::tma_load_4d(base, &tmQ, 0, h, c * 64, b, &bar_c[st]);
          tc::tma_load_4d(base + TILE, &tmdO, 0, h, c * 64, b, &bar_c[st]);
          tc::bulk_load(base + 2 * TILE, a.lse + rb, 256, &bar_c[st]);
          tc::bulk_load(base + 2 * TILE + 256, a.Dbuf + rb, 256, &bar_c[st]);
          ++nc[st];
        }
        tc::mbar_arrive(&meta_empty[k % MR]);  // the record has been read
        ++tcn;
      }
      // End marker: a consumer record with the end flag.
      if (alive && take_stage(23)) {
        crec(gx)->flags = kRecEnd;
        tc::mbar_arrive(&bar_c[gx % NST]);
      }
      // After an abort, let the copies already issued land before the CTA exits.
      if (*reinterpret_cast<volatile int*>(&abort_s)) {
        for (int x = 0; x < 2; ++x)
          if (nkv[x] > 0) tc::mbar_wait(&bar_kv[x], (nkv[x] - 1) & 1);
        for (int st = 0; st < NST; ++st)
          if (nc[st] > 0) tc::mbar_wait(&bar_c[st], (nc[st] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kKVMma) {
    // ------------------------------------------------------------ MMA warp
    const uint32_t tS = tm, tP = tm + 64, tdV = tm + 128, tdK = tm + 192;
    const uint64_t dKV = tc::desc_km(tc::su32(kvbuf));
    const uint64_t dRingKm = tc::desc_km(tc::su32(ring)), dRingMn = tc::desc_mn(tc::su32(ring));
    constexpr uint64_t kStage = kKVStageBytes >> 4, kTileStep = TILE >> 4;
    bool issued = false;
    // The products of consumer x are issued in the order dV(x), S^T(x + 1), dK(x),
    // dPo^T(x + 1): S^T(x + 1) overwrites w P^T(x), which only dV(x) reads, and dPo^T(x + 1)
    // overwrites dS^T(x), which only dK(x) reads; so S^T(x + 1) runs while the element warps
    // still form dS^T(x), and they find it done when they move on.
    auto issue_st = [&](int y, const KVConsRec& r) -> bool {  // S^T(y) = K Q^T
      if ((r.flags & kRecFirst) && !W(&bar_kv[r.kb], (r.tc >> 1) & 1, 25, r.tc, y)) return false;
      const uint64_t dk = dKV + (2 * r.kb) * kTileStep;
      const uint64_t dq = dRingKm + (y % NST) * kStage;
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tS, dk, dq, kIdKm, 0u);
      tc::commit_warp(&bar_s1);
      issued = true;
      return true;
    };
    auto issue_dpt = [&](int y, const KVConsRec& r) {  // dPo^T(y) = V dO^T
      const uint64_t dv = dKV + (2 * r.kb + 1) * kTileStep;
      const uint64_t ddo = dRingKm + (y % NST) * kStage + kTileStep;
      tc::mma4_ss<tc::kKStepKm, tc::kKStepKm>(tP, dv, ddo, kIdKm, 0u);
      tc::commit_warp(&bar_s2);
      if (r.flags & kRecLast) tc::commit_warp(&kv_empty[r.kb]);  // the tile's K, V are read
    };
    int nend = 0x7fffffff, x = 0;
    KVConsRec rx;  // record of consumer x
    bool ok = W(&bar_c[0], 0, 24, -1, 0);
    if (ok) {
      rx = *crec(0);
      if (rx.flags & kRecEnd) {
        nend = 0;
      } else {
        ok = issue_st(0, rx);
        if (ok) issue_dpt(0, rx);
      }
    }
    for (x = 0; ok && x < nend; ++x) {
      // dV += (w P^T) dO as soon as w P^T is in, while the element warps form dS^T.
      if (!W(&op_v, x & 1, 26, rx.tc, x)) break;
      tc::fence_after();
      if ((rx.flags & kRecFirst) && rx.tc >= 1 && !W(&acc_empty, (rx.tc - 1) & 1, 27, rx.tc, x)) break;
      const uint64_t bq = dRingMn + (x % NST) * kStage, bdo = bq + kTileStep;
      // The A columns of the four K steps' query pairs: 0, 8, 32, 40.
      tc::mma4_ts<8, 32, 40, tc::kKStepMn>(tdV, tS, bdo, kIdMn, (rx.flags & kRecFirst) ? 0u : 1u);
      // S^T(x + 1), if there is a next consumer.
      if (!W(&bar_c[(x + 1) % NST], ((x + 1) / NST) & 1, 24, rx.tc, x + 1)) break;
      const KVConsRec rn = *crec(x + 1);
      const bool more = !(rn.flags & kRecEnd);
      if (more && !issue_st(x + 1, rn)) break;
      // dK += dS^T Q once dS^T is in.
      if (!W(&op_k, x & 1, 32, rx.tc, x)) break;
      tc::fence_after();
      tc::mma4_ts<8, 32, 40, tc::kKStepMn>(tdK, tP, bq, kIdMn, (rx.flags & kRecFirst) ? 0u : 1u);
      tc::commit_warp(&ring_empty[x % NST]);
      if (rx.flags & kRecLast) tc::commit_warp(&acc_full);
      if (!more) {
        nend = x + 1;
        break;
      }
      issue_dpt(x + 1, rn);
      rx = rn;
    }
    // No product may still be running when TMEM is released (after an abort in particular).
    if (issued) {
      tc::commit_warp(&drain);
      if (!tc::mbar_wait(&drain, 0) && lane == 0) flag_timeout(a.err, 28, blockIdx.x, -1, x);
    }
  } else {
    // ------------------------------------------------------------ element-wise warps
    const int cq = lane & 3, g = lane >> 2, quarter = warp & 3, hc = warp >> 2;
    const uint32_t lane_q = (uint32_t)(32 * quarter) << 16;
    const uint32_t tb = tm + lane_q + 32 * hc;  // this warp's 32 columns of S^T
    const float scale = 1.0f / sqrtf((float)DH);
    const float sl2 = scale * kLog2e;
    // A finished tile's dK and dV from TMEM, straight to global memory.
    auto write_out = [&](const KVConsRec& r) -> bool {
      if (!W(&acc_full, r.tc & 1, 31, r.tc, -1)) return false;
      tc::fence_after();
      float ov[4][4], ok[4][4];
      tc::ld16x256_x4(tm + 128 + lane_q + 32 * hc, ov);
      tc::ld16x256_x4(tm + 192 + lane_q + 32 * hc, ok);
      tc::ld_wait(ov);
      tc::ld_wait(ok);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty);
      const int64_t ktok0 = ((int64_t)r.b * a.nC * 64 + (int64_t)r.j * 64) * ts + r.h * DH;
      bf16* dkg = reinterpret_cast<bf16*>(a.dk) + ktok0;
      bf16* dvg = reinterpret_cast<bf16*>(a.dv) + ktok0;
      const int r0 = 16 * quarter + g;
#pragma unroll
      for (int n = 0; n < 4; ++n) {  // key rows r0, r0 + 8; columns 32hc + 8n + 2cq (+1)
        const int col = 32 * hc + 8 * n + 2 * cq;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int64_t off = (int64_t)(r0 + 8 * half) * ts + col;
          float k0 = ok[n][2 * half] * scale, k1 = ok[n][2 * half + 1] * scale;
          float v0 = ov[n][2 * half], v1 = ov[n][2 * half + 1];
          if (a.acc_dkv) {
            const __nv_bfloat162 kk = *reinterpret_cast<const __nv_bfloat162*>(dkg + off);
            const __nv_bfloat162 vv = *reinterpret_cast<const __nv_bfloat162*>(dvg + off);
            k0 += __low2float(kk);
            k1 += __high2float(kk);
            v0 += __low2float(vv);
            v1 += __high2float(vv);
          }
          *reinterpret_cast<uint32_t*>(dkg + off) = pack_bf16(k0, k1);
          *reinterpret_cast<uint32_t*>(dvg + off) = pack_bf16(v0, v1);
        }
      }
      return true;
    };
    // A tile is written out after the next consumer's operands are in (its products run
    // meanwhile), so that the wait for the tile's last products leaves the pipe busy.
    KVConsRec pend;
    bool have_pend = false, alive = true;
    for (int x = 0;; ++x) {
      if (!W(&bar_c[x % NST], (x / NST) & 1, 29, -1, x)) {
        alive = false;
        break;
      }  // record and rows are in
      const KVConsRec r = *crec(x);
      if (r.flags & kRecEnd) break;
      const unsigned char* sb = ring + (x % NST) * kKVStageBytes;
      const float* lrow = reinterpret_cast<const float*>(sb + 2 * TILE) + 32 * hc;
      const float* drow = lrow + 64;
      // w P^T = exp2(S^T sl2 - LSE log2 e + log2 w): the fusion weight rides in the exponent,
      // and the 1/sqrt(dh) of dS^T goes onto dK once per tile.
      const float lw = __log2f(r.w);
      // P^T from S^T, and w P^T into TMEM over the columns just read.
      if (!W(&bar_s1, x & 1, 30, r.tc, x)) {
        alive = false;
        break;
      }
      float p[4][4];
      tc::ld16x256_x4(tb, p);
      tc::ld_wait(p);
      uint32_t pv[8];
      const uint64_t sl2x2 = tc::f2(sl2, sl2), nl2e = tc::f2(-kLog2e, -kLog2e), lwx2 = tc::f2(lw, lw);
#pragma unroll
      for (int n = 0; n < 4; ++n) {  // columns are queries 32hc + 8n + 2cq (+1)
        const uint64_t l2 = *reinterpret_cast<const uint64_t*>(lrow + 8 * n + 2 * cq);
        const uint64_t off = tc::fma2(l2, nl2e, lwx2);  // log2 w - LSE log2 e of both columns
        float x0, x1, x2, x3;
        tc::uf2(tc::fma2(tc::f2(p[n][0], p[n][1]), sl2x2, off), x0, x1);
        tc::uf2(tc::fma2(tc::f2(p[n][2], p[n][3]), sl2x2, off), x2, x3);
        p[n][0] = tc::ex2(x0);
        p[n][1] = tc::ex2(x1);
        p[n][2] = tc::ex2(x2);
        p[n][3] = tc::ex2(x3);
        pv[2 * n] = pack_bf16(p[n][0], p[n][1]);
        pv[2 * n + 1] = pack_bf16(p[n][2], p[n][3]);
      }
      // w P^T and dS^T as TMEM A operands (keys are rows): the pair of queries
      // (32hc + 8n + 2cq, +1) of key rows g and g + 8 goes to column 32hc + 4n + cq, inside
      // the 32 columns this warp has read.
      tc::st16x128_x4(tb, pv);
      tc::st_wait();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&op_v);
      // dS^T from dPo^T.
      if (!W(&bar_s2, x & 1, 33, r.tc, x)) {
        alive = false;
        break;
      }
      float dp[4][4];
      tc::ld16x256_x4(tb + 64, dp);
      tc::ld_wait(dp);
      uint32_t dv[8];
      const uint64_t neg1 = tc::f2(-1.f, -1.f);
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const uint64_t d2 = *reinterpret_cast<const uint64_t*>(drow + 8 * n + 2 * cq);
        float a0, a1, b0, b1;
        tc::uf2(tc::mul2(tc::f2(p[n][0], p[n][1]), tc::fma2(d2, neg1, tc::f2(dp[n][0], dp[n][1]))), a0, a1);
        tc::uf2(tc::mul2(tc::f2(p[n][2], p[n][3]), tc::fma2(d2, neg1, tc::f2(dp[n][2], dp[n][3]))), b0, b1);
        dv[2 * n] = pack_bf16(a0, a1);
        dv[2 * n + 1] = pack_bf16(b0, b1);
      }
      tc::st16x128_x4(tb + 64, dv);
      tc::st_wait();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&op_k);
      if (have_pend) {
        have_pend = false;
        if (!write_out(pend)) {
          alive = false;
          break;
        }
      }
      if (r.flags & kRecLast) {
        pend = r;
        have_pend = true;
      }
    }
    if (alive && have_pend) write_out(pend);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::tmem_dealloc(tm, 256);
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
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long ntiles = (long long)a.nC * a.H * a.B;
  const int grid = (int)std::min<long long>(ntiles, 2LL * sms);  // two CTAs per SM (TMEM: 256 columns each)
  // Heads per tile block: as many as keep their Q, dO, K and V within about the size of L2
  // (128 MB; measured against 24, 48 and 96 MB blocks and blocks of every head: 48 MB and
  // smaller are slower, the larger ones alike).
  BwdArgs b2 = a;
  const long long per_head = 4LL * 64 * 64 * 2 * std::max(a.nQ, a.nC);
  b2.kv_hb = (int)std::max<long long>(1, std::min<long long>(a.H, (128LL << 20) / per_head));
  launch_begin("gca_bwd_kv", s);
  gca_bwd_kv_tc_kernel<<<grid, kKVThreads, kKVSmem, s>>>(b2, tq, tdo, tk, tv);
  return launch_end("gca_bwd_kv", s);
}

}  // namespace gca
