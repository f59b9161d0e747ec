// Host-side declarations shared by the entry points (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gca.h"

namespace gca {

struct ErrWord;

// Launch bookkeeping: every kernel launch goes through launch_begin/launch_end so that
// the library can count launches and, when profiling is on, time them with events.
void launch_begin(const char* name, cudaStream_t s);
cudaError_t launch_end(const char* name, cudaStream_t s);

// Records `msg` as the calling thread's error detail and returns `s`.
int set_error_detail(const char* msg);

// Sets the dynamic shared-memory limit of `fn` once per device.
cudaError_t allow_smem(const void* fn, int bytes);

// TMA tensor map of a [B][rows][H][dh] bf16 tensor whose box is one head's 64 x dh
// tile, 128-byte swizzled (tmap.cu).  batch_stride_elems = 0: one tensor shared by all
// sequences.
cudaError_t make_head_tmap(CUtensorMap* out, const void* base, int dh, int H, int64_t rows, int B,
                           int64_t batch_stride_elems);

// TMA tensor map of a row-major [rows][cols] bf16 matrix whose box is 64 columns by
// box_rows rows, 128-byte swizzled (tmap.cu).
cudaError_t make_rows_tmap(CUtensorMap* out, const void* base, int64_t cols, int64_t rows, int box_rows);
// Token rows of a [chunks][65][cols] bf16 tensor (64 tokens and an LMK row per chunk) as
// 128-row boxes of two chunks' tokens, 64 columns wide, 128-byte swizzled (tmap.cu).
cudaError_t make_chunk_token_tmap(CUtensorMap* out, const void* base, int64_t cols, int64_t chunks);
// Landmark rows [batches][rows][D] bf16 with free row and batch strides (in elements;
// batch stride 0 = one table for every sequence) as boxes of 64 dims x box_rows rows.
cudaError_t make_lmk_tmap(CUtensorMap* out, const void* base, int64_t D, int64_t rows, int64_t batches,
                          int64_t row_stride, int64_t batch_stride, int box_rows);
// The same matrix as a TMA store target: 32 x 32 boxes, 64-byte swizzle (tmap.cu).
cudaError_t make_store_tmap(CUtensorMap* out, const void* base, int64_t cols, int64_t rows);

// Argument checks of gca_retrieve_topk other than the workspace (api.cu); records the
// error detail and returns the status of the first problem, or GCA_OK.
gca_status check_retrieve_args(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride, const void* k_lmk,
                               int64_t k_batch_stride, gca_dtype dtype, int B, int nQ, int nC, int D, int topk,
                               int causal_offset, int use_gumbel, int group, const int32_t* idx,
                               const float* scores);

// ---- retrieval (retrieve.cu)
struct RetrieveArgs {
  const void* q; int64_t q_rs, q_bs;
  const void* k; int64_t k_bs;
  int bf16;
  int B, nQ, nC, D, topk, off;
  int gumbel; uint64_t seed; int group;
  const uint64_t* seed_dev;  // when set, the kernels take the seed from here at launch
  int32_t* idx; float* scores;
  ErrWord* err;
  void* part;  // partial-candidate buffer (may be null when nsplit == 1)
};
// Plan: number of candidate splits per row (or row block) for the chosen kernel.
struct RetrievePlan {
  int rowwise;   // 1: one CTA per (row, split) streaming kernel; 0: 64-row tile kernel
  int nsplit;    // splits of the candidate range
  int seg;       // candidates per split
  int tc_ns[2];  // tcgen05 scoring (bf16, TMA-compatible layouts): candidate segments per
  int tc_sl[2];  //   128-row block and 256-candidate tiles per segment, without [0] and
                 //   with [1] noise; two partial lists (column halves) per segment and row
  size_t part_bytes;  // enough for whichever row-block kernel the launch picks
};
RetrievePlan retrieve_plan(int B, int nQ, int nC, int topk, int off);
cudaError_t launch_retrieve(const RetrieveArgs& a, const RetrievePlan& p, cudaStream_t s);
// tcgen05 scoring of 128 query rows x 256-candidate tiles with the top-k in the epilogue
// (retrieve_tc.cu): whether a call can take it, and the stage-1 launch (2 tc_ns[noise] lists).
bool retrieve_tc_eligible(const RetrieveArgs& a);
cudaError_t launch_retrieve_tc(const RetrieveArgs& a, const RetrievePlan& p, cudaStream_t s);

// ---- GCA forward (gca_fwd.cu)
struct FwdArgs {
  const void* q; const void* k; const void* v; int64_t kv_bs;
  int bf16, B, nQ, nC, H, dh;
  const int32_t* idx; const float* scores; int topk, shift;
  void* o; float* lse; ErrWord* err;
};
cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s);

// ---- one-softmax attention over a list of key blocks (block_attn.cu):
// mode 0: sliding-window causal self-attention (K/V of the query's own sequence, nC = nQ);
// mode 1: chunked cross-attention over the valid retrieved chunks of row c - shift.
struct BlockAttnArgs {
  const void* q; const void* k; const void* v; int64_t kv_bs;
  int bf16, B, nQ, nC, H, dh;
  int mode, window;                          // window in tokens (mode 0), a multiple of 64
  const int32_t* idx; int topk, shift;       // mode 1
  void* o; float* lse; int accumulate;       // lse [B][nQ][H][64]
  ErrWord* err;
};
cudaError_t launch_block_attn(const BlockAttnArgs& a, cudaStream_t s);

// ---- backward of the sliding-window attention (window_bwd.cu)
struct WindowBwdArgs {
  const void* q; const void* k; const void* v;  // [B][nQ*64][H][dh]
  const void* o; const void* dout;               // window output (not accumulated) and its gradient
  const float* lse;                              // [B][nQ][H][64] from the forward
  float* Dbuf;                                   // [B][nQ][H][64] workspace: rowsum(dO * O)
  void* dq; void* dk; void* dv;
  int bf16, B, nQ, H, dh, window, accumulate;
  ErrWord* err;
  // mode 0: sliding window (K/V as long as Q, nC = nQ).  mode 1: CCA, query chunk c over
  // the valid retrieved chunks of row c - shift (K/V [B][nC*64][H][dh]), key chunk j over
  // the query chunks whose row retrieved it (csr_off [B][nC+1], csr_ent [B][nQ*topk]).
  int mode, nC;
  const int32_t* idx; int topk, shift;
  const int32_t* csr_off; const int32_t* csr_ent; int32_t* csr_cur;
};
cudaError_t launch_window_backward(const WindowBwdArgs& a, cudaStream_t s);

// ---- gather of retrieved chunks into a compact buffer (gather.cu)
struct GatherArgs {
  const void* k_src; const void* v_src; int64_t src_bs;  // store [B][nC*64][H][dh]; batch stride in elements
  int esize, B, nQ, nC, H, dh, topk;
  const int32_t* idx;                                    // [B][nQ][topk]
  void* k_dst; void* v_dst;                              // [B][nQ*topk*64][H][dh]
  int32_t* idx_local;                                    // [B][nQ][topk]: slot index r*topk+m, or -1
  ErrWord* err;
};
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s);

// ---- GCA backward (gca_bwd.cu)
struct BwdArgs {
  const void* q; const void* k; const void* v;
  int bf16, B, nQ, nC, H, dh;
  const int32_t* idx; const float* scores; int topk, shift;
  const void* dout; const float* lse;
  void* dq; void* dk; void* dv; float* dscores; int acc_dkv;
  ErrWord* err;
  float* Dbuf;      // [B][nQ][H][topk][64]
  float* dwp;       // [B][nQ][H][topk]
  int32_t* csr_off; // [B][nC+1]
  int32_t* csr_ent; // [B][nQ*topk]
  int32_t* csr_cur; // [B][nC]
  float* wrow;      // [B][nQ][topk] fusion weight of every slot (written by the tensor-core query side)
  int32_t* kv_ctr;  // tile counter of the persistent key side (zeroed by the dscores kernel)
  int kv_hb;        // heads per tile block of the key side (set at its launch)
};
cudaError_t launch_backward(const BwdArgs& a, cudaStream_t s);
// Tensor-core (tcgen05) query-side and key-side passes, bf16 with dh = 64 (gca_bwd_tc.cu).
cudaError_t launch_bwd_q_tc(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_kv_tc(const BwdArgs& a, cudaStream_t s);

// ---- chunk / landmark encoder (encoder.cu), bf16, encoder head dim 64
struct EncoderArgs {
  const void* x;  // [B][nC*65][d]: per chunk 64 token rows, then the LMK row
  int B, nC, d, H;
  const float *ln1_g, *ln1_b, *b_qkv, *b_o, *ln2_g, *ln2_b, *b_1, *b_2;
  const void *w_qkv, *w_o, *w_1, *w_2, *w_kv;  // [N][K] row-major
  void* y;      // [B][nC*65][d]
  void* k;      // [B][nC*64][d]
  void* v;      // [B][nC*64][d]
  void* k_lmk;  // [B][nC][d]
  void* bufA;   // workspace [M][d]
  void* bufU;   // workspace [M][d]
  void* bufF;   // workspace [M][4d]
  ErrWord* err;
};
cudaError_t launch_chunk_encoder(const EncoderArgs& a, cudaStream_t s);

// ---- CSR of consumers per key chunk (gca_bwd.cu), also used by the score backward.
// Rows r in [0, nrows) of idx [B][ld_rows][topk] are entries e = r*topk + m.
cudaError_t launch_csr(const int32_t* idx, int B, int ld_rows, int nrows, int topk, int nC,
                       int32_t* off, int32_t* ent, int32_t* cur, ErrWord* err, cudaStream_t s);

// ---- landmark gradients (scores_bwd.cu)
struct ScoresBwdArgs {
  const void* q; int64_t q_rs, q_bs;
  const void* k; int64_t k_bs;
  int bf16, B, nQ, nC, D;
  const int32_t* idx; const float* ds; int topk;
  void* dq; int dq_bf16; int64_t dq_rs, dq_bs; int dq_acc;
  float* dk; ErrWord* err;
  int32_t* csr_off; int32_t* csr_ent; int32_t* csr_cur;
  int scan;  // set by the launcher: key chunks scan idx instead of reading the CSR
};
cudaError_t launch_scores_backward(const ScoresBwdArgs& a, cudaStream_t s);

}  // namespace gca
