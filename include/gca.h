/*
 * gca.h - C ABI of the GB300 (sm_103a) library for Grouped Cross-Attention (GCA) with
 * causal chunk retrieval.
 *
 * The method (paper "Efficient Length-Generalizable Attention via Causal Retrieval for
 * Long-Context Language Modeling"; sources cited below):
 *   - a sequence is cut into chunks of S = 64 tokens, each chunk summarised by a
 *     landmark vector (Paper-Notes page, section 整体框架 / framework);
 *   - retrieval: the landmark of chunk i scores every earlier chunk's landmark and keeps
 *     the top-k (Paper-Notes page, 关键设计 / key design, "causal retrieval"; OpenReview
 *     forum page, abstract); during training Gumbel noise perturbs the selection
 *     (Paper-Notes page, 关键设计, "Gumbel top-k");
 *   - fusion: every token of the NEXT chunk attends to each retrieved chunk with its own
 *     softmax and the k results are summed with softmax(retrieval score) weights, so
 *     the scores receive gradient (Paper-Notes page, 关键设计, "Grouped Cross-Attention"
 *     and 亮点与洞察 / insights).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or retains them.  Every call is asynchronous on `stream`.
 *   - Sizes: S = 64 tokens per chunk (fixed).  B sequences, nQ query chunks, nC key
 *     chunks, H heads of size dh, landmark dimension D, top-k = `topk`.
 *   - Layouts are row-major with the last index contiguous.  "elements" strides count
 *     elements of the tensor's own dtype.
 *   - `ws` is caller-owned device workspace of at least the size returned by the
 *     matching *_workspace_size function, 256-byte aligned.  Its first 256 bytes are a
 *     sticky device error word: zero it once after allocation; kernels only ever set
 *     bits in it; gca_check_error() reads and clears it.  Different concurrent calls
 *     must use different workspaces.
 *   - Errors: argument problems are reported synchronously (nothing is launched).
 *     A bad retrieved index met by a kernel (outside [-1, nC)) is treated as an empty
 *     slot and flagged in the error word; call gca_check_error() to see it.
 */
#ifndef GCA_H
#define GCA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GCA_API __attribute__((visibility("default")))
#else
#define GCA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* gca_stream_t;

typedef enum {
  GCA_OK = 0,
  GCA_ERR_INVALID_ARG = 1,  /* a pointer, size, stride or flag is out of range          */
  GCA_ERR_UNSUPPORTED = 2,  /* valid but not provided (e.g. dh not 32/64, topk > 16)    */
  GCA_ERR_WORKSPACE = 3,    /* ws is NULL, misaligned or smaller than required          */
  GCA_ERR_CUDA = 4,         /* a CUDA runtime call failed; see gca_last_error_detail()  */
  GCA_ERR_DEVICE_INDEX = 5, /* (gca_check_error) a kernel met idx outside [-1, nC)      */
  GCA_ERR_TIMEOUT = 6       /* (gca_check_error) a bounded wait inside a kernel ran out  */
} gca_status;

typedef enum { GCA_F32 = 0, GCA_BF16 = 1 } gca_dtype;

enum { GCA_CHUNK = 64, GCA_MAX_TOPK = 16 };

/* Human-readable name of a status. */
GCA_API const char* gca_status_string(gca_status s);
/* Text of the last error raised on the calling host thread ("" if none). */
GCA_API const char* gca_last_error_detail(void);

/* ---------------------------------------------------------------------------------
 * gca_retrieve_topk - causal landmark scoring + per-row top-k.
 *
 * Paper-Notes page, 关键设计 (causal retrieval; Gumbel top-k); OpenReview abstract.
 * For every sequence b and query row i, with candidates j = 0 .. n_i - 1 where
 * n_i = min(nC, i + causal_offset):
 *     s_ij   = <q_lmk[b,i,:], k_lmk[b,j,:]> / sqrt(D)       (float32 accumulation)
 *     key_ij = s_ij + g_ij   if use_gumbel, else s_ij       (float32)
 *     g_ij   = -log(-log U),  U = ((h >> 41) + 0.5) / 2^23,
 *     h      = splitmix64 output number (ctr + 1) from state `seed`,
 *     ctr    = group << 56 | b << 48 | i << 24 | j.
 * The min(topk, n_i) candidates with the largest keys are written in descending key
 * order (equal keys: lower j first).  Unused slots get idx = -1 and score = -inf.
 * The call picks its kernels from the shape (a streaming scan for up to 8 query rows;
 * tensor-core score tiles with the selection in their epilogue for large bf16 problems;
 * 64-row tiles otherwise).  All apply the same order and tie rule; their float32 sums
 * may round differently, so only keys within that rounding of each other can be
 * ordered differently by different kernels.  A given shape always takes the same
 * kernels, and its result does not depend on how the candidates are split.
 *
 *   q_lmk   [B][nQ][D] at q_row_stride / q_batch_stride elements (row stride >= D,
 *           a multiple of 8 elements for bf16 and 4 for f32; strides allow reading the
 *           landmark rows straight out of a larger tensor).
 *   k_lmk   [B][nC][D], rows contiguous, batch stride k_batch_stride (>= nC*D, or 0 to
 *           share one landmark set among all sequences).
 *   dtype   GCA_F32 or GCA_BF16 (both landmark tensors).
 *   D       bf16: a multiple of 64 in 64..1024; f32: a multiple of 32 in 32..512.
 *   topk    1 .. 16.   causal_offset >= 0 (0 in training; nC at decode).
 *   use_gumbel: requires B <= 256, nQ, nC <= 2^24 and 0 <= group < 256.
 *   idx     [B][nQ][topk] int32 out.   scores [B][nQ][topk] float32 out (clean s).
 *   ws      >= gca_retrieve_workspace_size(B, nQ, nC, topk, causal_offset) bytes.
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_retrieve_workspace_size(int B, int nQ, int nC, int topk, int causal_offset);
GCA_API gca_status gca_retrieve_topk(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride,
                             const void* k_lmk, int64_t k_batch_stride, gca_dtype dtype,
                             int B, int nQ, int nC, int D, int topk, int causal_offset,
                             int use_gumbel, uint64_t seed, int group, int32_t* idx,
                             float* scores, void* ws, size_t ws_bytes, gca_stream_t stream);
/* gca_retrieve_topk_dseed - gca_retrieve_topk with the noise seed in device memory: the
 * kernels read the one uint64 at `seed` when they run, not when the call is made.  A
 * captured CUDA graph of a training step can then draw fresh noise on every replay (a
 * kernel in the graph, or a copy before each replay, writes the next seed).  `seed` is a
 * device pointer, 8-byte aligned, that the caller keeps alive while the work runs; it is
 * only read.  Every other argument, the results and the errors are those of
 * gca_retrieve_topk with that seed value; a NULL or misaligned `seed` returns
 * GCA_ERR_INVALID_ARG before anything is launched. */
GCA_API gca_status gca_retrieve_topk_dseed(const void* q_lmk, int64_t q_row_stride,
                                   int64_t q_batch_stride, const void* k_lmk,
                                   int64_t k_batch_stride, gca_dtype dtype, int B, int nQ,
                                   int nC, int D, int topk, int causal_offset, int use_gumbel,
                                   const uint64_t* seed, int group, int32_t* idx,
                                   float* scores, void* ws, size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_retrieve_topk_noalloc - gca_retrieve_topk for callers that cannot allocate.
 *
 * The paper has no counterpart: this is a convenience of the library.  Some callers
 * cannot allocate device memory where they retrieve: a plug-in inside a host
 * application whose allocator already owns all of the GPU's memory, a latency-bound
 * decode loop where a cudaMalloc would synchronise the device and stall other streams,
 * or a plain C caller with no device allocator of its own.  This entry point takes the
 * arguments of gca_retrieve_topk without the workspace and keeps its scratch (the
 * per-split candidate lists and an error word) in one static device array of
 * gca_retrieve_noalloc_max_scratch() = 4 MiB (+256 bytes), which every GPU that loads
 * the library holds until the process exits.
 *   - A problem whose candidate scratch is larger (gca_retrieve_workspace_size() minus
 *     256 bytes above 4 MiB) returns GCA_ERR_UNSUPPORTED with an explanation: decode
 *     at 16M context with up to 16 sequences and training-size problems fit, a
 *     1M-token prefill does not.
 *   - Nothing is allocated (no cudaMalloc or cudaFree).  The first call on a device
 *     looks up the array's device address (cudaGetSymbolAddress) with that device
 *     current; make that first call before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents.  Calls
 *     that can overlap on the GPU (several streams or host threads) race on it; issue
 *     them on one stream.
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_retrieve_noalloc_max_scratch(void);
GCA_API gca_status gca_retrieve_topk_noalloc(const void* q_lmk, int64_t q_row_stride,
                                     int64_t q_batch_stride, const void* k_lmk,
                                     int64_t k_batch_stride, gca_dtype dtype, int B, int nQ,
                                     int nC, int D, int topk, int causal_offset,
                                     int use_gumbel, uint64_t seed, int group, int32_t* idx,
                                     float* scores, gca_stream_t stream);
/* gca_retrieve_noalloc_check_error - gca_check_error() for the static array of
 * gca_retrieve_topk_noalloc on the current device: synchronises `stream`, reads and clears
 * the array's device error word.  Returns GCA_OK, GCA_ERR_TIMEOUT (a bounded wait ran out:
 * the idx/scores of that call are not valid), GCA_ERR_DEVICE_INDEX or GCA_ERR_CUDA.  Each
 * gca_retrieve_topk_noalloc call clears the word when it starts, so check after a call and
 * before the next one.  Argument errors of a rejected call are returned by that call and
 * leave the word untouched. */
GCA_API gca_status gca_retrieve_noalloc_check_error(gca_stream_t stream, int* bad_value);
/* Test hook: gca_selftest_timeout() run against the same array's error word (a wait on a
 * barrier that nothing arrives at runs out after `spins` probes and records
 * GCA_ERR_TIMEOUT; no fault or hang), so that a test can see the error reach
 * gca_retrieve_noalloc_check_error(). */
GCA_API gca_status gca_retrieve_noalloc_selftest_timeout(uint32_t spins, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_forward - grouped cross-attention over the retrieved chunks.
 *
 * Paper-Notes page, 关键设计 ("Grouped Cross-Attention"): each retrieved chunk gets its
 * own softmax; the k outputs are fused with softmax-normalised retrieval scores.
 * Query chunk c uses retrieval row r = c - shift (shift = 1: the next-chunk rule of
 * training, where row r's landmark sits at the end of chunk r; shift = 0: decode).
 * For each valid slot m of row r (j = idx[b,r,m] >= 0) and head h:
 *     A_m = softmax(Q_c K_j^T / sqrt(dh)) V_j      (64 x 64 logits, no mask)
 *     O_c = sum_m w_m A_m,   w = softmax over valid slots of scores[b,r,:]
 * Chunks with r < 0 or without a valid slot get O = 0.
 *
 *   q, o    [B][nQ*64][H][dh] contiguous, dtype `dtype`.
 *   k, v    [B][nC*64][H][dh]; kv_batch_stride elements between sequences
 *           (nC*64*H*dh when contiguous; 0 = all sequences share one store).
 *   idx, scores [B][nQ][topk] (idx in [-1, nC); scores float32).
 *   lse     [B][nQ][H][topk][64] float32 out: log-sum-exp of each slot's scaled
 *           logits (natural log), -inf for slots that are not valid; kept for backward.
 *   dh      32 or 64.   topk 1..16.   shift 0 or 1.
 *   ws      >= gca_forward_workspace_size() bytes (error word only).
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_forward_workspace_size(void);
GCA_API gca_status gca_forward(const void* q, const void* k, const void* v, int64_t kv_batch_stride,
                       gca_dtype dtype, int B, int nQ, int nC, int H, int dh,
                       const int32_t* idx, const float* scores, int topk, int shift,
                       void* o, float* lse, void* ws, size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_window_forward - sliding-window causal self-attention.
 *
 * Paper-Notes page, 损失函数/训练策略 (training strategy): the attention block runs
 * sliding-window self-attention (W = 512) beside the top-k retrieval.  Token t attends to
 * tokens t - window + 1 .. t of its own sequence (fewer at the start) with one softmax of
 * the dh^-1/2-scaled logits.  With accumulate != 0 the result is added to o (the block's
 * sum of this sublayer and gca_forward's output); otherwise o is overwritten.
 *
 *   q, k, v, o [B][L][H][dh] contiguous, dtype `dtype`; L a multiple of 64.
 *   lse     [B][L/64][H][64] float32 out: log-sum-exp of each row's scaled logits.
 *   window  a multiple of 64 in 64..4032.   dh 32 or 64.
 *   ws      >= gca_forward_workspace_size() bytes (error word only).
 * ------------------------------------------------------------------------------- */
GCA_API gca_status gca_window_forward(const void* q, const void* k, const void* v, gca_dtype dtype, int B,
                              int L, int H, int dh, int window, void* o, float* lse, int accumulate,
                              void* ws, size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_window_backward - gradients of gca_window_forward.
 *
 * With P the masked row softmax (from the saved LSE) and D = rowsum(dO * O):
 *     dS = P * (dO V^T - D),  dQ = dS K / sqrt(dh),  dK = dS^T Q / sqrt(dh),  dV = P^T dO.
 * Deterministic (no atomics): a query-side and a key-side pass.
 *
 *   q, k, v, lse, window: as passed to / produced by gca_window_forward.
 *   o       [B][L][H][dh] the window attention's own output (before any accumulation
 *           onto another sublayer's output; that sum is linear, so dout is the same).
 *   dout    [B][L][H][dh] gradient of o.
 *   dq, dk, dv [B][L][H][dh] out (accumulate != 0: added to).
 *   ws      >= gca_window_backward_workspace_size(B, L, H) bytes.
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_window_backward_workspace_size(int B, int L, int H);
GCA_API gca_status gca_window_backward(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, gca_dtype dtype, int B, int L,
                               int H, int dh, int window, void* dq, void* dk, void* dv,
                               int accumulate, void* ws, size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_cca_forward - chunked cross-attention over the retrieved chunks (ablation).
 *
 * Paper-Notes page, 关键设计 ("Grouped Cross-Attention"): the variant GCA is contrasted
 * with.  The valid retrieved chunks of row r = c - shift are concatenated and query chunk
 * c attends to them with ONE softmax; the retrieval scores take no part.  Chunks without a
 * valid slot get O = 0 (unchanged when accumulating) and LSE = -inf.
 *
 *   q, k, v, kv_batch_stride, idx, topk, shift: as for gca_forward (no scores).
 *   o       [B][nQ*64][H][dh] out (accumulate != 0: added to).
 *   lse     [B][nQ][H][64] float32 out.
 *   ws      >= gca_forward_workspace_size() bytes (error word; idx outside [-1, nC) is
 *           flagged there and skipped).
 * ------------------------------------------------------------------------------- */
GCA_API gca_status gca_cca_forward(const void* q, const void* k, const void* v, int64_t kv_batch_stride,
                           gca_dtype dtype, int B, int nQ, int nC, int H, int dh, const int32_t* idx,
                           int topk, int shift, void* o, float* lse, int accumulate, void* ws,
                           size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_selftest_timeout - exercise the device error path of a wait that runs out.
 *
 * Launches one CTA that waits, with the library's bounded mbarrier wait limited to
 * `spins` probes, on a barrier that nothing ever arrives at.  The wait runs out, the CTA
 * records GCA_ERR_TIMEOUT (wait site 30) in the error word of `ws` and exits; no fault,
 * trap or hang.  gca_check_error(ws) then returns GCA_ERR_TIMEOUT and clears the word, and
 * the context stays usable.  For tests of the failure path.
 *
 *   ws      >= 256 bytes (the error word).   spins in 1..2^20.
 * ------------------------------------------------------------------------------- */
GCA_API gca_status gca_selftest_timeout(void* ws, size_t ws_bytes, uint32_t spins, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_cca_backward - gradients of gca_cca_forward.
 *
 * With P the joint row softmax of a query chunk over its valid retrieved chunks (from the
 * saved LSE) and D = rowsum(dO * O):  dS = P * (dO V^T - D),  dQ = dS K / sqrt(dh),
 * dK_j += dS^T Q / sqrt(dh),  dV_j += P^T dO  for every retrieved chunk j.  The scores take
 * no part in CCA, so there is no score gradient.  Deterministic (no atomics): a query-side
 * pass, and a key-side pass over each chunk's consumers in entry order.
 *
 *   q, k, v, idx, topk, shift, lse: as passed to / produced by gca_cca_forward (K/V
 *           contiguous per sequence: no shared store).
 *   o       [B][nQ*64][H][dh] CCA's own output (before any accumulation).
 *   dout    [B][nQ*64][H][dh] gradient of o.
 *   dq [B][nQ*64][H][dh], dk, dv [B][nC*64][H][dh] out (accumulate != 0: added to).  Query
 *           chunks without a valid slot get dq = 0, chunks never retrieved dk = dv = 0.
 *   ws      >= gca_cca_backward_workspace_size(B, nQ, nC, H, topk) bytes (error word,
 *           D rows, consumer lists); idx outside [-1, nC) is flagged there and skipped.
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_cca_backward_workspace_size(int B, int nQ, int nC, int H, int topk);
GCA_API gca_status gca_cca_backward(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, gca_dtype dtype, int B, int nQ,
                            int nC, int H, int dh, const int32_t* idx, int topk, int shift,
                            void* dq, void* dk, void* dv, int accumulate, void* ws,
                            size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_chunk_encoder_forward - the chunk / landmark encoder and the shared K/V transform.
 *
 * Paper-Notes page, 整体框架 (framework): the lower layers' output, with an LMK token
 * closing every 64-token chunk, passes a bidirectional Transformer encoder that yields
 * the chunk representations and the landmark representations shared by the upper
 * layers; 关键设计 / GCA: one K/V transform serves all of them.  Read as one pre-LN
 * encoder layer applied to every chunk on its own (the pages give neither depth nor
 * form), with dh = d / H:
 *     u = x + MHA(LN1(x)) W_o^T + b_o     attention over the chunk's 65 rows, no mask,
 *                                         logits scaled by dh^-1/2;
 *     y = u + GELU(LN2(u) W_1^T + b_1) W_2^T + b_2      (erf GELU, LayerNorm eps 1e-5);
 *     k_lmk = y at the LMK rows;   K, V = (y at the token rows) W_K^T, W_V^T.
 *
 *   x       [B][nC*65][d] bf16: per chunk its 64 token rows, then its LMK row.
 *   w       weights: matrices bf16 [out][in] row-major (w_qkv [3d][d] with the Q, K, V
 *           blocks in that order and heads contiguous inside each; w_o [d][d]; w_1 [4d][d];
 *           w_2 [d][4d]; w_kv [2d][d], K rows first); biases and LayerNorm gains/shifts
 *           float32 ([3d], [d], [4d], [d]; [d]).  Caller-owned device memory.
 *   y       [B][nC*65][d] bf16 out: the encoder's output rows.
 *   k, v    [B][nC*64][d] bf16 out: GCA's keys and values, i.e. [B][L][H'][dh'] for any
 *           head split H' dh' = d of the upper layers.
 *   k_lmk   [B][nC][d] bf16 out: the landmark representations (retrieval's k_lmk, D = d).
 *   dtype   GCA_BF16 (GCA_ERR_UNSUPPORTED otherwise).   d a multiple of 128 in 128..1024,
 *           H = d / 64 (encoder head dim 64).  All pointers 16-byte aligned.
 *   ws      >= gca_chunk_encoder_workspace_size(B, nC, d) bytes: the error word and the
 *           intermediate rows (B*nC*65 x 6d bf16).
 * ------------------------------------------------------------------------------- */
typedef struct {
  const float* ln1_g; const float* ln1_b;
  const void* w_qkv;  const float* b_qkv;
  const void* w_o;    const float* b_o;
  const float* ln2_g; const float* ln2_b;
  const void* w_1;    const float* b_1;
  const void* w_2;    const float* b_2;
  const void* w_kv;
} gca_encoder_weights;
GCA_API size_t gca_chunk_encoder_workspace_size(int B, int nC, int d);
GCA_API gca_status gca_chunk_encoder_forward(const void* x, gca_dtype dtype, int B, int nC, int d, int H,
                                     const gca_encoder_weights* w, void* y, void* k, void* v, void* k_lmk,
                                     void* ws, size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_gather_chunks - copy the retrieved chunks' keys and values into a compact buffer.
 *
 * Paper-Notes page, 关键设计 / key design (inference memory offload): the past chunks'
 * K/V may live in host memory; only the k retrieved chunks are brought to the GPU.  The
 * copy is a GPU kernel driven by the device-side idx, so nothing returns to the host.
 * For each (b, r, m) with j = idx[b,r,m] in [0, nC): chunk j of the store (64 tokens x H
 * x dh of K and of V) goes to slot s = r*topk + m of the destination, and
 * idx_local[b,r,m] = s; other slots get idx_local = -1 and are left untouched.
 * gca_forward(q, k_dst, v_dst, kv_batch_stride = nQ*topk*64*H*dh, nC' = nQ*topk,
 * idx_local, scores, ...) then gives the same result as on the full store.
 *
 *   k_src, v_src [B][nC*64][H][dh] (src_batch_stride elements between sequences, 0 = one
 *           store shared by all).  Any memory the device can read: device memory, or
 *           pinned host memory (read directly by the GPU over its host link).
 *   k_dst, v_dst [B][nQ*topk*64][H][dh] device memory.   idx, idx_local [B][nQ][topk].
 *   dtype   GCA_F32 or GCA_BF16.   dh 32 or 64.   topk 1..16.   Pointers 16-byte aligned.
 *   ws      >= gca_gather_workspace_size() bytes (error word only); idx outside [-1, nC)
 *           is flagged there (GCA_ERR_DEVICE_INDEX) and treated as -1.
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_gather_workspace_size(void);
GCA_API gca_status gca_gather_chunks(const void* k_src, const void* v_src, int64_t src_batch_stride,
                             gca_dtype dtype, int B, int nQ, int nC, int H, int dh,
                             const int32_t* idx, int topk, void* k_dst, void* v_dst,
                             int32_t* idx_local, void* ws, size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_backward - gradients of gca_forward: dQ, dK, dV and the retrieval scores.
 *
 * The score gradient is what lets the retriever learn from the language-model loss
 * (Paper-Notes page, 研究背景与动机 / motivation and 亮点与洞察 / insights).  With
 * D_m[t] = <dO[t], A_m[t]> and dw_m = sum over tokens and heads of D_m:
 *     dscores[b,r,m] = w_m (dw_m - sum_n w_n dw_n)
 *     dS_m = w_m P_m * (dO V_j^T - D_m) / sqrt(dh)
 *     dQ_c = sum_m dS_m K_j,   dK_j += dS_m^T Q_c,   dV_j += w_m P_m^T dO_c
 *
 *   q, k, v, idx, scores, lse: as passed to / produced by gca_forward (K/V contiguous).
 *   dout    [B][nQ*64][H][dh] gradient of o.
 *   dq      [B][nQ*64][H][dh] out (chunks without a valid slot get 0).
 *   dk, dv  [B][nC*64][H][dh] out; every chunk is written (0 if never retrieved), or,
 *           with accumulate_dkv = 1, the gradient is added to their current contents.
 *   dscores [B][nQ][topk] float32 out, aligned with idx (0 for unused slots and rows).
 *   ws      >= gca_backward_workspace_size(B, nQ, nC, H, topk) bytes.
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_backward_workspace_size(int B, int nQ, int nC, int H, int topk);
GCA_API gca_status gca_backward(const void* q, const void* k, const void* v, gca_dtype dtype, int B,
                        int nQ, int nC, int H, int dh, const int32_t* idx, const float* scores,
                        int topk, int shift, const void* dout, const float* lse, void* dq,
                        void* dk, void* dv, float* dscores, int accumulate_dkv, void* ws,
                        size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_scores_backward - gradient of the scaled dot-product scores into the landmarks.
 *
 *     dq_lmk[b,i] (+)= sum_m dscores[b,i,m] k_lmk[b, idx[b,i,m]] / sqrt(D)
 *     dk_lmk[b,j]   = sum_{(i,m): idx[b,i,m] = j} dscores[b,i,m] q_lmk[b,i] / sqrt(D)
 * The Gumbel noise only chose the slots and carries no gradient.
 *
 *   q_lmk, k_lmk, dtype, strides: as for gca_retrieve_topk (k_batch_stride may not be 0).
 *   idx, dscores [B][nQ][topk].
 *   dq_lmk  output with its own dtype, row and batch strides (elements); with
 *           dq_accumulate = 1 the gradient is added to the current contents (used to
 *           push a second group's landmark gradient into the first group's output
 *           gradient at each chunk's last token).
 *   dk_lmk  [B][nC][D] float32 out, overwritten.
 *   ws      >= gca_scores_backward_workspace_size(B, nQ, nC, topk) bytes.
 * ------------------------------------------------------------------------------- */
GCA_API size_t gca_scores_backward_workspace_size(int B, int nQ, int nC, int topk);
GCA_API gca_status gca_scores_backward(const void* q_lmk, int64_t q_row_stride, int64_t q_batch_stride,
                               const void* k_lmk, int64_t k_batch_stride, gca_dtype dtype,
                               int B, int nQ, int nC, int D, const int32_t* idx,
                               const float* dscores, int topk, void* dq_lmk,
                               gca_dtype dq_dtype, int64_t dq_row_stride,
                               int64_t dq_batch_stride, int dq_accumulate, float* dk_lmk,
                               void* ws, size_t ws_bytes, gca_stream_t stream);

/* ---------------------------------------------------------------------------------
 * gca_check_error - synchronise `stream`, read and clear the device error word of `ws`.
 * Returns GCA_OK, GCA_ERR_TIMEOUT (a tensor-core completion wait gave up instead of
 * hanging; the results of that call are not valid), GCA_ERR_DEVICE_INDEX (with the
 * offending index in *bad_value when bad_value != NULL) or GCA_ERR_CUDA.
 * ------------------------------------------------------------------------------- */
GCA_API gca_status gca_check_error(void* ws, gca_stream_t stream, int* bad_value);

/* ---------------------------------------------------------------------------------
 * Instrumentation (host side, process-wide).
 *   gca_launch_count  - number of kernels this library has launched so far.
 *   gca_profile_begin - from now on, bracket every kernel launch with CUDA events on
 *                       its own stream (adds ~1 us per launch).
 *   gca_profile_end   - stop recording, wait for the events, and fill a table of
 *                       (kernel name, launches, total milliseconds); returns the number
 *                       of rows, reads them with gca_profile_row(i, ...).
 * ------------------------------------------------------------------------------- */
GCA_API uint64_t gca_launch_count(void);
GCA_API gca_status gca_profile_begin(void);
GCA_API int gca_profile_end(void);
GCA_API gca_status gca_profile_row(int i, const char** name, int* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* GCA_H */
