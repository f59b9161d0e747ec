// Host-side construction of TMA tensor maps for [B][rows][H][dh] bf16 tensors: one box is
// the 64 x dh tile of one head (64 consecutive tokens), written to shared memory with the
// 128-byte swizzle that the tcgen05 operand descriptors expect.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace gca {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_encode_err = cudaSuccess;

void load_encode() {
  cudaDriverEntryPointQueryResult q{};
  void* fn = nullptr;
  g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (g_encode_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
    g_encode_err = cudaErrorSymbolNotFound;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

cudaError_t make_head_tmap(CUtensorMap* out, const void* base, int dh, int H, int64_t rows, int B,
                           int64_t batch_stride_elems) {
  std::call_once(g_once, load_encode);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  // dims innermost first: dh, head, token, sequence.  A batch stride of 0 (one store
  // shared by every sequence) becomes a single-sequence map; kernels then use
  // sequence coordinate 0.
  const bool shared = batch_stride_elems == 0;
  cuuint64_t dims[4] = {(cuuint64_t)dh, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)(shared ? 1 : B)};
  cuuint64_t strides[3] = {(cuuint64_t)dh * 2, (cuuint64_t)H * dh * 2,
                           (cuuint64_t)(shared ? rows * H * dh * 2 : batch_stride_elems * 2)};
  cuuint32_t box[4] = {(cuuint32_t)dh, 1, 64, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_rows_tmap(CUtensorMap* out, const void* base, int64_t cols, int64_t rows, int box_rows) {
  std::call_once(g_once, load_encode);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  // dims innermost first: column, row.  The box is 64 columns (128 bytes, one swizzle
  // span) by box_rows rows; rows past the end read as zeros.
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_chunk_token_tmap(CUtensorMap* out, const void* base, int64_t cols, int64_t chunks) {
  std::call_once(g_once, load_encode);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  // [chunks][65][cols] viewed with a box of 64 columns x the first 64 rows x 2 chunks: the
  // token rows of two consecutive chunks, without their LMK rows, as one 128-row tile.
  cuuint64_t dims[3] = {(cuuint64_t)cols, 65, (cuuint64_t)chunks};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * 65};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_lmk_tmap(CUtensorMap* out, const void* base, int64_t D, int64_t rows, int64_t batches,
                          int64_t row_stride, int64_t batch_stride, int box_rows) {
  std::call_once(g_once, load_encode);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  // dims innermost first: landmark dim, row, sequence; the box is 64 dims (128 bytes) by
  // box_rows rows of one sequence.  A batch stride of 0 (one table shared by every
  // sequence) becomes a single-sequence map.
  const bool shared = batch_stride == 0;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)(shared ? 1 : batches)};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, (cuuint64_t)(shared ? rows * row_stride : batch_stride) * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_store_tmap(CUtensorMap* out, const void* base, int64_t cols, int64_t rows) {
  std::call_once(g_once, load_encode);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  // Box of 32 columns (64 bytes) by 32 rows, 64-byte swizzle: in shared memory 16-byte
  // unit u of row r sits at unit u ^ ((r >> 1) & 3) of the row's 64 bytes.
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gca
