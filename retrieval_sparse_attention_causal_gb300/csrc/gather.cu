// Gather of retrieved chunks from a K/V store into a compact device buffer.
//
// Paper-Notes page on "Efficient Length-Generalizable Attention via Causal Retrieval for
// Long-Context Language Modeling", 关键设计 / key design (inference memory offload): the
// past chunks' keys and values can stay in host memory and only the retrieved chunks are
// brought to the GPU.  The store may be any memory the device can address: device memory,
// or pinned host memory, which a GB300 reads directly over its host link.  The copy runs
// on the GPU from the device-side retrieval result, so no index ever goes back to the
// host; the GCA forward then runs on the compact buffer with slot-local indices.
#include "common.cuh"
#include "internal.h"

namespace gca {
namespace {

constexpr int kParts = 4;  // CTAs per retrieved chunk (each copies a quarter of K and of V)

__global__ void __launch_bounds__(256) gather_chunks_kernel(GatherArgs a) {
  const int slot = blockIdx.x / kParts, part = blockIdx.x % kParts;  // slot = r * topk + m
  const int b = blockIdx.y;
  const int64_t e = (int64_t)b * a.nQ * a.topk + slot;
  const int j = a.idx[e];
  const bool valid = j >= 0 && j < a.nC;
  if (threadIdx.x == 0 && part == 0) {
    if (j < -1 || j >= a.nC) flag_bad_index(a.err, j);
    a.idx_local[e] = valid ? slot : -1;
  }
  if (!valid) return;
  const int64_t chunk16 = (int64_t)64 * a.H * a.dh * a.esize / 16;  // 16-byte units per chunk
  const int64_t per16 = chunk16 / kParts;
  const int64_t src = ((int64_t)b * a.src_bs + (int64_t)j * 64 * a.H * a.dh) * a.esize / 16 + part * per16;
  const int64_t dst = ((int64_t)b * a.nQ * a.topk + slot) * chunk16 + part * per16;
  const uint4* ks = reinterpret_cast<const uint4*>(a.k_src) + src;
  const uint4* vs = reinterpret_cast<const uint4*>(a.v_src) + src;
  uint4* kd = reinterpret_cast<uint4*>(a.k_dst) + dst;
  uint4* vd = reinterpret_cast<uint4*>(a.v_dst) + dst;
  // Four 16-byte loads of each tensor in flight per thread before the stores.
  for (int64_t u = threadIdx.x; u < per16; u += 4 * blockDim.x) {
    uint4 k4[4], v4[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t w = u + x * blockDim.x;
      if (w < per16) {
        k4[x] = ks[w];  // plain global loads: valid for device memory and mapped host memory
        v4[x] = vs[w];
      }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t w = u + x * blockDim.x;
      if (w < per16) {
        kd[w] = k4[x];
        vd[w] = v4[x];
      }
    }
  }
}

}  // namespace

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s) {
  launch_begin("gather_chunks", s);
  gather_chunks_kernel<<<dim3(a.nQ * a.topk * kParts, a.B), 256, 0, s>>>(a);
  return launch_end("gather_chunks", s);
}

}  // namespace gca
