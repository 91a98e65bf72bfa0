// Packed-row gather for the tensor-core path: X_perm[p] = x[perm[p] / k],
// the activation row of each routed (token, slot) pair in the packed order
// of the bucketing pass, so that the grouped GEMM reads each group's rows as
// one contiguous TMA-addressable block.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int k,
                                                          int row_vecs, uint4* __restrict__ out,
                                                          int P) {
  pdl_wait();
  pdl_trigger();
  // kRows rows per CTA step, so that each thread has kRows loads in flight
  constexpr int kRows = 4;
  for (int p0 = blockIdx.x * kRows; p0 < P; p0 += gridDim.x * kRows) {
    size_t src[kRows], dst[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int p = p0 + u;
      src[u] = p < P ? (size_t)(perm[p] / k) * row_vecs : 0;
      dst[u] = (size_t)p * row_vecs;
    }
    for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
      uint4 val[kRows];
#pragma unroll
      for (int u = 0; u < kRows; ++u)
        if (p0 + u < P) val[u] = __ldg(x + src[u] + v);
#pragma unroll
      for (int u = 0; u < kRows; ++u)
        if (p0 + u < P) out[dst[u] + v] = val[u];
    }
  }
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, const int32_t* perm, int k, int d, void* out, int P,
                               cudaStream_t st) {
  if (P == 0) return cudaSuccess;
  const int steps = (P + 3) / 4;
  int grid = steps < tc_sm_count() * 16 ? steps : tc_sm_count() * 16;
  return launch_pdl(gather_rows_kernel, dim3(grid), 256, 0, st, static_cast<const uint4*>(x),
                    perm, k, d / 8, static_cast<uint4*>(out), P);
}

}  // namespace moe
