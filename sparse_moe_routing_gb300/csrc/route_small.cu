// Routing and bucketing of a small token batch in one launch.
//
// For decode-sized batches the router contraction, the routing rule and the
// counting/packing pass are each a few microseconds of work, and as three
// launches their fixed costs dominate. This kernel chains them inside one
// grid without any waiting:
//   1. every CTA computes the logits of 8 router rows (row E = the shared
//      gate) for one group of up to 8 tokens;
//   2. the last CTA of a token group to finish (a self-resetting arrival
//      counter per group) applies the routing rule to the group's tokens,
//      one warp per token;
//   3. the last token group to finish (one more counter) runs the counting
//      and packing pass over all T*k pairs in that CTA.
// Hand-over between CTAs is the fence-then-count pattern: writers make their
// results visible device-wide (__threadfence) before counting, the last
// arriver fences again and reads through L2. No CTA ever waits on another,
// so there is nothing to time out.
#include "bucket_core.cuh"
#include "router_core.cuh"

namespace moe {

constexpr int kSmallRows = 8;   // router rows per CTA (one per warp)
constexpr int kSmallTok = 8;    // tokens per token group

struct RouteSmallArgs {
  RouterArgs ra;
  TopkArgs ta;
  BucketArgs ba;
};

template <typename TA>
__global__ void __launch_bounds__(kSmallRows * 32) route_small_kernel(RouteSmallArgs p) {
  extern __shared__ int smem[];  // bucketing scratch (used by the last CTA)
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RouterArgs& ra = p.ra;
  Ctrl* ctrl = p.ba.ctrl;
  pdl_wait();
  pdl_trigger();

  // 1. logits of this CTA's rows for its token group
  const int rows = ra.E + (ra.w_shared ? 1 : 0);
  const int r = blockIdx.x * kSmallRows + warp;
  const int tg = blockIdx.y;
  const int t0 = tg * kSmallTok;
  if (r < rows) {
    const int nt = min(kSmallTok, ra.T - t0);
    const TA* wrow = r < ra.E ? static_cast<const TA*>(ra.W_router) + (size_t)r * ra.d
                              : static_cast<const TA*>(ra.w_shared);
    const TA* x = static_cast<const TA*>(ra.x) + (size_t)t0 * ra.d;
    float acc[kSmallTok];
    router_row_dots<TA, kSmallTok>(wrow, x, ra.d, nt, lane, acc);
#pragma unroll
    for (int t = 0; t < kSmallTok; ++t)
      if (lane == 0 && t < nt) ra.logits[(size_t)(t0 + t) * (ra.E + 1) + r] = acc[t];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&ctrl->arrive[tg], 1u);
    s_last = prev == gridDim.x - 1;
    if (s_last) ctrl->arrive[tg] = 0;  // every CTA of the group has counted
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // 2. routing rule for the group's tokens
  const int t = t0 + warp;
  if (t < p.ta.T) topk_token(p.ta, t, lane);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&ctrl->arrive_all, 1u);
    s_last = prev == gridDim.y - 1;
    if (s_last) ctrl->arrive_all = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // 3. counting and packing pass over all pairs
  bucket_body<kSmallRows>(p.ba, smem);
}

bool route_small_supported(int T, int E, int k) {
  return T >= 1 && T <= kSmallMaxTokens && E <= 512 && k <= 32 && T * k <= 32 * 512;
}

cudaError_t launch_route_small(const RouterArgs& ra, const TopkArgs& ta, const BucketArgs& ba,
                               bool bf16, cudaStream_t st) {
  if (ra.T == 0) return cudaSuccess;
  if (!route_small_supported(ra.T, ra.E, ta.k)) return cudaErrorInvalidValue;
  const int rows = ra.E + (ra.w_shared ? 1 : 0);
  const dim3 grid((rows + kSmallRows - 1) / kSmallRows, (ra.T + kSmallTok - 1) / kSmallTok);
  const size_t smem = (size_t)bucket_smem_words(kSmallRows, ba.E) * sizeof(int);
  RouteSmallArgs p{ra, ta, ba};
  if (bf16) return launch_pdl(route_small_kernel<__nv_bfloat16>, grid, kSmallRows * 32, smem, st, p);
  return launch_pdl(route_small_kernel<float>, grid, kSmallRows * 32, smem, st, p);
}

}  // namespace moe
