// Router kernels: logits z = W_router x (plus the shared-gate logit w_shared . x
// as column E), then the routing rule per token (router_core.cuh).
#include "router_core.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// logits: one warp per router row (row E = w_shared), up to 8 tokens per CTA.
// The CTA first copies its tokens' activation rows into shared memory (all
// loads in flight at once), so each warp's dot products wait on one round of
// weight loads instead of one round of activation loads per token.
// ---------------------------------------------------------------------------
template <typename TA, bool STAGE>
__global__ void __launch_bounds__(128) router_logits_kernel(RouterArgs a, int tok_per_cta) {
  constexpr int kTok = 8;
  constexpr int kVec = Chunk<TA>::kVec;
  extern __shared__ uint4 xs[];  // [nt][d / kVec] when STAGE
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = a.E + (a.w_shared ? 1 : 0);
  const int r = blockIdx.x * 4 + warp;
  pdl_wait();
  pdl_trigger();
  const int t0 = blockIdx.y * tok_per_cta;
  const int nt = min(tok_per_cta, a.T - t0);
  const int nvec = a.d / kVec;
  const TA* x = static_cast<const TA*>(a.x) + (size_t)t0 * a.d;
  if (STAGE) {
    const uint4* xg = reinterpret_cast<const uint4*>(x);
    for (int i = threadIdx.x; i < nt * nvec; i += blockDim.x) xs[i] = __ldg(xg + i);
    __syncthreads();
  }
  if (r >= rows) return;
  const TA* wrow = r < a.E ? static_cast<const TA*>(a.W_router) + (size_t)r * a.d
                           : static_cast<const TA*>(a.w_shared);
  float acc[kTok];
  if (STAGE) router_row_dots<TA, kTok>(wrow, xs, nvec, nt, lane, acc);
  else router_row_dots<TA, kTok>(wrow, reinterpret_cast<const uint4*>(x), nvec, nt, lane, acc);
#pragma unroll
  for (int t = 0; t < kTok; ++t)
    if (lane == 0 && t < nt) a.logits[(size_t)(t0 + t) * (a.E + 1) + r] = acc[t];
}

// ---------------------------------------------------------------------------
// routing rule: one warp per token (PL experts per lane)
// ---------------------------------------------------------------------------
template <int PL>
__global__ void __launch_bounds__(256) router_topk_kernel(TopkArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  pdl_wait();
  pdl_trigger();
  topk_token_pl<PL>(a, t, lane);
}

// ---------------------------------------------------------------------------
// shared gate only ("Shared expert computation": s_t = sigmoid(w_shared . x_t)),
// one warp per token
// ---------------------------------------------------------------------------
template <typename TA>
__global__ void __launch_bounds__(256) shared_gate_kernel(RouterArgs a, float* s_out) {
  constexpr int kVec = Chunk<TA>::kVec;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  pdl_wait();
  pdl_trigger();
  const TA* w = static_cast<const TA*>(a.w_shared);
  const TA* x = static_cast<const TA*>(a.x) + (size_t)t * a.d;
  float acc = 0.f;
  for (int c = lane; c < a.d / kVec; c += 32) {
    float wv[kVec], xv[kVec];
    Chunk<TA>::unpack(__ldg(reinterpret_cast<const uint4*>(w) + c), wv);
    Chunk<TA>::unpack(__ldg(reinterpret_cast<const uint4*>(x) + c), xv);
#pragma unroll
    for (int j = 0; j < kVec; ++j) acc = fmaf(wv[j], xv[j], acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) s_out[t] = 1.0f / (1.0f + expf(-acc));
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_shared_gate(const RouterArgs& ra, float* s_out, bool bf16, cudaStream_t st) {
  if (ra.T == 0) return cudaSuccess;
  const dim3 g((ra.T + 7) / 8);
  if (bf16) return launch_pdl(shared_gate_kernel<__nv_bfloat16>, g, 256, 0, st, ra, s_out);
  return launch_pdl(shared_gate_kernel<float>, g, 256, 0, st, ra, s_out);
}

cudaError_t launch_router_logits(const RouterArgs& ra, bool bf16, cudaStream_t st) {
  if (ra.T == 0) return cudaSuccess;
  const int rows = ra.E + (ra.w_shared ? 1 : 0);
  const size_t row_bytes = (size_t)ra.d * (bf16 ? 2 : 4);
  // tokens per CTA: up to 8, their activation rows within 32 KB of shared
  // memory; rows too long to stage one at a time are read from global memory
  int tpc = (int)(32768 / row_bytes);
  tpc = tpc < 1 ? 1 : (tpc > 8 ? 8 : tpc);
  const bool stage = row_bytes <= 48 * 1024;
  const size_t smem = stage ? (size_t)tpc * row_bytes : 0;
  dim3 g1((rows + 3) / 4, (ra.T + tpc - 1) / tpc);
  if (bf16)
    return stage ? launch_pdl(router_logits_kernel<__nv_bfloat16, true>, g1, 128, smem, st, ra, tpc)
                 : launch_pdl(router_logits_kernel<__nv_bfloat16, false>, g1, 128, 0, st, ra, tpc);
  return stage ? launch_pdl(router_logits_kernel<float, true>, g1, 128, smem, st, ra, tpc)
               : launch_pdl(router_logits_kernel<float, false>, g1, 128, 0, st, ra, tpc);
}

cudaError_t launch_router_topk(const TopkArgs& ta, cudaStream_t st) {
  if (ta.T == 0) return cudaSuccess;
  const dim3 g((ta.T + 7) / 8);
  if (ta.E <= 32) return launch_pdl(router_topk_kernel<1>, g, 256, 0, st, ta);
  if (ta.E <= 64) return launch_pdl(router_topk_kernel<2>, g, 256, 0, st, ta);
  if (ta.E <= 128) return launch_pdl(router_topk_kernel<4>, g, 256, 0, st, ta);
  if (ta.E <= 256) return launch_pdl(router_topk_kernel<8>, g, 256, 0, st, ta);
  return launch_pdl(router_topk_kernel<16>, g, 256, 0, st, ta);
}

}  // namespace moe
