// Router: logits z = W_router x (plus the shared-gate logit w_shared . x as
// column E), then the routing rule per token.
//
// Routing rules:
//  * softmax top-k ("How Treebeard routes Qwen3.6 MoE tokens", "Routing
//    math"; Edge0 "Softmax top-k"): p = softmax(z); the k largest; alpha =
//    p_sel / max(sum p_sel, clamp), times routed_scaling.
//  * sigmoid group top-k (Edge0 "Sigmoid group top-k"): s = sigmoid(z) in
//    fp32, selection score s + bias, contiguous groups ranked by the sum of
//    their two largest selection scores, best topk_group groups kept, the k
//    largest selection scores among them; alpha = s_sel / sum s_sel times
//    routed_scaling.
// Ties go to the lower expert (group) index; slots are written in
// descending score order. Softmax ranking uses the fp32 logits, which orders
// experts exactly as p does without the ties that rounding exp could create.
#include "common.cuh"
#include "kernels.h"

#include <math.h>

namespace moe {

// ---------------------------------------------------------------------------
// logits: one warp per router row (row E = w_shared), up to 8 tokens per CTA
// ---------------------------------------------------------------------------
template <typename TA>
__global__ void __launch_bounds__(128) router_logits_kernel(RouterArgs a) {
  constexpr int kTok = 8;
  constexpr int kVec = Chunk<TA>::kVec;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = a.E + (a.w_shared ? 1 : 0);
  const int r = blockIdx.x * 4 + warp;
  if (r >= rows) return;
  pdl_wait();
  pdl_trigger();
  const int t0 = blockIdx.y * kTok;
  const int nt = min(kTok, a.T - t0);
  const TA* wrow = r < a.E ? static_cast<const TA*>(a.W_router) + (size_t)r * a.d
                           : static_cast<const TA*>(a.w_shared);
  const TA* x = static_cast<const TA*>(a.x) + (size_t)t0 * a.d;
  float acc[kTok];
#pragma unroll
  for (int t = 0; t < kTok; ++t) acc[t] = 0.f;
  const int nvec = a.d / kVec;
#pragma unroll 2
  for (int c = lane; c < nvec; c += 32) {
    float w[kVec];
    Chunk<TA>::unpack(ldg_stream(wrow + (size_t)c * kVec), w);
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
      if (t < nt) {
        float xv[kVec];
        Chunk<TA>::unpack(__ldg(reinterpret_cast<const uint4*>(x + (size_t)t * a.d) + c), xv);
#pragma unroll
        for (int j = 0; j < kVec; ++j) acc[t] = fmaf(w[j], xv[j], acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kTok; ++t) {
    float v = warp_sum(acc[t]);
    if (lane == 0 && t < nt) a.logits[(size_t)(t0 + t) * (a.E + 1) + r] = v;
  }
}

// ---------------------------------------------------------------------------
// top-k: one warp per token; lane l owns experts l, l+32, ... (E <= 512)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void argmax_merge(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_merge(v, i, ov, oi);
  }
}

// NaN keys rank as -inf so that every unselected expert stays selectable.
__device__ __forceinline__ float rank_key(float v) { return isnan(v) ? -INFINITY : v; }

__global__ void __launch_bounds__(256) router_topk_kernel(TopkArgs a) {
  constexpr int kMaxPerLane = 16;  // E <= 512
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  pdl_wait();
  pdl_trigger();
  const float* z = a.logits + (size_t)t * (a.E + 1);
  const int E = a.E, k = a.k;

  float key[kMaxPerLane];   // ranking key per owned expert
  float val[kMaxPerLane];   // softmax: logit; sigmoid: raw score s
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    int e = lane + 32 * j;
    float zv = e < E ? z[e] : -INFINITY;
    if (a.kind == 0) {
      key[j] = e < E ? rank_key(zv) : -INFINITY;
      val[j] = zv;
    } else {
      float s = 1.0f / (1.0f + expf(-zv));
      float b = (a.bias && e < E) ? a.bias[e] : 0.0f;
      key[j] = e < E ? rank_key(s + b) : -INFINITY;
      val[j] = s;
    }
  }
  uint32_t taken = 0;  // bit j: expert lane+32j already selected
  // experts beyond E can never be selected
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j)
    if (lane + 32 * j >= E) taken |= 1u << j;

  if (a.kind == 1) {
    // group ranking: group g scores the sum of its two largest selection
    // scores (all members when a group has one member)
    const int G = E / a.n_group;
    float gscore = -INFINITY;
    // each group's top-2 is gathered by a warp-wide scan over its members
    uint32_t kept = 0;
    float my_gscore = -INFINITY;
    for (int g = 0; g < a.n_group; ++g) {
      float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j) {
        int e = lane + 32 * j;
        if (e < E && e / G == g) {
          float v = key[j];
          if (v > t1) { t2 = t1; t1 = v; } else if (v > t2) { t2 = v; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float o1 = __shfl_xor_sync(0xffffffffu, t1, o);
        float o2 = __shfl_xor_sync(0xffffffffu, t2, o);
        // merge two sorted pairs (t1 >= t2), (o1 >= o2) into the top two
        float n1 = fmaxf(t1, o1);
        float n2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
        t1 = n1; t2 = n2;
      }
      float sc = G >= 2 ? t1 + t2 : t1;
      if (lane == g) my_gscore = sc;
    }
    gscore = lane < a.n_group ? my_gscore : -INFINITY;
    for (int r = 0; r < a.topk_group; ++r) {
      float v = lane < a.n_group ? gscore : -INFINITY;
      int i = lane < a.n_group ? lane : 0x7fffffff;
      if (lane < a.n_group && ((kept >> lane) & 1u)) { v = -INFINITY; i = 0x7fffffff; }
      warp_argmax(v, i);
      if (i < a.n_group) kept |= 1u << i;
    }
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      int e = lane + 32 * j;
      if (e < E && !((kept >> (e / G)) & 1u)) taken |= 1u << j;
    }
  }

  // k rounds of warp arg-max over the untaken experts
  int my_id = 0;
  float my_val = 0.f;
  for (int s = 0; s < k; ++s) {
    float v = -INFINITY;
    int i = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      if (!((taken >> j) & 1u)) argmax_merge(v, i, key[j], lane + 32 * j);
    }
    warp_argmax(v, i);
    if (i == 0x7fffffff) i = 0;  // unreachable for validated shapes (k <= candidates)
    const int owner = i & 31, jj = i >> 5;
    float sv = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j)
      if (j == jj) sv = val[j];
    sv = __shfl_sync(0xffffffffu, sv, owner);
    if (lane == owner) taken |= 1u << jj;
    if (lane == s) { my_id = i; my_val = sv; }
  }

  float w;
  if (a.kind == 0) {
    // softmax over all E logits; renormalise the selected probabilities
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j)
      if (lane + 32 * j < E) m = fmaxf(m, val[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float S = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j)
      if (lane + 32 * j < E) S += expf(val[j] - m);
    S = warp_sum(S);
    float p = lane < k ? expf(my_val - m) / S : 0.f;
    float denom = fmaxf(warp_sum(p), a.renorm_clamp);
    w = p / denom * a.routed_scaling;
  } else {
    float s = lane < k ? my_val : 0.f;
    float denom = fmaxf(warp_sum(s), 1.17549435e-38f);
    w = s / denom * a.routed_scaling;
  }
  if (lane < k) {
    a.topk_ids[(size_t)t * k + lane] = my_id;
    a.weights[(size_t)t * k + lane] = w;
  }
  if (lane == 0 && a.s_shared && a.has_shared_logit)
    a.s_shared[t] = 1.0f / (1.0f + expf(-z[E]));
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
  dim3 g1((rows + 3) / 4, (ra.T + 7) / 8);
  if (bf16) return launch_pdl(router_logits_kernel<__nv_bfloat16>, g1, 128, 0, st, ra);
  return launch_pdl(router_logits_kernel<float>, g1, 128, 0, st, ra);
}

cudaError_t launch_router_topk(const TopkArgs& ta, cudaStream_t st) {
  if (ta.T == 0) return cudaSuccess;
  return launch_pdl(router_topk_kernel, dim3((ta.T + 7) / 8), 256, 0, st, ta);
}

}  // namespace moe
