// Unpermute-combine and residual ("How Treebeard routes Qwen3.6 MoE tokens",
// "Shared expert computation" and "Pseudocode": r_next = r_attention +
// (y_routed + y_shared); Airframe roadmap "Expert Combine": output = sum of
// weight_k * expert_k_output). The routing weights and the shared gate were
// already applied by the down projection, so each output row is
//   out[t] = r_attn[t] + ((sum over slots s, in slot order, of Y[pos[t*k+s]]) + Ys[t]),
// a fixed summation order (deterministic). One thread per float4 column.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// out[t] = r_attn[t] + ((sum over slots of Y[pos[t*k+s]]) + Ys[t])
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  const int t = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;  // float4 column
  if (c * 4 >= a.d) return;
  pdl_wait();
  pdl_trigger();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < a.k; ++s) {
    const int p = a.pos ? a.pos[(size_t)t * a.k + s] : t * a.k + s;
    const float4 y = reinterpret_cast<const float4*>(a.Y + (size_t)p * a.d)[c];
    acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
  }
  if (a.Ys) {
    const float4 y = reinterpret_cast<const float4*>(a.Ys + (size_t)t * a.d)[c];
    acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
  }
  const float4 r = reinterpret_cast<const float4*>(a.r_attn + (size_t)t * a.d)[c];
  float4 o;
  o.x = r.x + acc.x; o.y = r.y + acc.y; o.z = r.z + acc.z; o.w = r.w + acc.w;
  reinterpret_cast<float4*>(a.out + (size_t)t * a.d)[c] = o;
}

// Same sum with bf16 Y / Ys (the tensor-core path's intermediates).
__device__ __forceinline__ void add_bf16x4(float4& acc, const __nv_bfloat16* p) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  acc.x += bf16_lo(v.x); acc.y += bf16_hi(v.x); acc.z += bf16_lo(v.y); acc.w += bf16_hi(v.y);
}

__global__ void __launch_bounds__(256) combine_bf16_kernel(CombineArgs a) {
  const int t = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;  // 4-column group
  if (c * 4 >= a.d) return;
  pdl_wait();
  pdl_trigger();
  const __nv_bfloat16* Y = reinterpret_cast<const __nv_bfloat16*>(a.Y);
  const __nv_bfloat16* Ys = reinterpret_cast<const __nv_bfloat16*>(a.Ys);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < a.k; ++s) {
    const int p = a.pos ? a.pos[(size_t)t * a.k + s] : t * a.k + s;
    add_bf16x4(acc, Y + (size_t)p * a.d + c * 4);
  }
  if (Ys) add_bf16x4(acc, Ys + (size_t)t * a.d + c * 4);
  const float4 r = reinterpret_cast<const float4*>(a.r_attn + (size_t)t * a.d)[c];
  float4 o;
  o.x = r.x + acc.x; o.y = r.y + acc.y; o.z = r.z + acc.z; o.w = r.w + acc.w;
  reinterpret_cast<float4*>(a.out + (size_t)t * a.d)[c] = o;
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const int cols = a.d / 4;
  const dim3 g(a.T, (cols + 255) / 256);
  if (a.y_bf16) return launch_pdl(combine_bf16_kernel, g, 256, 0, st, a);
  return launch_pdl(combine_kernel, g, 256, 0, st, a);
}

}  // namespace moe
