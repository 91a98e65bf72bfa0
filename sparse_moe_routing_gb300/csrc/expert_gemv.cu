// Weight-streaming grouped expert GEMV on CUDA cores, and the combine.
//
// Routed expert ("How Treebeard routes Qwen3.6 MoE tokens", "Routed expert
// computation"; Edge0 "Experts"): h = SiLU(W_gate x) * (W_up x),
// e = W_down h; the routed output carries alpha ("weighted sum"), the shared
// expert carries its sigmoid gate s_t ("Shared expert computation"). The
// combine adds the routed slots in slot order, then the shared branch, then
// the residual ("Pseudocode": attention_residual + routed + shared).
//
// Work is organised by the packing of the bucketing pass ("Intel SYCL path":
// launch over active experts, reuse each loaded weight block across the
// expert's tokens, write back to the original token-slot position): CTA
// (slot, row block) streams a block of one active expert's weight rows from
// HBM exactly once per chunk of up to kTok of that expert's tokens, whose
// activations sit in shared memory as fp32.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kTok = 8;        // tokens per activation chunk
constexpr int kKc = 2048;      // input-dim elements per activation chunk
constexpr int kGuRows = 16;    // gate/up row pairs per CTA (2 per warp)
constexpr int kDnRows = 32;    // down rows per CTA (4 per warp)

struct GroupView {
  bool ok;
  int n;         // rows (tokens) in the group
  int row0;      // first packed row (routed) or 0 (shared)
  int width;     // intermediate width of this group
  bool shared;
  int g;
};

__device__ __forceinline__ GroupView resolve_group(const GemvArgs& a, int slot) {
  GroupView v{};
  if (slot < a.routed_slots) {
    if (slot >= *a.n_active) return v;
    const int g = a.active[slot];
    v.g = g;
    v.row0 = a.offsets[g];
    v.n = a.offsets[g + 1] - v.row0;
    v.width = a.I;
    v.shared = false;
  } else {
    v.g = a.E;
    v.row0 = 0;
    v.n = a.T;
    v.width = a.Is;
    v.shared = true;
  }
  v.ok = v.n > 0;
  return v;
}

// token index of packed row i of the group
__device__ __forceinline__ int group_token(const GemvArgs& a, const GroupView& v, int i) {
  return v.shared ? i : a.perm[v.row0 + i] / a.k;
}

// Loads activation rows [tok0, tok0+nt) x [k0, k0+kc) into smem as fp32.
template <typename TA>
__device__ __forceinline__ void stage_x(const GemvArgs& a, const GroupView& v, int tok0, int nt,
                                        int k0, int kc, float* xs) {
  const TA* x = static_cast<const TA*>(a.x);
  for (int idx = threadIdx.x; idx < nt * kc; idx += blockDim.x) {
    const int t = idx / kc, j = idx - t * kc;
    const int tok = group_token(a, v, tok0 + t);
    xs[t * kKc + j] = load_act(x, (size_t)tok * a.d + k0 + j);
  }
}

template <typename TW, typename TA>
__global__ void __launch_bounds__(256) gemv_gateup_kernel(GemvArgs a) {
  extern __shared__ float xs[];  // [kTok][kKc]
  constexpr int kVec = Chunk<TW>::kVec;
  const GroupView v = resolve_group(a, blockIdx.y);
  if (!v.ok) return;
  const int r_base = blockIdx.x * kGuRows;
  if (r_base >= v.width) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TW* Wg = static_cast<const TW*>(v.shared ? a.Wsg : a.Wg);
  const TW* Wu = static_cast<const TW*>(v.shared ? a.Wsu : a.Wu);
  if (!v.shared) {
    Wg += (size_t)v.g * a.I * a.d;
    Wu += (size_t)v.g * a.I * a.d;
  }
  float* H = v.shared ? a.Hs : a.H + (size_t)v.row0 * a.I;

  for (int tok0 = 0; tok0 < v.n; tok0 += kTok) {
    const int nt = min(kTok, v.n - tok0);
    float accg[2][kTok], accu[2][kTok];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int t = 0; t < kTok; ++t) accg[r][t] = accu[r][t] = 0.f;
    for (int k0 = 0; k0 < a.d; k0 += kKc) {
      const int kc = min(kKc, a.d - k0);
      __syncthreads();
      stage_x<TA>(a, v, tok0, nt, k0, kc, xs);
      __syncthreads();
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = r_base + warp * 2 + rr;
        if (r >= v.width) break;
        const TW* pg = Wg + (size_t)r * a.d + k0;
        const TW* pu = Wu + (size_t)r * a.d + k0;
#pragma unroll 4
        for (int c = lane; c < kc / kVec; c += 32) {
          float wg[kVec], wu[kVec];
          Chunk<TW>::unpack(ldg_stream(pg + c * kVec), wg);
          Chunk<TW>::unpack(ldg_stream(pu + c * kVec), wu);
#pragma unroll
          for (int t = 0; t < kTok; ++t) {
            if (t < nt) {
              const float* xr = xs + t * kKc + c * kVec;
#pragma unroll
              for (int j = 0; j < kVec; ++j) {
                accg[rr][t] = fmaf(wg[j], xr[j], accg[rr][t]);
                accu[rr][t] = fmaf(wu[j], xr[j], accu[rr][t]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = r_base + warp * 2 + rr;
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        const float g = warp_sum(accg[rr][t]);
        const float u = warp_sum(accu[rr][t]);
        if (lane == 0 && t < nt && r < v.width) H[(size_t)(tok0 + t) * v.width + r] = siluf_(g) * u;
      }
    }
  }
}

template <typename TW>
__global__ void __launch_bounds__(256) gemv_down_kernel(GemvArgs a) {
  extern __shared__ float hs[];  // [kTok][kKc]
  constexpr int kVec = Chunk<TW>::kVec;
  const GroupView v = resolve_group(a, blockIdx.y);
  if (!v.ok) return;
  const int r_base = blockIdx.x * kDnRows;
  if (r_base >= a.d) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TW* Wd = static_cast<const TW*>(v.shared ? a.Wsd : a.Wd);
  if (!v.shared) Wd += (size_t)v.g * a.d * a.I;
  const float* H = v.shared ? a.Hs : a.H + (size_t)v.row0 * a.I;
  float* Y = v.shared ? a.Ys : a.Y + (size_t)v.row0 * a.d;
  const int K = v.width;

  for (int tok0 = 0; tok0 < v.n; tok0 += kTok) {
    const int nt = min(kTok, v.n - tok0);
    float acc[4][kTok];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int t = 0; t < kTok; ++t) acc[r][t] = 0.f;
    for (int k0 = 0; k0 < K; k0 += kKc) {
      const int kc = min(kKc, K - k0);
      __syncthreads();
      for (int idx = threadIdx.x; idx < nt * kc; idx += blockDim.x) {
        const int t = idx / kc, j = idx - t * kc;
        hs[t * kKc + j] = H[(size_t)(tok0 + t) * K + k0 + j];
      }
      __syncthreads();
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int r = r_base + warp * 4 + rr;
        if (r >= a.d) break;
        const TW* pd = Wd + (size_t)r * K + k0;
#pragma unroll 2
        for (int c = lane; c < kc / kVec; c += 32) {
          float w[kVec];
          Chunk<TW>::unpack(ldg_stream(pd + c * kVec), w);
#pragma unroll
          for (int t = 0; t < kTok; ++t) {
            if (t < nt) {
              const float* hr = hs + t * kKc + c * kVec;
#pragma unroll
              for (int j = 0; j < kVec; ++j) acc[rr][t] = fmaf(w[j], hr[j], acc[rr][t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = r_base + warp * 4 + rr;
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        const float y = warp_sum(acc[rr][t]);
        if (lane == 0 && t < nt && r < a.d) {
          const int i = tok0 + t;
          const float scale = v.shared ? a.s_shared[i] : a.alpha[a.perm[v.row0 + i]];
          Y[(size_t)i * a.d + r] = scale * y;
        }
      }
    }
  }
}

// out[t] = r_attn[t] + ((sum over slots of Y[pos[t*k+s]]) + Ys[t])
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  const int t = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;  // float4 column
  if (c * 4 >= a.d) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < a.k; ++s) {
    const int p = a.pos[(size_t)t * a.k + s];
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

template <typename TW, typename TA>
static cudaError_t launch_gateup_t(const GemvArgs& a, cudaStream_t st) {
  const int slots = a.routed_slots + (a.has_shared ? 1 : 0);
  const size_t smem = (size_t)kTok * kKc * sizeof(float);
  const int wmax = a.has_shared && a.Is > a.I ? a.Is : a.I;
  static bool attr[64] = {};
  cudaError_t e = ensure_smem_limit(gemv_gateup_kernel<TW, TA>, (int)smem, attr);
  if (e != cudaSuccess) return e;
  gemv_gateup_kernel<TW, TA><<<dim3((wmax + kGuRows - 1) / kGuRows, slots), 256, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename TW>
static cudaError_t launch_down_t(const GemvArgs& a, cudaStream_t st) {
  const int slots = a.routed_slots + (a.has_shared ? 1 : 0);
  const size_t smem = (size_t)kTok * kKc * sizeof(float);
  static bool attr[64] = {};
  cudaError_t e = ensure_smem_limit(gemv_down_kernel<TW>, (int)smem, attr);
  if (e != cudaSuccess) return e;
  gemv_down_kernel<TW><<<dim3((a.d + kDnRows - 1) / kDnRows, slots), 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gemv_gateup(const GemvArgs& a, int act, int wdt, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (wdt == 0 && act == 0) return launch_gateup_t<float, float>(a, st);
  if (wdt == 1 && act == 1) return launch_gateup_t<__nv_bfloat16, __nv_bfloat16>(a, st);
  return cudaErrorNotSupported;
}

cudaError_t launch_gemv_down(const GemvArgs& a, int act, int wdt, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (wdt == 0 && act == 0) return launch_down_t<float>(a, st);
  if (wdt == 1 && act == 1) return launch_down_t<__nv_bfloat16>(a, st);
  return cudaErrorNotSupported;
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const int cols = a.d / 4;
  combine_kernel<<<dim3(a.T, (cols + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
