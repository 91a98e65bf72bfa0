// Direct-load grouped expert GEMV for batches of at most kGemvSmallTokens
// tokens (the same math as the streaming GEMV: "How Treebeard routes Qwen3.6
// MoE tokens", "Routed expert computation" and "Shared expert computation";
// Edge0 "Experts").
//
// With a few tokens an expert sees at most that many tokens, so each
// weight row feeds one dot product per token and the layer is a pure weight
// stream. Here one warp owns one gate/up row pair (or four down rows) and
// streams it with 16-byte no-allocate loads, kUnroll chunks per lane in
// flight, and no shared memory, barriers or waits: a whole layer's rows fit
// in one wave of warps, so the HBM queue is kept full by the number of warps
// rather than by a software pipeline. Activations (a few KB per token) are
// read through L1.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarps = 8;          // warps per CTA
constexpr int kUnroll = 4;         // 16-byte chunks per lane per row in flight
constexpr int kDnRows = 4;         // down rows per warp

struct SGroup {
  bool ok, shared;
  int g, n, row0, width;
};

// Group slot -> routed expert (active list order; or, in pair mode, the
// pair's expert) or the shared expert.
__device__ __forceinline__ SGroup group_at(const GemvArgs& a, int slot) {
  SGroup v{};
  if (a.pair_ids && slot < a.routed_slots) {
    v.g = a.pair_ids[slot];
    if (v.g < 0 || v.g >= a.E) {
      if (threadIdx.x == 0) report(a.ctrl, kDevBadId, kSiteGemvGateUp);
      return v;
    }
    v.row0 = slot;
    v.n = 1;
    v.width = a.I;
    v.ok = true;
    return v;
  }
  if (slot < a.routed_slots) {
    if (slot >= *a.n_active) return v;
    v.g = a.active[slot];
    v.row0 = a.offsets[v.g];
    v.n = a.offsets[v.g + 1] - v.row0;
    v.width = a.I;
  } else {
    v.shared = true;
    v.g = a.E;
    v.n = a.T;
    v.width = a.Is;
  }
  v.ok = v.n > 0;
  return v;
}

__device__ __forceinline__ void put(float* p, float v) { *p = v; }
__device__ __forceinline__ void put(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// h[i][row] = SiLU(W_gate[row] . x_i) * (W_up[row] . x_i) for the group's
// tokens i in [j0, j0 + nj), nj <= NT; one whole warp.
template <typename TW, int NT>
__device__ __forceinline__ void gateup_rows(const GemvArgs& a, const SGroup& v, int row,
                                            const TW* wg, const TW* wu, int j0, int nj,
                                            int lane) {
  constexpr int kVec = Chunk<TW>::kVec;
  const uint4* xr[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int i = j0 + j;
    int tok = 0;
    if (j < nj) tok = v.shared ? i : (a.pair_ids ? v.row0 + i : a.perm[v.row0 + i]) / a.k;
    xr[j] = reinterpret_cast<const uint4*>(static_cast<const TW*>(a.x) + (size_t)tok * a.d);
  }
  constexpr int NV = P2<2 * NT>::v;
  float acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0.f;
  const int nvec = a.d / kVec;
  for (int c0 = lane; c0 < nvec; c0 += 32 * kUnroll) {
    uint4 g4[kUnroll], u4[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + 32 * u;
      const bool in = c < nvec;
      g4[u] = in ? ldg_stream(wg + (size_t)c * kVec) : make_uint4(0, 0, 0, 0);
      u4[u] = in ? ldg_stream(wu + (size_t)c * kVec) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + 32 * u;
      if (c < nvec) {
        float gf[kVec], uf[kVec];
        Chunk<TW>::unpack(g4[u], gf);
        Chunk<TW>::unpack(u4[u], uf);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (j < nj) {
            float xf[kVec];
            Chunk<TW>::unpack(__ldg(xr[j] + c), xf);
#pragma unroll
            for (int e = 0; e < kVec; ++e) {
              acc[2 * j] = fmaf(gf[e], xf[e], acc[2 * j]);
              acc[2 * j + 1] = fmaf(uf[e], xf[e], acc[2 * j + 1]);
            }
          }
        }
      }
    }
  }
  const float sum = reduce_multi<NV>(acc, lane);
  const int per = 32 / NV;
  const int idx = lane / per;  // value index this lane holds: 2j gate, 2j+1 up
  const float up = __shfl_down_sync(0xffffffffu, sum, per);
  if ((lane % per) == 0 && (idx & 1) == 0 && idx / 2 < nj) {
    const int i = j0 + idx / 2;
    TW* H = static_cast<TW*>(v.shared ? a.Hs : a.H) +
            (v.shared ? (size_t)i * a.Is : (size_t)(v.row0 + i) * a.I);
    put(H + row, siluf_(sum) * up);
  }
}

template <typename TW, int NT>
__global__ void __launch_bounds__(kWarps * 32) gemv_small_gateup(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  const SGroup v = group_at(a, blockIdx.y);
  if (!v.ok) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  if (row >= v.width) return;
  const size_t rbase = v.shared ? (size_t)row * a.d : ((size_t)v.g * a.I + row) * a.d;
  const TW* wg = static_cast<const TW*>(v.shared ? a.Wsg : a.Wg) + rbase;
  const TW* wu = static_cast<const TW*>(v.shared ? a.Wsu : a.Wu) + rbase;
  // a group holds at most NT tokens unless a caller's ids repeat an expert
  // within a token; such groups are processed NT tokens at a time
  for (int j0 = 0; j0 < v.n; j0 += NT)
    gateup_rows<TW, NT>(a, v, row, wg, wu, j0, min(NT, v.n - j0), lane);
}

// scale_i * (W_down[col] . h_i) for kDnRows consecutive columns col0.. and
// the group's tokens i in [j0, j0 + nj); scale = the routing weight (routed)
// or the shared gate; one whole warp. put(r, i, value) stores each result
// (called by one lane per (column, token)).
template <typename TW, int NT, typename Put>
__device__ __forceinline__ void down_dots(const GemvArgs& a, const SGroup& v, int nr, const TW* Wd,
                                          const TW* Hb, int j0, int nj, int lane, Put put_result) {
  constexpr int kVec = Chunk<TW>::kVec;
  const int K = v.width;
  constexpr int NV = P2<kDnRows * NT>::v;
  float acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0.f;
  const int nvec = K / kVec;
  for (int c = lane; c < nvec; c += 32) {
    uint4 w4[kDnRows];
#pragma unroll
    for (int r = 0; r < kDnRows; ++r)
      w4[r] = r < nr ? ldg_stream(Wd + (size_t)r * K + (size_t)c * kVec) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (j < nj) {
        float hf[kVec];
        Chunk<TW>::unpack(__ldg(reinterpret_cast<const uint4*>(Hb + (size_t)(j0 + j) * K) + c),
                          hf);
#pragma unroll
        for (int r = 0; r < kDnRows; ++r) {
          float wf[kVec];
          Chunk<TW>::unpack(w4[r], wf);
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc[r * NT + j] = fmaf(wf[e], hf[e], acc[r * NT + j]);
        }
      }
    }
  }
  const float sum = reduce_multi<NV>(acc, lane);
  const int per = 32 / NV;
  const int idx = lane / per;
  if ((lane % per) == 0 && idx < kDnRows * NT) {
    const int r = idx / NT, j = idx - r * NT;
    if (r < nr && j < nj) {
      const int i = j0 + j;
      const float scale = v.shared ? a.s_shared[i]
                                   : a.alpha[a.pair_ids ? v.row0 + i : a.perm[v.row0 + i]];
      put_result(r, i, scale * sum);
    }
  }
}

// Y[i][col] for the group's tokens (packed rows, or token rows of Ys).
template <typename TW, int NT>
__device__ __forceinline__ void down_rows(const GemvArgs& a, const SGroup& v, int col0, int nr,
                                          const TW* Wd, const TW* Hb, int j0, int nj, int lane) {
  down_dots<TW, NT>(a, v, nr, Wd, Hb, j0, nj, lane, [&](int r, int i, float y) {
    float* Y = v.shared ? a.Ys + (size_t)i * a.d : a.Y + (size_t)(v.row0 + i) * a.d;
    Y[col0 + r] = y;
  });
}

template <typename TW, int NT>
__global__ void __launch_bounds__(kWarps * 32) gemv_small_down(GemvArgs a) {
  pdl_wait();
  pdl_trigger();
  const SGroup v = group_at(a, blockIdx.y);
  if (!v.ok) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = (blockIdx.x * kWarps + warp) * kDnRows;
  if (col0 >= a.d) return;
  const TW* Wd = static_cast<const TW*>(v.shared ? a.Wsd : a.Wd) +
                 (v.shared ? 0 : (size_t)v.g * a.d * a.I) + (size_t)col0 * v.width;
  const TW* Hb = static_cast<const TW*>(v.shared ? a.Hs : a.H) +
                 (v.shared ? 0 : (size_t)v.row0 * a.I);
  const int nr = min(kDnRows, a.d - col0);
  for (int j0 = 0; j0 < v.n; j0 += NT)
    down_rows<TW, NT>(a, v, col0, nr, Wd, Hb, j0, min(NT, v.n - j0), lane);
}

// Down + combine for pair groups: CTA b owns the kDnRows output columns
// 4b.. of every token; its warps compute those columns for every (token,
// slot) pair and for the shared expert (warp w: groups w, w + kWarps, ...),
// then the CTA adds them as the combine kernel does: out[t] = r_attn[t] +
// ((sum over slots s, in slot order) + shared). The same products and the
// same summation order, so the results are those of the two-kernel path.
constexpr int kDcMaxGroups = 2 * kWarps;
template <typename TW, int NT>
__global__ void __launch_bounds__(kWarps * 32) gemv_small_down_combine(GemvArgs a) {
  __shared__ float sy[kDcMaxGroups][kDnRows];                   // pair p = t * k + s
  __shared__ float sys[kGemvSmallTokens][kDnRows];             // shared expert, token t
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = blockIdx.x * kDnRows;
  const int nr = min(kDnRows, a.d - col0);
  for (int i = threadIdx.x; i < kDcMaxGroups * kDnRows; i += kWarps * 32) (&sy[0][0])[i] = 0.f;
  for (int i = threadIdx.x; i < kGemvSmallTokens * kDnRows; i += kWarps * 32) (&sys[0][0])[i] = 0.f;
  __syncthreads();
  const int G = a.routed_slots + (a.has_shared ? 1 : 0);
  for (int gi = warp; gi < G; gi += kWarps) {
    const SGroup v = group_at(a, gi);
    if (!v.ok) continue;  // a bad id (reported): the pair adds nothing
    const TW* Wd = static_cast<const TW*>(v.shared ? a.Wsd : a.Wd) +
                   (v.shared ? 0 : (size_t)v.g * a.d * a.I) + (size_t)col0 * v.width;
    const TW* Hb = static_cast<const TW*>(v.shared ? a.Hs : a.H) +
                   (v.shared ? 0 : (size_t)v.row0 * a.I);
    for (int j0 = 0; j0 < v.n; j0 += NT)
      down_dots<TW, NT>(a, v, nr, Wd, Hb, j0, min(NT, v.n - j0), lane, [&](int r, int i, float y) {
        if (v.shared) sys[i][r] = y;
        else sy[gi][r] = y;
      });
  }
  __syncthreads();
  if (threadIdx.x < a.T * kDnRows) {
    const int t = threadIdx.x / kDnRows, r = threadIdx.x - t * kDnRows;
    if (r < nr) {
      float acc = 0.f;
      for (int s = 0; s < a.k; ++s) acc += sy[t * a.k + s][r];
      if (a.has_shared) acc += sys[t][r];
      const size_t o = (size_t)t * a.d + col0 + r;
      a.out[o] = a.r_attn[o] + acc;
    }
  }
}

template <typename TW, int NT>
cudaError_t launch_small(const GemvArgs& a, bool down, cudaStream_t st) {
  const int slots = a.routed_slots + (a.has_shared ? 1 : 0);
  if (down) {
    const int cols_per_cta = kWarps * kDnRows;
    return launch_pdl(gemv_small_down<TW, NT>, dim3((a.d + cols_per_cta - 1) / cols_per_cta, slots),
                      kWarps * 32, 0, st, a);
  }
  const int wmax = a.has_shared && a.Is > a.I ? a.Is : a.I;
  return launch_pdl(gemv_small_gateup<TW, NT>, dim3((wmax + kWarps - 1) / kWarps, slots),
                    kWarps * 32, 0, st, a);
}

template <typename TW>
cudaError_t dispatch(const GemvArgs& a, bool down, cudaStream_t st) {
  // tokens per pass: the batch rounded up to a power of two (a routed pair
  // group holds one token; the shared expert holds all T)
  if (a.T <= 1) return launch_small<TW, 1>(a, down, st);
  if (a.T <= 2) return launch_small<TW, 2>(a, down, st);
  if (a.T <= 4) return launch_small<TW, 4>(a, down, st);
  if (a.T <= 8) return launch_small<TW, 8>(a, down, st);
  return cudaErrorInvalidValue;
}

}  // namespace

bool gemv_small_down_combine_ok(const GemvArgs& a) {
  return a.pair_ids != nullptr && a.T >= 1 && a.T <= kGemvSmallTokens &&
         a.routed_slots + (a.has_shared ? 1 : 0) <= kDcMaxGroups && a.d % kDnRows == 0;
}

cudaError_t launch_gemv_small_down_combine(const GemvArgs& a, int act, int wdt, cudaStream_t st) {
  if (!gemv_small_down_combine_ok(a) || a.d % 8 != 0 || a.I % 8 != 0 || a.Is % 8 != 0)
    return cudaErrorInvalidValue;
  const dim3 grid(a.d / kDnRows);
  if (wdt == 0 && act == 0) {
    if (a.T <= 1) return launch_pdl(gemv_small_down_combine<float, 1>, grid, kWarps * 32, 0, st, a);
    if (a.T <= 2) return launch_pdl(gemv_small_down_combine<float, 2>, grid, kWarps * 32, 0, st, a);
    if (a.T <= 4) return launch_pdl(gemv_small_down_combine<float, 4>, grid, kWarps * 32, 0, st, a);
    return launch_pdl(gemv_small_down_combine<float, 8>, grid, kWarps * 32, 0, st, a);
  }
  if (wdt == 1 && act == 1) {
    using B = __nv_bfloat16;
    if (a.T <= 1) return launch_pdl(gemv_small_down_combine<B, 1>, grid, kWarps * 32, 0, st, a);
    if (a.T <= 2) return launch_pdl(gemv_small_down_combine<B, 2>, grid, kWarps * 32, 0, st, a);
    if (a.T <= 4) return launch_pdl(gemv_small_down_combine<B, 4>, grid, kWarps * 32, 0, st, a);
    return launch_pdl(gemv_small_down_combine<B, 8>, grid, kWarps * 32, 0, st, a);
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_gemv_small(const GemvArgs& a, int act, int wdt, bool down, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (a.T > kGemvSmallTokens || a.d % 8 != 0 || a.I % 8 != 0 || a.Is % 8 != 0)
    return cudaErrorInvalidValue;
  if (wdt == 0 && act == 0) return dispatch<float>(a, down, st);
  if (wdt == 1 && act == 1) return dispatch<__nv_bfloat16>(a, down, st);
  return cudaErrorNotSupported;
}

}  // namespace moe
