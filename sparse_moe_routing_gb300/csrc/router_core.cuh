// Router device code shared by the router kernels: the logit dot products
// z = W_router x (plus the shared-gate logit w_shared . x as column E) and
// the routing rule per token.
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
#pragma once

#include "common.cuh"
#include "kernels.h"

#include <math.h>

namespace moe {

// Dot products of one router row with up to KTOK tokens whose activation
// rows (nvec 16-byte chunks each, consecutive) start at xr (shared or global
// memory), by one whole warp; afterwards every lane holds the sums acc[t] for
// t < nt. kRouterU weight chunks per lane are held in registers while the
// tokens stream past. Split into one pass over kRouterU * 32 chunks
// (router_dots_pass, weights through a loader wl(c) -> chunk c) and the
// reduction (router_dots_reduce), so that a caller streaming the row through
// shared memory in passes of that size gets the same sums bit for bit.
constexpr int kRouterU = 8;

template <typename TA, int KTOK, typename WL>
__device__ __forceinline__ void router_dots_pass(WL wl, const uint4* xr, int nvec, int nt, int c0,
                                                 float* acc) {
  constexpr int kVec = Chunk<TA>::kVec;
  float w[kRouterU][kVec];
#pragma unroll
  for (int u = 0; u < kRouterU; ++u) {
    const int c = c0 + 32 * u;
    Chunk<TA>::unpack(c < nvec ? wl(c) : make_uint4(0, 0, 0, 0), w[u]);
  }
#pragma unroll
  for (int t = 0; t < KTOK; ++t) {
    if (t < nt) {
      const uint4* xt = xr + (size_t)t * nvec;
      uint4 xv[kRouterU];
#pragma unroll
      for (int u = 0; u < kRouterU; ++u) {
        const int c = c0 + 32 * u;
        xv[u] = c < nvec ? xt[c] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kRouterU; ++u) {
        float xf[kVec];
        Chunk<TA>::unpack(xv[u], xf);
#pragma unroll
        for (int j = 0; j < kVec; ++j) acc[t] = fmaf(w[u][j], xf[j], acc[t]);
      }
    }
  }
}

template <int KTOK>
__device__ __forceinline__ void router_dots_reduce(float* acc, int nt, int lane) {
  if (nt == 1) {
    acc[0] = warp_sum(acc[0]);
    return;
  }
  constexpr int NV = P2<KTOK>::v;
  float v[NV];
#pragma unroll
  for (int t = 0; t < NV; ++t) v[t] = t < KTOK ? acc[t] : 0.f;
  const float sum = reduce_multi<NV>(v, lane);
  // lane l holds the total of token l / (32 / NV); gather them to every lane
#pragma unroll
  for (int t = 0; t < KTOK; ++t) acc[t] = __shfl_sync(0xffffffffu, sum, t * (32 / NV));
}

template <typename TA, int KTOK>
__device__ __forceinline__ void router_row_dots(const TA* wrow, const uint4* xr, int nvec, int nt,
                                                int lane, float* acc) {
  constexpr int kVec = Chunk<TA>::kVec;
#pragma unroll
  for (int t = 0; t < KTOK; ++t) acc[t] = 0.f;
  auto wl = [&](int c) { return ldg_stream(wrow + (size_t)c * kVec); };
  for (int c0 = lane; c0 < nvec; c0 += 32 * kRouterU)
    router_dots_pass<TA, KTOK>(wl, xr, nvec, nt, c0, acc);
  router_dots_reduce<KTOK>(acc, nt, lane);
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

// Order-preserving map of a non-NaN float to an unsigned key (larger float,
// larger key; -0 and +0 map to the same key). Every float maps above 0, so 0
// marks an expert that can no longer be selected.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_key_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Compare-exchange of two (key, slot) candidates so that the first is the
// better one: larger key, or equal key and lower slot (= lower expert index,
// since lane l's slot j holds expert l + 32 j).
__device__ __forceinline__ void cas_desc(uint32_t& ka, int& ja, uint32_t& kb, int& jb) {
  const bool swap = kb > ka || (kb == ka && jb < ja);
  const uint32_t tk = swap ? kb : ka;
  const int tj = swap ? jb : ja;
  kb = swap ? ka : kb;
  jb = swap ? ja : jb;
  ka = tk;
  ja = tj;
}

// The routing rule for token t, run by one whole warp (lane = lane index);
// PL = experts per lane (E <= 32 PL, PL a power of two). Logits are read
// through L2 (ld.global.cg).
//
// Selection: each lane sorts its PL candidates (bitonic network, best
// first); each of the k rounds then takes the warp's best lane head with two
// redux instructions (largest key, then lowest expert among equal keys) and
// the owning lane pops its head.
template <int PL>
__device__ __forceinline__ void topk_token_pl(const TopkArgs& a, int t, int lane) {
  const float* z = a.logits + (size_t)t * (a.E + 1);
  const int E = a.E, k = a.k;

  float key[PL];   // ranking key per owned expert
  float val[PL];   // softmax: logit; sigmoid: raw score s
  // every load issued before the first use (partial sums: two parts at most)
  float z0[PL], z1[PL];
  const bool two = a.nparts > 1;
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    const int e = lane + 32 * j;
    z0[j] = e < E ? __ldcg(z + e) : -INFINITY;
    z1[j] = (two && e < E) ? __ldcg(z + a.part_stride + e) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    int e = lane + 32 * j;
    const float zv = two ? z0[j] + z1[j] : z0[j];
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
  uint32_t taken = 0;  // bit j: expert lane+32j cannot be selected
#pragma unroll
  for (int j = 0; j < PL; ++j)
    if (lane + 32 * j >= E) taken |= 1u << j;

  if (a.kind == 1) {
    // group ranking: group g scores the sum of its two largest selection
    // scores (all members when a group has one member)
    const int G = E / a.n_group;
    uint32_t kept = 0;
    float my_gscore = -INFINITY;
    for (int g = 0; g < a.n_group; ++g) {
      float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
      for (int j = 0; j < PL; ++j) {
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
    const float gscore = lane < a.n_group ? my_gscore : -INFINITY;
    for (int r = 0; r < a.topk_group; ++r) {
      float v = lane < a.n_group ? gscore : -INFINITY;
      int i = lane < a.n_group ? lane : 0x7fffffff;
      if (lane < a.n_group && ((kept >> lane) & 1u)) { v = -INFINITY; i = 0x7fffffff; }
      warp_argmax(v, i);
      if (i < a.n_group) kept |= 1u << i;
    }
#pragma unroll
    for (int j = 0; j < PL; ++j) {
      int e = lane + 32 * j;
      if (e < E && !((kept >> (e / G)) & 1u)) taken |= 1u << j;
    }
  }

  // per-lane candidates, best first
  uint32_t ck[PL];
  int cj[PL];
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    ck[j] = ((taken >> j) & 1u) ? 0u : order_key(key[j]);
    cj[j] = j;
  }
#pragma unroll
  for (int size = 2; size <= PL; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int l = i ^ stride;
        if (l > i) {
          if ((i & size) == 0) cas_desc(ck[i], cj[i], ck[l], cj[l]);
          else cas_desc(ck[l], cj[l], ck[i], cj[i]);
        }
      }
    }
  }

  int my_id = 0;
  float my_val = 0.f;
  for (int s = 0; s < k; ++s) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, ck[0]);
    const uint32_t cand = ck[0] == m ? (uint32_t)(lane + 32 * cj[0]) : 0xffffffffu;
    // m == 0 (no candidate left) is unreachable for validated shapes
    const int i = (int)__reduce_min_sync(0xffffffffu, cand);
    const int owner = i & 31, jj = i >> 5;
    float sv = 0.f;
#pragma unroll
    for (int j = 0; j < PL; ++j)
      if (j == jj) sv = val[j];
    sv = __shfl_sync(0xffffffffu, sv, owner);
    if (lane == owner) {  // pop the head
#pragma unroll
      for (int j = 0; j + 1 < PL; ++j) {
        ck[j] = ck[j + 1];
        cj[j] = cj[j + 1];
      }
      ck[PL - 1] = 0u;
    }
    if (lane == s) { my_id = i; my_val = sv; }
  }

  float w;
  if (a.kind == 0) {
    // softmax over all E logits; renormalise the selected probabilities
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < PL; ++j)
      if (lane + 32 * j < E) m = fmaxf(m, val[j]);
    m = order_key_inv(__reduce_max_sync(0xffffffffu, order_key(rank_key(m))));
    float S = 0.f;
#pragma unroll
    for (int j = 0; j < PL; ++j)
      if (lane + 32 * j < E) S += expf(val[j] - m);
    S = warp_sum(S);
    float p = lane < k ? expf(my_val - m) / S : 0.f;
    float denom = fmaxf(warp_sum(p), a.renorm_clamp);
    w = p / denom * a.routed_scaling;
  } else {
    float sel = lane < k ? my_val : 0.f;
    float denom = fmaxf(warp_sum(sel), 1.17549435e-38f);
    w = sel / denom * a.routed_scaling;
  }
  if (lane < k) {
    a.topk_ids[(size_t)t * k + lane] = my_id;
    a.weights[(size_t)t * k + lane] = w;
  }
  if (lane == 0 && a.s_shared && a.has_shared_logit)
    a.s_shared[t] = 1.0f / (1.0f + expf(-__ldcg(z + E)));
}

}  // namespace moe
