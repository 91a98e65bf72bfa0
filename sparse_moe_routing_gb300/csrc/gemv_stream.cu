// Weight-streaming grouped expert GEMV (decode path), bulk-copy fed.
//
// Routed expert ("How Treebeard routes Qwen3.6 MoE tokens", "Routed expert
// computation"; Edge0 "Experts"): h = SiLU(W_gate x) * (W_up x), and
// e = alpha * W_down h (alpha = the routing weight, or the shared expert's
// sigmoid gate, "Shared expert computation").
//
// Organisation follows the packing of the bucketing pass ("Intel SYCL path":
// launch over active experts, reuse each loaded weight block across all of
// the expert's tokens). CTA = (group slot, block of weight rows). One
// producer warp streams the block's weight rows from HBM into shared memory
// with cp.async.bulk (the copy engine moves the bytes; no registers are tied
// up by loads in flight), completion tracked by mbarrier transaction counts.
// Eight consumer warps stage the group's activations (up to 8 tokens) once,
// then compute dot products from shared memory.
//
// Each consumer warp owns a private sub-ring of kSW stages and consumes its
// own units strictly in order, so no consumer ever waits on a phase more than
// one ahead of its stage (a parity wait cannot alias). A unit belongs to the
// warp row % 8 and lands in that warp's stage j % kSW, where j counts the
// warp's units in (token chunk, row, K segment) order; producer lane w fills
// warp w's sub-ring in the same order, independently of the other lanes.
//
// The token count is a template parameter and partial sums are reduced with a
// multi-value butterfly (N values across 32 lanes in N-1+log2(32/N) shuffles).
// Every wait is bounded (about one second; then the CTA records kDevTimeout
// in the workspace status word, stops waiting, lets in-flight copies land and
// returns).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kConsumers = 8;                      // consumer warps
constexpr int kStreamThreads = (kConsumers + 1) * 32;
constexpr int kSW = 2;                             // stages per consumer warp
constexpr int kStageBytes = 4096;                  // bytes per stage
constexpr int kStages = kConsumers * kSW;
constexpr int kRing = kStages * kStageBytes;       // 64 KB
constexpr int kTokMax = 8;
constexpr int kDnRows = 4;                         // down rows per unit

// ---------------------------------------------------------------------------
// mbarrier / bulk-copy wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void bar_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait by one lane: false if the CTA is aborting or the wait timed
// out (then the abort flag is raised and the timeout recorded).
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                         Ctrl* ctrl, uint32_t site) {
  if (bar_try(b, parity)) return true;
  const uint64_t t0 = gtimer();
  uint32_t n = 0;
  while (!bar_try(b, parity)) {
    if ((++n & 31u) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > 1000000000ull) {
        *abort_flag = 1;
        report(ctrl, kDevTimeout, site);
        return false;
      }
    }
  }
  return true;
}
// Warp-wide bounded wait: lane 0 waits, the outcome is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          Ctrl* ctrl, uint32_t site) {
  const int lane = threadIdx.x & 31;
  bool ok = lane == 0 ? bar_wait(b, parity, abort_flag, ctrl, site) : true;
  return __shfl_sync(0xffffffffu, ok, 0);
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(b))
      : "memory");
}
// named barrier among the consumer warps only (the producer never joins)
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

// ---------------------------------------------------------------------------
// groups, reductions, element access
// ---------------------------------------------------------------------------
struct Group {
  bool ok, shared;
  int g, n, row0, width;
};

__device__ __forceinline__ Group group_of(const GemvArgs& a, int slot) {
  Group v{};
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

// 8-element chunk c of a row (bf16 or f32) in shared memory, as floats
template <typename TW> struct Ch;
template <> struct Ch<__nv_bfloat16> {
  __device__ __forceinline__ static void get(const void* row, int c, float* w) {
    const uint4 v = reinterpret_cast<const uint4*>(row)[c];
    w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
  }
};
template <> struct Ch<float> {
  __device__ __forceinline__ static void get(const void* row, int c, float* w) {
    const float4 a = reinterpret_cast<const float4*>(row)[2 * c];
    const float4 b = reinterpret_cast<const float4*>(row)[2 * c + 1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
};

__device__ __forceinline__ float dot8(const float* w, const float* x, float acc) {
#pragma unroll
  for (int j = 0; j < 8; ++j) acc = fmaf(w[j], x[j], acc);
  return acc;
}

__device__ __forceinline__ void store_h(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_h(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Copies rows [tok0, tok0+nt) x [0, K) of the activations into xs (consumer
// threads only), 16 bytes at a time. by_token: rows of x through the group's
// tokens; else rows of H.
template <typename TS>
__device__ __forceinline__ void stage(const TS* src, const GemvArgs& a, const Group& v, int tok0,
                                      int nt, int K, bool by_token, TS* xs) {
  constexpr int kPer = 16 / sizeof(TS);
  const int nvec = K / kPer;
  for (int idx = threadIdx.x; idx < nt * nvec; idx += kConsumers * 32) {
    const int t = idx / nvec, c = idx - t * nvec;
    size_t row = (size_t)(tok0 + t);
    if (by_token && !v.shared) row = (size_t)(a.perm[v.row0 + tok0 + t] / a.k);
    reinterpret_cast<uint4*>(xs + (size_t)t * K)[c] =
        __ldg(reinterpret_cast<const uint4*>(src + row * K) + c);
  }
}

struct Smem {
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  volatile int* abort_flag;
  void* xs;
};

constexpr size_t kFixed = kRing + 2 * kStages * 8 + 16;

__device__ __forceinline__ Smem carve(uint8_t* base) {
  Smem s;
  s.ring = base;
  s.full = reinterpret_cast<uint64_t*>(base + kRing);
  s.empty = s.full + kStages;
  s.abort_flag = reinterpret_cast<volatile int*>(s.empty + kStages);
  s.xs = base + kFixed;
  return s;
}

__device__ __forceinline__ void init_bars(Smem& s) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      bar_init(&s.full[i], 1);
      bar_init(&s.empty[i], 1);
    }
    *s.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
}

__device__ __forceinline__ void finish(const Smem& s) {
  __syncthreads();
  if (*s.abort_flag && threadIdx.x == 0) {
    // let copies already in flight land before the CTA exits
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 2000000ull) {
    }
  }
  __syncthreads();
}

// stage and parity of the j-th unit of consumer warp w
__device__ __forceinline__ int stage_of(int w, int j) { return w * kSW + (j % kSW); }
__device__ __forceinline__ uint32_t parity_of(int j) { return (uint32_t)((j / kSW) & 1); }

// number of items i in [0, n) with i % kConsumers == w
__device__ __forceinline__ int items_of_warp(int n, int w) {
  return w < n ? (n - w + kConsumers - 1) / kConsumers : 0;
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU. Unit = (token chunk, row, K segment): the gate and the up
// segment of one row (kseg elements each).
// ---------------------------------------------------------------------------
template <int NT, typename TW>
__device__ __forceinline__ void gateup_consume(const GemvArgs& a, Smem& s, int chunk_idx,
                                               int nrows, int nseg, int kseg, int r_base, TW* H,
                                               int ldh, int tok0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TW* xs = static_cast<const TW*>(s.xs);
  const int seg_bytes = kseg * (int)sizeof(TW);
  const int my_rows = items_of_warp(nrows, warp);
  constexpr int NV = P2<2 * NT>::v;
  for (int rr = 0; rr < my_rows; ++rr) {
    const int row = warp + rr * kConsumers;
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0.f;
    for (int seg = 0; seg < nseg; ++seg) {
      const int j = (chunk_idx * my_rows + rr) * nseg + seg;
      const int st = stage_of(warp, j);
      const bool ok = warp_wait(&s.full[st], parity_of(j), s.abort_flag, a.ctrl, kSiteGemvGateUp);
      if (ok) {
        const uint8_t* g = s.ring + (size_t)st * kStageBytes;
        const uint8_t* u = g + seg_bytes;
        const int k0 = seg * kseg;
        const int cn = min(kseg, a.d - k0) / 8;
        for (int c = lane; c < cn; c += 32) {
          float wg[8], wu[8];
          Ch<TW>::get(g, c, wg);
          Ch<TW>::get(u, c, wu);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            float x[8];
            Ch<TW>::get(xs + (size_t)t * a.d + k0, c, x);
            acc[2 * t] = dot8(wg, x, acc[2 * t]);
            acc[2 * t + 1] = dot8(wu, x, acc[2 * t + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) bar_arrive(&s.empty[st]);
    }
    const float sum = reduce_multi<NV>(acc, lane);
    const int per = 32 / NV;
    const int idx = lane / per;
    const float up = __shfl_down_sync(0xffffffffu, sum, per);
    if ((lane % per) == 0 && (idx & 1) == 0 && idx / 2 < NT && !*s.abort_flag)
      store_h(H + (size_t)(tok0 + idx / 2) * ldh + r_base + row, siluf_(sum) * up);
  }
}

template <typename TW>
__global__ void __launch_bounds__(kStreamThreads, 2)
    gemv_gateup_stream(GemvArgs a, int rows_per_cta, int tok_chunk, int kseg) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  const Group v = group_of(a, blockIdx.y);
  if (!v.ok) return;
  const int r_base = blockIdx.x * rows_per_cta;
  if (r_base >= v.width) return;
  const int nrows = min(v.width, r_base + rows_per_cta) - r_base;
  const int nseg = (a.d + kseg - 1) / kseg;
  Smem s = carve(smem);
  init_bars(s);

  const TW* Wg = static_cast<const TW*>(v.shared ? a.Wsg : a.Wg);
  const TW* Wu = static_cast<const TW*>(v.shared ? a.Wsu : a.Wu);
  if (!v.shared) {
    Wg += (size_t)v.g * a.I * a.d;
    Wu += (size_t)v.g * a.I * a.d;
  }
  TW* H = static_cast<TW*>(v.shared ? a.Hs : a.H) + (v.shared ? 0 : (size_t)v.row0 * a.I);
  const int n_chunks = (v.n + tok_chunk - 1) / tok_chunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumers) {
    // ---------------------------------------------------------------- producer
    // Lane w refills consumer warp w's sub-ring, in that warp's unit order,
    // independently of the other lanes (no head-of-line blocking).
    if (lane < kConsumers) {
      const int w = lane;
      const int my_rows = items_of_warp(nrows, w);
      int j = 0;
      bool alive = true;
      for (int ch = 0; ch < n_chunks && alive; ++ch) {
        for (int rr = 0; rr < my_rows && alive; ++rr) {
          const int row = w + rr * kConsumers;
          for (int seg = 0; seg < nseg; ++seg, ++j) {
            const int st = stage_of(w, j);
            if (!bar_wait(&s.empty[st], parity_of(j) ^ 1u, s.abort_flag, a.ctrl,
                          kSiteGemvGateUp)) {
              alive = false;
              break;
            }
            const int k0 = seg * kseg;
            const uint32_t bytes = (uint32_t)(min(kseg, a.d - k0) * sizeof(TW));
            uint8_t* dst = s.ring + (size_t)st * kStageBytes;
            const size_t off = (size_t)(r_base + row) * a.d + k0;
            bar_expect(&s.full[st], 2 * bytes);
            bulk_g2s(dst, Wg + off, bytes, &s.full[st]);
            bulk_g2s(dst + (size_t)kseg * sizeof(TW), Wu + off, bytes, &s.full[st]);
          }
        }
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------------- consumers
    for (int ch = 0; ch < n_chunks; ++ch) {
      const int tok0 = ch * tok_chunk;
      const int nt = min(tok_chunk, v.n - tok0);
      consumers_sync();
      stage<TW>(static_cast<const TW*>(a.x), a, v, tok0, nt, a.d, true, static_cast<TW*>(s.xs));
      consumers_sync();
      switch (nt) {
        case 1: gateup_consume<1, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
        case 2: gateup_consume<2, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
        case 3: gateup_consume<3, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
        case 4: gateup_consume<4, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
        case 5: gateup_consume<5, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
        case 6: gateup_consume<6, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
        case 7: gateup_consume<7, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
        default: gateup_consume<8, TW>(a, s, ch, nrows, nseg, kseg, r_base, H, v.width, tok0); break;
      }
    }
  }
  finish(s);
}

// ---------------------------------------------------------------------------
// down x alpha. Unit = (token chunk, group of kDnRows rows, K segment).
// ---------------------------------------------------------------------------
template <int NT, typename TW>
__device__ __forceinline__ void down_consume(const GemvArgs& a, Smem& s, int chunk_idx,
                                             int ngroups, int nrows, int nseg, int kseg, int K,
                                             int r_base, float* Y, int tok0, const float* scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TW* hs = static_cast<const TW*>(s.xs);
  const int seg_bytes = kseg * (int)sizeof(TW);
  const int my_groups = items_of_warp(ngroups, warp);
  constexpr int NV = P2<kDnRows * NT>::v;
  for (int gi = 0; gi < my_groups; ++gi) {
    const int grp = warp + gi * kConsumers;
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0.f;
    for (int seg = 0; seg < nseg; ++seg) {
      const int j = (chunk_idx * my_groups + gi) * nseg + seg;
      const int st = stage_of(warp, j);
      const bool ok = warp_wait(&s.full[st], parity_of(j), s.abort_flag, a.ctrl, kSiteGemvDown);
      if (ok) {
        const uint8_t* base = s.ring + (size_t)st * kStageBytes;
        const int k0 = seg * kseg;
        const int cn = min(kseg, K - k0) / 8;
        for (int c = lane; c < cn; c += 32) {
          float h[NT][8];
#pragma unroll
          for (int t = 0; t < NT; ++t) Ch<TW>::get(hs + (size_t)t * K + k0, c, h[t]);
#pragma unroll
          for (int r = 0; r < kDnRows; ++r) {
            float w[8];
            Ch<TW>::get(base + (size_t)r * seg_bytes, c, w);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r * NT + t] = dot8(w, h[t], acc[r * NT + t]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) bar_arrive(&s.empty[st]);
    }
    const float sum = reduce_multi<NV>(acc, lane);
    const int per = 32 / NV;
    const int idx = lane / per;
    if ((lane % per) == 0 && idx < kDnRows * NT && !*s.abort_flag) {
      const int r = idx / NT, t = idx - r * NT;
      const int row = grp * kDnRows + r;
      if (row < nrows) Y[(size_t)(tok0 + t) * a.d + r_base + row] = scale[t] * sum;
    }
  }
}

template <typename TW>
__global__ void __launch_bounds__(kStreamThreads, 2)
    gemv_down_stream(GemvArgs a, int rows_per_cta, int tok_chunk, int kseg) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float scale[kTokMax];
  pdl_wait();
  pdl_trigger();
  const Group v = group_of(a, blockIdx.y);
  if (!v.ok) return;
  const int r_base = blockIdx.x * rows_per_cta;
  if (r_base >= a.d) return;
  const int nrows = min(a.d, r_base + rows_per_cta) - r_base;  // multiple of kDnRows
  const int ngroups = nrows / kDnRows;
  const int K = v.width;
  const int nseg = (K + kseg - 1) / kseg;
  Smem s = carve(smem);
  init_bars(s);

  const TW* Wd = static_cast<const TW*>(v.shared ? a.Wsd : a.Wd);
  if (!v.shared) Wd += (size_t)v.g * a.d * a.I;
  const TW* H =
      static_cast<const TW*>(v.shared ? a.Hs : a.H) + (v.shared ? 0 : (size_t)v.row0 * a.I);
  float* Y = v.shared ? a.Ys : a.Y + (size_t)v.row0 * a.d;
  const int n_chunks = (v.n + tok_chunk - 1) / tok_chunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumers) {
    // producer: lane w refills consumer warp w's sub-ring independently
    if (lane < kConsumers) {
      const int w = lane;
      const int my_groups = items_of_warp(ngroups, w);
      int j = 0;
      bool alive = true;
      for (int ch = 0; ch < n_chunks && alive; ++ch) {
        for (int gi = 0; gi < my_groups && alive; ++gi) {
          const int grp = w + gi * kConsumers;
          for (int seg = 0; seg < nseg; ++seg, ++j) {
            const int st = stage_of(w, j);
            if (!bar_wait(&s.empty[st], parity_of(j) ^ 1u, s.abort_flag, a.ctrl, kSiteGemvDown)) {
              alive = false;
              break;
            }
            const int k0 = seg * kseg;
            const int len = min(kseg, K - k0);
            const uint32_t bytes = (uint32_t)(len * sizeof(TW));
            uint8_t* dst = s.ring + (size_t)st * kStageBytes;
            const int row0 = r_base + grp * kDnRows;
            bar_expect(&s.full[st], kDnRows * bytes);
            if (len == K) {
              // whole rows: the unit's rows are contiguous in the bank
              bulk_g2s(dst, Wd + (size_t)row0 * K, kDnRows * bytes, &s.full[st]);
            } else {
              for (int r = 0; r < kDnRows; ++r)
                bulk_g2s(dst + (size_t)r * kseg * sizeof(TW), Wd + (size_t)(row0 + r) * K + k0,
                         bytes, &s.full[st]);
            }
          }
        }
      }
    }
    __syncwarp();
  } else {
    for (int ch = 0; ch < n_chunks; ++ch) {
      const int tok0 = ch * tok_chunk;
      const int nt = min(tok_chunk, v.n - tok0);
      consumers_sync();
      stage<TW>(H, a, v, tok0, nt, K, false, static_cast<TW*>(s.xs));
      if (threadIdx.x < nt) {
        const int i = tok0 + threadIdx.x;
        scale[threadIdx.x] = v.shared ? a.s_shared[i] : a.alpha[a.perm[v.row0 + i]];
      }
      consumers_sync();
      switch (nt) {
        case 1: down_consume<1, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
        case 2: down_consume<2, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
        case 3: down_consume<3, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
        case 4: down_consume<4, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
        case 5: down_consume<5, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
        case 6: down_consume<6, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
        case 7: down_consume<7, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
        default: down_consume<8, TW>(a, s, ch, ngroups, nrows, nseg, kseg, K, r_base, Y, tok0, scale); break;
      }
    }
  }
  finish(s);
}

// ---------------------------------------------------------------------------
// launch geometry
// ---------------------------------------------------------------------------
constexpr size_t kSmemCap = 227 * 1024;

int rows_for(int rows, int slots, int granule, int cap) {
  const long target = 4L * tc_sm_count();
  long per = ((long)rows * slots + target - 1) / target;
  per = ((per + granule - 1) / granule) * granule;
  if (per < granule) per = granule;
  if (per > cap) per = cap;
  return (int)per;
}

// tokens per activation chunk: at most 8, at most T, within shared memory
// (two CTAs per SM when the row is short enough)
int tok_chunk_for(int T, int K, int elem) {
  const size_t per = (size_t)K * elem;
  size_t n = (kSmemCap / 2 - kFixed) / per;
  if (n < 1) n = (kSmemCap - kFixed) / per;
  int c = (int)(n < (size_t)kTokMax ? n : (size_t)kTokMax);
  return c < T ? c : T;
}

template <typename TW>
cudaError_t launch_gateup(const GemvArgs& a, cudaStream_t st) {
  const int slots = a.routed_slots + (a.has_shared ? 1 : 0);
  const int wmax = a.has_shared && a.Is > a.I ? a.Is : a.I;
  const int chunk = tok_chunk_for(a.T, a.d, sizeof(TW));
  const int seg_cap = kStageBytes / 2 / (int)sizeof(TW);  // gate + up in one stage
  const int kseg = a.d <= seg_cap ? a.d : seg_cap;
  const size_t smem = kFixed + (size_t)chunk * a.d * sizeof(TW);
  static int limits[64] = {};
  cudaError_t e = ensure_smem_limit(gemv_gateup_stream<TW>, (int)smem, limits);
  if (e != cudaSuccess) return e;
  const int rpc = rows_for(wmax, slots, kConsumers, 64);
  return launch_pdl(gemv_gateup_stream<TW>, dim3((wmax + rpc - 1) / rpc, slots), kStreamThreads,
                    smem, st, a, rpc, chunk, kseg);
}

template <typename TW>
cudaError_t launch_down(const GemvArgs& a, cudaStream_t st) {
  const int slots = a.routed_slots + (a.has_shared ? 1 : 0);
  const int kmax = a.has_shared && a.Is > a.I ? a.Is : a.I;
  const int chunk = tok_chunk_for(a.T, kmax, sizeof(TW));
  const int seg_cap = kStageBytes / kDnRows / (int)sizeof(TW);
  const int kseg = kmax <= seg_cap ? kmax : seg_cap;
  const size_t smem = kFixed + (size_t)chunk * kmax * sizeof(TW);
  static int limits[64] = {};
  cudaError_t e = ensure_smem_limit(gemv_down_stream<TW>, (int)smem, limits);
  if (e != cudaSuccess) return e;
  const int rpc = rows_for(a.d, slots, kConsumers * kDnRows, 256);
  return launch_pdl(gemv_down_stream<TW>, dim3((a.d + rpc - 1) / rpc, slots), kStreamThreads,
                    smem, st, a, rpc, chunk, kseg);
}

}  // namespace

bool gemv_supported(int d, int kmax) {
  const size_t need = kFixed + (size_t)(d > kmax ? d : kmax) * sizeof(float);
  return need <= kSmemCap && d % 8 == 0 && kmax % 8 == 0;
}

cudaError_t launch_gemv_gateup(const GemvArgs& a, int act, int wdt, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (wdt == 0 && act == 0) return launch_gateup<float>(a, st);
  if (wdt == 1 && act == 1) return launch_gateup<__nv_bfloat16>(a, st);
  return cudaErrorNotSupported;
}

cudaError_t launch_gemv_down(const GemvArgs& a, int act, int wdt, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (wdt == 0 && act == 0) return launch_down<float>(a, st);
  if (wdt == 1 && act == 1) return launch_down<__nv_bfloat16>(a, st);
  return cudaErrorNotSupported;
}

}  // namespace moe
