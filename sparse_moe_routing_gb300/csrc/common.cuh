// Device-side helpers shared by the MoE layer kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------------------
// workspace control block (first 256 bytes of every workspace)
// ---------------------------------------------------------------------------
enum : uint32_t {
  kDevBadId = 1u << 0,     // an expert id outside [0, E) was seen
  kDevTimeout = 1u << 1,   // a bounded wait gave up
  kDevBadShape = 1u << 2,  // a device-side shape check failed
};

// Sites recorded in the upper 16 bits of the status word (first failure wins).
enum : uint32_t {
  kSiteBucket = 1,
  kSiteGemvGateUp = 2,
  kSiteGemvDown = 3,
  kSiteCombine = 4,
  kSiteTcGateUp = 5,
  kSiteTcDown = 6,
  kSiteTcRouter = 7,
  kSiteRouter = 8,
  kSiteDecode = 9,
};

struct Ctrl {
  uint32_t status;        // error bits (low 16) | first failing site (high 16)
  int32_t n_active;       // active routed experts (bucket)
  int32_t n_rowblocks;    // tensor-core path: (group, m-tile) row blocks
  int32_t pad0;
  uint32_t arrive_bucket; // self-resetting arrival counter (multi-CTA bucketing)
  int32_t pad1;
  // single-launch decode: grid-barrier arrivals, monotonic (every launch
  // adds two per block, so it is a multiple of the grid size between launches)
  unsigned long long grid_arrivals;
  int32_t pad[56];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");

__device__ __forceinline__ void report(Ctrl* c, uint32_t bits, uint32_t site) {
  uint32_t old = atomicOr(&c->status, bits);
  if ((old >> 16) == 0) atomicCAS(&c->status, old | bits, (old | bits) | (site << 16));
}

// ---------------------------------------------------------------------------
// element helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16-byte streaming load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Unpacks a 16-byte chunk of weights into floats. Element type selects the
// count: 8 bf16 or 4 f32 per chunk.
template <typename TW> struct Chunk;
template <> struct Chunk<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* w) {
    w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
  }
};
template <> struct Chunk<float> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* w) {
    w[0] = __uint_as_float(v.x); w[1] = __uint_as_float(v.y);
    w[2] = __uint_as_float(v.z); w[3] = __uint_as_float(v.w);
  }
};

__device__ __forceinline__ float load_act(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_act(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_act(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_act(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float sigmoidf_(float v) { return 1.0f / (1.0f + __expf(-v)); }
// SiLU with the fast division (reciprocal + multiply, 2 ulp): its result
// is rounded to bf16 or summed in fp32 right after, and the IEEE division
// made the tensor-core epilogues that apply it the slowest stage of the
// 4-bit gate/up kernel (1055 -> 891 us at the Mixtral shape). As v -> -inf
// the denominator overflows to inf and the quotient is 0, SiLU's limit.
__device__ __forceinline__ float siluf_(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// Programmatic dependent launch: every kernel is launched so that it may be
// scheduled while its predecessor on the stream finishes. pdl_wait() blocks
// until the predecessor grid has completed and its writes are visible, and
// must come before the kernel's first global memory access; pdl_trigger()
// then lets the successor grid be scheduled. Both are no-ops for a plain
// launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Default limit of every bounded on-device wait (about one second).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Multi-value butterfly: reduces N partial sums (N a power of two <= 32)
// across the warp in N-1+log2(32/N) shuffles; afterwards lane l holds the
// total of value l / (32/N).
template <int N>
__device__ __forceinline__ float reduce_multi(float (&v)[N], int lane) {
  int cnt = N;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (cnt > 1) {
      const int half = cnt / 2;
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      cnt = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}
// P2<X>::v = X rounded up to a power of two.
template <int X> struct P2 { static constexpr int v = 2 * P2<(X + 1) / 2>::v; };
template <> struct P2<1> { static constexpr int v = 1; };

}  // namespace moe
