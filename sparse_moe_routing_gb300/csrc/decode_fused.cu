// Single-launch layer forward for decode batches of a few tokens: the whole
// pipeline of "How Treebeard routes Qwen3.6 MoE tokens" ("Pseudocode": router,
// routing rule, selected SwiGLU experts weighted by alpha, sigmoid-gated
// shared expert, residual) in one kernel, with the expert ids kept on the
// device as in that page's "NVIDIA CUDA path" (device-routed selected-expert
// mat-vecs). At a few tokens the layer is a stream of weight rows, and a
// chain of separate launches spends much of its time between kernels; here
// the steps are phases of one cooperative launch (one block per SM)
// separated by bounded grid barriers:
//
//  1. routing-independent work spread over the grid: router logits
//     z = W_router x plus the shared-gate logit w_shared . x (column E) and
//     the shared expert's gate/up + SwiGLU rows;
//  -- grid barrier --
//  2. every block applies the routing rule to all tokens itself (the router
//     kernels' own routing code; a routing-only call, moe_route with this
//     path, runs phases 1-2 of this kernel so that its ids and weights are
//     the layer's), sorts the (token, slot) pairs by expert into chunks of at
//     most 8 pairs of one expert; block 0 writes topk_ids and weights;
//  3. routed gate/up + SwiGLU: (chunk, row) items in a contiguous range per
//     block; each weight row is read once per chunk and dotted with every
//     token of the chunk ("Intel SYCL path": one weight load serves all of
//     an expert's tokens);
//  -- grid barrier --
//  4. down x alpha and the combine, per token and output column: the slots
//     in slot order, the shared expert and the residual (a fixed order: the
//     result is deterministic).
//
// Two variants. The tensor-core variant (bf16, d a multiple of 1024, I and
// Is multiples of 128) contracts with mma.sync m16n8k16 on 2D TMA tiles
// (the tokens are the n = 8 side), splits phase 1 along K when its items
// would leave half of the grid idle, keeps h in mma fragment order, spreads
// phase 4 as (8-column group, chunk) items over the whole grid with each
// block's chunks of h copied to shared memory, and adds a third barrier
// before the combine. The CUDA-core variant (fp32, or other bf16 shapes)
// streams rows with 1D bulk copies, owns output columns per block in phase
// 4 and runs the shared expert's down rows in phase 2 on warps that route no
// token.
//
// Weight bytes reach the SM through one ring of 4 KB stages per warp: each
// warp copies the next segments of its own work into its ring (lane 0
// issues, completion counted by mbarrier transactions) and computes from
// shared memory, refilling each stage as soon as it has read it. No register
// holds a load in flight, so every SM keeps its rings (up to 192 KB) of
// weights in flight.
//
// Every wait is bounded (about one second; a block that gives up records
// kDevTimeout in the workspace's status word, lets its copies in flight land
// and returns).
#include <string.h>

#include "decode_mma.cuh"
#include "router_core.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;          // every warp streams and computes
constexpr int kSB = 4096;                      // bytes per ring stage
constexpr int kNT = 8;                         // pairs (tokens) per chunk
constexpr int kDnRows = 4;                     // output columns per phase-4 item
constexpr int kMaxStages = 4;                  // ring stages per warp, at most
// Profiling build (-DMOE_DECODE_PHASE_TIMES): thread 0 of every block
// records the globaltimer at each phase mark i in the control block's spare
// words, as the earliest and the latest block (u64 pair i at byte 40 + 16 i;
// the host seeds them with (max, 0) before a call). Marks: 0 start, 1 phase
// 1 done, 2 past barrier 1, 3 routing rule done, 4 grouping done, 5 phase 3
// done, 6 past barrier 2, 7 past barrier 3, 8 router tiles done, 9 shared
// gate/up done, 10 shared-gate row done, 11 down items done, 12 phase-4 h
// staged.
#ifdef MOE_DECODE_PHASE_TIMES
__device__ __forceinline__ void stamp(Ctrl* c, int i) {
  if (threadIdx.x == 0) {
    unsigned long long* t = reinterpret_cast<unsigned long long*>(&c->pad[2]);
    unsigned long long now;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    atomicMin(&t[2 * i], now);
    atomicMax(&t[2 * i + 1], now);
  }
}
#define STAMP(i) stamp(a.ctrl, i)
#else
#define STAMP(i)
#endif


// ---------------------------------------------------------------------------
// mbarriers, bulk copies, bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void bar_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
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
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(b))
      : "memory");
}
// 2D tile copy (tensor map, coordinates x along the contiguous dimension).
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(su32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ unsigned long long atom_add_release_u64(unsigned long long* p,
                                                                   unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

struct Block {
  uint8_t* ring;
  uint64_t* full;        // [kWarps * S]
  volatile int* abort_flag;
  volatile int* bar_flag;
  int S;
  Ctrl* ctrl;
  uint64_t limit;
};

// Bounded wait of one lane; on timeout the block's abort flag is raised and
// the timeout recorded. False once the block is aborting.
__device__ bool wait_bar(const Block& B, uint64_t* b, uint32_t parity) {
  if (bar_try(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!bar_try(b, parity)) {
    if ((++n & 31u) == 0) {
      if (*B.abort_flag) return false;
      if (globaltimer_ns() - t0 > B.limit) {
        *B.abort_flag = 1;
        report(B.ctrl, kDevTimeout, kSiteDecode);
        return false;
      }
    }
  }
  return true;
}

// Ring of warp w: its unit j sits in stage w*S + j%S with parity (j/S)&1.
__device__ __forceinline__ int stage_of(const Block& B, int w, uint32_t j) {
  return w * B.S + (int)(j % (uint32_t)B.S);
}

// The copies that fill one stage: up to kDnRows contiguous pieces.
struct Copies {
  const void* src[kDnRows];
  uint32_t bytes[kDnRows];
  uint32_t off[kDnRows];
  int n;
};

// A warp's unit sequence in one phase: items it, it + step, ... < it1, each
// cut into segments of `seg` elements of its K; `jn` counts the units issued.
struct Feed {
  int it, it1, step, e0;
  uint32_t jn;
};

// Issues the warp's next unit (if any) into its stage: describe(it, e0, cp,
// K, seg) gives the unit's copies, the item's length K and the segment
// length. Warp-uniform; lane 0 issues.
template <typename Describe>
__device__ __forceinline__ void issue(const Block& B, int w, Feed& f, Describe describe, int lane) {
  if (f.it >= f.it1) return;
  Copies cp;
  int K, seg;
  describe(f.it, f.e0, cp, K, seg);
  if (lane == 0) {
    const int st = stage_of(B, w, f.jn);
    uint32_t total = 0;
    for (int i = 0; i < cp.n; ++i) total += cp.bytes[i];
    bar_expect(&B.full[st], total);
    uint8_t* dst = B.ring + (size_t)st * kSB;
    for (int i = 0; i < cp.n; ++i) bulk_g2s(dst + cp.off[i], cp.src[i], cp.bytes[i], &B.full[st]);
  }
  ++f.jn;
  f.e0 += seg;
  if (f.e0 >= K) {
    f.e0 = 0;
    f.it += f.step;
  }
}

// Waits for the warp's unit j; null once the block is aborting.
__device__ const uint8_t* acquire(const Block& B, int w, uint32_t j, int lane) {
  const int st = stage_of(B, w, j);
  bool ok = lane == 0 ? wait_bar(B, &B.full[st], (j / (uint32_t)B.S) & 1u) : true;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok ? B.ring + (size_t)st * kSB : nullptr;
}
// The warp has read its unit j: order those reads before the copy that
// refills the stage (async proxy), then issue the next unit into it.
template <typename Refill>
__device__ __forceinline__ void release(uint32_t& j, Refill& refill) {
  __syncwarp();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  refill();
  ++j;
}

// ---------------------------------------------------------------------------
// grid barrier: a 64-bit arrival count that every block increments once per
// barrier and that never resets; with nb blocks a barrier completes when the
// count reaches the next multiple of nb (the count is a multiple of nb
// between launches: each launch adds two per block). One atomic per block;
// the last arriver is released by its own add.
// ---------------------------------------------------------------------------
__device__ bool grid_barrier(const Block& B, bool arrive) {
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = arrive && !*B.abort_flag;
    if (ok) {
      // release: the block's writes before the __syncthreads above are
      // ordered before the arrival; the polls below acquire the others'
      const unsigned long long nb = gridDim.x;
      const unsigned long long prev = atom_add_release_u64(&B.ctrl->grid_arrivals, 1ull);
      const unsigned long long target = (prev / nb + 1) * nb;
      if (prev + 1 != target) {
        const uint64_t t0 = globaltimer_ns();
        unsigned n = 0;
        while ((long long)(ld_acquire_u64(&B.ctrl->grid_arrivals) - target) < 0) {
          if ((++n & 255u) == 0 && globaltimer_ns() - t0 > B.limit) {
            ok = false;
            report(B.ctrl, kDevTimeout, kSiteDecode);
            break;
          }
        }
      }
    }
    *B.bar_flag = ok ? 1 : 0;
  }
  __syncthreads();
  // data other blocks wrote before the barrier may next be read by bulk
  // copies (the async proxy)
  asm volatile("fence.proxy.async;" ::: "memory");
  return *B.bar_flag != 0;
}

// ---------------------------------------------------------------------------
// shared-memory layout (identical on host and device)
// ---------------------------------------------------------------------------
struct Layout {
  int ring, full, part, ids, w, key, gpair, cstart, cexp, ssh, misc, y, ystride, bytes;
};
// Tensor-core variant: cross-warp partial sums of one 16-row block (gate and
// up, 16 rows x 8 tokens, per warp).
constexpr int kPartBytes = kWarps * 2 * 16 * 8 * 4;
__host__ __device__ inline Layout layout(int T, int k, int ncols, int S, bool mma) {
  const int P = T * k;
  Layout L;
  int o = 0;
  L.ring = o;   o += kWarps * S * kSB;
  L.full = o;   o += kWarps * S * 8;
  L.part = o;   o += mma ? kPartBytes : 0;
  L.ids = o;    o += P * 4;
  L.w = o;      o += P * 4;
  L.key = o;    o += P * 4;
  L.gpair = o;  o += P * 4;
  L.cstart = o; o += (P + 1) * 4;
  L.cexp = o;   o += P * 4;
  L.ssh = o;    o += T * 4;
  L.misc = o;   o += 16;
  o = (o + 15) & ~15;
  L.y = o;
  L.ystride = P + T;
  o += ncols * L.ystride * 4;
  L.bytes = o + 1024;  // slack to align the ring to 1024 bytes (swizzled TMA tiles)
  return L;
}
constexpr int kSmemBudget = 227 * 1024;

// Output columns are owned in groups of `gran` (4 on the CUDA cores, 8 for
// the tensor-core tiles): block b owns groups [b*ng/nb, (b+1)*ng/nb).
__host__ __device__ inline int quad_lo(int b, int nq, int nb) {
  return (int)((long long)b * nq / nb);
}
__host__ __device__ inline int max_cols(int d, int nb, int gran) {
  const int nq = d / gran;
  return gran * ((nq + nb - 1) / nb);
}
// Ring stages per warp that fit beside the tables (0: the shape does not fit).
__host__ __device__ inline int ring_stages(int T, int k, int ncols, bool mma) {
  for (int S = kMaxStages; S >= 2; --S)
    if (layout(T, k, ncols, S, mma).bytes <= kSmemBudget) return S;
  return 0;
}
// The tensor-core variant: bf16, K of the gate/up rows split into 64-wide
// segments over the 16 warps, 16-row blocks and 128-wide down segments.
__host__ __device__ inline bool mma_shape(int d, int I, int Is, bool bf16) {
  return bf16 && d % (64 * kWarps) == 0 && I % 128 == 0 && Is % 128 == 0;
}

// [lo, hi) of n equal items for this block.
__device__ __forceinline__ void block_range(int n, int& lo, int& hi) {
  lo = (int)((long long)blockIdx.x * n / gridDim.x);
  hi = (int)((long long)(blockIdx.x + 1) * n / gridDim.x);
}

// ---------------------------------------------------------------------------
// consumer arithmetic on one stage
// ---------------------------------------------------------------------------
// Independent partial sums per dot product, so that a few-token chunk still
// keeps several FMA chains in flight: 4 for one or two vectors, 2 for four,
// 1 for eight.
template <int NJ> struct Parts { static constexpr int v = NJ <= 2 ? 4 : (NJ <= 4 ? 2 : 1); };

// Gate/up stage: gate[seg] at offset 0, up[seg] at offset kSB/2, `len`
// elements starting at element e0 of the row; accumulates the dot products
// with tokens tok[0..nj) (acc[2j][.] gate, acc[2j+1][.] up, in partial sums).
template <typename TW, int NJ>
__device__ __forceinline__ void gateup_stage(const uint8_t* st, const TW* x, int d, const int* tok,
                                             int nj, int e0, int len, int lane,
                                             float (&acc)[2 * NJ][Parts<NJ>::v]) {
  constexpr int kVec = Chunk<TW>::kVec;
  constexpr int kP = Parts<NJ>::v;
  const uint4* g = reinterpret_cast<const uint4*>(st);
  const uint4* u = reinterpret_cast<const uint4*>(st + kSB / 2);
  const int nv = len / kVec;
  for (int c = lane; c < nv; c += 32) {
    float gf[kVec], uf[kVec];
    Chunk<TW>::unpack(g[c], gf);
    Chunk<TW>::unpack(u[c], uf);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < nj) {
        float xf[kVec];
        Chunk<TW>::unpack(
            __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok[j] * d + e0) + c), xf);
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          acc[2 * j][e % kP] = fmaf(gf[e], xf[e], acc[2 * j][e % kP]);
          acc[2 * j + 1][e % kP] = fmaf(uf[e], xf[e], acc[2 * j + 1][e % kP]);
        }
      }
    }
  }
}

// Down stage: kDnRows row segments of `len` elements at offsets r * kSB/4;
// accumulates their dot products with the fp32 vectors h_j (rows hrow[j] of
// a buffer of row stride hs, written earlier in this launch: read via L2)
// from element e0 (acc[r * NJ + j][.], in partial sums).
template <typename TW, int NJ>
__device__ __forceinline__ void down_stage(const uint8_t* st, const float* h, size_t hs,
                                           const int* hrow, int nj, int e0, int len, int lane,
                                           float (&acc)[kDnRows * NJ][Parts<NJ>::v]) {
  constexpr int kVec = Chunk<TW>::kVec;
  constexpr int kP = Parts<NJ>::v;
  const int nv = len / kVec;
  for (int c = lane; c < nv; c += 32) {
    float wf[kDnRows][kVec];
#pragma unroll
    for (int r = 0; r < kDnRows; ++r)
      Chunk<TW>::unpack(reinterpret_cast<const uint4*>(st + r * (kSB / kDnRows))[c], wf[r]);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < nj) {
        const float4* hp = reinterpret_cast<const float4*>(h + (size_t)hrow[j] * hs + e0) +
                           (size_t)c * (kVec / 4);
        float hf[kVec];
#pragma unroll
        for (int q = 0; q < kVec / 4; ++q) {
          const float4 v = __ldcg(hp + q);
          hf[4 * q] = v.x; hf[4 * q + 1] = v.y; hf[4 * q + 2] = v.z; hf[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int r = 0; r < kDnRows; ++r)
#pragma unroll
          for (int e = 0; e < kVec; ++e)
            acc[r * NJ + j][e % kP] = fmaf(wf[r][e], hf[e], acc[r * NJ + j][e % kP]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// per-item consumers (one warp; all stages of the item in order)
// ---------------------------------------------------------------------------
// Gate/up item: one gate/up row pair dotted with tokens tok[0..nj);
// h(j) -> out[orow[j] * ostride + r]. False once the block is aborting.
template <typename TW, int NJ, typename Refill>
__device__ bool gateup_item(const Block& B, int c, uint32_t& j, Refill& refill, const TW* x, int d,
                            const int* tok, int nj, float* out, const int* orow, size_t ostride,
                            int r, int lane) {
  constexpr int kSeg = kSB / 2 / sizeof(TW);
  constexpr int kP = Parts<NJ>::v;
  float part[2 * NJ][kP];
#pragma unroll
  for (int i = 0; i < 2 * NJ; ++i)
#pragma unroll
    for (int q = 0; q < kP; ++q) part[i][q] = 0.f;
  for (int e0 = 0; e0 < d; e0 += kSeg) {
    const uint8_t* st = acquire(B, c, j, lane);
    if (!st) return false;
    gateup_stage<TW, NJ>(st, x, d, tok, nj, e0, min(kSeg, d - e0), lane, part);
    release(j, refill);
  }
  float acc[2 * NJ];
#pragma unroll
  for (int i = 0; i < 2 * NJ; ++i) {
    acc[i] = part[i][0];
#pragma unroll
    for (int q = 1; q < kP; ++q) acc[i] += part[i][q];
  }
  const float sum = reduce_multi<2 * NJ>(acc, lane);
  constexpr int per = 32 / (2 * NJ);
  const float up = __shfl_down_sync(0xffffffffu, sum, per);
  const int idx = lane / per;  // value this lane holds: 2j gate, 2j+1 up
  if ((lane % per) == 0 && (idx & 1) == 0 && idx / 2 < nj) {
    int o = orow[0];
#pragma unroll
    for (int q = 1; q < NJ; ++q)
      if (q == idx / 2) o = orow[q];
    out[(size_t)o * ostride + r] = siluf_(sum) * up;
  }
  return true;
}

// Down item: kDnRows rows (row stride K) dotted with h rows hrow[0..nj); on
// return lane l < kDnRows * NJ holds the value of (row l / NJ, vector l % NJ).
template <typename TW, int NJ, typename Refill>
__device__ bool down_item(const Block& B, int c, uint32_t& j, Refill& refill, int K, const float* h,
                          size_t hs, const int* hrow, int nj, int lane, float& val) {
  constexpr int kSeg = kSB / kDnRows / sizeof(TW);
  constexpr int kP = Parts<NJ>::v;
  float part[kDnRows * NJ][kP];
#pragma unroll
  for (int i = 0; i < kDnRows * NJ; ++i)
#pragma unroll
    for (int q = 0; q < kP; ++q) part[i][q] = 0.f;
  for (int e0 = 0; e0 < K; e0 += kSeg) {
    const uint8_t* st = acquire(B, c, j, lane);
    if (!st) return false;
    down_stage<TW, NJ>(st, h, hs, hrow, nj, e0, min(kSeg, K - e0), lane, part);
    release(j, refill);
  }
  float acc[kDnRows * NJ];
#pragma unroll
  for (int i = 0; i < kDnRows * NJ; ++i) {
    acc[i] = part[i][0];
#pragma unroll
    for (int q = 1; q < kP; ++q) acc[i] += part[i][q];
  }
  constexpr int NV = kDnRows * NJ;  // 4, 8, 16 or 32: a power of two
  const float sum = reduce_multi<NV>(acc, lane);   // lane l holds value l / (32 / NV)
  val = __shfl_sync(0xffffffffu, sum, (lane * (32 / NV)) & 31);
  return true;
}

// dispatch on the chunk's pair count (rounded up to 1, 2, 4 or 8)
template <typename TW, typename Refill>
__device__ bool gateup_any(const Block& B, int c, uint32_t& j, Refill& refill, const TW* x, int d,
                           const int* tok, int nj, float* out, const int* orow, size_t ostride,
                           int r, int lane) {
  if (nj <= 1)
    return gateup_item<TW, 1>(B, c, j, refill, x, d, tok, nj, out, orow, ostride, r, lane);
  if (nj <= 2)
    return gateup_item<TW, 2>(B, c, j, refill, x, d, tok, nj, out, orow, ostride, r, lane);
  if (nj <= 4)
    return gateup_item<TW, 4>(B, c, j, refill, x, d, tok, nj, out, orow, ostride, r, lane);
  return gateup_item<TW, 8>(B, c, j, refill, x, d, tok, nj, out, orow, ostride, r, lane);
}
template <typename TW, typename Refill>
__device__ bool down_any(const Block& B, int c, uint32_t& j, Refill& refill, int K, const float* h,
                         size_t hs, const int* hrow, int nj, int lane, float& val, int& njp) {
  if (nj <= 1) {
    njp = 1;
    return down_item<TW, 1>(B, c, j, refill, K, h, hs, hrow, nj, lane, val);
  }
  if (nj <= 2) {
    njp = 2;
    return down_item<TW, 2>(B, c, j, refill, K, h, hs, hrow, nj, lane, val);
  }
  if (nj <= 4) {
    njp = 4;
    return down_item<TW, 4>(B, c, j, refill, K, h, hs, hrow, nj, lane, val);
  }
  njp = 8;
  return down_item<TW, 8>(B, c, j, refill, K, h, hs, hrow, nj, lane, val);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// The tensor maps of the tensor-core variant (128-byte swizzle, 64-wide
// boxes): gate/up banks [E*I][d] and shared [Is][d] with 16-row boxes, down
// banks [E*d][I] and shared [d][Is] with 8-row boxes.
struct DecodeMaps {
  CUtensorMap g, u, sg, su, dn, sdn, r;  // r: router [E][d]
};

// A warp's tensor-core down items (see dn_run in the kernel) and the state of
// its ring feed.
struct DnPlan {
  int it0, it1, step, nroute, nchs, obase, nqg, hc0;
  const uint2* hs;
};
struct DnFeed {
  int fit, fk;
  uint32_t jn;
};

template <typename TW, int PL, bool MMA>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap mg, const __grid_constant__ CUtensorMap mu,
                        const __grid_constant__ CUtensorMap msg, const __grid_constant__ CUtensorMap msu,
                        const __grid_constant__ CUtensorMap mdn, const __grid_constant__ CUtensorMap msdn,
                        const __grid_constant__ CUtensorMap mr, const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int T = a.T, k = a.k, E = a.E, d = a.d, I = a.I, Is = a.Is;
  const int P = T * k;
  const int nb = gridDim.x;
  constexpr int kGran = MMA ? 8 : 4;  // output columns per down item
  const int nq = d / kGran;
  const int q0 = quad_lo(blockIdx.x, nq, nb), q1 = quad_lo(blockIdx.x + 1, nq, nb);
  const int c0 = kGran * q0, ncols = kGran * (q1 - q0);
  const int S = ring_stages(T, k, max_cols(d, nb, kGran), MMA);
  const Layout Ly = layout(T, k, max_cols(d, nb, kGran), S, MMA);
  int* s_ids = reinterpret_cast<int*>(smem + Ly.ids);
  float* s_w = reinterpret_cast<float*>(smem + Ly.w);
  int* s_key = reinterpret_cast<int*>(smem + Ly.key);
  int* s_gpair = reinterpret_cast<int*>(smem + Ly.gpair);
  int* s_cstart = reinterpret_cast<int*>(smem + Ly.cstart);
  int* s_cexp = reinterpret_cast<int*>(smem + Ly.cexp);
  float* s_ssh = reinterpret_cast<float*>(smem + Ly.ssh);
  volatile int* s_misc = reinterpret_cast<volatile int*>(smem + Ly.misc);  // nch, abort, bar
  float* s_y = reinterpret_cast<float*>(smem + Ly.y);

  Block B;
  B.ring = smem + Ly.ring;
  B.full = reinterpret_cast<uint64_t*>(smem + Ly.full);
  B.abort_flag = s_misc + 1;
  B.bar_flag = s_misc + 2;
  B.S = S;
  B.ctrl = a.ctrl;
  B.limit = a.wait_ns;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t jr = 0;  // units this warp has consumed from its ring
  const bool route = a.ids_in == nullptr;
  // shared: the shared expert's work; sgate: its gate s_t is computed
  const bool shared = Is > 0 && !a.route_only;
  const bool sgate = a.route_only ? a.s_out != nullptr : Is > 0;
  const TW* x = static_cast<const TW*>(a.x);
  const TW* Wg = static_cast<const TW*>(a.Wg);
  const TW* Wu = static_cast<const TW*>(a.Wu);
  const TW* Wd = static_cast<const TW*>(a.Wd);
  const TW* Wsg = static_cast<const TW*>(a.Wsg);
  const TW* Wsu = static_cast<const TW*>(a.Wsu);
  const TW* Wsd = static_cast<const TW*>(a.Wsd);
  constexpr int kRowSeg = kSB / sizeof(TW);            // logit-row elements per stage
  constexpr int kPairSeg = kSB / 2 / sizeof(TW);       // gate/up elements per stage
  constexpr int kDnSeg = kSB / kDnRows / sizeof(TW);   // down-row elements per stage

  // The shared expert's down rows need only phase 1's results: in the
  // CUDA-core variant, when some warps have no token to route, they compute
  // this block's shared-expert columns while the others route. The
  // tensor-core variant keeps them in phase 4, where they hold up no phase.
  const bool sh_early = !MMA && shared && T < kWarps;
  auto down_items = [&](int it0, int it1, int step, int nroute, int nchs) {
    // items (4-column quad qi, chunk ci): ci < nroute a routed chunk, else a
    // shared-expert token chunk; results scaled into s_y
    auto describe = [&](int it, int e0, Copies& cp, int& K, int& seg) {
      const int qi = it / nchs, ci = it - qi * nchs;
      const int col = c0 + 4 * qi;
      const TW* w;
      if (ci < nroute) {
        K = I;
        w = Wd + ((size_t)s_cexp[ci] * d + col) * I;
      } else {
        K = Is;
        w = Wsd + (size_t)col * Is;
      }
      seg = kDnSeg;
      const uint32_t n = (uint32_t)(min(kDnSeg, K - e0) * sizeof(TW));
      cp.n = kDnRows;
#pragma unroll
      for (int rr = 0; rr < kDnRows; ++rr) {
        cp.src[rr] = w + (size_t)rr * K + e0;
        cp.bytes[rr] = n;
        cp.off[rr] = rr * (kSB / kDnRows);
      }
    };
    Feed f{it0, it1, step, 0, jr};
    auto refill = [&]() { issue(B, warp, f, describe, lane); };
    for (int i = 0; i < S; ++i) refill();
    for (int it = it0; it < it1 && !*B.abort_flag; it += step) {
      const int qi = it / nchs, ci = it - qi * nchs;
      const int col = c0 + 4 * qi;
      int hrow[kNT], slot[kNT];
      int nj, K;
      const float* h;
      if (ci < nroute) {
        const int cs = s_cstart[ci];
        nj = min(kNT, s_cstart[ci + 1] - cs);
#pragma unroll
        for (int q = 0; q < kNT; ++q) hrow[q] = slot[q] = s_gpair[cs + (q < nj ? q : 0)];
        h = a.H;
        K = I;
      } else {
        const int t0 = (ci - nroute) * kNT;
        nj = min(kNT, T - t0);
#pragma unroll
        for (int q = 0; q < kNT; ++q) {
          hrow[q] = t0 + (q < nj ? q : 0);
          slot[q] = P + hrow[q];
        }
        h = a.Hs;
        K = Is;
      }
      float v;
      int njp;
      if (!down_any<TW>(B, warp, jr, refill, K, h, (size_t)K, hrow, nj, lane, v, njp)) break;
      const int rr = lane / njp, q = lane - rr * njp;
      if (rr < kDnRows && q < nj) {
        int sl = slot[0];
#pragma unroll
        for (int z = 1; z < kNT; ++z)
          if (z == q) sl = slot[z];
        const float scale = sl < P ? s_w[sl] : s_ssh[sl - P];
        s_y[(size_t)(col - c0 + rr) * Ly.ystride + sl] = scale * v;
      }
    }
  };
  // Tensor-core down items (bf16): (8-column group qi, chunk ci), one warp
  // each; the chunk's slots (at most 8) are the A side of mma m16n8k16 and
  // the 8 columns its n side. Items are numbered column-major (it = qi * nchs
  // + ci, columns from group obase) or chunk-major (it = ci * nqg + qi).
  // With hs null a stage holds 8 columns x 128 k of the down bank (two
  // 64-wide swizzled boxes) and the chunk's h fragments for those k (written
  // in fragment order by the gate/up items); with hs set, the h fragments of
  // chunks hc0.. are copied to shared memory once for the whole block
  // (consecutively, K x 16 bytes each) and a stage holds 8 columns x 256 k
  // of the bank (four boxes), so that a warp may fill its ring before the h
  // rows exist.
  auto dn_decode = [&](const DnPlan& pl, int it, int& qi, int& ci) {
    if (pl.nqg) {
      ci = it / pl.nqg;
      qi = it - ci * pl.nqg;
    } else {
      qi = it / pl.nchs;
      ci = it - qi * pl.nchs;
    }
  };
  auto dn_refill = [&](const DnPlan& pl, DnFeed& f) {
    if (f.fit >= pl.it1 || *B.abort_flag) return;
    int qi, ci;
    dn_decode(pl, f.fit, qi, ci);
    const int col = 8 * (pl.obase + qi);
    const bool rt = ci < pl.nroute;
    const int K = rt ? I : Is;
    const int nbox = pl.hs ? min(4, (K - f.fk) / 64) : 2;
    if (lane == 0) {
      const int st = stage_of(B, warp, f.jn);
      bar_expect(&B.full[st], pl.hs ? 1024u * nbox : 4096u);
      uint8_t* dst = B.ring + (size_t)st * kSB;
      const int y = rt ? s_cexp[ci] * d + col : col;
      for (int b = 0; b < nbox; ++b)
        tma2d(dst + 1024 * b, rt ? &mdn : &msdn, &B.full[st], f.fk + 64 * b, y);
      if (!pl.hs) {
        const __nv_bfloat16* hf = reinterpret_cast<const __nv_bfloat16*>(rt ? a.H : a.Hs) +
                                  dmma::frag_index(rt ? ci : ci - pl.nroute, K, 0, f.fk);
        bulk_g2s(dst + 2048, hf, 2048u, &B.full[st]);
      }
    }
    ++f.jn;
    f.fk += 64 * nbox;
    if (f.fk >= K) {
      f.fk = 0;
      f.fit += pl.step;
    }
  };
  // fills the warp's ring with the plan's first units
  auto dn_prime = [&](const DnPlan& pl, DnFeed& f) {
    f.fit = pl.it0;
    f.fk = 0;
    f.jn = jr;
    for (int i = 0; i < S; ++i) dn_refill(pl, f);
  };
  auto dn_run = [&](const DnPlan& pl, DnFeed& f) {
    auto refill = [&]() { dn_refill(pl, f); };
    const int g = lane >> 2, t = lane & 3;
    const int kst = pl.hs ? 256 : 128;  // k per stage
    for (int it = pl.it0; it < pl.it1 && !*B.abort_flag; it += pl.step) {
      int qi, ci;
      dn_decode(pl, it, qi, ci);
      const int col = 8 * (pl.obase + qi);
      const bool rt = ci < pl.nroute;
      const int K = rt ? I : Is;
      int nj, hrow, slot;
      if (rt) {
        const int cs = s_cstart[ci];
        nj = min(kNT, s_cstart[ci + 1] - cs);
        hrow = s_gpair[cs + (g < nj ? g : 0)];
        slot = hrow;
      } else {
        const int t0 = (ci - pl.nroute) * kNT;
        nj = min(kNT, T - t0);
        hrow = t0 + (g < nj ? g : 0);
        slot = P + hrow;
      }
      const uint2* hc = nullptr;
      if (pl.hs) {
        size_t off = 0;
        for (int c = pl.hc0; c < ci; ++c) off += (size_t)(c < pl.nroute ? I : Is) * 2;
        hc = pl.hs + off;
      }
      float dd[4] = {0.f, 0.f, 0.f, 0.f};
      bool ok = true;
      for (int k0 = 0; k0 < K; k0 += kst) {
        const uint8_t* st = acquire(B, warp, jr, lane);
        if (!st) {
          ok = false;
          break;
        }
        const int nbox = pl.hs ? min(4, (K - k0) / 64) : 2;
        const uint2* af = pl.hs ? hc + (k0 >> 4) * 32 : reinterpret_cast<const uint2*>(st + 2048);
        dmma::down_tile(st, af, nbox, lane, dd);
        release(jr, refill);
      }
      if (!ok) break;
      if (g < nj) {
        const float scale = rt ? s_w[slot] : s_ssh[hrow];
        a.Yg[(size_t)(col + 2 * t) * Ly.ystride + slot] = scale * dd[0];
        a.Yg[(size_t)(col + 2 * t + 1) * Ly.ystride + slot] = scale * dd[1];
      }
    }
  };
  DnPlan pl4{};  // this warp's phase-4 items
  DnFeed f4{};
  // Tensor-core gate/up items (bf16), block-wide: item = (chunk, 16-row
  // block) of a routed expert (sh false: rows of W_gate/W_up, h rows = the
  // chunk's pairs) or of the shared expert (sh true: token chunk, rows of
  // Ws_gate/Ws_up, h rows = tokens). Warp w streams the 64-wide K segments
  // w, w + 16, ... of the item's rows; the 16 partial sums meet in shared
  // memory and are added in warp order, then SwiGLU gives bf16 h.
  auto gateup_items_mma = [&](int lo, int hi, bool sh, int KS) {
    const int R = sh ? Is : I;
    const int nrb = R / 16;
    const int per = d / 64 / kWarps / KS;  // K segments per warp and item
    const CUtensorMap* mgp = sh ? &msg : &mg;
    const CUtensorMap* mup = sh ? &msu : &mu;
    int fit = lo, fj = 0;
    uint32_t jn = jr;
    auto refill = [&]() {
      if (fit >= hi || *B.abort_flag) return;
      if (lane == 0) {
        const int base = fit / KS, ks = fit - base * KS;
        const int c = base / nrb, rb = base - c * nrb;
        const int y = (sh ? 0 : s_cexp[c] * I) + rb * 16;
        const int st = stage_of(B, warp, jn);
        bar_expect(&B.full[st], 4096u);
        uint8_t* dst = B.ring + (size_t)st * kSB;
        const int k0 = (warp + kWarps * (ks * per + fj)) * 64;
        tma2d(dst, mgp, &B.full[st], k0, y);
        tma2d(dst + 2048, mup, &B.full[st], k0, y);
      }
      ++jn;
      if (++fj == per) {
        fj = 0;
        ++fit;
      }
    };
    for (int i = 0; i < S; ++i) refill();
    float* part = reinterpret_cast<float*>(smem + Ly.part);
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(a.x);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(sh ? a.Hs : a.H);
    const int g = lane >> 2, t = lane & 3;
    uint32_t xf0[8], xf1[8];
    int xc = -1;
    for (int it = lo; it < hi; ++it) {
      const int base = it / KS, ks = it - base * KS;
      const int c = base / nrb, rb = base - c * nrb;
      int nj, cs = 0;
      if (sh) {
        nj = min(kNT, T - c * kNT);
      } else {
        cs = s_cstart[c];
        nj = min(kNT, s_cstart[c + 1] - cs);
      }
      const bool valid = g < nj;
      const int tok = sh ? c * kNT + (valid ? g : 0) : s_gpair[cs + (valid ? g : 0)] / k;
      const int s0 = ks * per;  // first K segment of the item
      if (per <= 2 && c * KS + ks != xc) {
        // the chunk's token fragments for this warp's segments, kept while
        // the chunk lasts and loaded before its first tile lands
        dmma::x_frags(xb, d, tok, valid, (warp + kWarps * s0) * 64, lane, xf0);
        if (per == 2) dmma::x_frags(xb, d, tok, valid, (warp + kWarps * (s0 + 1)) * 64, lane, xf1);
        xc = c * KS + ks;
      }
      float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < per; ++j) {
        uint32_t f[8];
        if (per <= 2) {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = j ? xf1[e] : xf0[e];
        } else {
          dmma::x_frags(xb, d, tok, valid, (warp + kWarps * (s0 + j)) * 64, lane, f);
        }
        const uint8_t* st = acquire(B, warp, jr, lane);
        if (!st) break;
        dmma::gateup_tile(st, f, lane, dg, du);
        release(jr, refill);
      }
      float* pw = part + warp * 256;  // [gate, up][16 rows][8 tokens]
      pw[g * 8 + 2 * t] = dg[0];
      pw[g * 8 + 2 * t + 1] = dg[1];
      pw[(g + 8) * 8 + 2 * t] = dg[2];
      pw[(g + 8) * 8 + 2 * t + 1] = dg[3];
      pw[128 + g * 8 + 2 * t] = du[0];
      pw[128 + g * 8 + 2 * t + 1] = du[1];
      pw[128 + (g + 8) * 8 + 2 * t] = du[2];
      pw[128 + (g + 8) * 8 + 2 * t + 1] = du[3];
      __syncthreads();
      if (threadIdx.x < 128) {
        const int r = threadIdx.x >> 3, q = threadIdx.x & 7;
        float gs = 0.f, us = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          gs += part[w * 256 + r * 8 + q];
          us += part[w * 256 + 128 + r * 8 + q];
        }
        if (q < nj) {
          if (KS == 1) {
            // h in fragment order for the down items: chunk c, slot q, k = 16 rb + r
            out[dmma::frag_index(c, R, q, rb * 16 + r)] = __float2bfloat16_rn(siluf_(gs) * us);
          } else {
            // (shared expert only) partial sums of part ks, [ks][gate/up][t][row]
            const size_t o = ((size_t)ks * 2 * T + c * kNT + q) * Is + rb * 16 + r;
            a.Gs[o] = gs;
            a.Gs[o + (size_t)T * Is] = us;
          }
        }
      }
      __syncthreads();
    }
  };
  // Tensor-core router contraction (bf16), block-wide: item = (token chunk,
  // tile of 16 router rows; rows past E read as zeros); the K split and the
  // warp-ordered sum are those of gateup_items_mma.
  auto router_items_mma = [&](int lo, int hi, int ntiles, int KS) {
    const int per = d / 64 / kWarps / KS;  // K segments per warp and item
    int fit = lo, fj = 0;
    uint32_t jn = jr;
    auto refill = [&]() {
      if (fit >= hi || *B.abort_flag) return;
      if (lane == 0) {
        const int base = fit / KS, ks = fit - base * KS;
        const int tile = base % ntiles;
        const int st = stage_of(B, warp, jn);
        bar_expect(&B.full[st], 2048u);
        tma2d(B.ring + (size_t)st * kSB, &mr, &B.full[st], (warp + kWarps * (ks * per + fj)) * 64,
              tile * 16);
      }
      ++jn;
      if (++fj == per) {
        fj = 0;
        ++fit;
      }
    };
    for (int i = 0; i < S; ++i) refill();
    float* part = reinterpret_cast<float*>(smem + Ly.part);
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(a.x);
    const int g = lane >> 2, t = lane & 3;
    uint32_t xf0[8], xf1[8];
    int xc = -1;
    for (int it = lo; it < hi; ++it) {
      const int base = it / KS, ks = it - base * KS;
      const int c = base / ntiles, tile = base - c * ntiles;
      const int nj = min(kNT, T - c * kNT);
      const bool valid = g < nj;
      const int tok = c * kNT + (valid ? g : 0);
      const int s0 = ks * per;  // first K segment of the item
      if (per <= 2 && c * KS + ks != xc) {
        dmma::x_frags(xb, d, tok, valid, (warp + kWarps * s0) * 64, lane, xf0);
        if (per == 2) dmma::x_frags(xb, d, tok, valid, (warp + kWarps * (s0 + 1)) * 64, lane, xf1);
        xc = c * KS + ks;
      }
      float dr[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < per; ++j) {
        uint32_t f[8];
        if (per <= 2) {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = j ? xf1[e] : xf0[e];
        } else {
          dmma::x_frags(xb, d, tok, valid, (warp + kWarps * (s0 + j)) * 64, lane, f);
        }
        const uint8_t* st = acquire(B, warp, jr, lane);
        if (!st) break;
        dmma::router_tile(st, f, lane, dr);
        release(jr, refill);
      }
      float* pw = part + warp * 256;
      pw[g * 8 + 2 * t] = dr[0];
      pw[g * 8 + 2 * t + 1] = dr[1];
      pw[(g + 8) * 8 + 2 * t] = dr[2];
      pw[(g + 8) * 8 + 2 * t + 1] = dr[3];
      __syncthreads();
      if (threadIdx.x < 128) {
        const int r = threadIdx.x >> 3, q = threadIdx.x & 7;
        const int col = tile * 16 + r;
        if (q < nj && col < E) {
          float z = 0.f;
          for (int w = 0; w < kWarps; ++w) z += part[w * 256 + r * 8 + q];
          // (a K split's parts go to consecutive [T][E+1] planes)
          a.logits[(size_t)ks * T * (E + 1) + (size_t)(c * kNT + q) * (E + 1) + col] = z;
        }
      }
      __syncthreads();
    }
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps * S; ++i) bar_init(&B.full[i], 1);
    s_misc[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  STAMP(0);

  // Tensor-core variant: phase 1's contractions are split in ks1 parts along
  // K when the unsplit items would leave more than half of the grid idle
  // (partial sums: router logits in ks1 planes added by the routing rule,
  // shared gate/up in Gs, turned into h in phase 2). It depends on the
  // shape only, so that a routing-only call splits as the layer does.
  static_assert(kDecodeKSplit == 2, "the routing rule adds at most two partial logits");
  int ks1 = 1;
  if constexpr (MMA) {
    const int nte = route ? (E + 15) / 16 : 0;
    const int nc = (T + kNT - 1) / kNT;
    const int n1 = nc * nte + (Is > 0 ? nc * (Is / 16) : 0);
    if ((d / 64 / kWarps) % kDecodeKSplit == 0 && n1 * kDecodeKSplit <= nb) ks1 = kDecodeKSplit;
  }

  // shared h from the K parts of phase 1 (this block's share of the T x Is
  // values, in fragment order for the down items), in phase 2 by warps that
  // route no token, or by all threads once routing is done
  auto shared_h = [&](int tid, int nthr) {
    const int n = T * Is;
    const int lo = (int)((long long)blockIdx.x * n / nb), hi = (int)((long long)(blockIdx.x + 1) * n / nb);
    __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(a.Hs);
    for (int i = lo + tid; i < hi; i += nthr) {
      const int t = i / Is, r = i - t * Is;
      float gs = __ldcg(a.Gs + i), us = __ldcg(a.Gs + (size_t)T * Is + i);
      for (int q = 1; q < ks1; ++q) {
        gs += __ldcg(a.Gs + (size_t)q * 2 * T * Is + i);
        us += __ldcg(a.Gs + (size_t)(q * 2 + 1) * T * Is + i);
      }
      hs[dmma::frag_index(t / kNT, Is, t % kNT, r)] = __float2bfloat16_rn(siluf_(gs) * us);
    }
  };
  const bool split_h = MMA && shared && ks1 > 1;
  // ------------------------------------------------------------- phase 1
  // logit items (token chunk, row): router rows 0..E-1 (route mode), then the
  // shared-gate row E when the gate is not given; then shared gate/up items
  // (token chunk, row). Items are balanced over blocks by their stage count.
  {
    const bool slogit = sgate && (route || a.s_in == nullptr);
    int tpc = (int)(32768 / ((size_t)d * sizeof(TW)));  // the router kernel's token chunks
    tpc = tpc < 1 ? 1 : (tpc > 8 ? 8 : tpc);
    const int ntc = (T + tpc - 1) / tpc;
    // (the tensor-core variant contracts the router rows and the shared-gate
    // row block-wide below)
    const int nlr = MMA ? 0 : (route ? E : 0) + (slogit ? 1 : 0);
    const int nL = nlr * ntc;
    const int nsh = (T + kNT - 1) / kNT;
    // (the tensor-core variant runs the shared gate/up rows block-wide after
    // the logit rows, so only the logit rows are balanced here)
    const int nS = (shared && !MMA) ? Is * nsh : 0;
    const long long cl = (d + kRowSeg - 1) / kRowSeg, cs = (d + kPairSeg - 1) / kPairSeg;
    const long long ctot = nL * cl + nS * cs;
    auto first_item = [&](long long cost) -> int {  // first item starting at or after cost
      if (cost <= nL * cl) return (int)((cost + cl - 1) / cl);
      return nL + (int)((cost - nL * cl + cs - 1) / cs);
    };
    const int lo = first_item(ctot * blockIdx.x / nb);
    const int hi = first_item(ctot * (blockIdx.x + 1) / nb);
    auto logit_row = [&](int it) -> const TW* {
      const int r = (route && !MMA) ? it / ntc : E;
      return r < E ? static_cast<const TW*>(a.W_router) + (size_t)r * d
                   : static_cast<const TW*>(a.w_shared);
    };
    auto describe = [&](int it, int e0, Copies& cp, int& K, int& seg) {
      K = d;
      if (it < nL) {
        seg = kRowSeg;
        cp.n = 1;
        cp.src[0] = logit_row(it) + e0;
        cp.bytes[0] = (uint32_t)(min(kRowSeg, d - e0) * sizeof(TW));
        cp.off[0] = 0;
      } else {
        seg = kPairSeg;
        const int r = (it - nL) % Is;
        const uint32_t n = (uint32_t)(min(kPairSeg, d - e0) * sizeof(TW));
        cp.n = 2;
        cp.src[0] = Wsg + (size_t)r * d + e0;
        cp.src[1] = Wsu + (size_t)r * d + e0;
        cp.bytes[0] = cp.bytes[1] = n;
        cp.off[0] = 0;
        cp.off[1] = kSB / 2;
      }
    };
    Feed f{lo + warp, hi, kWarps, 0, jr};
    auto refill = [&]() { issue(B, warp, f, describe, lane); };
    for (int i = 0; i < S; ++i) refill();
    const int nvec = d / Chunk<TW>::kVec;
    for (int it = lo + warp; it < hi && !*B.abort_flag; it += kWarps) {
      if (it < nL) {
        const int tc = it % ntc;
        const int r = (route && !MMA) ? it / ntc : E;
        const int t0 = tc * tpc, nt = min(tpc, T - t0);
        float acc[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[t] = 0.f;
        bool ok = true;
        for (int e0 = 0; e0 < d; e0 += kRowSeg) {
          const uint8_t* st = acquire(B, warp, jr, lane);
          if (!st) {
            ok = false;
            break;
          }
          const int cbase = e0 / Chunk<TW>::kVec;
          auto wl = [&](int cc) { return reinterpret_cast<const uint4*>(st)[cc - cbase]; };
          router_dots_pass<TW, 8>(wl, reinterpret_cast<const uint4*>(x + (size_t)t0 * d), nvec,
                                  nt, cbase + lane, acc);
          release(jr, refill);
        }
        if (!ok) break;
        router_dots_reduce<8>(acc, nt, lane);
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (lane == 0 && t < nt) a.logits[(size_t)(t0 + t) * (E + 1) + r] = acc[t];
      } else {
        const int sc = (it - nL) / Is, r = (it - nL) - sc * Is;
        const int t0 = sc * kNT, nj = min(kNT, T - t0);
        int tok[kNT];
#pragma unroll
        for (int q = 0; q < kNT; ++q) tok[q] = t0 + (q < nj ? q : 0);
        if (!gateup_any<TW>(B, warp, jr, refill, x, d, tok, nj, a.Hs, tok, (size_t)Is, r, lane))
          break;
      }
    }
    if constexpr (MMA) {
      // one list of block-wide items, router tiles of 16 experts first, then
      // the shared expert's 16-row blocks, each cut into ks1 K parts, cut
      // evenly over the blocks
      const int nte = route ? (E + 15) / 16 : 0;
      const int nR = ((T + kNT - 1) / kNT) * nte * ks1;
      const int nSh = shared ? nsh * (Is / 16) * ks1 : 0;
      int blo, bhi;
      block_range(nR + nSh, blo, bhi);
      // the shared-gate row: K split over all threads of one block with no
      // item (block 0 when the items do not fill the grid, else the last
      // block), one accumulator per token, summed in lane order within a
      // warp and in warp order across warps
      if (slogit && blockIdx.x == (nR + nSh < nb ? 0 : nb - 1)) {
        const uint4* wv = reinterpret_cast<const uint4*>(a.w_shared);
        const uint4* xv = reinterpret_cast<const uint4*>(x);
        const int nv = d / 8;
        float acc[kDecodeMaxTokens];
#pragma unroll
        for (int t = 0; t < kDecodeMaxTokens; ++t) acc[t] = 0.f;
        for (int c = threadIdx.x; c < nv; c += kThreads) {
          float wf[8];
          Chunk<TW>::unpack(__ldg(wv + c), wf);
#pragma unroll
          for (int h = 0; h < kDecodeMaxTokens; h += 8) {
            if (h < T) {
              // eight token rows at once (rows past T repeat the last one)
              uint4 xr[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) xr[u] = __ldg(xv + (size_t)min(h + u, T - 1) * nv + c);
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                float xf[8];
                Chunk<TW>::unpack(xr[u], xf);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h + u] = fmaf(wf[e], xf[e], acc[h + u]);
              }
            }
          }
        }
        float* part = reinterpret_cast<float*>(smem + Ly.part);
#pragma unroll
        for (int t = 0; t < kDecodeMaxTokens; ++t) {
          if (t < T) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) part[warp * kDecodeMaxTokens + t] = v;
          }
        }
        __syncthreads();
        if (threadIdx.x < T) {
          float z = 0.f;
          for (int w = 0; w < kWarps; ++w) z += part[w * kDecodeMaxTokens + threadIdx.x];
          a.logits[(size_t)threadIdx.x * (E + 1) + E] = z;
        }
        __syncthreads();
        STAMP(10);
      }
      router_items_mma(min(blo, nR), min(bhi, nR), nte, ks1);
      if (blo < nR) STAMP(8);
      if (shared) gateup_items_mma(max(blo, nR) - nR, max(bhi, nR) - nR, true, ks1);
      if (shared && bhi > nR) STAMP(9);
    }
  }
  STAMP(1);
  if (!grid_barrier(B, !(a.stall && blockIdx.x == 0))) goto drain;
  STAMP(2);

  // ------------------------------------------------------------- phase 2
  if (split_h && T < kWarps && warp >= T) shared_h(threadIdx.x - T * 32, kThreads - T * 32);
  if (route) {
    if (warp < T) {
      TopkArgs ta{};
      ta.logits = a.logits;
      ta.bias = a.kind == MOE_ROUTER_SIGMOID_GROUP_TOPK ? a.bias : nullptr;
      ta.topk_ids = s_ids;
      ta.weights = s_w;
      ta.s_shared = sgate ? s_ssh : nullptr;
      ta.T = T;
      ta.E = E;
      ta.k = k;
      ta.kind = a.kind;
      ta.n_group = a.n_group;
      ta.topk_group = a.topk_group;
      ta.has_shared_logit = sgate ? 1 : 0;
      ta.routed_scaling = a.routed_scaling;
      ta.renorm_clamp = a.renorm_clamp;
      ta.nparts = ks1;
      ta.part_stride = (size_t)T * (E + 1);
      topk_token_pl<PL>(ta, warp, lane);
    }
  } else {
    for (int p = threadIdx.x; p < P; p += kThreads) {
      s_ids[p] = a.ids_in[p];
      s_w[p] = a.w_in[p];
    }
    if (shared) {
      for (int t = threadIdx.x; t < T; t += kThreads)
        s_ssh[t] = a.s_in ? a.s_in[t]
                          : 1.0f / (1.0f + expf(-__ldcg(a.logits + (size_t)t * (E + 1) + E)));
    }
  }
  __syncthreads();
  if (split_h && T >= kWarps) {
    shared_h(threadIdx.x, kThreads);
    __syncthreads();
  }
  STAMP(3);
  if (sh_early && warp >= T) {
    const int nsh = (T + kNT - 1) / kNT;
    down_items(warp - T, (q1 - q0) * nsh, kWarps - T, 0, nsh);
  }
  if (route && blockIdx.x == 0) {
    for (int p = threadIdx.x; p < P; p += kThreads) {
      a.topk_ids[p] = s_ids[p];
      a.weights[p] = s_w[p];
    }
    if (a.route_only && a.s_out)
      for (int t = threadIdx.x; t < T; t += kThreads) a.s_out[t] = s_ssh[t];
  }
  if (a.route_only) return;
  // pairs sorted by (expert, pair id); ids outside [0, E) form no chunk
  for (int p = threadIdx.x; p < P; p += kThreads) {
    const int e = s_ids[p];
    const bool ok = e >= 0 && e < E;
    if (!ok && blockIdx.x == 0) report(a.ctrl, kDevBadId, kSiteDecode);
    s_key[p] = ok ? e : E;
  }
  __syncthreads();
  {
    // rank of pair p: G consecutive threads count over every G-th pair and
    // add their counts with shuffles (G a power of two, G P <= threads)
    int G = 16;
    while (G > 1 && G * P > kThreads) G >>= 1;
    const int p = threadIdx.x / G, sub = threadIdx.x & (G - 1);
    const int key = p < P ? s_key[p] : 0;
    int rank = 0;
    if (p < P)
      for (int q = sub; q < P; q += G) {
        const int kq = s_key[q];
        rank += (kq < key || (kq == key && q < p)) ? 1 : 0;
      }
    for (int o = G >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (p < P && sub == 0) s_gpair[rank] = p;
  }
  __syncthreads();
  // chunks: runs of one expert in the sorted order, cut every kNT pairs
  if (warp == 0) {
    int nch = 0, nvalid = 0, run0 = 0;
    for (int base = 0; base < P; base += 32) {
      const int r = base + lane;
      const int key = r < P ? s_key[s_gpair[r]] : E;
      const int prev = (r > 0 && r < P) ? s_key[s_gpair[r - 1]] : -1;
      const bool head = r < P && key < E && key != prev;
      // start of this pair's run: the last head at or before it
      const unsigned hm = __ballot_sync(0xffffffffu, head);
      const unsigned below = hm & (0xffffffffu >> (31 - lane));
      const int my_run0 = below ? base + 31 - __clz(below) : run0;
      const bool cut = r < P && key < E && ((r - my_run0) % kNT) == 0;
      const unsigned cm = __ballot_sync(0xffffffffu, cut);
      if (cut) {
        const int ch = nch + __popc(cm & ((1u << lane) - 1u));
        s_cstart[ch] = r;
        s_cexp[ch] = key;
      }
      nch += __popc(cm);
      nvalid += __popc(__ballot_sync(0xffffffffu, r < P && key < E));
      run0 = __shfl_sync(0xffffffffu, my_run0, 31);
    }
    if (lane == 0) {
      s_cstart[nch] = nvalid;
      s_misc[0] = nch;
    }
  }
  __syncthreads();
  {
    const int nch = s_misc[0];
    STAMP(4);
    if constexpr (MMA) {
      // phase 4's plan: (8-column group, chunk) items over the whole grid,
      // evenly, chunk-major, so that a block's range touches one or two
      // chunks, whose h fragments are copied to shared memory once when
      // they fit; the results go to the workspace and meet after one more
      // barrier. With h in shared memory the rings are filled before the
      // barrier.
      const int nsh = shared ? (T + kNT - 1) / kNT : 0;
      int lo4, hi4;
      block_range(nq * (nch + nsh), lo4, hi4);
      pl4 = DnPlan{lo4 + warp, hi4, kWarps, nch, nch + nsh, 0, nq, 0, nullptr};
      if (lo4 < hi4) {
        const int hc0 = lo4 / nq, hc1 = (hi4 - 1) / nq;
        size_t bytes = 0;
        for (int c = hc0; c <= hc1; ++c) bytes += (size_t)(c < nch ? I : Is) * 16;
        if (bytes <= (size_t)kPartBytes) {
          pl4.hc0 = hc0;
          pl4.hs = reinterpret_cast<const uint2*>(smem + Ly.part);
        }
      }
    }
    // ----------------------------------------------------------- phase 3
    int lo, hi;
    if constexpr (MMA) {
      block_range(nch * (I / 16), lo, hi);
      gateup_items_mma(lo, hi, false, 1);
      lo = hi = 0;  // the per-warp rows below have no work
    } else {
      block_range(nch * I, lo, hi);
    }
    auto describe = [&](int it, int e0, Copies& cp, int& K, int& seg) {
      K = d;
      seg = kPairSeg;
      const int ch = it / I, r = it - ch * I;
      const size_t rb = ((size_t)s_cexp[ch] * I + r) * d + e0;
      const uint32_t n = (uint32_t)(min(kPairSeg, d - e0) * sizeof(TW));
      cp.n = 2;
      cp.src[0] = Wg + rb;
      cp.src[1] = Wu + rb;
      cp.bytes[0] = cp.bytes[1] = n;
      cp.off[0] = 0;
      cp.off[1] = kSB / 2;
    };
    Feed f{lo + warp, hi, kWarps, 0, jr};
    auto refill = [&]() { issue(B, warp, f, describe, lane); };
    for (int i = 0; i < S; ++i) refill();
    for (int it = lo + warp; it < hi && !*B.abort_flag; it += kWarps) {
      const int ch = it / I, r = it - ch * I;
      const int cs = s_cstart[ch], nj = min(kNT, s_cstart[ch + 1] - cs);
      int tok[kNT], prow[kNT];
#pragma unroll
      for (int q = 0; q < kNT; ++q) {
        prow[q] = s_gpair[cs + (q < nj ? q : 0)];
        tok[q] = prow[q] / k;
      }
      if (!gateup_any<TW>(B, warp, jr, refill, x, d, tok, nj, a.H, prow, (size_t)I, r, lane))
        break;
    }
    if constexpr (MMA) {
      if (pl4.hs) dn_prime(pl4, f4);
    }
  }
  STAMP(5);
  if (!grid_barrier(B, true)) goto drain;
  STAMP(6);

  // ------------------------------------------------------------- phase 4
  {
    const int nch = s_misc[0];
    const int nsh = (shared && !sh_early) ? (T + kNT - 1) / kNT : 0;
    if constexpr (MMA) {
      if (pl4.hs) {
        const int lo4 = pl4.it0 - warp, hi4 = pl4.it1;
        uint4* dst = reinterpret_cast<uint4*>(smem + Ly.part);
        size_t o = 0;
        for (int c = lo4 / nq; c <= (hi4 - 1) / nq; ++c) {
          const bool rt = c < nch;
          const int K = rt ? I : Is;
          const uint4* src = reinterpret_cast<const uint4*>(
              reinterpret_cast<const __nv_bfloat16*>(rt ? a.H : a.Hs) +
              dmma::frag_index(rt ? c : c - nch, K, 0, 0));
          for (int i = threadIdx.x; i < K; i += kThreads) dst[o + i] = __ldcg(src + i);
          o += K;
        }
      }
      __syncthreads();
      STAMP(12);
      if (!pl4.hs) dn_prime(pl4, f4);
      dn_run(pl4, f4);
      STAMP(11);
    } else {
      down_items(warp, (q1 - q0) * (nch + nsh), kWarps, nch, nch + nsh);
    }
  }
  if constexpr (MMA) {
    if (!grid_barrier(B, true)) goto drain;
  }
  __syncthreads();
  STAMP(7);
  if (*B.abort_flag) goto drain;
  // out = r_attn + ((sum over slots, in slot order) + shared)
  for (int i = threadIdx.x; i < T * ncols; i += kThreads) {
    const int t = i / ncols, cc = i - t * ncols;
    const float* yr = (MMA ? a.Yg + (size_t)c0 * Ly.ystride : s_y) + (size_t)cc * Ly.ystride;
    float acc = 0.f;
    for (int s = 0; s < k; ++s) {
      const int p = t * k + s;
      if (s_key[p] < E) acc += MMA ? __ldcg(yr + p) : yr[p];
    }
    if (shared) acc += MMA ? __ldcg(yr + P + t) : yr[P + t];
    const size_t o = (size_t)t * d + c0 + cc;
    a.out[o] = a.r_attn[o] + acc;
  }
  return;

drain:
  // a wait gave up (here or in another block): let this block's copies in
  // flight land before its shared memory is released
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  __syncthreads();
}

template <typename TW, int PL, bool MMA>
cudaError_t launch_pl(const DecodeArgs& a, cudaStream_t st) {
  static int attr[64] = {};
  const int nb = tc_sm_count();
  const int ncols = max_cols(a.d, nb, MMA ? 8 : 4);
  const int S = ring_stages(a.T, a.k, ncols, MMA);
  if (S == 0) return cudaErrorInvalidValue;
  const Layout L = layout(a.T, a.k, ncols, S, MMA);
  cudaError_t e = ensure_smem_limit(decode_fused_kernel<TW, PL, MMA>, L.bytes, attr);
  if (e != cudaSuccess) return e;
  DecodeMaps m;
  memset(&m, 0, sizeof(m));
  if (MMA) {
    const uint64_t E = a.E, I = a.I, d = a.d, Is = a.Is;
    bool ok = a.route_only ||
              (tc_make_map(&m.g, a.Wg, E * I, d, 16) && tc_make_map(&m.u, a.Wu, E * I, d, 16) &&
               tc_make_map(&m.dn, a.Wd, E * d, I, 8));
    if (ok && Is > 0 && !a.route_only)
      ok = tc_make_map(&m.sg, a.Wsg, Is, d, 16) && tc_make_map(&m.su, a.Wsu, Is, d, 16) &&
           tc_make_map(&m.sdn, a.Wsd, d, Is, 8);
    if (ok && a.W_router) ok = tc_make_map(&m.r, a.W_router, E, d, 16);
    if (!ok) return cudaErrorInvalidValue;
  }
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nb);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.bytes;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel<TW, PL, MMA>, m.g, m.u, m.sg, m.su, m.dn,
                            m.sdn, m.r, a);
}

template <typename TW, bool MMA>
cudaError_t launch_tw(const DecodeArgs& a, cudaStream_t st) {
  if (a.E <= 32) return launch_pl<TW, 1, MMA>(a, st);
  if (a.E <= 64) return launch_pl<TW, 2, MMA>(a, st);
  if (a.E <= 128) return launch_pl<TW, 4, MMA>(a, st);
  if (a.E <= 256) return launch_pl<TW, 8, MMA>(a, st);
  return launch_pl<TW, 16, MMA>(a, st);
}

}  // namespace

bool decode_fused_supported(int T, int d, int E, int k, int I, int Is, int act, int wdt) {
  if (T < 1 || T > kDecodeMaxTokens || E > 512 || k > 32) return false;
  if (!((act == MOE_BF16 && wdt == MOE_BF16) || (act == MOE_F32 && wdt == MOE_F32))) return false;
  if (d % 8 != 0 || I % 8 != 0 || Is % 8 != 0) return false;
  const bool mma = mma_shape(d, I, Is, act == MOE_BF16);
  return ring_stages(T, k, max_cols(d, tc_sm_count(), mma ? 8 : 4), mma) > 0;
}

bool decode_fused_mma(int d, int I, int Is) { return mma_shape(d, I, Is, true); }

cudaError_t launch_decode_fused(const DecodeArgs& a, bool bf16, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (!bf16) return launch_tw<float, false>(a, st);
  if (mma_shape(a.d, a.I, a.Is, true)) return launch_tw<__nv_bfloat16, true>(a, st);
  return launch_tw<__nv_bfloat16, false>(a, st);
}

}  // namespace moe
