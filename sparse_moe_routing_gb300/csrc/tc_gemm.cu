// Persistent grouped GEMM on the fifth-generation tensor cores (sm_103a):
// TMA tile loads (128-byte swizzle) feed a multi-stage mbarrier pipeline, one
// elected thread issues tcgen05.mma (bf16 x bf16 -> fp32) into a
// double-buffered TMEM accumulator, and four epilogue warps drain TMEM with
// tcgen05.ld and apply the fused epilogue while the next tile accumulates.
//
// Three uses, one kernel template:
//  * gate/up ("How Treebeard routes Qwen3.6 MoE tokens", "Routed expert
//    computation"; Edge0 "Experts"): per active expert, H = SiLU(X W_gate^T)
//    * (X W_up^T); the gate and up tiles of the same 128 intermediate columns
//    share one N = 256 instruction, so SwiGLU is applied straight from TMEM;
//  * down: Y = alpha * (H W_down^T), the routing weight (or, for the shared
//    expert, its sigmoid gate) applied in the epilogue;
//  * router ("Routing math": z_t = W_router x_t) for large token batches:
//    one dense problem, fp32 logits out.
// Work items are (group, 128-row block, N tile); groups are the active
// experts packed by the bucketing pass ("Intel SYCL path": launch over
// active experts, load each weight block once per token block) plus the
// shared expert as group E. CTAs stride over the item list.
//
// Every wait is bounded: a wait that exceeds about one second records
// kDevTimeout in the workspace status word and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// Warp roles: warp 0 TMA producer, warp 1 MMA issuer + TMEM owner, warps 2-5
// epilogue, and (4-bit weights only) warps 6-13 dequantise the B stages and
// warp 14 brings their raw codes.
constexpr int BM = 128, BK = 64;
constexpr uint32_t kTmemCols = 512;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `bar` with the given parity; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 63u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 128-byte-swizzled, K-major shared-memory matrix descriptor: rows of 128 B,
// 8-row atoms 1024 B apart (stride byte offset), version bits for tcgen05.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(p)), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p))
               : "memory");
  return v;
}
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

struct TileInfo {
  int g, m, nt, row0, rows;
  bool shared;
};

// Item t -> (row block, N tile). Items walk bands of kBandRows consecutive
// row blocks N tile by N tile, so the CTAs in flight at one time share each
// weight tile across the row blocks of a band (one DRAM read, the rest L2
// hits) while the band's activation rows stay L2-resident. The last band may
// be narrower; the map is a bijection onto [0, n_rb) x [0, n_tiles).
constexpr int kBandRows = 8;

template <int MODE>
__device__ __forceinline__ TileInfo decode_tile(const TcArgs& a, int t, int n_rb) {
  TileInfo ti;
  const int span = kBandRows * a.n_tiles;
  const int band = t / span;
  const int rb0 = band * kBandRows;
  const int width = min(kBandRows, n_rb - rb0);
  const int w = t - band * span;
  const int rb = rb0 + w % width;
  ti.nt = w / width;
  if (MODE == kTcRouter) {
    ti.g = 0;
    ti.m = rb;
    ti.row0 = 0;
    ti.rows = a.T;
    ti.shared = false;
  } else if (a.shared_only) {
    ti.g = a.E;
    ti.m = rb;
    ti.row0 = 0;
    ti.rows = a.T;
    ti.shared = true;
  } else {
    const int2 r = a.rowblocks[rb];
    ti.g = r.x;
    ti.m = r.y;
    if (ti.g < a.E) {
      ti.row0 = a.offsets[ti.g];
      ti.rows = a.offsets[ti.g + 1] - ti.row0;
      ti.shared = false;
    } else {
      ti.row0 = 0;
      ti.rows = a.T;
      ti.shared = true;
    }
  }
  return ti;
}

__device__ __forceinline__ void give_up(const TcArgs& a, volatile int* abort_flag, int site) {
  *abort_flag = 1;
  report(a.ctrl, kDevTimeout, site);
}

// Down epilogue staging: per epilogue warp, 32 rows x 128 B of bf16 output
// (64 columns), rows padded to 144 B so that both the row-wise writes and the
// column-wise reads of the transpose are free of bank conflicts.
constexpr int kEpiRowBytes = 144;
constexpr int kEpiWarpBytes = 32 * kEpiRowBytes;

// 4-bit weights: warps 6 .. 6 + kDequantWarps - 1 dequantise the B stages,
// one B row (of 256) per thread; warp 6 + kDequantWarps brings the raw codes.
constexpr int kDequantWarps = 8;

// Shared-memory plan of one CTA (1024-byte aligned stages). bf16: kStages
// stages of A + B, filled by one TMA producer and freed by the MMA. 4-bit:
// three rings. kStages A stages (TMA, freed by the MMA); kCStages raw-code
// stages (TMA from a second producer warp, freed by the dequant warps once
// they have read them); kBStages dequantised B stages (filled by the dequant
// warps, freed by the MMA). The code ring runs furthest ahead, so that the
// dequantisation of a stage never waits for its codes to cross DRAM; the A
// ring only has to land before the MMA reaches it. EPI: the down epilogue's
// staging rows (the other modes leave that shared memory to the pipeline).
//
// RB = row blocks per work item. RB = 2 ("paired" items, used for 4-bit
// banks): two 128-row blocks of one group share each B stage (two A tiles
// per stage, two MMAs per k-block into two 256-column accumulators that fill
// TMEM), halving the B traffic and the dequantisation per flop; the
// accumulator is then single-buffered.
// NB = rows of the largest B tile the plan holds: 256, or 128 for bf16
// gate/up items with 64 + 64-column N tiles (decode batches).
// AR = rows of the A tile TMA brings per stage: 128, or 64 / 16 for bf16
// decode batches whose groups all hold at most that many rows. The MMA still
// reads 128 A rows from the stage's base; rows past AR hold whatever the
// following shared memory holds and only feed accumulator rows past the
// group's last row, which the epilogue never stores.
// The narrower plans (NB < 256 or AR < 128) fit as many stages as 227 KB
// allows, at most 12, so that more weight bytes are in flight per SM.
template <bool Q4, int RB, bool EPI, int NB = 256, int AR = 128>
struct SmemPlan {
  static_assert(NB == 256 || (NB == 128 && !Q4 && RB == 1), "128-row B plan: bf16, unpaired");
  static_assert(AR == 128 || ((AR == 64 || AR == 16) && !Q4 && RB == 1), "short A: bf16, unpaired");
  static constexpr int kStageA = AR * BK * 2;  // bytes of one A stage
  static constexpr int kStageB = NB * BK * 2;  // bytes of one B stage
  static constexpr int kStageQ = 256 * (BK / 2);  // raw 4-bit codes of one B stage
  static constexpr size_t kEpiBytes = EPI ? 4 * (size_t)kEpiWarpBytes : 0;
  static constexpr size_t kAvail = 227 * 1024 - 2048 - kEpiBytes;
  static constexpr int kFit = (int)(kAvail / (kStageA + kStageB));
  static constexpr bool kNarrow = !Q4 && RB == 1 && (NB < 256 || AR < 128);
  static constexpr int kBStages = Q4 ? ((EPI && RB == 2) ? 2 : 3) : 0;
  static constexpr int kCStages = Q4 ? 4 : 0;
  static constexpr int kQ4Fit =
      (int)((kAvail - (size_t)kBStages * kStageB - (size_t)kCStages * kStageQ) /
            ((size_t)RB * kStageA));
  static constexpr int kStages =
      Q4 ? (kQ4Fit > 5 ? 5 : kQ4Fit)
         : (kNarrow ? (kFit > 12 ? 12 : kFit) : (RB == 2 ? (EPI ? 3 : 4) : 4));
  static constexpr int kNAcc = 2 / RB;   // accumulator buffers of RB x 256 TMEM columns
  static constexpr int kThreadsCta = Q4 ? 192 + 32 * kDequantWarps + 32 : 192;
  static constexpr size_t kA = 0;
  static constexpr size_t kB = kA + (size_t)kStages * RB * kStageA;
  static constexpr size_t kQ = kB + (size_t)(Q4 ? kBStages : kStages) * kStageB;
  static constexpr size_t kEpi = kQ + (size_t)kCStages * kStageQ;
  static constexpr size_t kBars = kEpi + kEpiBytes;
  // full and empty per A (+ B for bf16) stage; rawfull and rawempty per code
  // stage; bfull and bempty per B stage; tfull and tempty per accumulator
  // (two slots each); then the TMEM address word and the abort flag
  static constexpr size_t kBarBytes =
      ((2 * kStages + 2 * kCStages + 2 * kBStages + 4) * 8 + 8 + 127) / 128 * 128;
  static constexpr size_t kBytes = 1024 + kBars + kBarBytes;
  static_assert(kBytes <= 227 * 1024, "shared memory plan exceeds 227 KB");
  static_assert(!Q4 || kStages >= 3, "4-bit plan: at least three A stages");
};

// The (scale, min) arrays of the B row a dequant thread owns: bank row and
// base pointers (gate/up: rows 0-127 gate, 128-255 up of N tile nt; down:
// 256 rows of N tile nt).
struct QRow {
  const __nv_bfloat16* qs;
  const __nv_bfloat16* qm;
  size_t grow;
};
template <int MODE>
__device__ __forceinline__ QRow q_row(const TcArgs& a, const TileInfo& ti, int r) {
  QRow q;
  if (MODE == kTcGateUp) {
    q.grow = (size_t)ti.g * a.brows_routed + (size_t)ti.nt * 128 + (r & 127);
    q.qs = r < 128 ? a.qs0 : a.qs1;
    q.qm = r < 128 ? a.qm0 : a.qm1;
  } else {
    q.grow = (size_t)ti.g * a.brows_routed + (size_t)ti.nt * 256 + r;
    q.qs = a.qs0;
    q.qm = a.qm0;
  }
  return q;
}

// bf16 element j (0..7) of a 16-byte vector, as raw bits.
__device__ __forceinline__ uint32_t bf16_at(const uint4& v, int j) {
  const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
  return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Dequantises one B row of a stage: 64 4-bit codes (one affine group) into
// 64 bf16 w = scale * q + min, written in the 128-byte-swizzled K-major
// layout that a bf16 TMA tile would have. Arithmetic in packed bf16: a code
// nibble e becomes the bf16 128 + e by OR-ing it into 0x4300 (2^7, mantissa
// e), 128 is subtracted exactly, and one fused multiply-add rounds
// scale * q + min once.
__device__ __forceinline__ void dequant_row(const uint8_t* q_row_src, uint8_t* b_stage, int r,
                                            uint32_t scale_bits, uint32_t min_bits) {
  const __nv_bfloat162 s2 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)scale_bits),
                                                __ushort_as_bfloat16((unsigned short)scale_bits));
  const __nv_bfloat162 m2 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)min_bits),
                                                __ushort_as_bfloat16((unsigned short)min_bits));
  const __nv_bfloat162 b128 = __float2bfloat162_rn(128.0f);
  const uint4 c0 = reinterpret_cast<const uint4*>(q_row_src)[0];
  const uint4 c1 = reinterpret_cast<const uint4*>(q_row_src)[1];
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  uint8_t* row_base = b_stage + (r >> 3) * 1024 + (r & 7) * 128;
  auto deq = [&](uint32_t pair_bits) {  // (128 + e_lo, 128 + e_hi) -> (w_lo, w_hi)
    __nv_bfloat162 q = *reinterpret_cast<__nv_bfloat162*>(&pair_bits);
    const __nv_bfloat162 w = __hfma2(__hsub2(q, b128), s2, m2);
    return *reinterpret_cast<const uint32_t*>(&w);
  };
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    // word c holds elements 8c..8c+7, the even element in the low nibble:
    // element e at bits 4e..4e+3
    const uint32_t x = words[c];
    const uint32_t h04 = deq((x & 0x000F000Fu) | 0x43004300u);          // e0, e4
    const uint32_t h15 = deq(((x >> 4) & 0x000F000Fu) | 0x43004300u);   // e1, e5
    const uint32_t h26 = deq(((x >> 8) & 0x000F000Fu) | 0x43004300u);   // e2, e6
    const uint32_t h37 = deq(((x >> 12) & 0x000F000Fu) | 0x43004300u);  // e3, e7
    st_shared_v4(row_base + ((c ^ (r & 7)) << 4), __byte_perm(h04, h15, 0x5410),
                 __byte_perm(h26, h37, 0x5410), __byte_perm(h04, h15, 0x7632),
                 __byte_perm(h26, h37, 0x7632));
  }
}

template <int MODE, bool Q4, int RB, int NB, int AR>
__global__ void __launch_bounds__(SmemPlan<Q4, RB, MODE == kTcDown, NB, AR>::kThreadsCta, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmB3,
                   const TcArgs a) {
  using SP = SmemPlan<Q4, RB, MODE == kTcDown, NB, AR>;
  constexpr int STAGES = SP::kStages;
  constexpr int kStageA = SP::kStageA;
  constexpr int kStageB = SP::kStageB;
  constexpr int NACC = SP::kNAcc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + SP::kA;
  uint8_t* sB = smem + SP::kB;
  uint8_t* sQ = smem + SP::kQ;
  uint8_t* sEpi = smem + SP::kEpi;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SP::kBars);  // A (+ B for bf16) landed
  uint64_t* empty = full + STAGES;
  uint64_t* rawfull = empty + STAGES;           // Q4 only: raw codes landed
  uint64_t* rawempty = rawfull + SP::kCStages;  // Q4 only: codes read by every dequant warp
  uint64_t* bfull = rawempty + SP::kCStages;    // Q4 only: B stage dequantised
  uint64_t* bempty = bfull + SP::kBStages;      // Q4 only: B stage consumed
  uint64_t* tfull = bempty + SP::kBStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int site = MODE == kTcGateUp ? kSiteTcGateUp : (MODE == kTcDown ? kSiteTcDown : kSiteTcRouter);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < SP::kCStages; ++s) {
      mbar_init(&rawfull[s], 1);
      mbar_init(&rawempty[s], kDequantWarps);  // one arrival per dequant warp
    }
    for (int s = 0; s < SP::kBStages; ++s) {
      mbar_init(&bfull[s], kDequantWarps);  // one arrival per dequant warp
      mbar_init(&bempty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t lim = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  pdl_wait();
  pdl_trigger();

  const int n_rb = (MODE == kTcRouter || a.shared_only) ? (a.T + BM - 1) / BM : *a.n_rowblocks;
  const int total = n_rb * a.n_tiles;
  const int nkb = a.K / BK;

  // Every role loop below is run by its whole warp, so that each warp reaches
  // the closing CTA barrier converged; lane 0 issues the TMA copies and the
  // MMAs. A wait's outcome is lane 0's, broadcast to the warp.
  if (warp == 0) {
    // -------------------------------------------------------------- producer
    // A tiles (+ bf16 B tiles) land on full[]; 4-bit codes come from their
    // own producer warp.
    const uint32_t stage_bytes = Q4 ? kStageA : kStageA + a.bn * BK * 2;
    int stage = 0;
    uint32_t ph = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
      const TileInfo ti = decode_tile<MODE>(a, t, n_rb);
      const CUtensorMap* mA = ti.shared ? &tmA1 : &tmA0;
      const CUtensorMap* mB0 = ti.shared ? &tmB2 : &tmB0;
      const CUtensorMap* mB1 = ti.shared ? &tmB3 : &tmB1;
      const int arow = ti.row0 + ti.m * BM;
      const int bhalf = MODE == kTcGateUp ? a.bn / 2 : a.bn;
      const int brow = (ti.shared || MODE == kTcRouter ? 0 : ti.g * a.brows_routed) +
                       ti.nt * bhalf;
      const bool two = RB == 2 && (ti.m + 1) * BM < ti.rows;  // second row block present
      const uint32_t item_bytes = stage_bytes + (two ? kStageA : 0);
      for (int kb = 0; kb < nkb; ++kb) {
        bool ok = lane == 0 ? mbar_wait(&empty[stage], ph ^ 1u, lim) : true;
        ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort_flag;
        if (!ok) {
          if (lane == 0) give_up(a, abort_flag, site);
          alive = false;
          break;
        }
        if (lane == 0) {
          uint64_t* bar = &full[stage];
          mbar_expect_tx(bar, item_bytes);
          tma_load_2d(sA + stage * RB * kStageA, mA, bar, kb * BK, arow);
          if (two) tma_load_2d(sA + (stage * RB + 1) * kStageA, mA, bar, kb * BK, arow + BM);
          if (!Q4) {
            uint8_t* b_dst = sB + stage * kStageB;
            tma_load_2d(b_dst, mB0, bar, kb * BK, brow);
            if (MODE == kTcGateUp)
              tma_load_2d(b_dst + bhalf * BK * 2, mB1, bar, kb * BK, brow);
          }
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16(BM, a.bn);
    int stage = 0, acc = 0, bs = 0;
    uint32_t ph = 0, aph = 0, bph = 0;
    bool alive = true;
    if (a.stall) {
      // failure self-test: wait on the first accumulator's full barrier,
      // which only this warp would complete, until the wait gives up
      bool ok = lane == 0 ? mbar_wait(&tfull[0], 0u, lim) : true;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) give_up(a, abort_flag, site);
        alive = false;
      }
    }
    for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
      bool two = false;
      if (RB == 2) {
        const TileInfo ti = decode_tile<MODE>(a, t, n_rb);
        two = (ti.m + 1) * BM < ti.rows;
      }
      bool ok = lane == 0 ? mbar_wait(&tempty[acc], aph ^ 1u, lim) : true;
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort_flag;
      if (!ok) {
        if (lane == 0) give_up(a, abort_flag, site);
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256 * RB);
      for (int kb = 0; kb < nkb; ++kb) {
        ok = true;
        if (lane == 0) {
          ok = mbar_wait(&full[stage], ph, lim);             // the A (+ bf16 B) tiles
          if (Q4 && ok) ok = mbar_wait(&bfull[bs], bph, lim);  // the dequantised B stage
        }
        ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort_flag;
        if (!ok) {
          if (lane == 0) give_up(a, abort_flag, site);
          alive = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t b_base = smem_u32(sB + (Q4 ? bs : stage) * kStageB);
#pragma unroll
          for (int j = 0; j < RB; ++j) {
            if (j == 0 || two) {
              const uint32_t a_base = smem_u32(sA + (stage * RB + j) * kStageA);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                mma_bf16(d_tmem + j * 256, sw128_desc(a_base + k * 32),
                         sw128_desc(b_base + k * 32), idesc, (kb | k) != 0 ? 1u : 0u);
              }
            }
          }
          mma_commit(&empty[stage]);
          if (Q4) mma_commit(&bempty[bs]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
        if (Q4 && ++bs == SP::kBStages) {
          bs = 0;
          bph ^= 1u;
        }
      }
      if (!alive) break;
      if (lane == 0) mma_commit(&tfull[acc]);
      __syncwarp();
      if (++acc == NACC) {
        acc = 0;
        aph ^= 1u;
      }
    }
  } else if (warp < 6) {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
      const TileInfo ti = decode_tile<MODE>(a, t, n_rb);
      bool ok = lane == 0 ? mbar_wait(&tfull[acc], aph, lim) : true;
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort_flag;
      if (!ok) {
        if (lane == 0) give_up(a, abort_flag, site);
        break;
      }
      tc_fence_after();
      for (int j = 0; j < RB; ++j) {
        const int mb = ti.m + j;  // row block of this accumulator
        if (j > 0 && mb * BM >= ti.rows) break;
        const uint32_t tbase =
            tmem_base + (uint32_t)(acc * 256 * RB + j * 256) + ((uint32_t)(q * 32) << 16);
        const int i = mb * BM + r;  // row inside the group
        const bool valid = i < ti.rows;
        if (MODE == kTcGateUp) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(ti.shared ? a.out_shared : a.out_routed);
          __nv_bfloat16* dst = out + (size_t)(ti.row0 + i) * a.ld_out + ti.nt * (a.bn / 2);
          const int half = a.bn / 2;
          for (int c0 = 0; c0 < half; c0 += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(tbase + c0, g);
            tmem_ld32(tbase + half + c0, u);
            tmem_ld_wait();
            if (valid) {
              uint32_t h[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
                const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
                h[j] = pack_bf16x2(siluf_(g0) * u0, siluf_(g1) * u1);
              }
#pragma unroll
              for (int v = 0; v < 4; ++v)
                st_global_v4(dst + c0 + 8 * v, h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
            }
          }
        } else if (MODE == kTcDown) {
          // Each thread scales and packs its own row (64 columns = 128 B per
          // step) into the warp's staging rows; the warp then stores 4 rows x
          // 128 B per instruction, whole cache lines instead of 16 B pieces of
          // 32 rows.
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(ti.shared ? a.out_shared : a.out_routed);
          float scale = 0.f;
          if (valid) scale = ti.shared ? a.s_shared[i] : a.alpha[a.perm[ti.row0 + i]];
          uint8_t* wbuf = sEpi + (size_t)(warp - 2) * kEpiWarpBytes;
          uint8_t* myrow = wbuf + lane * kEpiRowBytes;
          const int rsub = lane >> 3, ch = lane & 7;  // store phase: row in a group of 4, chunk
          for (int c0 = 0; c0 < a.bn; c0 += 64) {
            uint32_t v0[32], v1[32];
            tmem_ld32(tbase + c0, v0);
            tmem_ld32(tbase + c0 + 32, v1);
            tmem_ld_wait();
            auto pk = [&](const uint32_t* v, int o) {
              return pack_bf16x2(scale * __uint_as_float(v[o]), scale * __uint_as_float(v[o + 1]));
            };
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              st_shared_v4(myrow + 16 * w, pk(v0, 8 * w), pk(v0, 8 * w + 2), pk(v0, 8 * w + 4),
                           pk(v0, 8 * w + 6));
              st_shared_v4(myrow + 64 + 16 * w, pk(v1, 8 * w), pk(v1, 8 * w + 2), pk(v1, 8 * w + 4),
                           pk(v1, 8 * w + 6));
            }
            __syncwarp();
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const int rr = 4 * g + rsub;                  // row within the warp's 32
              const int gi = mb * BM + q * 32 + rr;       // row inside the group
              const uint4 v = ld_shared_v4(wbuf + rr * kEpiRowBytes + ch * 16);
              __nv_bfloat16* dst = out + (size_t)(ti.row0 + gi) * a.ld_out + ti.nt * a.bn + c0;
              if (gi < ti.rows) st_global_v4(dst + ch * 8, v.x, v.y, v.z, v.w);
            }
            __syncwarp();
          }
        } else {
          float* out = static_cast<float*>(a.out_routed) + (size_t)i * a.ld_out + ti.nt * a.bn;
          for (int c0 = 0; c0 < a.bn; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + c0, v);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
              for (int j = 0; j < 32; ++j) out[c0 + j] = __uint_as_float(v[j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == NACC) {
        acc = 0;
        aph ^= 1u;
      }
    }
  } else if (Q4 && warp >= 6 + kDequantWarps) {
    // ------------------------------------------------------- code producer
    // Raw 4-bit codes of each (tile, k-block) into the code ring, as soon as
    // every dequant warp has read the stage's previous contents.
    int cs = 0;
    uint32_t cph = 0;
    bool alive = true;
    const uint32_t code_bytes = a.bn * (BK / 2);
    for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
      const TileInfo ti = decode_tile<MODE>(a, t, n_rb);
      const CUtensorMap* mB0 = ti.shared ? &tmB2 : &tmB0;
      const CUtensorMap* mB1 = ti.shared ? &tmB3 : &tmB1;
      const int bhalf = MODE == kTcGateUp ? a.bn / 2 : a.bn;
      const int brow = (ti.shared ? 0 : ti.g * a.brows_routed) + ti.nt * bhalf;
      for (int kb = 0; kb < nkb; ++kb) {
        bool ok = lane == 0 ? mbar_wait(&rawempty[cs], cph ^ 1u, lim) : true;
        ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort_flag;
        if (!ok) {
          if (lane == 0) give_up(a, abort_flag, site);
          alive = false;
          break;
        }
        if (lane == 0) {
          uint64_t* bar = &rawfull[cs];
          mbar_expect_tx(bar, code_bytes);
          uint8_t* q_dst = sQ + cs * SP::kStageQ;
          tma_load_2d(q_dst, mB0, bar, kb * (BK / 2), brow);
          if (MODE == kTcGateUp) tma_load_2d(q_dst + bhalf * (BK / 2), mB1, bar, kb * (BK / 2), brow);
        }
        __syncwarp();
        if (++cs == SP::kCStages) {
          cs = 0;
          cph ^= 1u;
        }
      }
    }
  } else if (Q4) {
    // --------------------------------------------------------------- dequant
    // The dequant warps follow the producers' (tile, k-block) order: wait for
    // the code stage and a free B stage, write the bf16 B stage, make the
    // generic-proxy writes visible to the tensor core's async proxy, then
    // arrive on bfull[] and rawempty[] (one arrival per warp each). Thread r
    // owns B row r. When a row's group count is a multiple of 8, its scales
    // and mins are read 8 groups (16 B) at a time, one block of 8 k-blocks
    // ahead of use.
    const int r = threadIdx.x - 192;  // B row of this thread
    const bool vec = (a.qgroups & 7) == 0;
    int cs = 0, bs = 0;
    uint32_t cph = 0, bph = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
      const TileInfo ti = decode_tile<MODE>(a, t, n_rb);
      const QRow qr = q_row<MODE>(a, ti, r);
      const uint4* sv = reinterpret_cast<const uint4*>(qr.qs + qr.grow * a.qgroups);
      const uint4* mv = reinterpret_cast<const uint4*>(qr.qm + qr.grow * a.qgroups);
      uint4 sc{}, mn{}, sc_next{}, mn_next{};
      if (vec) {
        sc_next = __ldg(sv);
        mn_next = __ldg(mv);
      }
      for (int kb = 0; kb < nkb; ++kb) {
        uint32_t sbits, mbits;
        if (vec) {
          if ((kb & 7) == 0) {
            sc = sc_next;
            mn = mn_next;
            if (kb + 8 < nkb) {
              sc_next = __ldg(sv + (kb >> 3) + 1);
              mn_next = __ldg(mv + (kb >> 3) + 1);
            }
          }
          sbits = bf16_at(sc, kb & 7);
          mbits = bf16_at(mn, kb & 7);
        } else {
          const size_t gi = qr.grow * a.qgroups + kb;
          sbits = __bfloat16_as_ushort(qr.qs[gi]);
          mbits = __bfloat16_as_ushort(qr.qm[gi]);
        }
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&rawfull[cs], cph, lim);
          if (ok) ok = mbar_wait(&bempty[bs], bph ^ 1u, lim);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort_flag;
        if (!ok) {
          if (lane == 0) give_up(a, abort_flag, site);
          alive = false;
          break;
        }
        dequant_row(sQ + cs * SP::kStageQ + r * 32, sB + bs * kStageB, r, sbits, mbits);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bfull[bs]);
          mbar_arrive(&rawempty[cs]);
        }
        if (++cs == SP::kCStages) {
          cs = 0;
          cph ^= 1u;
        }
        if (++bs == SP::kBStages) {
          bs = 0;
          bph ^= 1u;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // let copies and MMAs already in flight land before the CTA exits
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols));
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D bf16 view [rows][cols] (cols contiguous), box = 64 cols x box_rows rows,
// 128-byte swizzle. A null or empty view yields a map over a 1-row dummy of
// the same base that no tile ever addresses.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !base) return false;
  if (rows == 0) rows = 1;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tc_sm_count() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 1;
}

namespace {

template <int MODE, bool Q4, int RB, int NB = 256, int AR = 128>
cudaError_t launch_tc(const TcMaps& maps, const TcArgs& a, int max_items, cudaStream_t st) {
  using SP = SmemPlan<Q4, RB, MODE == kTcDown, NB, AR>;
  static int attr[64] = {};
  cudaError_t e = ensure_smem_limit(tc_gemm_kernel<MODE, Q4, RB, NB, AR>, (int)SP::kBytes, attr);
  if (e != cudaSuccess) return e;
  int grid = tc_sm_count();
  if (max_items < grid) grid = max_items;
  if (grid < 1) grid = 1;
  return launch_pdl(tc_gemm_kernel<MODE, Q4, RB, NB, AR>, dim3(grid), SP::kThreadsCta, SP::kBytes, st,
                    maps.A0, maps.A1, maps.B0, maps.B1, maps.B2, maps.B3, a);
}

// 2D uint8 view of 4-bit codes [rows][K/2 bytes], box = 32 bytes (one 64-code
// group) x box_rows rows, no swizzle.
bool make_map_q4(CUtensorMap* m, const void* codes, uint64_t rows, uint64_t K, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !codes) return false;
  if (rows == 0) rows = 1;
  cuuint64_t dims[2] = {K / 2, rows};
  cuuint64_t strides[1] = {K / 2};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  return make_map(m, base, rows, cols, box_rows);
}

bool tc_make_map_q4(CUtensorMap* m, const void* codes, uint64_t rows, uint64_t K,
                    uint32_t box_rows) {
  return make_map_q4(m, codes, rows, K, box_rows);
}

cudaError_t launch_tc_gemm(int mode, const TcMaps& maps, const TcArgs& a, int max_items,
                           cudaStream_t st) {
  if (mode == kTcRouter) return launch_tc<kTcRouter, false, 1>(maps, a, max_items, st);
  if (mode != kTcGateUp && mode != kTcDown) return cudaErrorInvalidValue;
  const bool up = mode == kTcGateUp;
  if (a.qs0) {
    if (a.pair)
      return up ? launch_tc<kTcGateUp, true, 2>(maps, a, max_items, st)
                : launch_tc<kTcDown, true, 2>(maps, a, max_items, st);
    return up ? launch_tc<kTcGateUp, true, 1>(maps, a, max_items, st)
              : launch_tc<kTcDown, true, 1>(maps, a, max_items, st);
  }
  if (a.pair) return cudaErrorInvalidValue;  // paired items are built for 4-bit banks only
  // the A maps' box height is a.arows: 128, or 64 / 16 for decode batches
  if (a.arows != 128 && a.arows != 64 && a.arows != 16) return cudaErrorInvalidValue;
  if (up && a.bn <= 128) {
    if (a.arows == 16) return launch_tc<kTcGateUp, false, 1, 128, 16>(maps, a, max_items, st);
    if (a.arows == 64) return launch_tc<kTcGateUp, false, 1, 128, 64>(maps, a, max_items, st);
    return launch_tc<kTcGateUp, false, 1, 128>(maps, a, max_items, st);
  }
  if (up) {
    if (a.arows == 16) return launch_tc<kTcGateUp, false, 1, 256, 16>(maps, a, max_items, st);
    if (a.arows == 64) return launch_tc<kTcGateUp, false, 1, 256, 64>(maps, a, max_items, st);
    return launch_tc<kTcGateUp, false, 1>(maps, a, max_items, st);
  }
  if (a.arows == 16) return launch_tc<kTcDown, false, 1, 256, 16>(maps, a, max_items, st);
  if (a.arows == 64) return launch_tc<kTcDown, false, 1, 256, 64>(maps, a, max_items, st);
  return launch_tc<kTcDown, false, 1>(maps, a, max_items, st);
}

}  // namespace moe
