// Kernel argument blocks and launchers of the MoE layer (host + device).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_route.h"

namespace moe {

struct Ctrl;

struct RouterArgs {
  const void* x;          // [T][d] act dtype
  const void* W_router;   // [E][d]
  const void* w_shared;   // [d] or null (then no column E)
  float* logits;          // [T][E+1] f32
  int T, d, E;
};

struct TopkArgs {
  const float* logits;    // [T][E+1]
  const float* bias;      // [E] or null
  int32_t* topk_ids;      // [T][k]
  float* weights;         // [T][k]
  float* s_shared;        // [T] or null
  int T, E, k, kind, n_group, topk_group, has_shared_logit;
  float routed_scaling, renorm_clamp;
  // logits of experts held as nparts partial sums (0 or 1: one; at most 2)
  // at logits + i * part_stride, added in part order; column E in part 0 only
  int nparts;
  size_t part_stride;
};

struct BucketArgs {
  const int32_t* ids;     // [P]
  int32_t* counts;        // [E]
  int32_t* offsets;       // [E+1]
  int32_t* active;        // [E]
  int32_t* n_active;      // [1] (may point into Ctrl)
  int32_t* perm;          // [P]
  int32_t* pos;           // [P]
  Ctrl* ctrl;
  int P, E;
  // tensor-core path work list (null when unused): row blocks of bm rows,
  // one int2 {group, m_tile} each, largest groups first; shared group = E
  int2* rowblocks;
  int32_t* n_rowblocks;
  int bm, shared_rows;    // shared_rows = T when a shared expert exists, else 0
  int pair;               // 1: list pairs of row blocks (m even), for paired GEMM items
};

// Grouped GEMV over the packed rows ("groups" = active routed experts, then
// the shared expert as group E).
struct GemvArgs {
  const void* x;            // [T][d] act dtype
  const int32_t* perm;      // packed row -> pair id
  const int32_t* active;
  const int32_t* offsets;   // [E+1]
  const int32_t* n_active;  // device count
  const float* alpha;       // [P] flattened routing weights
  const float* s_shared;    // [T]
  const void* Wg; const void* Wu; const void* Wd;              // routed banks
  const void* Wg_scale; const void* Wg_min;                    // q4 only
  const void* Wu_scale; const void* Wu_min;
  const void* Wd_scale; const void* Wd_min;
  const void* Wsg; const void* Wsu; const void* Wsd;           // shared expert
  void* H;                  // [P][I] weight dtype (bf16 or f32)
  void* Hs;                 // [T][Is] weight dtype
  float* Y;                 // [P][d] f32 (alpha applied)
  float* Ys;                // [T][d] f32 (s_shared applied)
  Ctrl* ctrl;
  int T, d, E, k, I, Is, P;
  int routed_slots;         // grid.y entries for routed groups (= min(E, P))
  int has_shared;
  // direct-load GEMV only: when set, every routed (token, slot) pair is its
  // own group (expert ids[p], one token p / k, packed row p), so no
  // bucketing pass is needed; routed_slots = P
  const int32_t* pair_ids;
  // down + combine in one kernel (pair groups only, see
  // gemv_small_down_combine_ok): out = r_attn + the combined slots
  const float* r_attn;      // [T][d]
  float* out;               // [T][d]
};
// Whether the few-token down kernel can also do the combine (pair groups,
// at most two groups per warp of a column's CTA).
bool gemv_small_down_combine_ok(const GemvArgs& a);
cudaError_t launch_gemv_small_down_combine(const GemvArgs& a, int act, int wdt, cudaStream_t st);

// Single-launch decode kernel (decode_fused.cu): the whole layer for a few
// tokens in one cooperative launch. Route mode (ids_in null): router
// contraction, routing rule, experts, combine; given-ids mode: the expert
// half for caller-given ids and weights.
struct DecodeArgs {
  const void* x;            // [T][d] act dtype (= weight dtype)
  const float* r_attn;      // [T][d]
  const void* W_router;     // [E][d] (route mode)
  const float* bias;        // [E] or null (sigmoid family)
  const void* w_shared;     // [d] shared-gate vector (null without a shared expert)
  const int32_t* ids_in;    // given-ids mode: [T][k]; null in route mode
  const float* w_in;        // given-ids mode: [T][k]
  const float* s_in;        // given shared gate [T], or null (computed from w_shared)
  const void* Wg; const void* Wu; const void* Wd;   // routed banks
  const void* Wsg; const void* Wsu; const void* Wsd;  // shared expert
  float* out;               // [T][d]
  int32_t* topk_ids;        // route mode outputs [T][k]
  float* weights;
  float* logits;            // workspace [T][E+1] x kDecodeKSplit (partial sums of a K split)
  float* H;                 // workspace [T*k][I] fp32
  float* Hs;                // workspace [T][Is] fp32
  float* Yg;                // workspace [d][T*k + T]: per-column slot results (tensor-core variant)
  float* Gs;                // workspace [kDecodeKSplit][2][T][Is]: shared gate/up partial sums
  Ctrl* ctrl;
  int T, d, E, k, I, Is;
  int kind, n_group, topk_group;
  float routed_scaling, renorm_clamp;
  uint64_t wait_ns;         // limit of the grid-barrier waits
  int stall;                // failure self-test: block 0 never arrives at the first barrier
  int route_only;           // 1: routing only (moe_route): logits, rule, topk_ids / weights
  float* s_out;             // route only: the shared gate [T], or null
};
constexpr int kDecodeMaxTokens = 16;
// The tensor-core variant splits K of its first-phase contractions over this
// many blocks when the items would otherwise leave most of the grid idle.
constexpr int kDecodeKSplit = 2;
// Shapes the single-launch decode kernel takes (T <= kDecodeMaxTokens,
// f32 or bf16 weights and activations alike, E <= 512, k <= 32).
bool decode_fused_supported(int T, int d, int E, int k, int I, int Is, int act, int wdt);
// Whether bf16 shapes (d, I, Is) take the kernel's tensor-core variant.
bool decode_fused_mma(int d, int I, int Is);
cudaError_t launch_decode_fused(const DecodeArgs& a, bool bf16, cudaStream_t st);

struct CombineArgs {
  const float* r_attn;      // [T][d]
  const float* Y;           // [P][d] f32, or bf16 when y_bf16
  const float* Ys;          // [T][d] or null (same dtype as Y)
  const int32_t* pos;       // [P], or null: pair p at row p
  float* out;               // [T][d]
  int T, d, k;
  int y_bf16;
};

// Tensor-core grouped GEMM (tc_gemm.cu).
enum TcMode { kTcGateUp = 0, kTcDown = 1, kTcRouter = 2 };

struct TcArgs {
  const int2* rowblocks;       // (group, m-tile) list from the bucketing pass
  const int32_t* n_rowblocks;  // device count of row blocks
  const int32_t* offsets;      // [E+1] packed-row offsets per routed expert
  const int32_t* perm;         // packed row -> pair id
  const float* alpha;          // [P] routing weights (down)
  const float* s_shared;       // [T] shared gate (down)
  void* out_routed;            // H | Y (bf16, packed rows) | logits (f32)
  void* out_shared;            // Hs | Ys (bf16, token rows)
  Ctrl* ctrl;
  int E, T, K;                 // K: reduction length (multiple of 64)
  int ld_out;                  // output row stride in elements
  int n_tiles;                 // N tiles per row block
  int bn;                      // N of one MMA (gate/up: 128 gate + 128 up)
  int brows_routed;            // rows of one routed expert in the 2D B view
  // 4-bit affine weights (null for bf16): per-row group scale and min, bf16
  // [rows][K/64]; 0 = gate (or down), 1 = up
  const __nv_bfloat16* qs0;
  const __nv_bfloat16* qm0;
  const __nv_bfloat16* qs1;
  const __nv_bfloat16* qm1;
  int qgroups;                 // K / 64
  // 1: each row-block entry is a pair of 128-row blocks (m, m + 1) sharing
  // the B tiles (the bucketing pass then lists every second block); 4-bit
  // banks only
  int pair;
  // 1: the launch's items are the shared expert's alone (row blocks of the T
  // token rows, no row-block list), for a shared expert of another width
  int shared_only;
  // box height of the A maps (gate/up and down, bf16): 128, or 64 / 16 when
  // every group holds at most that many rows
  int arows;
  uint64_t wait_ns;            // limit of every bounded wait (0: about one second)
  int stall;                   // failure self-test: the MMA warp waits on a flag nothing sets
};

// The six operand maps: A routed/shared, B0/B1 routed, B2/B3 shared.
struct TcMaps {
  CUtensorMap A0, A1, B0, B1, B2, B3;
};

// Encodes a 2D bf16 TMA map [rows][cols] with a 64-column x box_rows box and
// 128-byte swizzle; false if the driver entry point or the encoding fails.
bool tc_make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);
// Encodes a 2D uint8 TMA map of 4-bit codes [rows][K/2], box 32 B x box_rows.
bool tc_make_map_q4(CUtensorMap* m, const void* codes, uint64_t rows, uint64_t K,
                    uint32_t box_rows);
cudaError_t launch_tc_gemm(int mode, const TcMaps& maps, const TcArgs& a, int max_items,
                           cudaStream_t st);
cudaError_t launch_gather_rows(const void* x, const int32_t* perm, int k, int d, void* out, int P,
                               cudaStream_t st);
int tc_sm_count();

// Raises `kernel`'s dynamic shared-memory opt-in limit to at least `bytes`
// on the current device; `limits` holds the value set so far per device
// ordinal (< 64), so the attribute is only set when a launch needs more.
template <typename K>
inline cudaError_t ensure_smem_limit(K kernel, int bytes, int* limits) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (bytes <= 48 * 1024 || limits[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) limits[dev] = bytes;
  return e;
}

// Launches `kernel` with programmatic stream serialization: its CTAs may be
// scheduled (and run their set-up) while the previous kernel on the stream
// is still finishing. Every kernel of this library calls pdl_wait() before
// its first global memory access, so only launch latency and set-up overlap.
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

// Host-side argument checks shared by the entry points (api.cu): the layer
// configuration, and the subset routing needs (the routing entry points
// accept configurations whose expert banks are outside the library's limits).
moe_status_t validate_cfg(const moe_cfg_t* c);
moe_status_t validate_route_cfg(const moe_cfg_t* c);
// Records the CUDA error behind a MOE_ERR_CUDA for moe_last_cuda_error.
void set_last_cuda_error(cudaError_t e);

// One launcher per kernel; each returns the launch's cudaError_t.
cudaError_t launch_router_logits(const RouterArgs& ra, bool bf16, cudaStream_t st);
cudaError_t launch_router_topk(const TopkArgs& ta, cudaStream_t st);
cudaError_t launch_shared_gate(const RouterArgs& ra, float* s_out, bool bf16, cudaStream_t st);
// Bucketing: one CTA (launch_bucket) up to kBucketOneCta pairs, else
// launch_bucket_hist then launch_bucket_pack over bucket_ctas(P) segments,
// with per-CTA histograms (then bases) in cta_hist [bucket_ctas(P)][E] ints.
constexpr int kBucketOneCta = 4096;
int bucket_ctas(int P);
cudaError_t launch_bucket(const BucketArgs& a, cudaStream_t st);
cudaError_t launch_bucket_hist(const BucketArgs& a, int* cta_hist, cudaStream_t st);
cudaError_t launch_bucket_pack(const BucketArgs& a, const int* cta_base, cudaStream_t st);
// act: 0 f32, 1 bf16; wdt: 0 f32, 1 bf16, 2 q4
cudaError_t launch_gemv_gateup(const GemvArgs& a, int act, int wdt, cudaStream_t st);
cudaError_t launch_gemv_down(const GemvArgs& a, int act, int wdt, cudaStream_t st);
// Direct-load GEMV for batches of at most kGemvSmallTokens tokens
// (gemv_small.cu): down = false runs gate/up + SwiGLU, true runs down x alpha.
constexpr int kGemvSmallTokens = 8;
cudaError_t launch_gemv_small(const GemvArgs& a, int act, int wdt, bool down, cudaStream_t st);
// True when the GEMV kernels can stage at least one token of width d and kmax.
bool gemv_supported(int d, int kmax);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);

}  // namespace moe
