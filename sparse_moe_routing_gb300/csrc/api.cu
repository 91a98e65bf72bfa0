// C ABI of the MoE layer forward: argument validation, workspace plan and the
// launch sequence on the caller's stream. See include/moe_route.h.
#include "moe_route.h"

#include <math.h>
#include <atomic>
#include <stdint.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kTcBm = 128;  // token rows per tensor-core tile

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct Plan {
  size_t ctrl, logits, s_shared, counts, offsets, active, perm, pos, rowblocks, cta_hist;
  size_t H, Hs, Y, Ys, Xperm, Gs, total;
};

// Token batches at or above this size take the tensor-core path under
// MOE_PATH_AUTO (when the shape allows it). Measured per layer at the Qwen3.6
// shape (direct-load GEMV / tensor cores): T=4 57 / 68 us, T=5 83 / 89 us,
// T=6 96 / 92 us, T=8 123 / 100 us.
constexpr int kTcMinTokens = 6;

// The tensor-core path: bf16 experts and activations, K dims multiples of the
// 64-element TMA box, N tiles of 128 (gate/up) and 256 (down), and a shared
// expert (if any) as wide as the routed ones.
// 4-bit affine banks are dequantised inside this path (one 64-code group per
// 64-element k-block); they are supported without a shared expert only.
bool tc_shape_ok(const moe_cfg_t& c) {
  if (c.act_dtype != MOE_BF16 || c.d_model % 256 != 0 || c.d_ff % 128 != 0) return false;
  if (c.expert_dtype == MOE_Q4_AFFINE_G64) return c.d_ff_shared == 0;
  return c.expert_dtype == MOE_BF16 && c.d_ff_shared % 128 == 0;
}
// A shared expert of another width than the routed ones cannot be one more
// group of their grouped GEMMs (other N tiling, and another K for down): it
// runs as its own gate/up and down launches of the same kernels.
bool shared_apart(const moe_cfg_t& c) {
  return c.d_ff_shared > 0 && c.d_ff_shared != c.d_ff;
}

// The router contraction on the tensor cores: bf16, E a multiple of 32 (N
// tiles of 32 or 64 logits), d a multiple of the 64-element box, and enough
// tokens to fill 128-row tiles usefully (below this the CUDA-core router is
// as fast, measured at T=64, and needs no separate shared-gate launch).
constexpr int kTcRouterMinTokens = 128;
bool use_tc_router(const moe_cfg_t& c) {
  return c.act_dtype == MOE_BF16 && c.n_experts % 32 == 0 && c.n_experts <= 512 &&
         c.d_model % 64 == 0 && c.T >= kTcRouterMinTokens;
}
// N tile of the tensor-core router: 32 logits for small batches (more CTAs
// share the router weights), 64 for large ones.
int tc_router_bn(const moe_cfg_t& c) {
  return (c.T <= 1024 || c.n_experts % 64 != 0) ? 32 : 64;
}

// The single-launch decode kernel runs when asked for (MOE_PATH_FUSED), and
// is MOE_PATH_AUTO's choice for kFusedMinTokens..kDecodeMaxTokens tokens
// when its tensor-core variant takes the shape (bf16) and the shape is one
// where it was measured faster: d_model <= 2048 (each warp keeps its token
// fragments in registers) and expert widths <= 1024 (a block's chunks of h
// fit shared memory). Per layer (single launch / GEMV chain / tensor-core
// path): Qwen3.6 shape T=1 31 / 21 / - us, T=2 43 / 35 / - us, T=3 51 / 47 /
// - us, T=4 57 / 56 / - us, T=5 67 / 84 / - us, T=6 70 / 97 / - us, T=8
// 80 / - / 93 us, T=12 115 / - / 125 us, T=16 133 / - / 143 us;
// sigmoid-group shape T=4 57 / 61 us, T=5 60 / 87 us, T=8 76 / - / 90 us,
// T=16 106 / - / 113 us; but the Mixtral shape (d_model 4096, width 14336)
// T=8 545 / - / 398 us, and at width 1408 T=8 135 / - / 128 us (64 experts)
// and 284 / - / 163 us (60 experts, 5632-wide shared expert). Below
// kFusedMinTokens the GEMV chain stays: its
// launches cost less than the kernel's three grid barriers and in-kernel
// routing.
constexpr int kFusedMinTokens = 4;
bool fused_ok(const moe_cfg_t& c) {
  return decode_fused_supported(c.T, c.d_model, c.n_experts, c.top_k, c.d_ff, c.d_ff_shared,
                                c.act_dtype, c.expert_dtype);
}
bool auto_fused(const moe_cfg_t& c) {
  return c.path == MOE_PATH_AUTO && c.T >= kFusedMinTokens && c.T <= kDecodeMaxTokens &&
         c.act_dtype == MOE_BF16 && c.expert_dtype == MOE_BF16 && c.d_model <= 2048 &&
         c.d_ff <= 1024 && c.d_ff_shared <= 1024 &&
         decode_fused_mma(c.d_model, c.d_ff, c.d_ff_shared) && fused_ok(c);
}
bool use_fused(const moe_cfg_t& c) {
  return (c.path == MOE_PATH_FUSED && fused_ok(c)) || auto_fused(c);
}

bool use_tc(const moe_cfg_t& c) {
  if (!tc_shape_ok(c)) return false;
  if (c.path == MOE_PATH_TC || c.expert_dtype == MOE_Q4_AFFINE_G64) return true;
  return c.path == MOE_PATH_AUTO && c.T >= kTcMinTokens && !auto_fused(c);
}

// Failure self-test state (moe_inject_stall): the kernel family whose next
// launch stalls, and the wait limit of that launch.
std::atomic<int> g_stall_kernel{0};
std::atomic<uint64_t> g_stall_wait_ns{0};

// Takes the one-shot stall for kernel family `kid` if it is armed: returns
// the wait limit of the launch and sets *stall.
uint64_t take_stall(int kid, int* stall) {
  int want = kid;
  *stall = 0;
  if (g_stall_kernel.load(std::memory_order_relaxed) == kid &&
      g_stall_kernel.compare_exchange_strong(want, 0)) {
    *stall = 1;
    return g_stall_wait_ns.load();
  }
  return kWaitLimitNs;
}

// Batches of a few tokens on the GEMV path treat every (token, slot) pair
// as its own group (at most a handful of pairs share an expert), which needs
// no bucketing pass.
bool gemv_pairs(const moe_cfg_t& c) {
  return !use_tc(c) && !use_fused(c) && c.T <= kGemvSmallTokens;
}

// Paired GEMM items (two 128-row blocks per B tile) for 4-bit banks whose
// routed experts average at least two row blocks each: pairing halves the
// dequantisation per flop, which bounds those kernels (Mixtral-shape 4-bit
// gate/up 1440 -> 1335 us). For bf16 banks the single-buffered accumulator
// of paired items costs more than the B traffic it saves (Mixtral-shape bf16
// layer 1211 -> 1431 us), so they stay unpaired.
bool use_pair(const moe_cfg_t& c) {
  return use_tc(c) && c.expert_dtype == MOE_Q4_AFFINE_G64 &&
         (long long)c.T * c.top_k >= 2LL * kTcBm * c.n_experts;
}

Plan make_plan(const moe_cfg_t& c) {
  Plan p{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t T = c.T, E = c.n_experts, P = (size_t)c.T * c.top_k;
  const size_t d = c.d_model, I = c.d_ff, Is = c.d_ff_shared;
  p.ctrl = take(sizeof(Ctrl));
  const bool small = T <= (size_t)kDecodeMaxTokens;
  p.logits = take(T * (E + 1) * 4 * (small ? kDecodeKSplit : 1));
  p.s_shared = take(T * 4);
  p.counts = take(E * 4);
  p.offsets = take((E + 1) * 4);
  p.active = take(E * 4);
  p.perm = take(P * 4);
  p.pos = take(P * 4);
  p.rowblocks = take(((P + T) / kTcBm + E + 2) * 8);
  p.cta_hist = take((size_t)bucket_ctas((int)P) * E * 4);
  // (the single-launch decode kernel's tensor-core variant keeps h in mma
  // fragment order: up to P chunks, or ceil(T/8) shared chunks, of 8 slots)
  p.H = take(small ? P * I * 16 : P * I * 4);
  const size_t hs_frag = (T + 7) / 8 * Is * 16;
  p.Hs = take(small && hs_frag > T * Is * 4 ? hs_frag : T * Is * 4);
  p.Y = take(small && d * (P + T) > P * d ? d * (P + T) * 4 : P * d * 4);
  p.Ys = take(Is ? T * d * 4 : 0);
  p.Xperm = take(tc_shape_ok(c) ? P * d * 2 : 0);
  p.Gs = take(small ? kDecodeKSplit * 2 * T * Is * 4 : 0);
  p.total = off;
  return p;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

moe_status_t validate_cfg(const moe_cfg_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d_model <= 0 || (c->d_model % 8) != 0) return MOE_ERR_INVALID_ARG;
  if (c->n_experts < 1 || c->top_k < 1 || c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->d_ff <= 0 || (c->d_ff % 8) != 0) return MOE_ERR_INVALID_ARG;
  if (c->d_ff_shared < 0 || (c->d_ff_shared % 8) != 0) return MOE_ERR_INVALID_ARG;
  if (c->router == MOE_ROUTER_SIGMOID_GROUP_TOPK) {
    if (c->n_group < 1 || (c->n_experts % c->n_group) != 0) return MOE_ERR_INVALID_ARG;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_INVALID_ARG;
    if ((long long)c->topk_group * (c->n_experts / c->n_group) < c->top_k)
      return MOE_ERR_INVALID_ARG;
    if (c->n_group > 32) return MOE_ERR_UNSUPPORTED;
  } else if (c->router != MOE_ROUTER_SOFTMAX_TOPK) {
    return MOE_ERR_INVALID_ARG;
  }
  if (!isfinite(c->routed_scaling) || !isfinite(c->renorm_clamp) || c->renorm_clamp < 0.f)
    return MOE_ERR_INVALID_ARG;
  if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->expert_dtype != MOE_F32 && c->expert_dtype != MOE_BF16 &&
      c->expert_dtype != MOE_Q4_AFFINE_G64)
    return MOE_ERR_INVALID_ARG;
  if (c->path < MOE_PATH_AUTO || c->path > MOE_PATH_FUSED) return MOE_ERR_INVALID_ARG;
  // limits of the library (kernel templates and shared-memory plans)
  if (c->n_experts > 512 || c->top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (c->expert_dtype == MOE_F32 && c->act_dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (c->expert_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (!gemv_supported(c->d_model, c->d_ff > c->d_ff_shared ? c->d_ff : c->d_ff_shared))
    return MOE_ERR_UNSUPPORTED;
  if ((c->path == MOE_PATH_TC || c->expert_dtype == MOE_Q4_AFFINE_G64) && !tc_shape_ok(*c))
    return MOE_ERR_UNSUPPORTED;
  if (c->expert_dtype == MOE_Q4_AFFINE_G64 && c->path == MOE_PATH_GEMV) return MOE_ERR_UNSUPPORTED;
  if (c->path == MOE_PATH_FUSED &&
      !decode_fused_supported(c->T > 0 ? c->T : 1, c->d_model, c->n_experts, c->top_k, c->d_ff,
                              c->d_ff_shared, c->act_dtype, c->expert_dtype))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t validate_route_cfg(const moe_cfg_t* c) {
  moe_status_t s = validate_cfg(c);
  if (s != MOE_OK && s != MOE_ERR_UNSUPPORTED) return s;
  if (c->n_experts > 512 || c->top_k > 32 || c->n_group > 32) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

namespace {

moe_status_t check_workspace(const moe_cfg_t* c) {
  if (!c->workspace || ((uintptr_t)c->workspace & 255u)) return MOE_ERR_WORKSPACE;
  if (c->workspace_bytes < make_plan(*c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
T* at(const moe_cfg_t* c, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(c->workspace) + off);
}

}  // namespace

// Last CUDA error seen by a call of this thread (moe_last_cuda_error).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

namespace {

moe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  g_last_cuda_error = e;
  return MOE_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// measurement: launch counter and optional event bracketing of one kernel
// ---------------------------------------------------------------------------
std::atomic<unsigned long long> g_launches{0};
struct TraceState {
  int kernel = 0;
  cudaEvent_t* starts = nullptr;
  cudaEvent_t* stops = nullptr;
  int n = 0;
  int* count = nullptr;
} g_trace;

// Runs one kernel launcher, counting it and bracketing it with the traced
// events when its family is being traced.
// While the stream is being captured into a CUDA graph, the records become
// external event nodes, so every replay still timestamps the kernel.
cudaError_t trace_record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cudaErrorUnknown;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

// NVTX range names per kernel family (host-side ranges around each launch,
// visible to nsys / ncu --nvtx; free when no tool is attached).
const char* kernel_name(int kid) {
  switch (kid) {
    case MOE_KERNEL_ROUTER_LOGITS: return "moe:router_logits";
    case MOE_KERNEL_ROUTER_TOPK: return "moe:router_topk";
    case MOE_KERNEL_SHARED_GATE: return "moe:shared_gate";
    case MOE_KERNEL_BUCKET: return "moe:bucket";
    case MOE_KERNEL_GEMV_GATEUP: return "moe:gemv_gateup";
    case MOE_KERNEL_GEMV_DOWN: return "moe:gemv_down";
    case MOE_KERNEL_COMBINE: return "moe:combine";
    case MOE_KERNEL_TC_GATEUP: return "moe:tc_gateup";
    case MOE_KERNEL_TC_DOWN: return "moe:tc_down";
    case MOE_KERNEL_GATHER: return "moe:gather";
    case MOE_KERNEL_TC_ROUTER: return "moe:tc_router";
    case MOE_KERNEL_DECODE: return "moe:decode_fused";
  }
  return "moe:kernel";
}

template <typename F>
cudaError_t run(int kid, cudaStream_t st, F&& launch) {
  struct Range {
    explicit Range(const char* n) { nvtxRangePushA(n); }
    ~Range() { nvtxRangePop(); }
  } range(kernel_name(kid));
  const bool tr = g_trace.kernel == kid && g_trace.n > 0;
  const int slot = tr ? (*g_trace.count % g_trace.n) : 0;
  if (tr && trace_record(g_trace.starts[slot], st) != cudaSuccess) return cudaErrorUnknown;
  cudaError_t e = launch();
  if (e != cudaSuccess) {
    g_last_cuda_error = e;
    return e;
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (tr) {
    if (trace_record(g_trace.stops[slot], st) != cudaSuccess) return cudaErrorUnknown;
    ++*g_trace.count;
  }
  return cudaSuccess;
}

bool bank_ok(const moe_bank_t& b, int dt) {
  if (!b.w || !aligned16(b.w)) return false;
  if (dt == MOE_Q4_AFFINE_G64) return b.scale && b.minv && aligned16(b.scale) && aligned16(b.minv);
  return true;
}

RouterArgs router_args(const void* x, const void* W_router, const void* w_shared,
                       const moe_cfg_t* c, float* s_shared) {
  const Plan p = make_plan(*c);
  return RouterArgs{x, W_router, s_shared ? w_shared : nullptr, at<float>(c, p.logits), c->T,
                    c->d_model, c->n_experts};
}

TopkArgs topk_args(const RouterArgs& ra, const float* bias, const moe_cfg_t* c, int32_t* ids,
                   float* w, float* s_shared) {
  TopkArgs ta{};
  ta.logits = ra.logits;
  ta.bias = c->router == MOE_ROUTER_SIGMOID_GROUP_TOPK ? bias : nullptr;
  ta.topk_ids = ids;
  ta.weights = w;
  ta.s_shared = s_shared;
  ta.T = c->T;
  ta.E = c->n_experts;
  ta.k = c->top_k;
  ta.kind = c->router;
  ta.n_group = c->n_group;
  ta.topk_group = c->topk_group;
  ta.has_shared_logit = ra.w_shared ? 1 : 0;
  ta.routed_scaling = c->routed_scaling;
  ta.renorm_clamp = c->renorm_clamp;
  return ta;
}

moe_status_t enqueue_route(const void* x, const void* W_router, const float* bias,
                           const void* w_shared, const moe_cfg_t* c, int32_t* ids, float* w,
                           float* s_shared, cudaStream_t st) {
  const RouterArgs ra = router_args(x, W_router, w_shared, c, s_shared);
  TopkArgs ta = topk_args(ra, bias, c, ids, w, s_shared);
  const bool bf16 = c->act_dtype == MOE_BF16;
  cudaError_t e;
  if (use_tc_router(*c)) {
    // tensor-core router: logits [T][E] (column E unused), then the shared
    // gate from its own warp-per-token dot product
    const int bn = tc_router_bn(*c);
    TcMaps m{};
    if (!tc_make_map(&m.A0, x, c->T, c->d_model, 128) ||
        !tc_make_map(&m.B0, W_router, c->n_experts, c->d_model, bn))
      return MOE_ERR_CUDA;
    m.A1 = m.A0;
    m.B1 = m.B2 = m.B3 = m.B0;
    TcArgs a{};
    a.out_routed = ra.logits;
    a.ctrl = at<Ctrl>(c, 0);
    a.E = c->n_experts;
    a.T = c->T;
    a.K = c->d_model;
    a.ld_out = c->n_experts + 1;
    a.bn = bn;
    a.n_tiles = c->n_experts / bn;
    const int items = (c->T + kTcBm - 1) / kTcBm * a.n_tiles;
    e = run(MOE_KERNEL_TC_ROUTER, st, [&] { return launch_tc_gemm(kTcRouter, m, a, items, st); });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    ta.has_shared_logit = 0;
    if (s_shared) {
      RouterArgs rs{x, nullptr, w_shared, ra.logits, c->T, c->d_model, 0};
      e = run(MOE_KERNEL_SHARED_GATE, st, [&] { return launch_shared_gate(rs, s_shared, bf16, st); });
      if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
  } else {
    e = run(MOE_KERNEL_ROUTER_LOGITS, st, [&] { return launch_router_logits(ra, bf16, st); });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return cuda_status(run(MOE_KERNEL_ROUTER_TOPK, st, [&] { return launch_router_topk(ta, st); }));
}

BucketArgs bucket_args(const int32_t* ids, const moe_cfg_t* c, int32_t* counts,
                       int32_t* offsets, int32_t* active, int32_t* n_active, int32_t* perm,
                       int32_t* pos) {
  BucketArgs b{};
  b.ids = ids;
  b.counts = counts;
  b.offsets = offsets;
  b.active = active;
  b.n_active = n_active;
  b.perm = perm;
  b.pos = pos;
  b.ctrl = at<Ctrl>(c, 0);
  b.P = c->T * c->top_k;
  b.E = c->n_experts;
  b.rowblocks = nullptr;
  if (use_tc(*c)) {
    // the tensor-core path walks (group, 128-row block) work items
    const Plan p = make_plan(*c);
    b.rowblocks = at<int2>(c, p.rowblocks);
    b.n_rowblocks = &at<Ctrl>(c, 0)->n_rowblocks;
    b.bm = kTcBm;
    b.shared_rows = (c->d_ff_shared > 0 && !shared_apart(*c)) ? c->T : 0;
    b.pair = use_pair(*c) ? 1 : 0;
  }
  return b;
}

moe_status_t enqueue_bucket(const int32_t* ids, const moe_cfg_t* c, int32_t* counts,
                            int32_t* offsets, int32_t* active, int32_t* n_active, int32_t* perm,
                            int32_t* pos, cudaStream_t st) {
  const BucketArgs b = bucket_args(ids, c, counts, offsets, active, n_active, perm, pos);
  if (bucket_ctas(b.P) == 1)
    return cuda_status(run(MOE_KERNEL_BUCKET, st, [&] { return launch_bucket(b, st); }));
  int* cta_hist = at<int>(c, make_plan(*c).cta_hist);
  cudaError_t e = run(MOE_KERNEL_BUCKET, st, [&] { return launch_bucket_hist(b, cta_hist, st); });
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(run(MOE_KERNEL_BUCKET, st, [&] { return launch_bucket_pack(b, cta_hist, st); }));
}

// Routing and bucketing of the layer's own batch.
moe_status_t enqueue_route_bucket(const void* x, const void* W_router, const float* bias,
                                  const void* w_shared, const moe_cfg_t* c, int32_t* ids,
                                  float* w, float* s_shared, cudaStream_t st) {
  const Plan p = make_plan(*c);
  moe_status_t s = enqueue_route(x, W_router, bias, w_shared, c, ids, w, s_shared, st);
  if (s != MOE_OK || gemv_pairs(*c)) return s;
  return enqueue_bucket(ids, c, at<int32_t>(c, p.counts), at<int32_t>(c, p.offsets),
                        at<int32_t>(c, p.active), &at<Ctrl>(c, 0)->n_active,
                        at<int32_t>(c, p.perm), at<int32_t>(c, p.pos), st);
}

// Tensor-core sequence: gather X_perm, grouped gate/up (+SwiGLU) and down
// (x alpha) GEMMs over the (group, row block, N tile) items, bf16 combine.
moe_status_t enqueue_experts_tc(const void* x, const float* r_attn, const float* alpha,
                                const float* s_shared, moe_bank_t Wg, moe_bank_t Wu,
                                moe_bank_t Wd, const void* Wsg, const void* Wsu, const void* Wsd,
                                const moe_cfg_t* c, float* out, cudaStream_t st,
                                bool ids_distinct) {
  const Plan p = make_plan(*c);
  Ctrl* ctrl = at<Ctrl>(c, 0);
  const int T = c->T, d = c->d_model, E = c->n_experts, k = c->top_k, I = c->d_ff;
  const int Is = c->d_ff_shared, P = T * k;
  const bool apart = shared_apart(*c);
  const bool shared = Is > 0 && !apart;  // the shared expert is a group of the routed launches
  void* xperm = at<void>(c, p.Xperm);
  void* H = at<void>(c, p.H);
  void* Hs = at<void>(c, p.Hs);
  void* Y = at<void>(c, p.Y);
  void* Ys = at<void>(c, p.Ys);
  const int32_t* perm = at<int32_t>(c, p.perm);

  cudaError_t e = run(MOE_KERNEL_GATHER, st,
                      [&] { return launch_gather_rows(x, perm, k, d, xperm, P, st); });
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  const int max_rb = (P + kTcBm - 1) / kTcBm + (P < E ? P : E) + 1 +
                     (shared ? (T + kTcBm - 1) / kTcBm + 1 : 0);
  TcArgs a{};
  a.rowblocks = at<int2>(c, p.rowblocks);
  a.n_rowblocks = &ctrl->n_rowblocks;
  a.offsets = at<int32_t>(c, p.offsets);
  a.perm = perm;
  a.alpha = alpha;
  a.s_shared = s_shared;
  a.ctrl = ctrl;
  a.E = E;
  a.T = T;
  a.pair = use_pair(*c) ? 1 : 0;

  const bool q4 = c->expert_dtype == MOE_Q4_AFFINE_G64;
  // A tiles only as tall as the tallest group can be: with ids from the
  // routing rule (k distinct experts per token) every routed group holds at
  // most T rows, and the shared expert holds T
  const uint32_t arows = (!q4 && ids_distinct) ? (T <= 16 ? 16u : (T <= 64 ? 64u : 128u)) : 128u;
  a.arows = (int)arows;
  auto bmap = [&](CUtensorMap* mp, const void* w, uint64_t rows, uint64_t K, uint32_t box) {
    return q4 ? tc_make_map_q4(mp, w, rows, K, box) : tc_make_map(mp, w, rows, K, box);
  };
  // gate/up: A = X_perm (routed) / x (shared), B = gate and up rows (4-bit
  // codes for q4 banks, dequantised in the kernel). N tile = bn/2 gate + bn/2
  // up columns: 128 + 128, or 64 + 64 when the bf16 work list is too short
  // for 4 waves of 256-wide items (decode batches: finer items even out the
  // last wave of the weight stream)
  const int gu_bn = (!q4 && (long long)max_rb * (I / 128) < 4LL * tc_sm_count()) ? 128 : 256;
  const uint32_t gu_rows = gu_bn / 2;
  TcMaps m{};
  bool ok = tc_make_map(&m.A0, xperm, P, d, arows) && tc_make_map(&m.A1, x, T, d, arows) &&
            bmap(&m.B0, Wg.w, (uint64_t)E * I, d, gu_rows) &&
            bmap(&m.B1, Wu.w, (uint64_t)E * I, d, gu_rows);
  if (q4) {
    a.qs0 = static_cast<const __nv_bfloat16*>(Wg.scale);
    a.qm0 = static_cast<const __nv_bfloat16*>(Wg.minv);
    a.qs1 = static_cast<const __nv_bfloat16*>(Wu.scale);
    a.qm1 = static_cast<const __nv_bfloat16*>(Wu.minv);
    a.qgroups = d / 64;
  }
  if (ok && shared)
    ok = tc_make_map(&m.B2, Wsg, Is, d, gu_rows) && tc_make_map(&m.B3, Wsu, Is, d, gu_rows);
  if (!ok) return MOE_ERR_CUDA;
  if (!shared) {
    m.B2 = m.B0;
    m.B3 = m.B1;
  }
  a.out_routed = H;
  a.out_shared = Hs;
  a.K = d;
  a.ld_out = I;
  a.n_tiles = I / gu_rows;
  a.bn = gu_bn;
  a.brows_routed = I;
  a.wait_ns = take_stall(MOE_KERNEL_TC_GATEUP, &a.stall);
  e = run(MOE_KERNEL_TC_GATEUP, st,
          [&] { return launch_tc_gemm(kTcGateUp, m, a, max_rb * a.n_tiles, st); });
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const int shared_rb = (T + kTcBm - 1) / kTcBm;
  if (apart) {
    // the shared expert alone: A = x, B = its gate and up rows, out Hs [T][Is]
    TcMaps ms{};
    if (!tc_make_map(&ms.A1, x, T, d, arows) || !tc_make_map(&ms.B2, Wsg, Is, d, gu_rows) ||
        !tc_make_map(&ms.B3, Wsu, Is, d, gu_rows))
      return MOE_ERR_CUDA;
    ms.A0 = ms.A1;
    ms.B0 = ms.B2;
    ms.B1 = ms.B3;
    TcArgs as = a;
    as.shared_only = 1;
    as.pair = 0;
    as.ld_out = Is;
    as.n_tiles = Is / gu_rows;
    as.wait_ns = take_stall(MOE_KERNEL_TC_GATEUP, &as.stall);
    e = run(MOE_KERNEL_TC_GATEUP, st,
            [&] { return launch_tc_gemm(kTcGateUp, ms, as, shared_rb * as.n_tiles, st); });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  // down: A = H (routed) / Hs (shared), B = down rows; alpha in the epilogue
  TcMaps m2{};
  ok = tc_make_map(&m2.A0, H, P, I, arows) && bmap(&m2.B0, Wd.w, (uint64_t)E * d, I, 256);
  if (q4) {
    a.qs0 = static_cast<const __nv_bfloat16*>(Wd.scale);
    a.qm0 = static_cast<const __nv_bfloat16*>(Wd.minv);
    a.qs1 = a.qm1 = nullptr;
    a.qgroups = I / 64;
  }
  if (ok && shared)
    ok = tc_make_map(&m2.A1, Hs, T, Is, arows) && tc_make_map(&m2.B2, Wsd, d, Is, 256);
  if (!ok) return MOE_ERR_CUDA;
  if (!shared) {
    m2.A1 = m2.A0;
    m2.B2 = m2.B0;
  }
  m2.B1 = m2.B0;
  m2.B3 = m2.B2;
  a.out_routed = Y;
  a.out_shared = Ys;
  a.K = I;
  a.ld_out = d;
  a.n_tiles = d / 256;
  a.bn = 256;
  a.brows_routed = d;
  a.wait_ns = take_stall(MOE_KERNEL_TC_DOWN, &a.stall);
  e = run(MOE_KERNEL_TC_DOWN, st,
          [&] { return launch_tc_gemm(kTcDown, m2, a, max_rb * a.n_tiles, st); });
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (apart) {
    // the shared expert's down alone: A = Hs, B = its down rows, out Ys x s_t
    TcMaps ms{};
    if (!tc_make_map(&ms.A1, Hs, T, Is, arows) || !tc_make_map(&ms.B2, Wsd, d, Is, 256))
      return MOE_ERR_CUDA;
    ms.A0 = ms.A1;
    ms.B0 = ms.B1 = ms.B3 = ms.B2;
    TcArgs as = a;
    as.shared_only = 1;
    as.pair = 0;
    as.K = Is;
    as.qs0 = as.qm0 = nullptr;
    as.wait_ns = take_stall(MOE_KERNEL_TC_DOWN, &as.stall);
    e = run(MOE_KERNEL_TC_DOWN, st,
            [&] { return launch_tc_gemm(kTcDown, ms, as, shared_rb * as.n_tiles, st); });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  CombineArgs cb{r_attn, static_cast<const float*>(Y),
                 Is > 0 ? static_cast<const float*>(Ys) : nullptr, at<int32_t>(c, p.pos), out,
                 T, d, k, 1};
  return cuda_status(run(MOE_KERNEL_COMBINE, st, [&] { return launch_combine(cb, st); }));
}

moe_status_t enqueue_experts(const void* x, const float* r_attn, const int32_t* ids,
                             const float* alpha, const float* s_shared, moe_bank_t Wg,
                             moe_bank_t Wu, moe_bank_t Wd, const void* Wsg, const void* Wsu,
                             const void* Wsd, const moe_cfg_t* c, float* out, cudaStream_t st,
                             bool ids_distinct) {
  if (use_tc(*c))
    return enqueue_experts_tc(x, r_attn, alpha, s_shared, Wg, Wu, Wd, Wsg, Wsu, Wsd, c, out, st,
                              ids_distinct);
  const Plan p = make_plan(*c);
  Ctrl* ctrl = at<Ctrl>(c, 0);
  GemvArgs g{};
  g.x = x;
  g.perm = at<int32_t>(c, p.perm);
  g.active = at<int32_t>(c, p.active);
  g.offsets = at<int32_t>(c, p.offsets);
  g.n_active = &ctrl->n_active;
  g.alpha = alpha;
  g.s_shared = s_shared;
  g.Wg = Wg.w; g.Wu = Wu.w; g.Wd = Wd.w;
  g.Wg_scale = Wg.scale; g.Wg_min = Wg.minv;
  g.Wu_scale = Wu.scale; g.Wu_min = Wu.minv;
  g.Wd_scale = Wd.scale; g.Wd_min = Wd.minv;
  g.Wsg = Wsg; g.Wsu = Wsu; g.Wsd = Wsd;
  g.H = at<float>(c, p.H);
  g.Hs = at<float>(c, p.Hs);
  g.Y = at<float>(c, p.Y);
  g.Ys = at<float>(c, p.Ys);
  g.ctrl = ctrl;
  g.T = c->T; g.d = c->d_model; g.E = c->n_experts; g.k = c->top_k;
  g.I = c->d_ff; g.Is = c->d_ff_shared; g.P = c->T * c->top_k;
  g.routed_slots = g.P < g.E ? g.P : g.E;
  g.has_shared = c->d_ff_shared > 0 ? 1 : 0;
  const bool pairs = gemv_pairs(*c);
  if (pairs) {
    g.pair_ids = ids;
    g.routed_slots = g.P;
  }
  const int act = c->act_dtype == MOE_BF16 ? 1 : 0;
  const int wdt = c->expert_dtype == MOE_F32 ? 0 : (c->expert_dtype == MOE_BF16 ? 1 : 2);
  // batches of a few tokens: one warp per weight row, direct loads; larger
  // ones: the bulk-copy streaming kernels, which stage up to 8 tokens
  const bool small = c->T <= kGemvSmallTokens;
  cudaError_t e = run(MOE_KERNEL_GEMV_GATEUP, st, [&] {
    return small ? launch_gemv_small(g, act, wdt, false, st) : launch_gemv_gateup(g, act, wdt, st);
  });
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  g.r_attn = r_attn;
  g.out = out;
  if (small && gemv_small_down_combine_ok(g)) {
    // one kernel for down and combine (a token's few pairs and its shared
    // expert fit one CTA per output column group): one launch fewer on the
    // latency-bound single-token path
    return cuda_status(run(MOE_KERNEL_GEMV_DOWN, st, [&] {
      return launch_gemv_small_down_combine(g, act, wdt, st);
    }));
  }
  e = run(MOE_KERNEL_GEMV_DOWN, st, [&] {
    return small ? launch_gemv_small(g, act, wdt, true, st) : launch_gemv_down(g, act, wdt, st);
  });
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  CombineArgs cb{r_attn, g.Y, g.has_shared ? g.Ys : nullptr,
                 pairs ? nullptr : at<int32_t>(c, p.pos), out, c->T, c->d_model, c->top_k, 0};
  return cuda_status(run(MOE_KERNEL_COMBINE, st, [&] { return launch_combine(cb, st); }));
}

// The single-launch decode kernel: route mode (ids null: the whole layer,
// writing topk_ids / weights) or given-ids mode (the expert half for the
// caller's ids, weights and optional shared gate).
moe_status_t enqueue_fused(const void* x, const float* r_attn, const void* W_router,
                           const float* bias, const int32_t* ids_in, const float* w_in,
                           const float* s_in, moe_bank_t Wg, moe_bank_t Wu, moe_bank_t Wd,
                           const void* Wsg, const void* Wsu, const void* Wsd, const void* w_shared,
                           const moe_cfg_t* c, float* out, int32_t* ids_out, float* w_out,
                           cudaStream_t st, float* s_out = nullptr, bool route_only = false) {
  const Plan p = make_plan(*c);
  DecodeArgs a{};
  a.route_only = route_only ? 1 : 0;
  a.s_out = s_out;
  a.x = x;
  a.r_attn = r_attn;
  a.W_router = W_router;
  a.bias = bias;
  a.w_shared = w_shared;
  a.ids_in = ids_in;
  a.w_in = w_in;
  a.s_in = s_in;
  a.Wg = Wg.w; a.Wu = Wu.w; a.Wd = Wd.w;
  a.Wsg = Wsg; a.Wsu = Wsu; a.Wsd = Wsd;
  a.out = out;
  a.topk_ids = ids_out;
  a.weights = w_out;
  a.logits = at<float>(c, p.logits);
  a.H = at<float>(c, p.H);
  a.Hs = at<float>(c, p.Hs);
  a.Yg = at<float>(c, p.Y);
  a.Gs = at<float>(c, p.Gs);
  a.ctrl = at<Ctrl>(c, 0);
  a.T = c->T; a.d = c->d_model; a.E = c->n_experts; a.k = c->top_k;
  a.I = c->d_ff; a.Is = c->d_ff_shared;
  a.kind = c->router;
  a.n_group = c->n_group;
  a.topk_group = c->topk_group;
  a.routed_scaling = c->routed_scaling;
  a.renorm_clamp = c->renorm_clamp;
  a.wait_ns = take_stall(MOE_KERNEL_DECODE, &a.stall);
  const bool bf16 = c->act_dtype == MOE_BF16;
  return cuda_status(run(MOE_KERNEL_DECODE, st, [&] { return launch_decode_fused(a, bf16, st); }));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_ROUTE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: outside the library's limits";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace null, too small or misaligned";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or launch failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK: a device-side check failed";
  }
  return "unknown moe_status_t";
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

moe_status_t moe_trace_kernel(int kernel, void* const* starts, void* const* stops, int n,
                              int* count) {
  if (kernel == 0) {
    g_trace = TraceState{};
    return MOE_OK;
  }
  if (kernel < MOE_KERNEL_ROUTER_LOGITS || kernel > MOE_KERNEL_DECODE || n <= 0 || !starts ||
      !stops || !count)
    return MOE_ERR_INVALID_ARG;
  g_trace.kernel = kernel;
  g_trace.starts = (cudaEvent_t*)starts;
  g_trace.stops = (cudaEvent_t*)stops;
  g_trace.n = n;
  g_trace.count = count;
  *count = 0;
  return MOE_OK;
}

moe_status_t moe_inject_stall(int kernel, uint32_t wait_us) {
  if (kernel == 0) {
    g_stall_kernel.store(0);
    return MOE_OK;
  }
  if (kernel != MOE_KERNEL_TC_GATEUP && kernel != MOE_KERNEL_TC_DOWN && kernel != MOE_KERNEL_DECODE)
    return MOE_ERR_INVALID_ARG;
  g_stall_wait_ns.store((uint64_t)(wait_us ? wait_us : 1) * 1000ull);
  g_stall_kernel.store(kernel);
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_cfg_t* cfg) {
  moe_status_t s = validate_cfg(cfg);
  if (s != MOE_OK && s != MOE_ERR_UNSUPPORTED) return 0;
  return make_plan(*cfg).total;
}

moe_status_t moe_workspace_init(const moe_cfg_t* cfg, void* stream) {
  if (!cfg || !cfg->workspace || ((uintptr_t)cfg->workspace & 255u) ||
      cfg->workspace_bytes < sizeof(Ctrl))
    return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(cfg->workspace, 0, sizeof(Ctrl), (cudaStream_t)stream));
}

moe_status_t moe_read_device_status(const moe_cfg_t* cfg, void* stream, uint32_t* info) {
  if (!cfg || !cfg->workspace || cfg->workspace_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(&word, cfg->workspace, sizeof(word), cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  // a wait that gave up may leave the grid-barrier and arrival counters
  // mid-count: after a timeout every control word is reset (no kernel of
  // this workspace is running once the stream has synchronised)
  const size_t clear = (word & kDevTimeout) ? sizeof(Ctrl) : sizeof(word);
  if (cudaMemsetAsync(cfg->workspace, 0, clear, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (info) *info = word;
  if (word & kDevTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (word & 0xFFFFu) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

moe_status_t moe_route(const void* x, const void* W_router, const float* expert_bias,
                       const void* w_shared, const moe_cfg_t* cfg, int32_t* topk_ids,
                       float* weights, float* s_shared, void* stream) {
  moe_status_t s = validate_route_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_workspace(cfg)) != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !W_router || !topk_ids || !weights) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_router) || !aligned16(topk_ids) || !aligned16(weights))
    return MOE_ERR_INVALID_ARG;
  if (s_shared && (!w_shared || !aligned16(w_shared) || !aligned16(s_shared)))
    return MOE_ERR_INVALID_ARG;
  if (expert_bias && !aligned16(expert_bias)) return MOE_ERR_INVALID_ARG;
  if (use_fused(*cfg))  // the routing phases of the single-launch kernel
    return enqueue_fused(x, nullptr, W_router, expert_bias, nullptr, nullptr, nullptr, moe_bank_t{},
                         moe_bank_t{}, moe_bank_t{}, nullptr, nullptr, nullptr,
                         s_shared ? w_shared : nullptr, cfg, nullptr, topk_ids, weights,
                         (cudaStream_t)stream, s_shared, true);
  return enqueue_route(x, W_router, expert_bias, w_shared, cfg, topk_ids, weights, s_shared,
                       (cudaStream_t)stream);
}

moe_status_t moe_bucket(const int32_t* topk_ids, const moe_cfg_t* cfg, int32_t* counts,
                        int32_t* offsets, int32_t* active, int32_t* n_active, int32_t* perm,
                        int32_t* pos, void* stream) {
  moe_status_t s = validate_cfg(cfg);
  if (s != MOE_OK && s != MOE_ERR_UNSUPPORTED) return s;
  if (cfg->n_experts > 512) return MOE_ERR_UNSUPPORTED;
  if ((s = check_workspace(cfg)) != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  const void* ptrs[] = {topk_ids, counts, offsets, active, n_active, perm, pos};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return enqueue_bucket(topk_ids, cfg, counts, offsets, active, n_active, perm, pos,
                        (cudaStream_t)stream);
}

moe_status_t moe_experts_forward(const void* x, const float* r_attn, const int32_t* topk_ids,
                                 const float* weights, const float* s_shared, moe_bank_t W_gate,
                                 moe_bank_t W_up, moe_bank_t W_down, const void* Ws_gate,
                                 const void* Ws_up, const void* Ws_down, const void* w_shared,
                                 const moe_cfg_t* cfg, float* out, void* stream) {
  moe_status_t s = validate_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_workspace(cfg)) != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  const void* ptrs[] = {x, r_attn, topk_ids, weights, out};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (!bank_ok(W_gate, cfg->expert_dtype) || !bank_ok(W_up, cfg->expert_dtype) ||
      !bank_ok(W_down, cfg->expert_dtype))
    return MOE_ERR_INVALID_ARG;
  const bool shared = cfg->d_ff_shared > 0;
  if (shared) {
    const void* sp[] = {Ws_gate, Ws_up, Ws_down};
    for (const void* q : sp)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if (!s_shared && !w_shared) return MOE_ERR_INVALID_ARG;
    if ((s_shared && !aligned16(s_shared)) || (w_shared && !aligned16(w_shared)))
      return MOE_ERR_INVALID_ARG;
  }
  if ((const void*)out == x) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (use_fused(*cfg))
    return enqueue_fused(x, r_attn, nullptr, nullptr, topk_ids, weights, shared ? s_shared : nullptr,
                         W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, shared ? w_shared : nullptr,
                         cfg, out, nullptr, nullptr, st);
  const Plan p = make_plan(*cfg);
  if (shared && !s_shared) {
    // shared gate only: the router with zero routed rows
    RouterArgs ra{x, nullptr, w_shared, at<float>(cfg, p.logits), cfg->T, cfg->d_model, 0};
    const bool bf16 = cfg->act_dtype == MOE_BF16;
    cudaError_t e = run(MOE_KERNEL_SHARED_GATE, st, [&] {
      return launch_shared_gate(ra, at<float>(cfg, p.s_shared), bf16, st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    s_shared = at<float>(cfg, p.s_shared);
  }
  if (!gemv_pairs(*cfg)) {
    s = enqueue_bucket(topk_ids, cfg, at<int32_t>(cfg, p.counts), at<int32_t>(cfg, p.offsets),
                       at<int32_t>(cfg, p.active), &at<Ctrl>(cfg, 0)->n_active,
                       at<int32_t>(cfg, p.perm), at<int32_t>(cfg, p.pos), st);
    if (s != MOE_OK) return s;
  }
  return enqueue_experts(x, r_attn, topk_ids, weights, s_shared, W_gate, W_up, W_down, Ws_gate,
                         Ws_up, Ws_down, cfg, out, st, /*ids_distinct=*/false);
}

moe_status_t moe_layer_forward(const void* x, const float* r_attn, const void* W_router,
                               const float* expert_bias, moe_bank_t W_gate, moe_bank_t W_up,
                               moe_bank_t W_down, const void* Ws_gate, const void* Ws_up,
                               const void* Ws_down, const void* w_shared, const moe_cfg_t* cfg,
                               float* out, int32_t* topk_ids, float* weights, void* stream) {
  moe_status_t s = validate_cfg(cfg);
  if (s != MOE_OK) return s;
  if ((s = check_workspace(cfg)) != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  const void* ptrs[] = {x, r_attn, W_router, out, topk_ids, weights};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (expert_bias && !aligned16(expert_bias)) return MOE_ERR_INVALID_ARG;
  if (!bank_ok(W_gate, cfg->expert_dtype) || !bank_ok(W_up, cfg->expert_dtype) ||
      !bank_ok(W_down, cfg->expert_dtype))
    return MOE_ERR_INVALID_ARG;
  const bool shared = cfg->d_ff_shared > 0;
  if (shared) {
    const void* sp[] = {Ws_gate, Ws_up, Ws_down, w_shared};
    for (const void* q : sp)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  }
  if ((const void*)out == x) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (use_fused(*cfg))
    return enqueue_fused(x, r_attn, W_router, expert_bias, nullptr, nullptr, nullptr, W_gate, W_up,
                         W_down, Ws_gate, Ws_up, Ws_down, shared ? w_shared : nullptr, cfg, out,
                         topk_ids, weights, st);
  const Plan p = make_plan(*cfg);
  float* s_sh = shared ? at<float>(cfg, p.s_shared) : nullptr;
  s = enqueue_route_bucket(x, W_router, expert_bias, shared ? w_shared : nullptr, cfg, topk_ids,
                           weights, s_sh, st);
  if (s != MOE_OK) return s;
  return enqueue_experts(x, r_attn, topk_ids, weights, s_sh, W_gate, W_up, W_down, Ws_gate, Ws_up,
                         Ws_down, cfg, out, st, /*ids_distinct=*/true);
}

}  // extern "C"
