/*
 * moe_route.h - C ABI of the sparse mixture-of-experts layer forward on one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The layer (the pages "How Treebeard routes Qwen3.6 MoE tokens", sections
 * "The short version", "Routing math", "Routed expert computation", "Shared
 * expert computation" and "Pseudocode"; Edge0 "MoE Routing and Experts",
 * sections "Experts", "Softmax top-k" and "Sigmoid group top-k"):
 *
 *   z_t      = W_router x_t                                (router logits)
 *   ids_t    = TopK(score(z_t), k)                         (routing rule)
 *   alpha_t  = normalised weights of the selected experts
 *   y_routed = sum_i alpha_t[i] * W_down_i (SiLU(W_gate_i x_t) * (W_up_i x_t))
 *   s_t      = sigmoid(w_shared . x_t)
 *   y_shared = s_t * Ws_down (SiLU(Ws_gate x_t) * (Ws_up x_t))
 *   out_t    = r_attn_t + (y_routed + y_shared)
 *
 * Conventions shared by every call:
 *   - Every tensor is caller-owned DEVICE memory, row-major and contiguous,
 *     16-byte aligned (checked: MOE_ERR_INVALID_ARG). The library allocates
 *     no device memory; scratch lives in a caller-provided workspace of
 *     moe_workspace_bytes(cfg) bytes, 256-byte aligned.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = the legacy default stream): it validates its arguments on the
 *     host, enqueues kernels and returns. No call synchronises the stream
 *     except moe_read_device_status. Nothing is copied to the host.
 *   - Host-side validation errors are returned synchronously and enqueue
 *     nothing. A failed launch returns MOE_ERR_CUDA.
 *   - Problems found on the device (an expert id out of range, a bounded wait
 *     that timed out) never fault or trap: the kernel records a code in the
 *     workspace's status word and keeps every access in bounds; the results of
 *     that call are then unspecified. moe_read_device_status reports and clears
 *     the word. The word is sticky across calls until read.
 *   - Calls that share a workspace must not run concurrently on the GPU.
 *   - No exception crosses this ABI.
 *
 * Shapes (T tokens, d = d_model, E routed experts, k = top_k, I = d_ff,
 * Is = d_ff_shared, P = T*k routed (token, slot) pairs):
 *   x         [T][d]     act_dtype (F32 or BF16); the post-attention,
 *                        RMS-normalised hidden state (normalisation is the
 *                        caller's, upstream of this layer)
 *   r_attn    [T][d]     f32, the attention residual
 *   out       [T][d]     f32; may alias r_attn (in-place residual update),
 *                        must not alias anything else
 *   W_router  [E][d]     act_dtype; row e scores expert e
 *   expert_bias [E]      f32, sigmoid family only (selection only); NULL = 0
 *   w_shared  [d]        act_dtype, the shared expert's scalar gate vector
 *   W_gate, W_up   banks [E][I][d]   expert_dtype (input dim contiguous)
 *   W_down         bank  [E][d][I]
 *   Ws_gate, Ws_up [Is][d], Ws_down [d][Is]   act_dtype
 *   topk_ids  [T][k]     int32, slots in descending score order
 *   weights   [T][k]     f32, alpha of each slot
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ROUTE_ABI_VERSION 1

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null pointer, bad shape, misalignment, aliasing */
  MOE_ERR_UNSUPPORTED = 2,    /* valid but outside the library's limits */
  MOE_ERR_WORKSPACE = 3,      /* workspace null, too small or misaligned */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded on-device wait gave up */
  MOE_ERR_DEVICE_CHECK = 6    /* a device-side check failed (e.g. id >= E) */
} moe_status_t;

typedef enum {
  /* "Routing math" (Treebeard page) / "Softmax top-k" (Edge0 page):
   * p = softmax(z) over all E experts; the k largest p; alpha_i =
   * p_i / max(sum of selected p, renorm_clamp) times routed_scaling. */
  MOE_ROUTER_SOFTMAX_TOPK = 0,
  /* "Sigmoid group top-k" (Edge0 page): s = sigmoid(z) in fp32; selection
   * score s + expert_bias; E/n_group contiguous experts per group ranked by
   * the sum of their two largest selection scores; the best topk_group groups
   * kept; the k largest selection scores inside them; alpha_i = s_i / sum of
   * selected s, times routed_scaling. */
  MOE_ROUTER_SIGMOID_GROUP_TOPK = 1
} moe_router_kind_t;

typedef enum {
  MOE_F32 = 0,
  MOE_BF16 = 1,
  /* 4-bit affine, group 64 (Edge0 tier table): w = scale * q + min with
   * q in 0..15, one (scale, min) pair of bf16 per 64 consecutive input-dim
   * elements, two codes per byte, the even element in the low nibble.
   * Bank layout: codes uint8 [E][N][K/2], scale and min bf16 [E][N][K/64]. */
  MOE_Q4_AFFINE_G64 = 2
} moe_dtype_t;

/* Expert-path selection for moe_layer_forward / moe_experts_forward. */
typedef enum {
  MOE_PATH_AUTO = 0,   /* by shape: with bf16 experts the single launch of
                          MOE_PATH_FUSED for 4 <= T <= 16 when its tensor-core
                          variant takes the shape and it is narrow enough
                          (d_model 1024 or 2048, d_ff and d_ff_shared
                          multiples of 128 up to 1024); otherwise CUDA-core
                          GEMV for T <= 5 and the tensor-core grouped GEMM
                          for T >= 6; 4-bit experts always take the
                          tensor-core path. moe_route follows the same
                          choice for its routing kernels. */
  MOE_PATH_GEMV = 1,   /* CUDA-core weight-streaming GEMV at any T */
  MOE_PATH_TC = 2,     /* tcgen05 grouped GEMM: bf16 or 4-bit experts with bf16
                          activations, d_model % 256 == 0, d_ff % 128 == 0,
                          d_ff_shared % 128 == 0 (a shared expert as wide as
                          the routed ones is one more group of their GEMMs,
                          one of another width runs as its own launches;
                          4-bit: no shared expert); other shapes return
                          MOE_ERR_UNSUPPORTED (and MOE_PATH_AUTO then uses
                          the GEMV path) */
  MOE_PATH_FUSED = 3   /* one cooperative launch (one block per SM) for the
                          whole layer, the device-routed decode of the
                          Treebeard page's "NVIDIA CUDA path": routing,
                          expert grouping, gate/up, down and combine as
                          phases split by bounded grid barriers (bf16
                          shapes as above contract on tensor cores with
                          mma.sync; others stream on CUDA cores).
                          1 <= T <= 16, bf16 (or fp32) banks and activations
                          alike, E <= 512, k <= 32; otherwise
                          MOE_ERR_UNSUPPORTED. moe_route with this path
                          runs the kernel's routing phases only, so that
                          its ids and weights are those of the layer. */
} moe_path_t;

typedef struct {
  int32_t T;             /* tokens, >= 0 (T = 0 enqueues nothing) */
  int32_t d_model;       /* d, multiple of 8 */
  int32_t n_experts;     /* E, 1..512 */
  int32_t top_k;         /* k, 1..min(E, 32) */
  int32_t d_ff;          /* I, multiple of 8 */
  int32_t d_ff_shared;   /* Is, multiple of 8; 0 = no shared expert */
  int32_t router;        /* moe_router_kind_t */
  int32_t n_group;       /* sigmoid family: E % n_group == 0, n_group <= 32 */
  int32_t topk_group;    /* sigmoid family: topk_group * E/n_group >= k */
  float routed_scaling;  /* multiplies alpha after normalisation (1 for Qwen) */
  float renorm_clamp;    /* softmax family: denominator floor (2^-14) */
  int32_t act_dtype;     /* moe_dtype_t of x, W_router, w_shared, shared expert */
  int32_t expert_dtype;  /* moe_dtype_t of the routed banks */
  int32_t path;          /* moe_path_t */
  void* workspace;       /* device scratch, >= moe_workspace_bytes(cfg) bytes */
  size_t workspace_bytes;
} moe_cfg_t;

/* One routed expert bank. F32/BF16: w = [E][N][K] values. Q4: w = codes,
 * scale/minv as described for MOE_Q4_AFFINE_G64; otherwise scale/minv NULL. */
typedef struct {
  const void* w;
  const void* scale;
  const void* minv;
} moe_bank_t;

/* Kernel families launched by this library (for moe_trace_kernel). */
typedef enum {
  MOE_KERNEL_ROUTER_LOGITS = 1, /* router contraction (+ shared-gate logit) */
  MOE_KERNEL_ROUTER_TOPK = 2,   /* routing rule, one warp per token */
  MOE_KERNEL_SHARED_GATE = 3,   /* shared gate alone (moe_experts_forward) */
  MOE_KERNEL_BUCKET = 4,        /* counting and packing pass (1 or 2 launches) */
  MOE_KERNEL_GEMV_GATEUP = 5,   /* CUDA-core gate/up + SwiGLU (direct-load or streaming) */
  MOE_KERNEL_GEMV_DOWN = 6,     /* CUDA-core down x alpha (direct-load or streaming) */
  MOE_KERNEL_COMBINE = 7,       /* unpermute, shared branch, residual */
  MOE_KERNEL_TC_GATEUP = 8,     /* tensor-core grouped gate/up + SwiGLU */
  MOE_KERNEL_TC_DOWN = 9,       /* tensor-core grouped down x alpha */
  MOE_KERNEL_GATHER = 10,       /* packed-row gather of x (tensor-core path) */
  MOE_KERNEL_TC_ROUTER = 11,    /* tensor-core router contraction (T >= 128, bf16) */
  MOE_KERNEL_DECODE = 12        /* single-launch decode kernel (MOE_PATH_FUSED) */
} moe_kernel_t;

/* Returns the ABI version (MOE_ROUTE_ABI_VERSION). */
MOE_API int moe_abi_version(void);

/* Human-readable name of a status code. Never NULL; static storage. */
MOE_API const char* moe_status_string(moe_status_t status);

/* Text of the last CUDA error behind a MOE_ERR_CUDA returned to the calling
 * thread ("no error" if none). Static storage. */
MOE_API const char* moe_last_cuda_error(void);

/* Number of kernel launches this library has enqueued in this process (all
 * devices, all streams). For measurement: the difference across a region is
 * the number of this library's kernels launched in it. */
MOE_API uint64_t moe_launch_count(void);

/* Measurement aid. While enabled, every launch of kernel family `kernel`
 * (moe_kernel_t) is bracketed by cudaEventRecord(starts[i], stream) before
 * and cudaEventRecord(stops[i], stream) after, on the stream it is launched
 * on, with i = *count % n; *count (host memory) is reset to 0 here and
 * incremented per traced launch. starts/stops are cudaEvent_t handles owned
 * by the caller, valid until tracing is turned off with kernel = 0. The
 * state is process-wide and not thread-safe. */
MOE_API moe_status_t moe_trace_kernel(int kernel, void* const* starts, void* const* stops,
                                      int n, int* count);

/* Failure-detection self-test: the next launch of kernel family `kernel`
 * (MOE_KERNEL_TC_GATEUP, MOE_KERNEL_TC_DOWN or MOE_KERNEL_DECODE) waits on a
 * flag that nothing sets, and every bounded wait of that launch gives up
 * after wait_us microseconds instead of about one second. The launch then
 * records MOE_ERR_DEVICE_TIMEOUT in its workspace's status word, lets its
 * copies in flight land, frees its tensor memory and returns; the call's
 * outputs are unspecified. One-shot and process-wide; kernel = 0 disarms.
 * Returns MOE_ERR_INVALID_ARG for any other kernel family. */
MOE_API moe_status_t moe_inject_stall(int kernel, uint32_t wait_us);

/* Workspace bytes needed by every call below for this cfg (the workspace
 * fields of cfg are ignored). Returns 0 if cfg is invalid. */
MOE_API size_t moe_workspace_bytes(const moe_cfg_t* cfg);

/* Zeroes the workspace's control words (status word and counters). Must be
 * enqueued once on a freshly allocated workspace before its first use. */
MOE_API moe_status_t moe_workspace_init(const moe_cfg_t* cfg, void* stream);

/* Synchronises `stream`, reads the workspace's device status word, clears
 * it, and returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_CHECK.
 * If info is non-NULL it receives the raw word (bit 0 bad id, bit 1 wait
 * timeout, upper 16 bits: first failing site). After a timeout it also
 * resets every control word of the workspace (a wait that gave up can leave
 * a grid-barrier count behind), so the workspace is usable again. */
MOE_API moe_status_t moe_read_device_status(const moe_cfg_t* cfg, void* stream,
                                    uint32_t* info);

/* Routing only ("Routing math" steps z -> p -> TopK -> renormalise;
 * "Sigmoid group top-k" steps 1-5). Writes topk_ids [T][k] (descending
 * score, ties to the lower expert id), weights [T][k] and, if s_shared is
 * non-NULL, the shared gate s_t = sigmoid(w_shared . x_t) [T] (requires
 * w_shared). expert_bias is ignored for the softmax family. */
MOE_API moe_status_t moe_route(const void* x, const void* W_router,
                       const float* expert_bias, const void* w_shared,
                       const moe_cfg_t* cfg, int32_t* topk_ids, float* weights,
                       float* s_shared, void* stream);

/* Routing without a workspace, for callers that cannot allocate device
 * memory (a plugin whose host framework owns every allocation and offers no
 * allocator; a serving loop that must not allocate once running, because an
 * allocation can synchronise the device). The pages have no counterpart:
 * this is a packaging of moe_route, with the same arguments and outputs,
 * except that the router logits live in a fixed array inside the library
 * (4 MiB, held on every device that loads the library until exit) instead
 * of cfg->workspace, which is ignored. Allocates nothing.
 * - Routing follows moe_route's CUDA-core router at every T (moe_route
 *   uses a tensor-core router contraction from 128 bf16 tokens; the two
 *   logits may differ in their last bits, so near-tied ids may differ).
 * - Errors: moe_route's argument checks and codes, without the workspace
 *   check; in addition T * (E + 1) above 1,048,576 returns
 *   MOE_ERR_UNSUPPORTED. A failed lookup or launch returns MOE_ERR_CUDA
 *   with its text in moe_last_cuda_error.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture. A device reset invalidates the lookup: do
 *   not call this entry point on a device after resetting it.
 * - All calls share the array, which keeps the last call's logits: calls
 *   whose kernels overlap on the GPU (two streams, two threads) race on it
 *   and must be serialised by the caller.
 * - Its launches are not counted by moe_launch_count nor traced. */
MOE_API moe_status_t moe_route_static(const void* x, const void* W_router,
                                      const float* expert_bias, const void* w_shared,
                                      const moe_cfg_t* cfg, int32_t* topk_ids, float* weights,
                                      float* s_shared, void* stream);

/* Counting and packing pass ("Intel SYCL path", steps 1-3 of the Treebeard
 * page) over given routing ids [T][k]: counts [E] pairs per expert, offsets
 * [E+1] exclusive scan, active [E] the experts with a pair in ascending id
 * (n_active [1] of them; entries past n_active unspecified), perm [P] the
 * pair ids t*k+slot packed by expert (ascending pair id within an expert)
 * and pos [P] its inverse. All outputs device int32. Ids outside [0, E) are
 * counted as expert E-1 and flagged in the status word. */
MOE_API moe_status_t moe_bucket(const int32_t* topk_ids, const moe_cfg_t* cfg,
                        int32_t* counts, int32_t* offsets, int32_t* active,
                        int32_t* n_active, int32_t* perm, int32_t* pos,
                        void* stream);

/* Expert half of the layer for given routing ("Routed expert computation",
 * "Shared expert computation", the residual add of "Pseudocode"):
 * out = r_attn + sum_slot weights * expert(x) + s_shared * shared(x).
 * s_shared [T] f32 may be NULL, in which case the gate is computed from
 * w_shared; both NULL is invalid when d_ff_shared > 0. Ids outside [0, E)
 * are flagged in the status word (MOE_ERR_DEVICE_CHECK from
 * moe_read_device_status) and every access stays in bounds; the outputs of
 * the tokens involved are then unspecified. */
MOE_API moe_status_t moe_experts_forward(const void* x, const float* r_attn,
                                 const int32_t* topk_ids, const float* weights,
                                 const float* s_shared,
                                 moe_bank_t W_gate, moe_bank_t W_up,
                                 moe_bank_t W_down, const void* Ws_gate,
                                 const void* Ws_up, const void* Ws_down,
                                 const void* w_shared, const moe_cfg_t* cfg,
                                 float* out, void* stream);

/* The whole layer forward (the Treebeard page's "Pseudocode", x already
 * normalised): router, routing rule, bucketing, routed experts, shared
 * expert, combine and residual. Also writes the routing artefacts
 * topk_ids [T][k] and weights [T][k], which are final once written. */
MOE_API moe_status_t moe_layer_forward(const void* x, const float* r_attn,
                               const void* W_router, const float* expert_bias,
                               moe_bank_t W_gate, moe_bank_t W_up,
                               moe_bank_t W_down, const void* Ws_gate,
                               const void* Ws_up, const void* Ws_down,
                               const void* w_shared, const moe_cfg_t* cfg,
                               float* out, int32_t* topk_ids, float* weights,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
