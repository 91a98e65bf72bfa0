// Counting and packing pass over the routed (token, slot) pairs ("How
// Treebeard routes Qwen3.6 MoE tokens", "Intel SYCL path", steps 1-3): count
// pairs per expert, exclusive-scan the counts into offsets, list the active
// experts, and pack every pair id t*k+slot under its expert, in ascending
// pair order within an expert (a stable counting sort).
//
// One CTA of 32 warps. Warp w owns a contiguous segment of the pairs and a
// private histogram row, so the packing phase needs no atomics: a warp ranks
// equal experts inside each 32-pair batch with __match_any_sync and advances
// its own cursors.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBucketThreads = 1024;
constexpr int kBucketWarps = kBucketThreads / 32;

// Exclusive scan of n (<= 32*16) ints held in smem `v` by warp 0; writes
// `out[0..n]` (out[n] = total). Returns nothing; caller syncs.
__device__ void warp0_exclusive_scan(const int* v, int* out, int n) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) / 32;
  const int b = lane * per, e = min(n, b + per);
  int local = 0;
  for (int i = b; i < e; ++i) local += v[i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - local;
  for (int i = b; i < e; ++i) { out[i] = run; run += v[i]; }
  if (lane == 31) out[n] = incl;
}

__global__ void __launch_bounds__(kBucketThreads) bucket_kernel(BucketArgs a) {
  extern __shared__ int smem[];
  const int E = a.E, P = a.P;
  int* hist = smem;                       // [32][E]: counts, then warp bases
  int* cnt = hist + kBucketWarps * E;     // [E]
  int* offs = cnt + E;                    // [E+1]
  int* flag = offs + E + 1;               // [E]
  int* aoff = flag + E;                   // [E+1]
  int* order = aoff + E + 1;              // [E+1]  ranked group ids
  int* nblk = order + E + 1;              // [E+1]  row blocks per ranked group
  int* bofs = nblk + E + 1;               // [E+2]  exclusive scan of nblk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < kBucketWarps * E; i += kBucketThreads) hist[i] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  const int seg = (P + kBucketWarps - 1) / kBucketWarps;
  const int s0 = min(P, warp * seg), s1 = min(P, s0 + seg);
  bool bad = false;
  for (int i = s0 + lane; i < s1; i += 32) {
    int e = a.ids[i];
    if (e < 0 || e >= E) { bad = true; e = E - 1; }
    atomicAdd(&hist[warp * E + e], 1);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(a.ctrl, kDevBadId, kSiteBucket);
  __syncthreads();

  for (int e = tid; e < E; e += kBucketThreads) {
    int run = 0;
    for (int w = 0; w < kBucketWarps; ++w) {
      int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    cnt[e] = run;
    flag[e] = run > 0 ? 1 : 0;
  }
  __syncthreads();
  if (warp == 0) {
    warp0_exclusive_scan(cnt, offs, E);
    __syncwarp();
    warp0_exclusive_scan(flag, aoff, E);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kBucketThreads) {
    a.counts[e] = cnt[e];
    a.offsets[e] = offs[e];
    if (flag[e]) a.active[aoff[e]] = e;
  }
  if (tid == 0) {
    a.offsets[E] = offs[E];
    *a.n_active = aoff[E];
  }

  // stable packing: warp w places its segment in order after the pairs of
  // lower warps (hist now holds each warp's base inside each expert)
  for (int base = s0; base < s1; base += 32) {
    const int i = base + lane;
    const bool valid = i < s1;
    int e = -1;
    if (valid) {
      e = a.ids[i];
      if (e < 0 || e >= E) e = E - 1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int p = 0;
    if (valid) {
      p = offs[e] + hist[warp * E + e] + rank;
      a.perm[p] = i;
      a.pos[i] = p;
    }
    __syncwarp();
    if (valid && rank == 0) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }

  // row-block work list for the tensor-core path: groups ordered by size
  // (largest first, ties by lower id), then the blocks of bm rows of each
  if (a.rowblocks) {
    __syncthreads();
    // rank of group g among groups with rows (shared group E included)
    const int G = E + (a.shared_rows > 0 ? 1 : 0);
    for (int g = tid; g < G; g += kBucketThreads) {
      const int ng = g < E ? cnt[g] : a.shared_rows;
      int r = 0;
      if (ng > 0) {
        for (int h = 0; h < G; ++h) {
          const int nh = h < E ? cnt[h] : a.shared_rows;
          r += (nh > ng || (nh == ng && h < g)) ? 1 : 0;
        }
        order[r] = g;
        nblk[r] = (ng + a.bm - 1) / a.bm;
      }
    }
    __syncthreads();
    // groups with rows occupy ranks [0, n_nonempty)
    const int n_nonempty = aoff[E] + (a.shared_rows > 0 ? 1 : 0);
    if (warp == 0) warp0_exclusive_scan(nblk, bofs, n_nonempty);
    __syncthreads();
    for (int r = warp; r < n_nonempty; r += kBucketWarps) {
      const int g = order[r];
      for (int m = lane; m < nblk[r]; m += 32) a.rowblocks[bofs[r] + m] = make_int2(g, m);
    }
    if (tid == 0) *a.n_rowblocks = bofs[n_nonempty];
  }
}

cudaError_t launch_bucket(const BucketArgs& a, cudaStream_t st) {
  if (a.P == 0) return cudaSuccess;
  const int words = kBucketWarps * a.E + a.E + (a.E + 1) + a.E + (a.E + 1) +
                    3 * (a.E + 1) + 1;
  const size_t smem = (size_t)words * sizeof(int);
  // raise the opt-in limit when this E needs more than the default
  static int attr[64] = {};
  cudaError_t e = ensure_smem_limit(bucket_kernel, (int)smem, attr);
  if (e != cudaSuccess) return e;
  return launch_pdl(bucket_kernel, 1, kBucketThreads, smem, st, a);
}

}  // namespace moe
