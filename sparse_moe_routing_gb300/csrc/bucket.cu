// Bucketing kernels (algorithm and source in bucket_core.cuh).
//
// Up to kBucketOneCta pairs: one CTA of 32 warps does the whole pass.
// Larger batches: two kernels over kSegCtas-pair segments.
//  1. bucket_hist: each CTA histograms its segment into cta_hist[b][E]; the
//     last CTA to finish (self-resetting arrival counter) turns the
//     histograms into per-CTA bases (exclusive prefix over CTAs per expert),
//     publishes counts, offsets, the active list and the row-block list.
//  2. bucket_pack: each CTA recounts its segment per warp and places its
//     pairs at offsets[e] + its CTA base + its warp base, stable.
#include "bucket_core.cuh"

namespace moe {

constexpr int kBucketWarps = 32;
constexpr int kPackWarps = 8;
constexpr int kSegPairs = 256 * 8;  // pairs per CTA of the multi-CTA pass

__global__ void __launch_bounds__(kBucketWarps * 32) bucket_kernel(BucketArgs a) {
  extern __shared__ int smem[];
  pdl_wait();
  pdl_trigger();
  bucket_body<kBucketWarps>(a, smem);
}

__global__ void __launch_bounds__(kPackWarps * 32) bucket_hist_kernel(BucketArgs a, int* cta_hist) {
  extern __shared__ int smem[];
  __shared__ int s_last;
  constexpr int kThreads = kPackWarps * 32;
  const int E = a.E, tid = threadIdx.x, b = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const int s0 = min(a.P, b * kSegPairs), s1 = min(a.P, s0 + kSegPairs);
  int* hist = smem;  // [E]
  for (int e = tid; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int i = s0 + tid; i < s1; i += kThreads) {
    int e = __ldcg(a.ids + i);
    if (e < 0 || e >= E) { bad = true; e = E - 1; }
    atomicAdd(&hist[e], 1);
  }
  if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0) report(a.ctrl, kDevBadId, kSiteBucket);
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) cta_hist[(size_t)b * E + e] = hist[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&a.ctrl->arrive_bucket, 1u);
    s_last = prev == gridDim.x - 1;
    if (s_last) a.ctrl->arrive_bucket = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  int* cnt = smem;                   // [E]
  int* offs = cnt + E;               // [E+1]
  int* flag = offs + E + 1;          // [E]
  int* aoff = flag + E;              // [E+1]
  int* order = aoff + E + 1;         // [E+1]
  int* nblk = order + E + 1;         // [E+1]
  int* bofs = nblk + E + 1;          // [E+2]
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(
      smem + ((bucket_smem_words(0, E) - 2 * kRankKeys) & ~1));  // [kRankKeys]
  // per-CTA bases: exclusive prefix over CTAs of each expert's counts, eight
  // CTAs' counts loaded at a time so their L2 round trips overlap
  const int nb = (int)gridDim.x;
  for (int e = tid; e < E; e += kThreads) {
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += 8) {
      int c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        c[u] = b0 + u < nb ? __ldcg(cta_hist + (size_t)(b0 + u) * E + e) : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (b0 + u < nb) cta_hist[(size_t)(b0 + u) * E + e] = run;
        run += c[u];
      }
    }
    cnt[e] = run;
  }
  __syncthreads();
  publish_counts<kPackWarps>(a, cnt, offs, flag, aoff);
  if (a.rowblocks) publish_rowblocks<kPackWarps>(a, cnt, aoff, order, nblk, bofs, keys);
}

__global__ void __launch_bounds__(kPackWarps * 32) bucket_pack_kernel(BucketArgs a,
                                                                      const int* cta_base) {
  extern __shared__ int smem[];
  constexpr int kThreads = kPackWarps * 32;
  const int E = a.E, tid = threadIdx.x, b = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const int s0 = min(a.P, b * kSegPairs), s1 = min(a.P, s0 + kSegPairs);
  int* hist = smem;  // [kPackWarps][E]
  warp_histograms<kPackWarps>(a, s0, s1, hist);
  for (int e = tid; e < E; e += kThreads) {
    int run = a.offsets[e] + cta_base[(size_t)b * E + e];
    for (int w = 0; w < kPackWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  pack_pairs<kPackWarps>(a, s0, s1, hist);
}

int bucket_ctas(int P) { return P <= kBucketOneCta ? 1 : (P + kSegPairs - 1) / kSegPairs; }

cudaError_t launch_bucket(const BucketArgs& a, cudaStream_t st) {
  if (a.P == 0) return cudaSuccess;
  const size_t smem = (size_t)bucket_smem_words(kBucketWarps, a.E) * sizeof(int);
  // raise the opt-in limit when this E needs more than the default
  static int attr[64] = {};
  cudaError_t e = ensure_smem_limit(bucket_kernel, (int)smem, attr);
  if (e != cudaSuccess) return e;
  return launch_pdl(bucket_kernel, 1, kBucketWarps * 32, smem, st, a);
}

cudaError_t launch_bucket_hist(const BucketArgs& a, int* cta_hist, cudaStream_t st) {
  if (a.P == 0) return cudaSuccess;
  const size_t smem = (size_t)bucket_smem_words(0, a.E) * sizeof(int);
  return launch_pdl(bucket_hist_kernel, bucket_ctas(a.P), kPackWarps * 32, smem, st, a, cta_hist);
}

cudaError_t launch_bucket_pack(const BucketArgs& a, const int* cta_base, cudaStream_t st) {
  if (a.P == 0) return cudaSuccess;
  const size_t smem = (size_t)kPackWarps * a.E * sizeof(int);
  return launch_pdl(bucket_pack_kernel, bucket_ctas(a.P), kPackWarps * 32, smem, st, a, cta_base);
}

}  // namespace moe
