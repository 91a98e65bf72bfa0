// Counting and packing pass over the routed (token, slot) pairs ("How
// Treebeard routes Qwen3.6 MoE tokens", "Intel SYCL path", steps 1-3): count
// pairs per expert, exclusive-scan the counts into offsets, list the active
// experts, and pack every pair id t*k+slot under its expert, in ascending
// pair order within an expert (a stable counting sort).
//
// Run by one CTA of NW warps. Warp w owns a contiguous segment of the pairs
// and a private histogram row, so the packing phase needs no atomics: a warp
// ranks equal experts inside each 32-pair batch with __match_any_sync and
// advances its own cursors. The expert ids are read through L2 (ld.global.cg)
// because the multi-CTA pass reads them in two kernels.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Row-block ranking holds one 64-bit key per group (E + 1 groups, E <= 512)
// in a buffer of this many entries.
constexpr int kRankKeys = 1024;

// Shared-memory words bucket_body<NW> needs for E experts: the per-warp
// histograms, the scan arrays, and the 8-byte-aligned sort keys.
__host__ __device__ constexpr int bucket_smem_words(int nw, int E) {
  return nw * E + E + (E + 1) + E + (E + 1) + 3 * (E + 1) + 1 + 1 + 2 * kRankKeys;
}

// Exclusive scan of n (<= 32*16) ints held in smem `v` by warp 0; writes
// `out[0..n]` (out[n] = total). The caller syncs.
__device__ __forceinline__ void warp0_exclusive_scan(const int* v, int* out, int n) {
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

// From per-expert counts cnt[E] in shared memory: offsets (exclusive scan),
// the active list and its length, written to the outputs; flag and aoff are
// scratch [E] and [E+1] (aoff[E] = number of active experts). All threads of
// the CTA call it; it ends synchronised.
template <int NW>
__device__ __forceinline__ void publish_counts(const BucketArgs& a, const int* cnt, int* offs,
                                               int* flag, int* aoff) {
  constexpr int kThreads = NW * 32;
  const int E = a.E, tid = threadIdx.x;
  for (int e = tid; e < E; e += kThreads) flag[e] = cnt[e] > 0 ? 1 : 0;
  __syncthreads();
  if (tid < 32) {
    warp0_exclusive_scan(cnt, offs, E);
    __syncwarp();
    warp0_exclusive_scan(flag, aoff, E);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) {
    a.counts[e] = cnt[e];
    a.offsets[e] = offs[e];
    if (flag[e]) a.active[aoff[e]] = e;
  }
  if (tid == 0) {
    a.offsets[E] = offs[E];
    *a.n_active = aoff[E];
  }
  __syncthreads();
}

// Row-block work list for the tensor-core path: groups ordered by size
// (largest first, ties by lower id; the shared expert is group E with
// shared_rows rows), then the blocks of bm rows of each (every second block
// when a.pair: each entry then stands for blocks m and m + 1). The order comes
// from ranking (rows descending, id ascending) keys in `keys` (E + 1 8-byte
// entries) by counting; order, nblk: [E+1], bofs: [E+2] scratch. All
// threads of the CTA call it.
template <int NW>
__device__ __forceinline__ void publish_rowblocks(const BucketArgs& a, const int* cnt,
                                                  const int* aoff, int* order, int* nblk,
                                                  int* bofs, unsigned long long* keys) {
  constexpr int kThreads = NW * 32;
  const int E = a.E, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // every group within one row block (decode-sized batches): the order does
  // not matter for balance, so take the active experts in id order, then the
  // shared expert
  bool big = a.shared_rows > a.bm;
  for (int g = tid; g < E; g += kThreads) big |= cnt[g] > a.bm;
  if (!__syncthreads_or(big)) {
    for (int e = tid; e < E; e += kThreads)
      if (cnt[e] > 0) a.rowblocks[aoff[e]] = make_int2(e, 0);
    if (tid == 0) {
      if (a.shared_rows > 0) a.rowblocks[aoff[E]] = make_int2(E, 0);
      *a.n_rowblocks = aoff[E] + (a.shared_rows > 0 ? 1 : 0);
    }
    return;
  }
  const int G = E + (a.shared_rows > 0 ? 1 : 0);
  // key: (0xFFFFFFFF - rows) << 32 | id, distinct for the groups with rows;
  // empty groups get the largest key and take no rank
  for (int g = tid; g < G; g += kThreads) {
    const int ng = g < E ? cnt[g] : a.shared_rows;
    keys[g] = ng > 0 ? ((unsigned long long)(0xFFFFFFFFu - (uint32_t)ng) << 32) | (uint32_t)g
                     : ~0ull;
  }
  __syncthreads();
  // a group's rank = the number of keys below its own: groups with rows
  // occupy ranks [0, n_nonempty) in ascending key order
  const int n_nonempty = aoff[E] + (a.shared_rows > 0 ? 1 : 0);
  for (int g = tid; g < G; g += kThreads) {
    const unsigned long long kg = keys[g];
    if (kg == ~0ull) continue;
    int r = 0;
#pragma unroll 8
    for (int h = 0; h < G; ++h) r += keys[h] < kg ? 1 : 0;
    const int ng = (int)(0xFFFFFFFFu - (uint32_t)(kg >> 32));
    order[r] = g;
    const int blocks = (ng + a.bm - 1) / a.bm;
    nblk[r] = a.pair ? (blocks + 1) / 2 : blocks;  // list entries: pairs when paired
  }
  __syncthreads();
  if (warp == 0) warp0_exclusive_scan(nblk, bofs, n_nonempty);
  __syncthreads();
  const int step = a.pair ? 2 : 1;
  for (int r = warp; r < n_nonempty; r += NW) {
    const int g = order[r];
    for (int m = lane; m < nblk[r]; m += 32) a.rowblocks[bofs[r] + m] = make_int2(g, m * step);
  }
  if (tid == 0) *a.n_rowblocks = bofs[n_nonempty];
}

// Counts the pairs [s0, s1) into per-warp histogram rows hist[NW][E] (warp w
// takes the w-th contiguous sub-segment); ids outside [0, E) are flagged and
// counted as E-1 so that every access stays in bounds. Ends synchronised.
template <int NW>
__device__ __forceinline__ void warp_histograms(const BucketArgs& a, int s0, int s1, int* hist) {
  constexpr int kThreads = NW * 32;
  const int E = a.E, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < NW * E; i += kThreads) hist[i] = 0;
  __syncthreads();
  const int seg = (s1 - s0 + NW - 1) / NW;
  const int w0 = min(s1, s0 + warp * seg), w1 = min(s1, w0 + seg);
  bool bad = false;
  for (int i = w0 + lane; i < w1; i += 32) {
    int e = __ldcg(a.ids + i);
    if (e < 0 || e >= E) { bad = true; e = E - 1; }
    atomicAdd(&hist[warp * E + e], 1);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(a.ctrl, kDevBadId, kSiteBucket);
  __syncthreads();
}

// Stable packing of the pairs [s0, s1): hist[w][e] holds warp w's first
// packed position for expert e; warp w places its sub-segment in order,
// ranking equal experts inside each 32-pair batch with __match_any_sync.
template <int NW>
__device__ __forceinline__ void pack_pairs(const BucketArgs& a, int s0, int s1, int* hist) {
  const int E = a.E, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = (s1 - s0 + NW - 1) / NW;
  const int w0 = min(s1, s0 + warp * seg), w1 = min(s1, w0 + seg);
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool valid = i < w1;
    int e = -1;
    if (valid) {
      e = __ldcg(a.ids + i);
      if (e < 0 || e >= E) e = E - 1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid) {
      const int p = hist[warp * E + e] + rank;
      a.perm[p] = i;
      a.pos[i] = p;
    }
    __syncwarp();
    if (valid && rank == 0) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
}

// The whole pass in one CTA of NW warps.
template <int NW>
__device__ __forceinline__ void bucket_body(const BucketArgs& a, int* smem) {
  constexpr int kThreads = NW * 32;
  const int E = a.E, P = a.P, tid = threadIdx.x;
  int* hist = smem;                  // [NW][E]: counts, then warp bases
  int* cnt = hist + NW * E;          // [E]
  int* offs = cnt + E;               // [E+1]
  int* flag = offs + E + 1;          // [E]
  int* aoff = flag + E;              // [E+1]
  int* order = aoff + E + 1;         // [E+1]  ranked group ids
  int* nblk = order + E + 1;         // [E+1]  row blocks per ranked group
  int* bofs = nblk + E + 1;          // [E+2]  exclusive scan of nblk
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(
      smem + ((bucket_smem_words(NW, E) - 2 * kRankKeys) & ~1));  // [kRankKeys]

  warp_histograms<NW>(a, 0, P, hist);
  for (int e = tid; e < E; e += kThreads) {
    int run = 0;
    for (int w = 0; w < NW; ++w) run += hist[w * E + e];
    cnt[e] = run;
  }
  __syncthreads();
  publish_counts<NW>(a, cnt, offs, flag, aoff);
  // warp bases inside each expert's packed range
  for (int e = tid; e < E; e += kThreads) {
    int run = offs[e];
    for (int w = 0; w < NW; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  pack_pairs<NW>(a, 0, P, hist);
  if (a.rowblocks) {
    __syncthreads();
    publish_rowblocks<NW>(a, cnt, aoff, order, nblk, bofs, keys);
  }
}

}  // namespace moe
