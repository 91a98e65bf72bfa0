// Tensor-core arithmetic of the single-launch decode kernel's weight stream
// (bf16 weights and activations): a few tokens against 2D weight tiles that
// TMA lands in shared memory with the 128-byte swizzle (rows of 64 bf16, the
// 16-byte chunk c of row r stored at chunk c ^ (r % 8)).
//
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) takes the narrow token side as
// its n = 8 dimension:
//  * gate/up: D[16 weight rows][8 tokens] += W[16 rows][16 k] x X^T[16 k][8 tokens]
//    (A from the weight tile by ldmatrix, B from the token rows of x);
//  * down:    D[16 pair slots][8 columns] += H[16 slots][16 k] x Wd^T[16 k][8 columns]
//    (A from h rows stored in fragment order, of which only the first 8
//    slots exist, B from the down tile by ldmatrix).
// Fragment layouts (PTX ISA, mma.m16n8k16 with .bf16): lane = 4 g + t;
// A regs (row g, k 2t..2t+1), (row g+8, k 2t..), (row g, k 2t+8..), (row g+8,
// k 2t+8..); B regs (k 2t..2t+1, col g), (k 2t+8.., col g); D regs (row g,
// cols 2t, 2t+1), (row g+8, cols 2t, 2t+1).
#pragma once

#include "common.cuh"

namespace moe {
namespace dmma {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Address of 16-byte chunk c of row r in a 128-byte-swizzled tile at `base`
// (1024-byte aligned).
__device__ __forceinline__ uint32_t sw(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * 128) + (uint32_t)(((c ^ (r & 7)) & 7) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two bf16 at element k of row `row` of a [rows][ld] bf16 array (k even),
// read through the read-only path (inputs of the launch).
__device__ __forceinline__ uint32_t ld_pair_ro(const __nv_bfloat16* p, size_t row, size_t ld, int k) {
  return __ldg(reinterpret_cast<const unsigned int*>(p + row * ld + k));
}
// B fragments of one 64-wide K segment for token slot g = lane / 4 (row
// tok_g of x, zeros when the slot is empty): for k16 step s, registers 2 s
// (k 2t..2t+1) and 2 s + 1 (k 2t+8..2t+9), t = lane % 4. Loaded ahead of the
// weight tile they meet.
__device__ __forceinline__ void x_frags(const __nv_bfloat16* x, int d, int tok_g, bool valid_g,
                                        int k0, int lane, uint32_t (&xb)[8]) {
  const int t = lane & 3;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    xb[2 * s] = valid_g ? ld_pair_ro(x, (size_t)tok_g, (size_t)d, k0 + 16 * s + 2 * t) : 0u;
    xb[2 * s + 1] = valid_g ? ld_pair_ro(x, (size_t)tok_g, (size_t)d, k0 + 16 * s + 8 + 2 * t) : 0u;
  }
}

// Gate/up: one stage holds the gate tile (16 rows x 64 k) at `st` and the up
// tile at `st + 2048`; xb holds the tokens' fragments for the same k.
// Accumulates D fragments (rows x token slots).
__device__ __forceinline__ void gateup_tile(const uint8_t* st, const uint32_t (&xb)[8], int lane,
                                            float (&dg)[4], float (&du)[4]) {
  const uint32_t bg = smem_addr(st), bu = bg + 2048;
  const int r = lane & 15, hi = lane >> 4;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(sw(bg, r, 2 * s + hi), a0, a1, a2, a3);
    mma16816(dg, a0, a1, a2, a3, xb[2 * s], xb[2 * s + 1]);
    ldsm_x4(sw(bu, r, 2 * s + hi), a0, a1, a2, a3);
    mma16816(du, a0, a1, a2, a3, xb[2 * s], xb[2 * s + 1]);
  }
}

// Router: one 16-row x 64-k tile of the router at `st`; accumulates its dot
// products with the tokens whose fragments xb holds.
__device__ __forceinline__ void router_tile(const uint8_t* st, const uint32_t (&xb)[8], int lane,
                                            float (&dr)[4]) {
  const uint32_t br = smem_addr(st);
  const int r = lane & 15, hi = lane >> 4;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(sw(br, r, 2 * s + hi), a0, a1, a2, a3);
    mma16816(dr, a0, a1, a2, a3, xb[2 * s], xb[2 * s + 1]);
  }
}

// Down: one stage holds nbox (2 or 4) tiles of 8 output columns x 64 k
// (1 KB each, at st + 1024 b); af holds the chunk's h rows for those k in mma
// fragment order (for k16 step j and lane, 8 bytes: the A registers (slot g,
// k 2t..2t+1) and (slot g, k 2t+8..2t+9)), either in the same stage or in a
// block-wide copy of the chunk. Rows 8..15 of the A tile do not exist
// (zero). Accumulates the D fragment (slots x columns).
__device__ __forceinline__ void down_tile(const uint8_t* st, const uint2* af, int nbox, int lane,
                                          float (&dd)[4]) {
  const uint32_t base = smem_addr(st);
  const int n = lane & 7, q = lane >> 3;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    if (b < nbox) {
      const uint32_t bb = base + 1024u * b;
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        // chunks 4 s2 .. 4 s2 + 3 of the 8 column rows: b0/b1 of k16 steps 2 s2, 2 s2 + 1
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sw(bb, n, 4 * s2 + q), b0, b1, b2, b3);
        const uint2 a0 = af[(4 * b + 2 * s2) * 32 + lane];
        const uint2 a1 = af[(4 * b + 2 * s2 + 1) * 32 + lane];
        mma16816(dd, a0.x, 0u, a0.y, 0u, b0, b1);
        mma16816(dd, a1.x, 0u, a1.y, 0u, b2, b3);
      }
    }
  }
}

// Index (in bf16 elements) of h(slot q, k) of fragment-ordered chunk c, for
// rows of K elements: [chunk][K/16 steps][32 lanes][a0 lo, a0 hi, a2 lo, a2 hi].
__device__ __forceinline__ size_t frag_index(int c, int K, int q, int k) {
  const int step = k >> 4, kk = k & 15;
  const int lane = 4 * q + ((kk & 7) >> 1);
  return (((size_t)c * (K >> 4) + step) * 32 + lane) * 4 + (kk >> 3) * 2 + (kk & 1);
}

}  // namespace dmma
}  // namespace moe
