// attn_fold.cuh - decode attention on the warp-level f16 tensor cores, shared
// by the one-kernel decode step and the split-K decode attention kernel.
//
// One warp folds one 16-key block of one KV head for the two query heads of
// its group (tinyllm L10.1 "Candle model runner ...", section 2.4: scores
// q . k_j / sqrt(D), softmax over the visible keys, probability-weighted
// values): S = Q K^T with the two queries as MMA rows 0 and 1 (rows 2..15
// zero), the softmax of each head's 16 scores in fp32, O = P V with P rounded
// to f16, fp32 accumulation throughout.  The keys and values arrive by TMA in
// boxes of 16 rows x min(D, 64) f16 columns; with D >= 64 a box row is 128
// bytes and its 16-byte chunks are XOR-swizzled by the row (the 128-byte
// swizzle), so the 8 rows one ldmatrix reads at one column hit 8 different
// bank groups.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tc_common.cuh"

namespace dec {

// Where the K (or V) rows of one 16-slot block of one KV head land in shared
// memory (one "slab": 16 rows x D columns, in boxes of kBoxDims columns).
template <int D>
struct KvSlab {
  static constexpr int kBoxDims = D >= 64 ? 64 : D;
  static constexpr int kBoxes = D / kBoxDims;
  static constexpr int kRowBytes = kBoxDims * 2;
  static constexpr int kBoxBytes = 16 * kRowBytes;
  static constexpr int kBytes = kBoxes * kBoxBytes;
  static constexpr bool kSwizzle = kBoxDims == 64;
  // byte offset of (row r, the 8 dims from d, d a multiple of 8) in the slab
  static __device__ __forceinline__ int chunk(int r, int d) {
    const int bx = d / kBoxDims, c = (d % kBoxDims) >> 3;
    return bx * kBoxBytes + r * kRowBytes + ((kSwizzle ? (c ^ (r & 7)) : c) << 4);
  }
};

__device__ __forceinline__ void af_ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void af_ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void af_mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t af_pack_half(float x, float y) {
  const uint32_t lo = __half_as_ushort(__float2half_rn(x));
  const uint32_t hi = __half_as_ushort(__float2half_rn(y));
  return lo | (hi << 16);
}

// Fold `nkeys` (<= 16; <= 0: an empty block) keys of the K and V slabs at
// Ks / Vs (shared memory, KvSlab<D> layout) for the query rows q0, q1 (f16
// [D] each in shared memory; zrow: D f16 zeros).  Whole warp.  Lanes 0..7
// write o_out[h][d] (h = lane / 4; float, [2][D] in shared memory) and lanes
// 0 and 4 write m_out[h] / l_out[h] (the block's max and sum of exp(s - max);
// -inf and 0 for an empty block).  Value rows past nkeys must hold finite
// numbers (their probabilities are 0, and 0 * NaN is NaN).
template <int D>
__device__ __forceinline__ void fold16(const __half* q0, const __half* q1, const __half* zrow, const uint8_t* Ks,
                                       const uint8_t* Vs, int nkeys, float scale, float* o_out, float* m_out,
                                       float* l_out) {
  const int lane = threadIdx.x & 31;
  constexpr int kNT = D / 16;  // value n-tiles of 8 dims per half of the head
  float mh = -INFINITY, lh = 0.f;
  uint32_t P4[4] = {0u, 0u, 0u, 0u};
  if (nkeys > 0) {
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int qr = lane & 15;
    const uint32_t qa = smem_u32(qr == 0 ? q0 : qr == 1 ? q1 : zrow) + (lane >> 4) * 16;
    const int key = (lane & 7) + ((lane >> 4) << 3), doff = ((lane >> 3) & 1) * 8;
    const uint32_t kb = smem_u32(Ks);
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
      uint32_t A[4], B[4], A2[4], B2[4];
      af_ldsm4(qa + kk * 32, A);
      af_ldsm4(kb + KvSlab<D>::chunk(key, kk * 16 + doff), B);
      af_ldsm4(qa + kk * 32 + 32, A2);
      af_ldsm4(kb + KvSlab<D>::chunk(key, kk * 16 + 16 + doff), B2);
      af_mma_f16(s[0], A, B[0], B[1]);
      af_mma_f16(s[1], A, B[2], B[3]);
      af_mma_f16(s2[0], A2, B2[0], B2[1]);
      af_mma_f16(s2[1], A2, B2[2], B2[3]);
    }
    // row lane>>2 (a query head for lanes 0..7): keys nt*8 + 2*(lane&3) + e
    float sc[2][2];
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kx = nt * 8 + 2 * (lane & 3) + e;
        sc[nt][e] = kx < nkeys ? (s[nt][e] + s2[nt][e]) * scale : -INFINITY;
        mx = fmaxf(mx, sc[nt][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    float p[2][2], ps = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[nt][e] = sc[nt][e] == -INFINITY ? 0.f : expf(sc[nt][e] - mx);
        ps += p[nt][e];
      }
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    mh = mx;
    lh = ps;
    // P as the A operand: rows 8..15 are not query heads and stay zero
    P4[0] = af_pack_half(p[0][0], p[0][1]);
    P4[2] = af_pack_half(p[1][0], p[1][1]);
  }
  // O = P V in two halves of the head dimension (fewer live accumulators)
  const int vkey = (lane & 7) + ((lane >> 3) & 1) * 8, vd = (lane >> 4) * 8;
  const uint32_t vb = smem_u32(Vs);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    float oacc[kNT][4];
#pragma unroll
    for (int j = 0; j < kNT; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
    if (nkeys > 0) {
#pragma unroll
      for (int j = 0; j < kNT / 2; ++j) {
        uint32_t B[4];
        af_ldsm4t(vb + KvSlab<D>::chunk(vkey, (hf * kNT / 2 + j) * 16 + vd), B);
        af_mma_f16(oacc[2 * j], P4, B[0], B[1]);
        af_mma_f16(oacc[2 * j + 1], P4, B[2], B[3]);
      }
    }
    if (lane < 8) {
      const int h = lane >> 2;
#pragma unroll
      for (int j = 0; j < kNT; ++j)
        *reinterpret_cast<float2*>(o_out + h * D + hf * (D / 2) + 8 * j + 2 * (lane & 3)) =
            make_float2(oacc[j][0], oacc[j][1]);
    }
  }
  if (lane < 8 && (lane & 3) == 0) {
    m_out[lane >> 2] = mh;
    l_out[lane >> 2] = lh;
  }
}

// Write this lane's kDim values of a new K or V row (already f16-rounded) at
// row r of a slab (KvSlab<D> layout); with tail_zero, also zero rows r+1..15
// (value slots past the context).  Whole warp; lane holds dims lane*kDim.. .
template <int D>
__device__ __forceinline__ void patch_row(uint8_t* slab, int r, const __half* vals, bool tail_zero) {
  constexpr int kDim = D / 32;
  const int lane = threadIdx.x & 31;
  __half* st = reinterpret_cast<__half*>(slab + KvSlab<D>::chunk(r, (lane * kDim) & ~7)) + ((lane * kDim) & 7);
#pragma unroll
  for (int e = 0; e < kDim; ++e) st[e] = vals[e];
  if (tail_zero) {
    constexpr int kRB = KvSlab<D>::kRowBytes / 4;  // 32-bit words of a box row
    for (int i = lane; i < (15 - r) * KvSlab<D>::kBoxes * kRB; i += 32) {
      const int rr = r + 1 + i / (KvSlab<D>::kBoxes * kRB), rem = i % (KvSlab<D>::kBoxes * kRB);
      reinterpret_cast<uint32_t*>(slab + (rem / kRB) * KvSlab<D>::kBoxBytes + rr * KvSlab<D>::kRowBytes)[rem % kRB] = 0u;
    }
  }
}

}  // namespace dec
