// epilogue.cuh - the fused epilogues shared by every weight-product kernel
// (CUDA-core streaming, CUDA-core tiled, tcgen05).
#pragma once

#include "common.cuh"
#include "launch.h"

namespace dec {

// ---------------------------------------------------------------------------
// Fused epilogues of the weight products, shared by the streaming kernel and
// the tiled kernel.  tile[r * ld + t] holds y for weight row r0 + r and token
// row t0 + t (r < nrows, t < ntok; nrows is a multiple of 16).
//   QKV_RAW : y * rstd -> raw q|k|v (QK-norm/RoPE/cache write follow)
//   RESID   : x += y ; next GEMM input x * w_next ; 16-feature sum of squares
//   SWIGLU  : silu(rstd * gate) * (rstd * up), gate/up interleaved by 8 rows
//   LOGITS  : rstd * y -> logits ; argmax key per token (atomicMax)
// The RMSNorm before a product is split in two: its gain multiplies the
// product's input where that input is written (the RESID epilogue, the
// embedding), its 1/rms scales the product's output rows here.
// ---------------------------------------------------------------------------
template <typename AT, int EPI, int NT>
__device__ __forceinline__ void epilogue(const GemvArgs& a, const float* tile, int ld, int r0, int nrows, int t0,
                                         int ntok, const float* rstd_s, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int total = ntok * nrows;
  if (EPI == EPI_QKV_RAW) {
    for (int i = tid; i < total; i += NT) {
      const int t = i / nrows, r = i - t * nrows;
      a.out_f32[(size_t)(t0 + t) * a.rows + r0 + r] = tile[r * ld + t] * rstd_s[t];
    }
  } else if (EPI == EPI_RESID) {
    AT* XN = reinterpret_cast<AT*>(a.XN);
    const int nch = a.d / kSsqChunk;
    for (int base = warp * 32; base < total; base += NT) {  // whole warps; validity is per half-warp
      const int i = base + lane;
      const bool valid = i < total;
      const int t = i / nrows, r = i - t * nrows;
      float x = 0.f;
      if (valid) {
        const size_t off = (size_t)(t0 + t) * a.d + r0 + r;
        x = a.X_res[off] + tile[r * ld + t];
        a.X_res[off] = x;
        XN[off] = from_f32<AT>(x * a.w_next[r0 + r]);
      }
      const float sq = half_warp_sum(x * x);
      if (valid && (r & (kSsqChunk - 1)) == 0) a.SSQ_out[(size_t)(t0 + t) * nch + (r0 + r) / kSsqChunk] = sq;
    }
  } else if (EPI == EPI_SWIGLU) {
    AT* out = reinterpret_cast<AT*>(a.act_out);
    const int half = nrows / 2;
    for (int i = tid; i < ntok * half; i += NT) {
      const int t = i / half, j = i - t * half;
      const int grp = j / kGuGroup, jj = j % kGuGroup;
      const float g = tile[(grp * 2 * kGuGroup + jj) * ld + t] * rstd_s[t];
      const float u = tile[(grp * 2 * kGuGroup + kGuGroup + jj) * ld + t] * rstd_s[t];
      out[(size_t)(t0 + t) * a.F + (r0 / (2 * kGuGroup) + grp) * kGuGroup + jj] = from_f32<AT>(silu(g) * u);
    }
  } else {  // EPI_LOGITS
    for (int base = warp * 32; base < total; base += NT) {
      const int i = base + lane;
      const bool valid = i < total;
      const int t = i / nrows, r = i - t * nrows;
      unsigned long long key = 0ull;
      if (valid) {
        const float v = tile[r * ld + t] * rstd_s[t];
        if (a.out_f32) a.out_f32[(size_t)(t0 + t) * a.rows + r0 + r] = v;
        key = argmax_key(v, r0 + r);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
        key = other > key ? other : key;
      }
      if (valid && (r & 15) == 0) atomicMax(a.keys + t0 + t, key);
    }
  }
}

}  // namespace dec
