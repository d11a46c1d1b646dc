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

// One output row (0 <= j < D) of a query or key head after QK-norm and
// split-half RoPE: y and yp are the head's values at channel j and at its
// partner j +- D/2, rn the head's 1/rms.
__device__ __forceinline__ float qk_rope(const QkvFuse& f, int gh, int j, float y, float yp, float rn, int pos) {
  const int half = f.D / 2;
  const float* g = gh < f.H ? f.q_norm : f.k_norm;
  const int jj = j < half ? j : j - half;
  const int jp = j < half ? j + half : j - half;
  const float a_ = y * rn * g[j], b_ = yp * rn * g[jp];
  const float c = f.rope[((size_t)pos * half + jj) * 2], sn = f.rope[((size_t)pos * half + jj) * 2 + 1];
  return j < half ? a_ * c - b_ * sn : a_ * c + b_ * sn;
}

// Cache block holding position `pos` of the sequence of token row tt.
__device__ __forceinline__ int qkv_block(const QkvFuse& f, int tt, int pos) {
  return f.meta.tables[(size_t)f.meta.tok_seq[tt] * f.max_blocks + pos / f.B];
}

// Write output row j of head gh for absolute token row tt at position pos
// (cache block blk): queries to Q (fp32), keys and values to their slot (KT).
template <typename KT>
__device__ __forceinline__ void qkv_store(const QkvFuse& f, int tt, int gh, int j, float v, int pos, int blk) {
  if (gh < f.H) {
    f.Q[((size_t)tt * f.H + gh) * f.D + j] = v;
    return;
  }
  const int is_v = gh >= f.H + f.Hkv;
  const int h = gh - f.H - (is_v ? f.Hkv : 0);
  reinterpret_cast<KT*>(f.kv)[kv_offset(f.layer, blk, is_v, h, pos % f.B, f.n_blocks, f.Hkv, f.B, f.D) + j] =
      from_f32<KT>(v);
}

// Fused QKV epilogue over a tile of whole heads: y = acc * rstd; per query or
// key head RMSNorm over its D rows with the shared gain, then split-half RoPE
// at the token's position; queries to Q, keys and values into the cache.
// `rn` is scratch for [nrows / D][ntok] head norms; `sync` orders the phases.
template <typename KT, int NT, typename Sync>
__device__ __forceinline__ void epilogue_qkv_tile(const GemvArgs& a, const float* tile, int ld, int r0, int nrows,
                                                  int t0, int ntok, const float* rstd_s, float* rn, int* tpos,
                                                  int* tblk, int tid, Sync sync) {
  const QkvFuse& f = a.qf;
  const int D = f.D, heads = nrows / D;
  for (int i = tid; i < ntok * heads; i += NT) {
    const int t = i % ntok, hh = i / ntok;
    const float rs = rstd_s[t];
    float ss = 0.f;
    for (int j = 0; j < D; ++j) {
      const float y = tile[(hh * D + j) * ld + t] * rs;
      ss = fmaf(y, y, ss);
    }
    rn[hh * ntok + t] = 1.0f / sqrtf(ss / (float)D + a.eps);
  }
  for (int t = tid; t < ntok; t += NT) {
    const int pos = f.meta.tok_pos[t0 + t];
    tpos[t] = pos;
    tblk[t] = qkv_block(f, t0 + t, pos);
  }
  sync();
  const int half = D / 2;
  for (int i = tid; i < ntok * nrows; i += NT) {
    const int t = i / nrows, r = i - t * nrows;
    const int hh = r / D, j = r - hh * D;
    const int gh = (r0 + hh * D) / D;
    const float y = tile[r * ld + t] * rstd_s[t];
    float out = y;
    if (gh < f.H + f.Hkv) {
      const int rp = j < half ? r + half : r - half;
      out = qk_rope(f, gh, j, y, tile[rp * ld + t] * rstd_s[t], rn[hh * ntok + t], tpos[t]);
    }
    qkv_store<KT>(f, t0 + t, gh, j, out, tpos[t], tblk[t]);
  }
}

}  // namespace dec
