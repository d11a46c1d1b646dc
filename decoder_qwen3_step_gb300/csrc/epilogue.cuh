// epilogue.cuh - the fused epilogues shared by every weight-product kernel
// (CUDA-core streaming, CUDA-core tiled, tcgen05).
#pragma once

#include "common.cuh"
#include "launch.h"

namespace dec {

// ---------------------------------------------------------------------------
// Fused epilogues of the weight products, shared by every product kernel.
// The staged output tile is token-major: tile[t * ld + r] holds y for weight
// row r0 + r and token row t0 + t (r < nrows, t < ntok; nrows a multiple of
// 16, ld a multiple of 4, the tile 16-byte aligned), so a thread's 4
// consecutive rows are one conflict-free 128-bit shared-memory load.
//   QKV_RAW : y * rstd -> raw q|k|v (QK-norm/RoPE/cache write follow)
//   RESID   : x += y ; next GEMM input x * w_next ; 16-feature sum of squares
//   SWIGLU  : silu(rstd * gate) * (rstd * up), gate/up interleaved by 8 rows
//   LOGITS  : rstd * y -> logits ; argmax key per token (atomicMax)
// The RMSNorm before a product is split in two: its gain multiplies the
// product's input where that input is written (the RESID epilogue, the
// embedding), its 1/rms scales the product's output rows here.
// ---------------------------------------------------------------------------
// Store 4 consecutive values of the activation type (8 bytes of bf16 or 16 of fp32).
__device__ __forceinline__ void store4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void store4(bf16* p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float4 rows4(const float* tile, int ld, int r, int t) {
  return *reinterpret_cast<const float4*>(tile + t * ld + r);
}

// Every thread takes 4 consecutive weight rows of one token row: the
// residual, activations and logits move in 128-bit pieces, and the loads of
// U such pieces are issued before any store.
template <typename AT, int EPI, int NT>
__device__ __forceinline__ void epilogue(const GemvArgs& a, const float* tile, int ld, int r0, int nrows, int t0,
                                         int ntok, const float* rstd_s, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  // 4-row groups per token row, padded to a power of two so a flat index
  // splits with a shift and a mask (groups past nrows are skipped)
  const int nq = nrows / 4;
  const int nq_sh = nq > 1 ? 32 - __clz(nq - 1) : 0;
  const int total = ntok << nq_sh;
  if (EPI == EPI_QKV_RAW) {
    for (int i = tid; i < total; i += NT) {
      const int t = i >> nq_sh, r = (i & ((1 << nq_sh) - 1)) * 4;
      if (r >= nrows) continue;
      const float rs = rstd_s[t];
      const float4 y = rows4(tile, ld, r, t);
      store4(a.out_f32 + (size_t)(t0 + t) * a.rows + r0 + r, y.x * rs, y.y * rs, y.z * rs, y.w * rs);
    }
  } else if (EPI == EPI_RESID) {
    AT* XN = reinterpret_cast<AT*>(a.XN);
    const int nch = a.d / kSsqChunk;
    constexpr int U = 4;
    // whole warps; a 16-feature chunk is 4 consecutive lanes, valid or not together
    for (int base = warp * 32; base < total; base += NT * U) {
      float4 xr[U], wr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * NT + lane;
        xr[u] = wr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int t = i >> nq_sh, r = (i & ((1 << nq_sh) - 1)) * 4;
        if (i < total && r < nrows) {
          xr[u] = *reinterpret_cast<const float4*>(a.X_res + (size_t)(t0 + t) * a.d + r0 + r);
          wr[u] = *reinterpret_cast<const float4*>(a.w_next + r0 + r);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * NT + lane;
        const int t = i >> nq_sh, r = (i & ((1 << nq_sh) - 1)) * 4;
        const bool valid = i < total && r < nrows;
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
        if (valid) {
          const float4 y = rows4(tile, ld, r, t);
          x0 = xr[u].x + y.x;
          x1 = xr[u].y + y.y;
          x2 = xr[u].z + y.z;
          x3 = xr[u].w + y.w;
          const size_t off = (size_t)(t0 + t) * a.d + r0 + r;
          store4(a.X_res + off, x0, x1, x2, x3);
          store4(XN + off, x0 * wr[u].x, x1 * wr[u].y, x2 * wr[u].z, x3 * wr[u].w);
        }
        float sq = (x0 * x0 + x1 * x1) + (x2 * x2 + x3 * x3);
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        if (valid && (r & (kSsqChunk - 1)) == 0) a.SSQ_out[(size_t)(t0 + t) * nch + (r0 + r) / kSsqChunk] = sq;
      }
    }
  } else if (EPI == EPI_SWIGLU) {
    AT* out = reinterpret_cast<AT*>(a.act_out);
    const int ng = nrows / 8;  // groups of 4 outputs per token row (gate/up interleave in 8s)
    const int ng_sh = nq_sh - 1;  // padded like nq
    for (int i = tid; i < (ntok << ng_sh); i += NT) {
      const int t = i >> ng_sh, q = i & ((1 << ng_sh) - 1);
      if (q >= ng) continue;
      const int grp = q >> 1, jj = (q & 1) * 4;
      const float rs = rstd_s[t];
      const int rg = grp * 2 * kGuGroup + jj, ru = rg + kGuGroup;
      const float4 g4 = rows4(tile, ld, rg, t), u4 = rows4(tile, ld, ru, t);
      const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = silu(gv[e] * rs) * (uv[e] * rs);
      store4(out + (size_t)(t0 + t) * a.F + (r0 / (2 * kGuGroup) + grp) * kGuGroup + jj, o[0], o[1], o[2], o[3]);
    }
  } else {  // EPI_LOGITS
    for (int base = warp * 32; base < total; base += NT) {
      const int i = base + lane;
      const int t = i >> nq_sh, r = (i & ((1 << nq_sh) - 1)) * 4;
      const bool valid = i < total && r < nrows;
      unsigned long long key = 0ull;
      if (valid) {
        const float rs = rstd_s[t];
        const float4 y = rows4(tile, ld, r, t);
        const float yv[4] = {y.x, y.y, y.z, y.w};
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[e] = yv[e] * rs;
          const unsigned long long k = argmax_key(v[e], r0 + r + e);
          key = k > key ? k : key;
        }
        if (a.out_f32) store4(a.out_f32 + (size_t)(t0 + t) * a.rows + r0 + r, v[0], v[1], v[2], v[3]);
      }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
        key = other > key ? other : key;
      }
      // keys only grow: a local maximum at or below the key already stored (read
      // from L2, possibly stale, so never above the true value) cannot raise it
      if (valid && (r & 15) == 0 && key > __ldcg(a.keys + t0 + t)) atomicMax(a.keys + t0 + t, key);
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
  return table_block(f.meta.tables, f.meta.tok_seq[tt], pos / f.B, f.max_blocks, f.n_blocks, f.err);
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

// qkv_store for 4 consecutive rows j .. j+3 of one head (16 bytes of Q, or
// 4 cache elements).
template <typename KT>
__device__ __forceinline__ void qkv_store4(const QkvFuse& f, int tt, int gh, int j, const float* v, int pos, int blk) {
  if (gh < f.H) {
    store4(f.Q + ((size_t)tt * f.H + gh) * f.D + j, v[0], v[1], v[2], v[3]);
    return;
  }
  const int is_v = gh >= f.H + f.Hkv;
  const int h = gh - f.H - (is_v ? f.Hkv : 0);
  KT* p = reinterpret_cast<KT*>(f.kv) + kv_offset(f.layer, blk, is_v, h, pos % f.B, f.n_blocks, f.Hkv, f.B, f.D) + j;
  if constexpr (sizeof(KT) == 4) {
    store4(reinterpret_cast<float*>(p), v[0], v[1], v[2], v[3]);
  } else {
    __half2 lo = __floats2half2_rn(v[0], v[1]), hi = __floats2half2_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
  }
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
    for (int j = 0; j < D; j += 4) {
      const float4 y = rows4(tile, ld, hh * D + j, t);
      ss = fmaf(y.x * rs, y.x * rs, ss);
      ss = fmaf(y.y * rs, y.y * rs, ss);
      ss = fmaf(y.z * rs, y.z * rs, ss);
      ss = fmaf(y.w * rs, y.w * rs, ss);
    }
    rn[hh * ntok + t] = 1.0f / sqrtf(ss / (float)D + a.eps);
  }
  for (int t = tid; t < ntok; t += NT) {
    const int pos = f.meta.tok_pos[t0 + t];
    tpos[t] = pos;
    tblk[t] = qkv_block(f, t0 + t, pos);
  }
  sync();
  const int half = D / 2, nq = nrows / 4;  // D: a power of two; nrows: whole heads
  const int nq_sh = nq > 1 ? 32 - __clz(nq - 1) : 0, dsh = 31 - __clz(D);
  constexpr int U = 4;  // row groups per thread per pass: their loads in flight together
  for (int base = tid; base < (ntok << nq_sh); base += NT * U) {
    float4 g0[U], g1[U], cs0[U], cs1[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NT;
      const int t = i >> nq_sh, r = (i & ((1 << nq_sh) - 1)) * 4;
      if (i >= (ntok << nq_sh) || r >= nrows) continue;
      const int hh = r >> dsh, j = r & (D - 1);
      const int gh = (r0 >> dsh) + hh;
      if (gh < f.H + f.Hkv) {
        const float* g = gh < f.H ? f.q_norm : f.k_norm;
        const int jj = j < half ? j : j - half, jp = j < half ? j + half : j - half;
        g0[u] = __ldg(reinterpret_cast<const float4*>(g + j));
        g1[u] = __ldg(reinterpret_cast<const float4*>(g + jp));
        cs0[u] = __ldg(reinterpret_cast<const float4*>(f.rope + ((size_t)tpos[t] * half + jj) * 2));
        cs1[u] = __ldg(reinterpret_cast<const float4*>(f.rope + ((size_t)tpos[t] * half + jj) * 2 + 4));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NT;
      const int t = i >> nq_sh, r = (i & ((1 << nq_sh) - 1)) * 4;  // rows r .. r+3 of one head (D is a multiple of 4)
      if (i >= (ntok << nq_sh) || r >= nrows) continue;
      const int hh = r >> dsh, j = r & (D - 1);
      const int gh = (r0 >> dsh) + hh;
      const float rs = rstd_s[t];
      const float4 y4 = rows4(tile, ld, r, t);
      float out[4] = {y4.x * rs, y4.y * rs, y4.z * rs, y4.w * rs};
      if (gh < f.H + f.Hkv) {
        const int rp = j < half ? r + half : r - half;
        const float rn_ = rn[hh * ntok + t];
        const float ga[4] = {g0[u].x, g0[u].y, g0[u].z, g0[u].w}, gb[4] = {g1[u].x, g1[u].y, g1[u].z, g1[u].w};
        const float c4[4] = {cs0[u].x, cs0[u].z, cs1[u].x, cs1[u].z}, s4[4] = {cs0[u].y, cs0[u].w, cs1[u].y, cs1[u].w};
        const float4 p4 = rows4(tile, ld, rp, t);
        const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a_ = out[e] * rn_ * ga[e], b_ = pv[e] * rs * rn_ * gb[e];
          out[e] = j < half ? a_ * c4[e] - b_ * s4[e] : a_ * c4[e] + b_ * s4[e];
        }
      }
      qkv_store4<KT>(f, t0 + t, gh, j, out, tpos[t], tblk[t]);
    }
  }
}

}  // namespace dec
