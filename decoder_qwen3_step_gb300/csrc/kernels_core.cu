// kernels_core.cu - embedding, weight-streaming products with fused epilogues,
// QK-norm + RoPE + KV-cache write, argmax finalisation, weight packing.
//
// The step these kernels implement: tinyllm L10.1 "Candle model runner ...",
// section 2.4 "The Llama forward, one step" (RMSNorm, y = x W^T, the residual
// adds, SwiGLU, final norm and the tied LM head), with the Qwen3 switches of
// octlm "A real model in our own decoder" (rectangular q/o, QK-norm before
// RoPE, split-half RoPE).
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace dec {

// ---------------------------------------------------------------------------
// Embedding: x[t] = E[id_t] (an exact copy; bf16 rows widen exactly), the
// first layer's GEMM input x * w_attn, and the 16-feature sum-of-squares
// partials from which the QKV product forms 1/rms.  Also clears the argmax
// keys of this step's logits rows.
// ---------------------------------------------------------------------------
template <typename WT, typename AT>
__global__ void __launch_bounds__(256) k_embed(EmbedArgs a) {
  pdl_launch_next();
  pdl_wait_prev();
  const int t = blockIdx.x;
  int id = a.ids[t];
  if (id < 0 || id >= a.vocab) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrBadId);
    id = 0;
  }
  const WT* row = reinterpret_cast<const WT*>(a.E) + (size_t)id * a.d;
  AT* xn = reinterpret_cast<AT*>(a.XN) + (size_t)t * a.d;
  const int nch = a.d / kSsqChunk;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) {  // d is a multiple of 32: whole warps
    const float x = to_f32(row[c]);
    a.X[(size_t)t * a.d + c] = x;
    xn[c] = from_f32<AT>(x * a.w0[c]);
    const float s = half_warp_sum(x * x);
    if ((c & (kSsqChunk - 1)) == 0) a.SSQ[(size_t)t * nch + c / kSsqChunk] = s;
  }
  if (threadIdx.x == 0 && t < a.R) a.keys[t] = 0ull;
}

// ---------------------------------------------------------------------------
// Weight-streaming product for few tokens (decode).  A CTA owns 16
// consecutive weight rows, two per warp; lanes split K in 8-element pieces
// (128-bit loads of bf16, two of fp32), so each weight byte comes from HBM
// once and every token row staged in shared memory is read once per pair of
// rows.  Token rows go 8 at a time.
// ---------------------------------------------------------------------------
constexpr int kGemvMaxT = kGemvMaxTokens;  // above this the tiled kernel runs

template <typename WT, typename AT, int EPI>
__global__ void __launch_bounds__(kGemvThreads) k_gemv(GemvArgs a) {
  pdl_launch_next();
  pdl_wait_prev();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AT* xs = reinterpret_cast<AT*>(smem_raw);  // [kGemvTok][K]
  __shared__ __align__(16) float outs[kGemvTok * kGemvRows];  // token-major [token][row]
  __shared__ float rstd_s[kGemvTok];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kGemvRows;
  const int K = a.K;
  const WT* W = reinterpret_cast<const WT*>(a.W);
  const AT* X = reinterpret_cast<const AT*>(a.X);
  const WT* w0 = W + (size_t)(r0 + warp * 2) * K;
  const WT* w1 = w0 + K;

  for (int t0 = 0; t0 < a.T; t0 += kGemvTok) {
    const int tc = min(kGemvTok, a.T - t0);
    constexpr int kPer16 = 16 / sizeof(AT);
    const int pieces = K / kPer16;
    for (int i = threadIdx.x; i < tc * pieces; i += kGemvThreads) {
      const int t = i / pieces, p = i - t * pieces;
      const int src = a.x_row ? a.x_row[t0 + t] : t0 + t;
      reinterpret_cast<uint4*>(xs + (size_t)t * K)[p] = reinterpret_cast<const uint4*>(X + (size_t)src * K)[p];
    }
    if (warp < tc) {
      float r = 1.0f;
      if (a.ssq) r = row_rstd(a.ssq, a.x_row ? a.x_row[t0 + warp] : t0 + warp, a.d, a.eps);
      if (lane == 0) rstd_s[warp] = r;
    }
    __syncthreads();

    float acc0[kGemvTok], acc1[kGemvTok];
#pragma unroll
    for (int t = 0; t < kGemvTok; ++t) acc0[t] = acc1[t] = 0.f;
#pragma unroll 4
    for (int k = lane * 8; k < K; k += 256) {
      float wa[8], wb[8];
      load8(w0 + k, wa);
      load8(w1 + k, wb);
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t) {
        if (t < tc) {
          float x8[8];
          load8(xs + (size_t)t * K + k, x8);
          float s0 = acc0[t], s1 = acc1[t];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            s0 = fmaf(wa[e], x8[e], s0);
            s1 = fmaf(wb[e], x8[e], s1);
          }
          acc0[t] = s0;
          acc1[t] = s1;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kGemvTok; ++t) {
      const float v0 = warp_sum(acc0[t]);
      const float v1 = warp_sum(acc1[t]);
      if (lane == t) {
        outs[t * kGemvRows + warp * 2] = v0;
        outs[t * kGemvRows + warp * 2 + 1] = v1;
      }
    }
    __syncthreads();
    epilogue<AT, EPI, kGemvThreads>(a, outs, kGemvRows, r0, kGemvRows, t0, tc, rstd_s, threadIdx.x);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Tiled product for many tokens (prefill), true fp32 FFMA (no TF32): a CTA
// computes 128 tokens x 128 weight rows, K in steps of 16 through double-
// buffered shared memory; each thread owns an 8x8 register tile.  The output
// tile is staged through shared memory into the same fused epilogue.
// ---------------------------------------------------------------------------
constexpr int kTM = 128, kTN = 128, kTK = 16, kTThreads = 256;
constexpr int kTLd = kTM + 4;

template <typename WT, typename AT, int EPI>
__global__ void __launch_bounds__(kTThreads) k_gemm_tiled(GemvArgs a) {
  pdl_launch_next();
  pdl_wait_prev();
  extern __shared__ __align__(16) float tsm[];
  float* As = tsm;                      // [2][kTK][kTLd]   tokens
  float* Bs = tsm + 2 * kTK * kTLd;     // [2][kTK][kTLd]   weight rows
  float* tile = tsm;                    // epilogue, token-major [kTM][kTN + 4], aliases As/Bs
  __shared__ float rstd_s[kTM];
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int warp = tid >> 5, lane = tid & 31;
  const int K = a.K;
  const WT* W = reinterpret_cast<const WT*>(a.W);
  const AT* X = reinterpret_cast<const AT*>(a.X);
  const int lrow = tid >> 1, lk = (tid & 1) * 8;
  const int tok = m0 + lrow, feat = n0 + lrow;
  const bool va = tok < a.T, vw = feat < a.rows;
  const AT* xa = X + (size_t)(va ? (a.x_row ? a.x_row[tok] : tok) : 0) * K + lk;
  const WT* wr = W + (size_t)(vw ? feat : 0) * K + lk;

  for (int t = warp; t < kTM; t += kTThreads / 32) {
    float r = 1.0f;
    if (a.ssq && m0 + t < a.T) r = row_rstd(a.ssq, a.x_row ? a.x_row[m0 + t] : m0 + t, a.d, a.eps);
    if (lane == 0) rstd_s[t] = r;
  }

  float ra[8], rw[8];
  auto gload = [&](int k0) {
    if (va) load8(xa + k0, ra); else for (int e = 0; e < 8; ++e) ra[e] = 0.f;
    if (vw) load8(wr + k0, rw); else for (int e = 0; e < 8; ++e) rw[e] = 0.f;
  };
  auto sstore = [&](int buf) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      As[(buf * kTK + lk + e) * kTLd + lrow] = ra[e];
      Bs[(buf * kTK + lk + e) * kTLd + lrow] = rw[e];
    }
  };
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  gload(0);
  sstore(0);
  __syncthreads();
  for (int k0 = 0; k0 < K; k0 += kTK) {
    const int buf = (k0 / kTK) & 1;
    const bool more = k0 + kTK < K;
    if (more) gload(k0 + kTK);
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      const float* ar = As + (buf * kTK + kk) * kTLd;
      const float* br = Bs + (buf * kTK + kk) * kTLd;
      const float4 a0 = *reinterpret_cast<const float4*>(ar + ty * 4);
      const float4 a1 = *reinterpret_cast<const float4*>(ar + 64 + ty * 4);
      const float4 b0 = *reinterpret_cast<const float4*>(br + tx * 4);
      const float4 b1 = *reinterpret_cast<const float4*>(br + 64 + tx * 4);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (more) sstore(buf ^ 1);
    __syncthreads();
  }
  // stage the tile token-major for the epilogue: 4 consecutive rows per 128-bit store
  constexpr int kLd = kTN + 4;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = (i < 4 ? 0 : 64) + ty * 4 + (i & 3);
    *reinterpret_cast<float4*>(tile + t * kLd + tx * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4*>(tile + t * kLd + 64 + tx * 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
  __syncthreads();
  epilogue<AT, EPI, kTThreads>(a, tile, kLd, n0, min(kTN, a.rows - n0), m0, min(kTM, a.T - m0), rstd_s,
                               threadIdx.x);
}

// ---------------------------------------------------------------------------
// QK-norm + split-half RoPE + KV-cache write.  One warp per head of one token:
// query and key heads get RMSNorm over head_dim with their shared gain, then
// channel j rotates with j + D/2 by the angle of the token's absolute
// position (cos/sin from the table built in double precision); queries go to
// Q, keys and values to slot pos % B of block table[pos / B] (tinyllm L10.1
// section 2.4, section 3 "Where a key lands").
// ---------------------------------------------------------------------------
template <typename KT>
__global__ void k_qkv_post(QkvPostArgs a) {
  pdl_launch_next();
  pdl_wait_prev();
  extern __shared__ float buf[];  // [warps][D]
  const Dims& dm = a.dims;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = dm.D, half = D / 2;
  const int nq = dm.H, nk = dm.Hkv;
  const int width = (nq + 2 * nk) * D;
  const float* raw = a.raw + (size_t)t * width + (size_t)warp * D;
  const int pos = a.meta.tok_pos[t];
  const int seq = a.meta.tok_seq[t];
  const int blk = table_block(a.meta.tables, seq, pos / dm.B, dm.max_blocks, dm.n_blocks, a.err);
  const int slot = pos % dm.B;
  KT* kv = reinterpret_cast<KT*>(a.kv);
  float* mine = buf + warp * D;

  if (warp < nq + nk) {
    const float* g = warp < nq ? a.q_norm : a.k_norm;
    float ss = 0.f;
    for (int j = lane; j < D; j += 32) ss += raw[j] * raw[j];
    ss = warp_sum(ss);
    const float r = 1.0f / sqrtf(ss / (float)D + dm.eps);
    for (int j = lane; j < D; j += 32) mine[j] = raw[j] * r * g[j];
    __syncwarp();
    const float* cs = a.rope + (size_t)pos * half * 2;
    for (int j = lane; j < D; j += 32) {
      const int jj = j < half ? j : j - half;
      const float c = cs[2 * jj], s = cs[2 * jj + 1];
      const float y = j < half ? mine[j] * c - mine[j + half] * s : mine[j] * c + mine[j - half] * s;
      if (warp < nq) {
        a.Q[((size_t)t * nq + warp) * D + j] = y;
      } else {
        kv[kv_offset(a.layer, blk, 0, warp - nq, slot, dm.n_blocks, nk, dm.B, D) + j] = from_f32<KT>(y);
      }
    }
  } else {
    const int h = warp - nq - nk;
    for (int j = lane; j < D; j += 32)
      kv[kv_offset(a.layer, blk, 1, h, slot, dm.n_blocks, nk, dm.B, D) + j] = from_f32<KT>(raw[j]);
  }
}

__global__ void k_argmax_finalize(const unsigned long long* keys, int32_t* ids, int R) {
  pdl_launch_next();
  pdl_wait_prev();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < R) ids[r] = (int32_t)(0xFFFFFFFFu - (uint32_t)(keys[r] & 0xFFFFFFFFull));
}

template <typename WT>
__global__ void k_pack(WT* dst, const float* src, int rows, int cols, int mode) {
  const int64_t n = (int64_t)rows * cols;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / cols), c = (int)(i % cols);
    int dr = r;
    if (mode == PACK_GATE) dr = (r / kGuGroup) * 2 * kGuGroup + r % kGuGroup;
    if (mode == PACK_UP) dr = (r / kGuGroup) * 2 * kGuGroup + kGuGroup + r % kGuGroup;
    dst[(int64_t)dr * cols + c] = from_f32<WT>(src[i]);
  }
}

__global__ void k_f32_to_f16(const float* in, __half* out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = from_f32<__half>(in[i]);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_embed(const EmbedArgs& a, bool wbf16, cudaStream_t s) {
  if (wbf16)
    k_embed<bf16, bf16><<<a.T, 256, 0, s>>>(a);
  else
    k_embed<float, float><<<a.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename WT, typename AT, int EPI>
static cudaError_t gemv_one(const GemvArgs& a, cudaStream_t s) {
  if (a.T <= kGemvMaxT) {
    static SmemOptIn opt;
    const int smem = (int)((size_t)kGemvTok * a.K * sizeof(AT));
    cudaError_t e = opt.ensure(k_gemv<WT, AT, EPI>, smem);
    if (e != cudaSuccess) return e;
    k_gemv<WT, AT, EPI><<<a.rows / kGemvRows, kGemvThreads, smem, s>>>(a);
    return cudaGetLastError();
  }
  static SmemOptIn opt_t;
  const int smem = kTM * (kTN + 4) * (int)sizeof(float);
  cudaError_t e = opt_t.ensure(k_gemm_tiled<WT, AT, EPI>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.rows + kTN - 1) / kTN, (a.T + kTM - 1) / kTM);
  k_gemm_tiled<WT, AT, EPI><<<grid, kTThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gemv(const GemvArgs& a, int epi, bool wbf16, cudaStream_t s) {
  if (wbf16) {
    switch (epi) {
      case EPI_QKV_RAW: return gemv_one<bf16, bf16, EPI_QKV_RAW>(a, s);
      case EPI_RESID: return gemv_one<bf16, bf16, EPI_RESID>(a, s);
      case EPI_SWIGLU: return gemv_one<bf16, bf16, EPI_SWIGLU>(a, s);
      default: return gemv_one<bf16, bf16, EPI_LOGITS>(a, s);
    }
  }
  switch (epi) {
    case EPI_QKV_RAW: return gemv_one<float, float, EPI_QKV_RAW>(a, s);
    case EPI_RESID: return gemv_one<float, float, EPI_RESID>(a, s);
    case EPI_SWIGLU: return gemv_one<float, float, EPI_SWIGLU>(a, s);
    default: return gemv_one<float, float, EPI_LOGITS>(a, s);
  }
}

cudaError_t launch_qkv_post(const QkvPostArgs& a, int T, bool wbf16, cudaStream_t s) {
  const int warps = a.dims.H + 2 * a.dims.Hkv;
  const size_t smem = (size_t)warps * a.dims.D * sizeof(float);
  if (wbf16)
    k_qkv_post<__half><<<T, warps * 32, smem, s>>>(a);
  else
    k_qkv_post<float><<<T, warps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_argmax_finalize(const unsigned long long* keys, int32_t* ids, int R, cudaStream_t s) {
  k_argmax_finalize<<<(R + 255) / 256, 256, 0, s>>>(keys, ids, R);
  return cudaGetLastError();
}

cudaError_t launch_pack(void* dst, const float* src, int rows, int cols, int mode, bool wbf16, cudaStream_t s) {
  const int64_t n = (int64_t)rows * cols;
  const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  if (wbf16)
    k_pack<bf16><<<grid, 256, 0, s>>>(reinterpret_cast<bf16*>(dst), src, rows, cols, mode);
  else
    k_pack<float><<<grid, 256, 0, s>>>(reinterpret_cast<float*>(dst), src, rows, cols, mode);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_f16(const float* in, uint16_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  k_f32_to_f16<<<grid, 256, 0, s>>>(in, reinterpret_cast<__half*>(out), n);
  return cudaGetLastError();
}

}  // namespace dec
