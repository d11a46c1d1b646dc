// kernels_int4.cu - int4 group-symmetric projection weights: the load-time
// quantizer and the weight-streaming product that dequantizes in registers.
//
// tinyllm L10.1 "Candle model runner (Llama + bigram, int4), Rust KV cache,
// sampler and PCG32", section 2.5 "Int4 weights": per group of g = 32 input
// columns one f16 scale s = f16(max|W| / 7) and codes q = clamp(rint(W / s),
// -8, 7), rint rounding half to even and s the f16 value stored; column 2b in
// the low nibble of byte b, column 2b + 1 in the high nibble, four-bit two's
// complement; the effective weight is q * s.  The quantizer divides in f32,
// as the runner quantizes f32 weights at load; an all-zero group has s = 0
// and codes 0.
//
// Layout of one quantized matrix (rows x K): the codes, rows x K/2 bytes
// (row-major), then the scales, rows x K/32 f16 values.
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace dec {

constexpr int kI4Group = 32;

// One thread per (row, group): 32 weights -> 16 bytes of codes and one scale.
__global__ void k_quant_i4(uint8_t* __restrict__ nib, __half* __restrict__ scl, const float* __restrict__ src,
                           int rows, int K, int mode) {
  const int groups = K / kI4Group;
  const int64_t n = (int64_t)rows * groups;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / groups), g = (int)(i - (int64_t)r * groups);
    int dr = r;  // destination row: gate and up rows interleave in groups of kGuGroup
    if (mode == PACK_GATE) dr = (r / kGuGroup) * 2 * kGuGroup + r % kGuGroup;
    if (mode == PACK_UP) dr = (r / kGuGroup) * 2 * kGuGroup + kGuGroup + r % kGuGroup;
    const float* w = src + (size_t)r * K + (size_t)g * kI4Group;
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < kI4Group; ++e) amax = fmaxf(amax, fabsf(w[e]));
    const __half sh = __float2half_rn(amax / 7.0f);  // f32 division, one rounding to f16
    const float s = __half2float(sh);
    uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < kI4Group; ++e) {
      int q = 0;
      if (s != 0.0f) q = (int)fminf(fmaxf(rintf(w[e] / s), -8.0f), 7.0f);
      words[e >> 3] |= ((uint32_t)q & 0xFu) << (4 * (e & 7));  // column e: nibble e of the 16 bytes
    }
    *reinterpret_cast<uint4*>(nib + (size_t)dr * (K / 2) + (size_t)g * 16) =
        make_uint4(words[0], words[1], words[2], words[3]);
    scl[(size_t)dr * groups + g] = sh;
  }
}

// 16 codes (8 bytes, column order) as floats: the nibble xor 8 is q + 8 in
// [0, 15]; placed in the mantissa of 2^23, the offset comes off exactly
__device__ __forceinline__ void unpack16(uint2 q, float* w) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w[e] = __int_as_float(0x4B000000 | (((q.x >> (4 * e)) & 0xFu) ^ 8u)) - 8388616.0f;
    w[8 + e] = __int_as_float(0x4B000000 | (((q.y >> (4 * e)) & 0xFu) ^ 8u)) - 8388616.0f;
  }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

// ---------------------------------------------------------------------------
// Weight-streaming product on int4 weights, any number of token rows (8 at a
// time).  A CTA owns 16 consecutive rows (contiguous codes and scales), two
// per warp.  Its codes and scales are copied to shared memory asynchronously
// before the wait on the previous kernel: weights do not depend on it, so
// with programmatic dependent launch the copy overlaps that kernel's tail.
// Each code byte comes from HBM once, whatever the number of tokens.  A lane
// takes 16 codes of both rows per step (a warp step covers 512 columns); the
// dot product of each 16-code piece is scaled once by its group's scale.
// ---------------------------------------------------------------------------
template <typename AT, int EPI>
__global__ void __launch_bounds__(kGemvThreads, 3) k_gemv_i4(GemvArgs a) {
  pdl_launch_next();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int K = a.K, KB = K / 2, G = K / kI4Group;
  uint8_t* cs = smem_raw;                                          // [16][K/2] codes
  __half* ss = reinterpret_cast<__half*>(smem_raw + kGemvRows * KB);  // [16][K/32] scales
  AT* xs = reinterpret_cast<AT*>(smem_raw + kGemvRows * KB + kGemvRows * G * 2);  // [kGemvTok][K]
  __shared__ __align__(16) float outs[kGemvTok * kGemvRows];
  __shared__ float rstd_s[kGemvTok];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kGemvRows;
  const uint8_t* Wn = reinterpret_cast<const uint8_t*>(a.W);
  const uint8_t* Ws = Wn + (size_t)a.rows * KB;
  {
    const uint8_t* src = Wn + (size_t)r0 * KB;
    for (int i = threadIdx.x; i < kGemvRows * KB / 16; i += kGemvThreads) cp_async16(cs + 16 * i, src + 16 * i);
    const uint8_t* ssrc = Ws + (size_t)r0 * G * 2;
    for (int i = threadIdx.x; i < kGemvRows * G * 2 / 16; i += kGemvThreads)
      cp_async16(reinterpret_cast<uint8_t*>(ss) + 16 * i, ssrc + 16 * i);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  pdl_wait_prev();
  const AT* X = reinterpret_cast<const AT*>(a.X);
  const uint8_t* na = cs + (warp * 2) * KB;
  const uint8_t* nb = na + KB;
  const __half* sa = ss + (warp * 2) * G;
  const __half* sb = sa + G;

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
    if (t0 == 0) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();

    float acc0[kGemvTok], acc1[kGemvTok];
#pragma unroll
    for (int t = 0; t < kGemvTok; ++t) acc0[t] = acc1[t] = 0.f;
#pragma unroll 2
    for (int k = lane * 16; k < K; k += 512) {
      const uint2 qa = *reinterpret_cast<const uint2*>(na + k / 2);
      const uint2 qb = *reinterpret_cast<const uint2*>(nb + k / 2);
      const float fa = __half2float(sa[k / kI4Group]), fb = __half2float(sb[k / kI4Group]);
      float wa[16], wb[16];
      unpack16(qa, wa);
      unpack16(qb, wb);
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t) {
        if (t < tc) {
          float x[16];
          load8(xs + (size_t)t * K + k, x);
          load8(xs + (size_t)t * K + k + 8, x + 8);
          float da = 0.f, db = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            da = fmaf(wa[e], x[e], da);
            db = fmaf(wb[e], x[e], db);
          }
          acc0[t] = fmaf(fa, da, acc0[t]);
          acc1[t] = fmaf(fb, db, acc1[t]);
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

template <int EPI>
static cudaError_t gemv_i4_one(const GemvArgs& a, cudaStream_t s) {
  static SmemOptIn opt;
  const int smem = (int)((size_t)kGemvRows * (a.K / 2) + (size_t)kGemvRows * (a.K / kI4Group) * 2 +
                         (size_t)kGemvTok * a.K * sizeof(bf16));
  cudaError_t e = opt.ensure(k_gemv_i4<bf16, EPI>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.rows / kGemvRows, 1, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // weight loads overlap the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_i4<bf16, EPI>, a);
}

cudaError_t launch_gemv_i4(const GemvArgs& a, int epi, cudaStream_t s) {
  switch (epi) {
    case EPI_QKV_RAW: return gemv_i4_one<EPI_QKV_RAW>(a, s);
    case EPI_RESID: return gemv_i4_one<EPI_RESID>(a, s);
    case EPI_SWIGLU: return gemv_i4_one<EPI_SWIGLU>(a, s);
    default: return cudaErrorInvalidValue;  // the tied LM head stays bf16
  }
}

cudaError_t launch_quant_i4(void* nib, void* scl, const float* src, int rows, int K, int mode, cudaStream_t s) {
  const int64_t n = (int64_t)rows * (K / kI4Group);
  const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  k_quant_i4<<<grid, 256, 0, s>>>(reinterpret_cast<uint8_t*>(nib), reinterpret_cast<__half*>(scl), src, rows, K,
                                  mode);
  return cudaGetLastError();
}

}  // namespace dec
