// common.cuh - device-side layouts and helpers shared by the decoder kernels.
//
// Data layout in HBM (all row-major, 256-byte aligned sub-buffers):
//   X    fp32 [T, d]           residual stream
//   XN   act  [T, d]           x * (gain of the next RMSNorm), the GEMM input;
//                               the RMSNorm's 1/rms is applied as a row scale
//                               in the consuming GEMM's epilogue
//   SSQ  fp32 [T, d/16]        sum of x^2 over each 16-feature chunk of x
//   Q    fp32 [T, H, D]        queries after QK-norm and RoPE
//   ATT  act  [T, H*D]         attention output (input of the O projection)
//   ACT  act  [T, F]           silu(gate) * up (input of the down projection)
// act is fp32 in the parity mode and bf16 in the serving mode.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dec {

constexpr int kSsqChunk = 16;    // features per sum-of-squares partial
constexpr int kGuGroup = 8;      // gate/up rows interleave in groups of 8
constexpr int kDecodeChunk = 64;  // keys per split-K work item of decode attention (4 blocks of 16)

// Device error word bits (mirrors DEC_DEV_* in include/dec.h).
constexpr uint32_t kErrBadId = 1u;
constexpr uint32_t kErrTimeout = 2u;
constexpr uint32_t kErrCapacity = 4u;  // a kernel's fixed-size list overflowed (the host sizes grids to avoid it)
constexpr uint32_t kErrBounds = 8u;    // DEC_DEBUG builds: a block-table column or pool block id out of range
constexpr int kMaxPositions = 40960;    // the longest context a model may be built for (Qwen3's limit)

using bf16 = __nv_bfloat16;

// Shape of the decoder as the kernels see it.
struct Dims {
  int vocab, d, n_layers, H, Hkv, D, F;
  int B;        // block_tokens
  int n_blocks; // pool blocks
  int max_blocks; // block-table row stride in the metadata
  float eps;
};

// Per-step metadata in device memory (filled by one host->device copy).
struct StepMeta {
  const int32_t* ids;       // [T]
  const int32_t* tok_pos;   // [T] absolute position
  const int32_t* tok_seq;   // [T] sequence index
  const int32_t* seq_start; // [S+1]
  const int32_t* seq_ctx;   // [S] last position + 1
  const int32_t* row_tok;   // [R] token index of every logits row
  const int32_t* tables;    // [S, max_blocks]
  const int32_t* work;      // prefill attention tiles: [n_work, 3] = (seq, first token, n tokens)
};

// ---- programmatic dependent launch ------------------------------------------
// Let the next kernel of the stream begin launching (it still waits for this
// kernel's completion before it reads anything this kernel wrote).
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Wait until the previous kernel of the stream has completed and its writes
// are visible; a no-op for a kernel launched without programmatic serialisation.
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- element loads as fp32 ------------------------------------------------
__device__ __forceinline__ void load8(const float* p, float* v) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16* p, float* v) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is exact: the bits go to the top half
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load8(const __half* p, float* v) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }
// f32 -> f16 round to nearest even with subnormals and overflow to inf: the
// conversion the f16 KV store uses.
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// ---- reductions --------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Sum over the 16 lanes of a half-warp (xor butterfly; every lane gets the
// same bits because addition is commutative).  This is THE order in which a
// 16-feature chunk's sum of squares is formed, by every producer kernel.
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 1 / sqrt(mean(x^2) + eps) of token row t from its chunk partials, summed in
// one fixed order (lane-strided, then a warp butterfly).  Whole warp calls it.
__device__ __forceinline__ float row_rstd(const float* ssq, int t, int d, float eps) {
  const int nch = d / kSsqChunk;
  const float* p = ssq + (size_t)t * nch;
  float s = 0.f;
  for (int c = threadIdx.x & 31; c < nch; c += 32) s += p[c];
  s = warp_sum(s);
  return 1.0f / sqrtf(s / (float)d + eps);
}

// row_rstd for up to U consecutive token rows t0 .. t0+n-1 at once: every
// partial a lane adds is loaded before the first add (one round trip for
// d <= 2048), and each lane adds its partials in the same lane-strided order
// as row_rstd, so the result is the same.  Whole warp.
template <int U>
__device__ __forceinline__ void row_rstd_n(const float* ssq, int t0, int n, int d, float eps, float* out) {
  constexpr int kK = 4;  // partials per lane per pass
  const int nch = d / kSsqChunk, lane = threadIdx.x & 31;
  float s[U];
#pragma unroll
  for (int u = 0; u < U; ++u) s[u] = 0.f;
  for (int c0 = 0; c0 < nch; c0 += 32 * kK) {
    float v[U][kK];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < kK; ++k) {
        const int c = c0 + lane + 32 * k;
        v[u][k] = (u < n && c < nch) ? ssq[(size_t)(t0 + u) * nch + c] : 0.f;
      }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < kK; ++k) s[u] += v[u][k];
  }
#pragma unroll
  for (int u = 0; u < U; ++u) out[u] = 1.0f / sqrtf(warp_sum(s[u]) / (float)d + eps);
}

// Order-preserving 64-bit key of (logit, id): larger logit wins, then lower id.
__device__ __forceinline__ unsigned long long argmax_key(float v, int id) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

// silu(z) = z / (1 + e^-z) with the fast exponential and division (relative
// error about 1e-7); below -80 the value is below 1e-33 and is returned as 0.
__device__ __forceinline__ float silu(float z) { return z < -80.0f ? 0.0f : __fdividef(z, 1.0f + __expf(-z)); }

// Element offset of (layer, block, is_v, kv head, slot) in the KV slab buffer.
__host__ __device__ __forceinline__ int64_t kv_offset(int layer, int block, int is_v, int kv_head, int slot,
                                                      int n_blocks, int Hkv, int B, int D) {
  int64_t slab = ((int64_t)layer * n_blocks + block) * 2 + is_v;
  return slab * (int64_t)Hkv * B * D + ((int64_t)kv_head * B + slot) * D;
}

// Pool block id in column `col` of sequence s's block-table row (row stride
// max_blocks).  The host validates every table before a step; a DEC_DEBUG
// build checks again on the device: a column or id out of range sets
// kErrBounds in *err and yields block 0, so the access stays inside the pool
// (the step's results are then invalid, and the error word says so).
__device__ __forceinline__ int table_block(const int32_t* tables, int s, int col, int max_blocks, int n_blocks,
                                           uint32_t* err) {
#ifdef DEC_DEBUG
  if ((unsigned)col >= (unsigned)max_blocks) {
    atomicOr(err, kErrBounds);
    return 0;
  }
  const int blk = __ldg(tables + (size_t)s * max_blocks + col);
  if ((unsigned)blk >= (unsigned)n_blocks) {
    atomicOr(err, kErrBounds);
    return 0;
  }
  return blk;
#else
  (void)n_blocks;
  (void)err;
  return __ldg(tables + (size_t)s * max_blocks + col);
#endif
}

}  // namespace dec
