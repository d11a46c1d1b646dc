// kernels_attn_tc.cu - prefill attention of the serving mode (f16 KV cache)
// on the warp-level tensor cores.
//
// o_t = sum_{j <= pos(t)} softmax_j(q_t . k_j / sqrt(D)) v_j with query head h
// reading KV head floor(h * Hkv / H) (tinyllm L10.1 "Candle model runner ...",
// section 2.4).  Work tiles are those of the CUDA-core prefill kernel: up to
// 64 / G consecutive new tokens of one sequence and one KV head, the G query
// heads of the group stacked as the tile's 64 rows (row = token * G + head).
// Four warps own 16 rows each.  Keys come in tiles of 64 from the paged cache
// (16-byte asynchronous copies into padded shared rows, double-buffered); keys
// past the last position of the tile are zero-filled.  Per key tile a warp
// forms S = Q K^T (m16n8k16, f16 inputs, fp32 accumulation), applies the causal
// mask and the scale, folds S into an online softmax held in registers, and
// adds P V with P rounded to f16 (the accumulator layout of S is the operand
// layout of P).  Q is rounded to f16 once; the output is divided by the row
// sum and stored in the activation type.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

namespace {

constexpr int kTcRows = 64;   // query-head rows of a work tile
constexpr int kTcKeys = 64;   // keys per tile
constexpr int kTcWarps = 4;   // 16 rows each

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float x, float y) {
  const __half2 h = __floats2half2_rn(x, y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// 16 bytes global -> shared, cached in L2 only; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

template <int D>
struct TcLayout {
  static constexpr int LDH = D + 8;  // halfs per padded shared row (16 bytes of padding: conflict-free ldmatrix)
  static constexpr size_t q_bytes = (size_t)kTcRows * LDH * 2;
  static constexpr size_t kv_bytes = (size_t)kTcKeys * LDH * 2;
  static constexpr size_t total = q_bytes + 4 * kv_bytes;  // Q, then K and V of two stages
};

template <typename AT, int D, int G>
__global__ void __launch_bounds__(kTcWarps * 32, 2) k_attn_prefill_tc(AttnArgs a) {
  pdl_launch_next();
  pdl_wait_prev();
  using L = TcLayout<D>;
  constexpr int LDH = L::LDH, KS = D / 16, NT = kTcKeys / 8, ND = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  __half* Qs = reinterpret_cast<__half*>(smem);
  __half* Kst = reinterpret_cast<__half*>(smem + L::q_bytes);  // stage i: K at 2i, V at 2i+1
  const Dims& dm = a.dims;
  const int* w = a.meta.work + blockIdx.x * 3;
  const int s = w[0], tok0 = w[1], ntok = w[2];
  const int g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p0 = a.meta.tok_pos[tok0];
  const int p_last = p0 + ntok - 1;
  const __half* kv = reinterpret_cast<const __half*>(a.kv);

  // key tile kt of K and V into stage st (16-byte pieces, rows past p_last zero)
  auto load_tile = [&](int kt, int st) {
    __half* Kd = Kst + (size_t)(2 * st) * kTcKeys * LDH;
    __half* Vd = Kd + (size_t)kTcKeys * LDH;
    constexpr int kPieces = D / 8;  // per key row
    for (int i = tid; i < kTcKeys * kPieces; i += kTcWarps * 32) {
      const int kk = i / kPieces, c8 = (i % kPieces) * 8;
      const int j = kt * kTcKeys + kk;
      const bool in = j <= p_last;
      const int blk = in ? table_block(a.meta.tables, s, j / dm.B, dm.max_blocks, dm.n_blocks, a.err) : 0;
      const int slot = in ? j % dm.B : 0;
      const __half* ksrc = kv + kv_offset(a.layer, blk, 0, g, slot, dm.n_blocks, dm.Hkv, dm.B, D) + c8;
      const __half* vsrc = kv + kv_offset(a.layer, blk, 1, g, slot, dm.n_blocks, dm.Hkv, dm.B, D) + c8;
      cp16(smem_u32(Kd + kk * LDH + c8), ksrc, in ? 16u : 0u);
      cp16(smem_u32(Vd + kk * LDH + c8), vsrc, in ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  const int ntiles = p_last / kTcKeys + 1;
  load_tile(0, 0);
  // queries, rounded to f16 once (rows past the tile's tokens repeat its last token)
  for (int i = tid; i < kTcRows * (D / 4); i += kTcWarps * 32) {
    const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
    const int qi = min(r / G, ntok - 1), hh = r % G;
    const float4 v = *reinterpret_cast<const float4*>(a.Q + ((size_t)(tok0 + qi) * dm.H + g * G + hh) * D + c4);
    *reinterpret_cast<uint2*>(Qs + r * LDH + c4) = make_uint2(pack_half2(v.x, v.y), pack_half2(v.z, v.w));
  }
  __syncthreads();
  // this warp's 16 rows as A fragments for every k step
  uint32_t qf[KS][4];
  {
    const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, col = (lane >> 4) * 8;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) ldsm4(smem_u32(Qs + row * LDH + ks * 16 + col), qf[ks]);
  }
  // the two rows of this lane: r0 = warp*16 + lane/4 and r0 + 8; their positions
  const int r0 = warp * 16 + (lane >> 2);
  const int pos0 = p0 + min(r0 / G, ntok - 1), pos1 = p0 + min((r0 + 8) / G, ntok - 1);
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[ND][4];
#pragma unroll
  for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  for (int kt = 0; kt < ntiles; ++kt) {
    const int st = kt & 1;
    if (kt + 1 < ntiles) {
      load_tile(kt + 1, st ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const __half* Ks = Kst + (size_t)(2 * st) * kTcKeys * LDH;
    const __half* Vs = Ks + (size_t)kTcKeys * LDH;
    // S = Q K^T over the 64 keys (8 tiles of 8)
    float sc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b[4];
        const int key = n * 8 + ((lane >> 4) & 1) * 8 + (lane & 7), col = ks * 16 + ((lane >> 3) & 1) * 8;
        ldsm4(smem_u32(Ks + key * LDH + col), b);
        mma_f16(sc[n], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b[0], b[1]);
        mma_f16(sc[n + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b[2], b[3]);
      }
    }
    // causal mask and scale; the rows' running maxima
    const int kbase = kt * kTcKeys + (lane & 3) * 2;
    float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kbase + n * 8 + e;
        sc[n][e] = key <= pos0 ? sc[n][e] * a.scale : -INFINITY;
        sc[n][2 + e] = key <= pos1 ? sc[n][2 + e] * a.scale : -INFINITY;
        tm0 = fmaxf(tm0, sc[n][e]);
        tm1 = fmaxf(tm1, sc[n][2 + e]);
      }
    }
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
      tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, x));
      tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, x));
    }
    const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);  // finite: key 0 is visible to every row
    const float c0 = m0 == -INFINITY ? 0.f : expf(m0 - mn0), c1 = m1 == -INFINITY ? 0.f : expf(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    l0 *= c0;
    l1 *= c1;
#pragma unroll
    for (int n = 0; n < ND; ++n) {
      o[n][0] *= c0;
      o[n][1] *= c0;
      o[n][2] *= c1;
      o[n][3] *= c1;
    }
    // P = exp(S - m) (lane-partial row sums; the quad adds them at the end), then O += P V
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
      float p[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int n = 2 * kk + h;
        p[h][0] = sc[n][0] == -INFINITY ? 0.f : expf(sc[n][0] - m0);
        p[h][1] = sc[n][1] == -INFINITY ? 0.f : expf(sc[n][1] - m0);
        p[h][2] = sc[n][2] == -INFINITY ? 0.f : expf(sc[n][2] - m1);
        p[h][3] = sc[n][3] == -INFINITY ? 0.f : expf(sc[n][3] - m1);
        l0 += p[h][0] + p[h][1];
        l1 += p[h][2] + p[h][3];
      }
      const uint32_t a0 = pack_half2(p[0][0], p[0][1]), a1 = pack_half2(p[0][2], p[0][3]);
      const uint32_t a2 = pack_half2(p[1][0], p[1][1]), a3 = pack_half2(p[1][2], p[1][3]);
#pragma unroll
      for (int n = 0; n < ND; n += 2) {
        uint32_t b[4];
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, col = n * 8 + ((lane >> 4) & 1) * 8;
        ldsm4t(smem_u32(Vs + key * LDH + col), b);
        mma_f16(o[n], a0, a1, a2, a3, b[0], b[1]);
        mma_f16(o[n + 1], a0, a1, a2, a3, b[2], b[3]);
      }
    }
    __syncthreads();  // this stage is refilled by the next iteration's copies
  }
#pragma unroll
  for (int x = 1; x <= 2; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }
  AT* out = reinterpret_cast<AT*>(a.ATT);
  const float i0 = 1.0f / l0, i1 = 1.0f / l1;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = r0 + 8 * half, qi = r / G, hh = r % G;
    if (qi >= ntok) continue;
    AT* dst = out + ((size_t)(tok0 + qi) * dm.H + g * G + hh) * D + (lane & 3) * 2;
    const float inv = half ? i1 : i0;
#pragma unroll
    for (int n = 0; n < ND; ++n) {
      const float x0 = o[n][2 * half] * inv, x1 = o[n][2 * half + 1] * inv;
      if constexpr (sizeof(AT) == 2) {
        *reinterpret_cast<__nv_bfloat162*>(dst + n * 8) = __floats2bfloat162_rn(x0, x1);
      } else {
        dst[n * 8] = from_f32<AT>(x0);
        dst[n * 8 + 1] = from_f32<AT>(x1);
      }
    }
  }
}

template <typename AT, int D, int G>
cudaError_t launch_tc(const AttnArgs& a, int n_work, cudaStream_t s) {
  static SmemOptIn opt;
  constexpr size_t smem = TcLayout<D>::total;
  cudaError_t e = opt.ensure(k_attn_prefill_tc<AT, D, G>, (int)smem);
  if (e != cudaSuccess) return e;
  k_attn_prefill_tc<AT, D, G><<<dim3(n_work, a.dims.Hkv), kTcWarps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool attn_prefill_tc_eligible(const AttnArgs& a) {
  const int D = a.dims.D, G = a.dims.H / a.dims.Hkv;
  return (D == 32 || D == 64 || D == 128) && (G == 1 || G == 2 || G == 4) && a.dims.B == 16 &&
         kTcRows / G == prefill_tile_queries(G);
}

cudaError_t launch_attn_prefill_tc(const AttnArgs& a, int n_work, cudaStream_t s) {
  const int D = a.dims.D, G = a.dims.H / a.dims.Hkv;
#define DEC_TC_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_tc<bf16, DD, GG>(a, n_work, s);
  DEC_TC_CASE(128, 2)
  DEC_TC_CASE(128, 1)
  DEC_TC_CASE(128, 4)
  DEC_TC_CASE(64, 2)
  DEC_TC_CASE(64, 1)
  DEC_TC_CASE(64, 4)
  DEC_TC_CASE(32, 2)
  DEC_TC_CASE(32, 1)
  DEC_TC_CASE(32, 4)
#undef DEC_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dec
