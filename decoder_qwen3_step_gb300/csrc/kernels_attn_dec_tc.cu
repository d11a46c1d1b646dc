// kernels_attn_dec_tc.cu - decode attention of the serving mode (f16 KV
// cache, two query heads per KV head) on the warp-level tensor cores, with
// the QK-norm, RoPE and cache append of the new token fused in.
//
// o = sum_{j < ctx} softmax_j(q . k_j / sqrt(D)) v_j for the newest token of
// every sequence, query head h reading KV head h / 2 (tinyllm L10.1 "Candle
// model runner ...", section 2.4, at one token per sequence; QK-norm before
// split-half RoPE as octlm "A real model in our own decoder" switches them
// on).  grid (chunk, KV head, sequence), 4 warps; keys are cut into the same
// fixed 64-key chunks as the CUDA-core kernel (the cut depends only on the
// position), one chunk per CTA:
//   * one thread arms an mbarrier and warp 0 issues TMA copies of the chunk's
//     K and V blocks (boxes of 16 rows, 128-byte swizzle) - before the wait on
//     the previous kernel for every chunk but a sequence's last, whose keys
//     all predate the step;
//   * warps 0 and 1 form the group's two queries from the raw q|k|v row of
//     the QKV product (RMSNorm over the head, then RoPE at the token's
//     position); in the sequence's last chunk warps 2 and 3 form the new key
//     (normed and rotated) and value, store them to the cache as f16 and
//     patch the landed tile, value rows past the context zeroed;
//   * warp w folds block w on the tensor cores (fold16), the four warps'
//     states merge in warp order into one record per chunk and head, and the
//     last CTA of a (sequence, KV head) to finish merges the records in chunk
//     order and writes the attention output.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "attn_fold.cuh"
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBlocks = kDecodeChunk / 16;  // 16-key blocks per chunk
constexpr int kChunkCap = (kMaxPositions + kDecodeChunk - 1) / kDecodeChunk;

template <int D>
struct Smem {
  static constexpr int kSlab = KvSlab<D>::kBytes;
  static constexpr int kTile = 2 * kBlocks * kSlab;        // K blocks, then V blocks
  static constexpr int kQ = kTile;                         // f16 [2][D] queries
  static constexpr int kZ = kQ + 2 * D * 2;                // f16 [D] zeros
  static constexpr int kO = (kZ + D * 2 + 15) / 16 * 16;   // float [4][2][D]
  static constexpr int kM = kO + kWarps * 2 * D * 4;       // float [4][2] max, [4][2] sum
  static constexpr int kF = kM + 2 * kWarps * 2 * 4;       // float [2][kChunkCap] merge factors
  static constexpr int kB = kF + 2 * kChunkCap * 4;        // mbarrier, then two flags
  static constexpr int kTotal = kB + 16;
};

// This lane's kDim channels of row `row` of token t's raw q|k|v, after
// RMSNorm over the head (gain `norm`) and split-half RoPE at `pos` when norm
// is given.  Whole warp.
template <int D>
__device__ __forceinline__ void head_row(const AttnDecTcArgs& a, int t, int row, const float* norm, int pos,
                                         float (&v)[D / 32]) {
  constexpr int kDim = D / 32, half = D / 2;
  const int lane = threadIdx.x & 31;
  const int QR = (a.at.dims.H + 2 * a.at.dims.Hkv) * D;
  const float* p = a.raw + (size_t)t * QR + row + lane * kDim;
#pragma unroll
  for (int e = 0; e < kDim; ++e) v[e] = p[e];
  if (norm) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < kDim; ++e) ss = fmaf(v[e], v[e], ss);
    const float rn = 1.0f / sqrtf(warp_sum(ss) / (float)D + a.at.dims.eps);
    float y[kDim];
#pragma unroll
    for (int e = 0; e < kDim; ++e) y[e] = v[e] * rn * norm[lane * kDim + e];
#pragma unroll
    for (int e = 0; e < kDim; ++e) {
      const float yp = __shfl_xor_sync(0xffffffffu, y[e], 16);  // channel j +- D/2
      const int jd = lane * kDim + e, jj = jd < half ? jd : jd - half;
      const float cs = a.rope[((size_t)pos * half + jj) * 2], sn = a.rope[((size_t)pos * half + jj) * 2 + 1];
      v[e] = jd < half ? y[e] * cs - yp * sn : y[e] * cs + yp * sn;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) k_attn_decode_tc(const __grid_constant__ CUtensorMap tm_kv,
                                                             const __grid_constant__ AttnDecTcArgs a) {
  pdl_launch_next();
  using SM = Smem<D>;
  constexpr int kDim = D / 32, kSlab = SM::kSlab;
  const Dims& dm = a.at.dims;
  const int c = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int ctx = a.at.meta.seq_ctx[s], pos = ctx - 1;
  const int nch = (ctx + kDecodeChunk - 1) / kDecodeChunk;
  if (c >= nch) return;
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t* Ks = dsm;
  uint8_t* Vs = dsm + kBlocks * kSlab;
  __half* qs = reinterpret_cast<__half*>(dsm + SM::kQ);
  __half* zrow = reinterpret_cast<__half*>(dsm + SM::kZ);
  float* os = reinterpret_cast<float*>(dsm + SM::kO);
  float* ms = reinterpret_cast<float*>(dsm + SM::kM);
  float* ls = ms + kWarps * 2;
  float* fac = reinterpret_cast<float*>(dsm + SM::kF);
  uint64_t& bar = *reinterpret_cast<uint64_t*>(dsm + SM::kB);
  int& last_flag = *reinterpret_cast<int*>(dsm + SM::kB + 8);
  int& abort_flag = *reinterpret_cast<int*>(dsm + SM::kB + 12);
  const int t = a.at.meta.seq_start[s];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int keys_here = min(kDecodeChunk, ctx - c * kDecodeChunk);
  const int nblk = (keys_here + 15) / 16;

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < D; i += kThreads) zrow[i] = __float2half_rn(0.f);
  __syncthreads();
  // lane = (K or V, block, box): one TMA box of 16 rows each
  auto issue = [&]() {
    constexpr int kB = KvSlab<D>::kBoxes;
    if (lane == 0) mbar_expect_tx(&bar, 2 * kSlab * nblk);
    __syncwarp();
    if (lane < 2 * nblk * kB) {
      const int bx = lane % kB, j = (lane / kB) % nblk, is_v = lane / (kB * nblk);
      const int blk = a.at.meta.tables[(size_t)s * dm.max_blocks + c * kBlocks + j];
      const int row = (((a.at.layer * dm.n_blocks + blk) * 2 + is_v) * dm.Hkv + g) * 16;
      tma_load_2d((is_v ? Vs : Ks) + j * kSlab + bx * KvSlab<D>::kBoxBytes, &tm_kv, bx * KvSlab<D>::kBoxDims, row,
                  &bar);
    }
  };
  // Every key of a chunk before the last was written by an earlier step and
  // the metadata before this step's first kernel, so those copies start
  // before the wait on the previous kernel (the QKV product): they overlap
  // its tail.  The last chunk holds the position this step writes.
  const bool last = c == nch - 1;
  if (warp == 0 && !last) issue();
  pdl_wait_prev();
  if (warp == 0 && last) issue();
  if (warp < 2) {  // the group's two queries: QK-norm, RoPE, f16
    float v[kDim];
    head_row<D>(a, t, (2 * g + warp) * D, a.q_norm, pos, v);
#pragma unroll
    for (int e = 0; e < kDim; ++e) qs[warp * D + lane * kDim + e] = __float2half_rn(v[e]);
  }
  __half hv[kDim];
  if (last && warp >= 2) {  // the new key (QK-norm, RoPE) and value: to the cache as f16
    const int is_v = warp == 3;
    float v[kDim];
    head_row<D>(a, t, (is_v ? dm.H + dm.Hkv + g : dm.H + g) * D, is_v ? nullptr : a.k_norm, pos, v);
    const int blk = a.at.meta.tables[(size_t)s * dm.max_blocks + pos / 16];
    // the pool is the caller's writable slab buffer (AttnArgs carries it read-only for the other kernels)
    __half* dst = const_cast<__half*>(reinterpret_cast<const __half*>(a.at.kv)) +
                  kv_offset(a.at.layer, blk, is_v, g, pos % 16, dm.n_blocks, dm.Hkv, 16, D);
#pragma unroll
    for (int e = 0; e < kDim; ++e) {
      hv[e] = __float2half_rn(v[e]);
      dst[lane * kDim + e] = hv[e];
    }
  }
  const bool ok = mbar_wait(&bar, 0, &abort_flag, a.at.err);
  if (last && warp >= 2 && ok) {
    // the landed tile holds what the cache held at the new position: patch it
    // (value rows past the context become zeros: P V must not meet NaN bits)
    const int kk = pos - c * kDecodeChunk;
    patch_row<D>((warp == 3 ? Vs : Ks) + (kk / 16) * kSlab, kk % 16, hv, warp == 3);
  }
  __syncthreads();
  if (ok)
    fold16<D>(qs, qs + D, zrow, Ks + warp * kSlab, Vs + warp * kSlab, min(16, keys_here - warp * 16), a.at.scale,
              os + warp * 2 * D, ms + warp * 2, ls + warp * 2);
  __syncthreads();
  // the chunk's record per query head: the four warps merged in warp order
  // (after a wait that gave up: an empty record)
  for (int i = threadIdx.x; i < 2 * D; i += kThreads) {
    const int h = i / D, dd = i % D;
    float M = -INFINITY, L = 0.f, O = 0.f;
    if (ok) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ms[w * 2 + h]);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ms[w * 2 + h] == -INFINITY ? 0.f : expf(ms[w * 2 + h] - M);
        L = fmaf(ls[w * 2 + h], f, L);
        O = fmaf(os[(w * 2 + h) * D + dd], f, O);
      }
    }
    float* part = a.at.part + (((size_t)s * dm.H + 2 * g + h) * a.at.nchunk_cap + c) * (D + 2);
    if (dd == 0) {
      part[0] = M;
      part[1] = L;
    }
    part[2 + dd] = O;
  }
  if (!ok && threadIdx.x == 0) {  // let the copies land before shared memory goes away
    const uint64_t t0 = global_ns();
    while (!mbar_try(&bar, 0) && global_ns() - t0 < kWaitLimitNs) {
    }
  }

  // the last CTA of this (sequence, KV head) merges the chunk records in chunk order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_flag = atomicAdd(a.at.counters + s * dm.Hkv + g, 1) == nch - 1;
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  const float* base = a.at.part + ((size_t)s * dm.H + 2 * g) * a.at.nchunk_cap * (D + 2);
  if (warp < 2) {
    const float* ph = base + (size_t)warp * a.at.nchunk_cap * (D + 2);
    float mx = -INFINITY;
    for (int cc = lane; cc < nch; cc += 32) mx = fmaxf(mx, __ldcg(ph + cc * (D + 2)));
    mx = warp_max(mx);
    float sum = 0.f;
    for (int cc = lane; cc < nch; cc += 32) {
      const float f = expf(__ldcg(ph + cc * (D + 2)) - mx);
      fac[warp * kChunkCap + cc] = f;
      sum = fmaf(__ldcg(ph + cc * (D + 2) + 1), f, sum);
    }
    sum = warp_sum(sum);
    if (lane == 0) ms[warp] = sum;
  }
  __syncthreads();
  bf16* out = reinterpret_cast<bf16*>(a.at.ATT);
  for (int i = threadIdx.x; i < 2 * D; i += kThreads) {
    const int h = i / D, dd = i % D;
    const float* ph = base + (size_t)h * a.at.nchunk_cap * (D + 2) + 2 + dd;
    float O = 0.f;
#pragma unroll 4
    for (int cc = 0; cc < nch; ++cc) O = fmaf(__ldcg(ph + cc * (D + 2)), fac[h * kChunkCap + cc], O);
    out[((size_t)t * dm.H + 2 * g + h) * D + dd] = __float2bfloat16_rn(O / ms[h]);
  }
  if (threadIdx.x == 0) a.at.counters[s * dm.Hkv + g] = 0;
}

template <int D>
cudaError_t launch_d(const AttnDecTcArgs& a, const CUtensorMap* tm, int nchunk, cudaStream_t s) {
  static SmemOptIn opt;
  constexpr int smem = Smem<D>::kTotal;
  cudaError_t e = opt.ensure(k_attn_decode_tc<D>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nchunk, a.at.dims.Hkv, a.at.S);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // older chunks' copies overlap the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attn_decode_tc<D>, *tm, a);
}

}  // namespace

bool attn_decode_tc_eligible(const Dims& dm) {
  return dm.H == 2 * dm.Hkv && (dm.D == 32 || dm.D == 64 || dm.D == 128) && dm.B == 16;
}

cudaError_t launch_attn_decode_tc(const AttnDecTcArgs& a, const void* tm_kv, int nchunk, cudaStream_t s) {
  const CUtensorMap* tm = reinterpret_cast<const CUtensorMap*>(tm_kv);
  switch (a.at.dims.D) {
    case 32: return launch_d<32>(a, tm, nchunk, s);
    case 64: return launch_d<64>(a, tm, nchunk, s);
    case 128: return launch_d<128>(a, tm, nchunk, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dec
