// kernels_tc.cu - the weight products of many-token steps on the 5th-generation
// tensor cores (tcgen05 + TMEM, operands staged by TMA), bf16 x bf16 -> fp32.
//
// D[r, t] = sum_k W[r, k] X[t, k]: the weight tile is the M = 128 operand,
// a tile of 128 token rows the N operand, both K-major with the 128-byte
// swizzle; K advances 64 elements (one 128-byte swizzle row) per stage.
// Persistent: one CTA per SM walks the (weight tile, token tile) grid.
//   warp 0      TMA producer: 4-stage shared-memory ring (full/empty mbarriers)
//   warp 1      TMEM owner and MMA issuer (one elected lane); two 128-column
//               fp32 accumulators so the epilogue of one tile overlaps the
//               MMAs of the next
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, staged through
//               shared memory into the same fused epilogues as the CUDA-core
//               products (QKV, residual + next-norm input, SwiGLU, logits)
// Every mbarrier wait is bounded (about a second); on expiry the kernel sets
// the device error word, lets copies and MMAs in flight land, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

constexpr int kTcM = 128, kTcN = 128, kTcK = 64, kTcStages = 4;
constexpr int kTcEpiThreads = 256;  // 8 epilogue warps, two per TMEM lane quarter
constexpr int kTcThreads = 64 + kTcEpiThreads;
constexpr int kTcTileLd = kTcM + 4;  // epilogue tile, token-major [kTcN tokens][kTcTileLd]
constexpr uint32_t kTcStageA = kTcM * kTcK * 2;  // 16 KB
constexpr uint32_t kTcStageB = kTcN * kTcK * 2;  // 16 KB
constexpr uint32_t kTcAccCols = 128;             // fp32 columns per accumulator
struct TcShared {
  float rn[4 * kTcN];  // fused QKV epilogue: head norms [heads per tile][tokens]
  int tpos[kTcN], tblk[kTcN];  // fused QKV epilogue: position and cache block per token
  uint64_t full[kTcStages], empty[kTcStages], tfull[2], tempty[2], mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int consumed;  // stage loads the MMA warp has taken (for the teardown drain)
};

constexpr size_t kTcSmemBytes =
    1024 + (size_t)kTcStages * (kTcStageA + kTcStageB) + (size_t)kTcN * kTcTileLd * 4 + kTcN * 4 + sizeof(TcShared);

template <typename AT, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, GemvArgs a,
              uint32_t* err) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t tc_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kTcStages * kTcStageA;
  float* tile = reinterpret_cast<float*>(sB + kTcStages * kTcStageB);
  float* rstd_s = tile + kTcN * kTcTileLd;
  TcShared* sh = reinterpret_cast<TcShared*>(rstd_s + kTcN);
  volatile int* abort_flag = &sh->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = a.rows / kTcM;
  const int n_tiles = (a.T + kTcN - 1) / kTcN;
  const int n_total = m_tiles * n_tiles;
  const int nk = a.K / kTcK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->tfull[i], 1);
      mbar_init(&sh->tempty[i], kTcEpiThreads);
    }
    mbar_init(&sh->mma_done, 1);
    sh->abort_flag = 0;
    sh->consumed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh->tmem_base)),
                 "r"(2 * kTcAccCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  int issued = 0;  // producer: stage loads issued

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile_i = blockIdx.x; tile_i < n_total; tile_i += gridDim.x) {
        const int mt = tile_i % m_tiles, nt = tile_i / m_tiles;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&sh->empty[stage], phase ^ 1, abort_flag, err)) goto producer_done;
          mbar_expect_tx(&sh->full[stage], kTcStageA + kTcStageB);
          tma_load_2d(sA + stage * kTcStageA, &tmW, kb * kTcK, mt * kTcM, &sh->full[stage]);
          tma_load_2d(sB + stage * kTcStageB, &tmX, kb * kTcK, nt * kTcN, &sh->full[stage]);
          ++issued;
          if (++stage == kTcStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // tail: every stage released by the MMA commits before the CTA may exit
      for (int i = 0; i < kTcStages && !*abort_flag; ++i) {
        if (!mbar_wait(&sh->empty[stage], phase ^ 1, abort_flag, err)) break;
        if (++stage == kTcStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      constexpr uint32_t idesc = idesc_bf16(kTcM, kTcN);
      for (int tile_i = blockIdx.x; tile_i < n_total; tile_i += gridDim.x) {
        if (!mbar_wait(&sh->tempty[acc], acc_phase ^ 1, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * kTcAccCols;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&sh->full[stage], phase, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kTcStageA), b0 = smem_u32(sB + stage * kTcStageB);
#pragma unroll
          for (int k = 0; k < kTcK / 16; ++k)
            tc_mma(d, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc, (kb | k) != 0);
          tc_commit(&sh->empty[stage]);  // the stage is free once these MMAs have read it
          sh->consumed = sh->consumed + 1;
          if (++stage == kTcStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&sh->tfull[acc]);  // the accumulator is complete once every MMA above is
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      tc_commit(&sh->mma_done);
    }
  } else {
    // epilogue warps: TMEM lane quarter (warp % 4), rows 32*(warp%4) .. +31; warps 2..5
    // read columns 0..63 of the accumulator, warps 6..9 columns 64..127
    const int et = threadIdx.x - 64;
    const int quarter = warp & 3, chalf = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile_i = blockIdx.x; tile_i < n_total; tile_i += gridDim.x) {
      const int mt = tile_i % m_tiles, nt = tile_i / m_tiles;
      const int t0 = nt * kTcN, ntok = min(kTcN, a.T - t0);
      epi_bar<kTcEpiThreads>();  // the previous tile's epilogue is done with tile/rstd_s
      {  // 1/rms of this tile's tokens: warp w takes tokens 16w .. 16w+15, 8 at a time
        const int wq = et >> 5;
#pragma unroll 1
        for (int t8 = wq * 16; t8 < wq * 16 + 16; t8 += 8) {
          float r8[8];
          const int n = max(0, min(8, ntok - t8));
          if (a.ssq) {
            row_rstd_n<8>(a.ssq, t0 + t8, n, a.d, a.eps, r8);
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) r8[u] = 1.0f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (lane == u) rstd_s[t8 + u] = r8[u];
        }
      }
      const bool got = mbar_wait(&sh->tfull[acc], acc_phase, abort_flag, err);
      if (epi_any<kTcEpiThreads>(!got)) break;
      tc_fence_after();
#pragma unroll 1
      for (int slab = 0; slab < 2; ++slab) {
        const int col = chalf * 64 + slab * 32;
        uint32_t v[32];
        tc_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + acc * kTcAccCols + col, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) tile[(col + j) * kTcTileLd + row] = __uint_as_float(v[j]);
      }
      tc_fence_before();
      mbar_arrive(&sh->tempty[acc]);
      epi_bar<kTcEpiThreads>();
      if constexpr (EPI == EPI_QKV) {
        epilogue_qkv_tile<__half, kTcEpiThreads>(a, tile, kTcTileLd, mt * kTcM, kTcM, t0, ntok, rstd_s, sh->rn,
                                                 sh->tpos, sh->tblk, et, EpiBar<kTcEpiThreads>{});
      } else {
        epilogue<AT, EPI, kTcEpiThreads>(a, tile, kTcTileLd, mt * kTcM, kTcM, t0, ntok, rstd_s, et);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // let what is in flight land before the memory goes away
    if (threadIdx.x == 0) {
      for (int j = sh->consumed; j < issued; ++j) {
        const uint64_t t0 = global_ns();
        while (!mbar_try(&sh->full[j % kTcStages], (j / kTcStages) & 1) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    if (warp == 1) {
      const uint64_t t0 = global_ns();
      while (!mbar_try(&sh->mma_done, 0) && global_ns() - t0 < kWaitLimitNs) {
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kTcAccCols) : "memory");
  }
}

template <typename AT, int EPI>
static cudaError_t tc_one(const GemvArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX, int num_sms, uint32_t* err,
                          cudaStream_t s) {
  static SmemOptIn opt;
  cudaError_t e = opt.ensure(k_gemm_tc<AT, EPI>, (int)kTcSmemBytes);
  if (e != cudaSuccess) return e;
  const int tiles = (a.rows / kTcM) * ((a.T + kTcN - 1) / kTcN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  k_gemm_tc<AT, EPI><<<grid, kTcThreads, kTcSmemBytes, s>>>(*tmW, *tmX, a, err);
  return cudaGetLastError();
}

bool tc_eligible(const GemvArgs& a) { return a.rows % kTcM == 0 && a.K % kTcK == 0 && a.T > 0 && a.x_row == nullptr; }

cudaError_t launch_gemm_tc(const GemvArgs& a, int epi, const void* tmW, const void* tmX, int num_sms, uint32_t* err,
                           cudaStream_t s) {
  const CUtensorMap* w = reinterpret_cast<const CUtensorMap*>(tmW);
  const CUtensorMap* x = reinterpret_cast<const CUtensorMap*>(tmX);
  switch (epi) {
    case EPI_QKV_RAW: return tc_one<bf16, EPI_QKV_RAW>(a, w, x, num_sms, err, s);
    case EPI_QKV: return tc_one<bf16, EPI_QKV>(a, w, x, num_sms, err, s);
    case EPI_RESID: return tc_one<bf16, EPI_RESID>(a, w, x, num_sms, err, s);
    case EPI_SWIGLU: return tc_one<bf16, EPI_SWIGLU>(a, w, x, num_sms, err, s);
    default: return tc_one<bf16, EPI_LOGITS>(a, w, x, num_sms, err, s);
  }
}

}  // namespace dec
