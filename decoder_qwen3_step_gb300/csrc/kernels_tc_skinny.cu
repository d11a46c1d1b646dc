// kernels_tc_skinny.cu - weight products of decode steps (at most 32 token
// rows) on the tcgen05 tensor cores.
//
// D[r, t] = sum_k W[r, k] X[t, k] with the 128-row weight tile as the M
// operand and the (up to) 32 token rows as N = 32.  A step of 1..32 tokens
// only streams weights, so the grid is made wide by splitting K: the KS CTAs
// of one weight tile form a thread-block cluster, each multiplies its K range
// into its own TMEM, copies the 128 x 32 partial tile to shared memory, and
// after a cluster barrier CTA z sums rows [16z, 16z + 16) over the cluster's
// tiles in rank order through distributed shared memory (deterministic) and
// runs the fused epilogue on them.
//
// Launched with programmatic dependent launch: the TMA producer issues its
// first weight tiles before griddepcontrol.wait, so the weight stream of this
// product overlaps the tail of the previous kernel; activations, norms and
// the residual are touched only after the wait.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

constexpr int kSkM = 128, kSkN = 32, kSkK = 64, kSkStages = 4;
constexpr int kSkThreads = 192;
constexpr int kSkLd = kSkM + 4;     // partial tile, token-major [kSkN tokens][kSkLd]
constexpr int kSkRedLd = 64 + 4;    // reduced rows of one CTA (at most 64), token-major
constexpr uint32_t kSkStageA = kSkM * kSkK * 2;  // 16 KB
constexpr uint32_t kSkStageB = kSkN * kSkK * 2;  // 4 KB
constexpr uint32_t kSkCols = 32;

struct SkShared {
  float psq[4][kSkN];  // fused QKV: partial sums of squares [head in tile][token]
  float rn[4][kSkN];   // fused QKV: 1/rms per [head in tile][token]
  int tpos[kSkN], tblk[kSkN];
  uint64_t full[kSkStages], empty[kSkStages], tfull, mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int consumed;
};

constexpr size_t kSkSmemBytes = 1024 + (size_t)kSkStages * (kSkStageA + kSkStageB) + (size_t)kSkN * kSkLd * 4 +
                                (size_t)kSkN * kSkRedLd * 4 + kSkN * 4 + sizeof(SkShared);

__device__ __forceinline__ float4 dsmem_ld4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Split-K reduction of this CTA's rows [r_lo, r_lo + rows_per) over the KS
// partial tiles of the cluster (token-major, kSkLd apart) into red (kSkRedLd
// apart): 4 consecutive rows of one token per 16-byte load, 16 / KS such
// groups per thread and pass, every remote load of a pass issued before the
// first sum; each sum runs over the ranks in order.
template <int KS>
__device__ __forceinline__ void sk_reduce(const float* tile, float* red, int r_lo, int rows_per, int et) {
  constexpr int kG = 16 / KS;
  const int g4 = rows_per / 4, n = g4 * kSkN;
  for (int i0 = et; i0 < n; i0 += 128 * kG) {
    float4 v[kG][KS];
#pragma unroll
    for (int u = 0; u < kG; ++u) {
      const int i = i0 + u * 128, t = i / g4, rr = (i - t * g4) * 4;
      const uint32_t loc = smem_u32(tile + t * kSkLd + r_lo + rr);
#pragma unroll
      for (int q = 0; q < KS; ++q) {
        uint32_t ra;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(loc), "r"(q));
        v[u][q] = i < n ? dsmem_ld4(ra) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kG; ++u) {
      const int i = i0 + u * 128, t = i / g4, rr = (i - t * g4) * 4;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < KS; ++q) {
        sum.x += v[u][q].x;
        sum.y += v[u][q].y;
        sum.z += v[u][q].z;
        sum.w += v[u][q].w;
      }
      if (i < n) *reinterpret_cast<float4*>(red + t * kSkRedLd + rr) = sum;
    }
  }
}

template <typename AT, int EPI>
__global__ void __launch_bounds__(kSkThreads, 1)
    k_gemm_tc_skinny(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, GemvArgs a,
                     int ks, uint32_t* err) {
  extern __shared__ uint8_t sk_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sk_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kSkStages * kSkStageA;
  float* tile = reinterpret_cast<float*>(sB + kSkStages * kSkStageB);  // this CTA's partial, token-major
  float* red = tile + kSkN * kSkLd;                                     // reduced rows, token-major
  float* rstd_s = red + kSkN * kSkRedLd;
  SkShared* sh = reinterpret_cast<SkShared*>(rstd_s + kSkN);
  volatile int* abort_flag = &sh->abort_flag;

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int z = (int)cluster_rank();
  const int mt = blockIdx.x / ks;
  const int nkb = a.K / kSkK / ks;  // K blocks of this CTA
  const int kb0 = z * nkb;
  const int ntok = a.T;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSkStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    mbar_init(&sh->tfull, 1);
    mbar_init(&sh->mma_done, 1);
    sh->abort_flag = 0;
    sh->consumed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh->tmem_base)),
                 "r"(kSkCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  int issued = 0;

  if (warp == 0) {
    if (lane == 0) {
      // weight tiles first: they do not depend on the previous kernel
      const int pre = nkb < kSkStages ? nkb : kSkStages;
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(&sh->full[i], kSkStageA + kSkStageB);
        tma_load_2d(sA + i * kSkStageA, &tmW, (kb0 + i) * kSkK, mt * kSkM, &sh->full[i]);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * kSkStageB, &tmX, (kb0 + i) * kSkK, 0, &sh->full[i]);
      issued = pre;
      int stage = pre % kSkStages;
      uint32_t phase = pre == kSkStages ? 1 : 0;
      for (int i = pre; i < nkb; ++i) {
        if (!mbar_wait(&sh->empty[stage], phase ^ 1, abort_flag, err)) break;
        mbar_expect_tx(&sh->full[stage], kSkStageA + kSkStageB);
        tma_load_2d(sA + stage * kSkStageA, &tmW, (kb0 + i) * kSkK, mt * kSkM, &sh->full[stage]);
        tma_load_2d(sB + stage * kSkStageB, &tmX, (kb0 + i) * kSkK, 0, &sh->full[stage]);
        ++issued;
        if (++stage == kSkStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      for (int i = 0; i < kSkStages && !*abort_flag; ++i) {  // tail: all stages released
        if (!mbar_wait(&sh->empty[stage], phase ^ 1, abort_flag, err)) break;
        if (++stage == kSkStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      constexpr uint32_t idesc = idesc_bf16(kSkM, kSkN);
      bool ok = true;
      for (int i = 0; i < nkb; ++i) {
        if (!mbar_wait(&sh->full[stage], phase, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * kSkStageA), b0 = smem_u32(sB + stage * kSkStageB);
#pragma unroll
        for (int k = 0; k < kSkK / 16; ++k) tc_mma(tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc, (i | k) != 0);
        tc_commit(&sh->empty[stage]);
        sh->consumed = sh->consumed + 1;
        if (++stage == kSkStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (ok) tc_commit(&sh->tfull);
      tc_commit(&sh->mma_done);
    }
  } else {
    const int et = threadIdx.x - 64;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    pdl_wait();
    {  // 1/rms of the tokens: warp w takes tokens 8w .. 8w+7 at once
      const int t8 = (et >> 5) * 8;
      float r8[8];
      const int n = max(0, min(8, ntok - t8));
      if (a.ssq) {
        row_rstd_n<8>(a.ssq, t8, n, a.d, a.eps, r8);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) r8[u] = 1.0f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (lane == u) rstd_s[t8 + u] = r8[u];
    }
    const bool got = mbar_wait(&sh->tfull, 0, abort_flag, err);
    if (!epi_any(!got)) {
      tc_fence_after();
      uint32_t v[32];
      tc_ld32(tmem + ((uint32_t)(quarter * 32) << 16), v);
#pragma unroll
      for (int j = 0; j < 32; ++j) tile[j * kSkLd + row] = __uint_as_float(v[j]);
    }
  }

  cluster_sync();  // every partial tile of the cluster is in shared memory
  const int rows_per = ks <= 8 ? kSkM / ks : 16;
  const int r_lo = z * rows_per;
  const bool has_rows = !*abort_flag && r_lo < kSkM;
  const float* src = tile + r_lo;  // this CTA's reduced rows: element (row rr, token t) at src[t * src_ld + rr]
  int src_ld = kSkLd;
  if (warp >= 2) {
    const int et = threadIdx.x - 64;
    if (has_rows && ks > 1) {
      switch (ks) {  // every rank's partial of 4 rows in flight at once, summed in rank order
        case 2: sk_reduce<2>(tile, red, r_lo, rows_per, et); break;
        case 4: sk_reduce<4>(tile, red, r_lo, rows_per, et); break;
        case 8: sk_reduce<8>(tile, red, r_lo, rows_per, et); break;
        default: sk_reduce<16>(tile, red, r_lo, rows_per, et); break;
      }
      src = red;
      src_ld = kSkRedLd;
    }
    if constexpr (EPI != EPI_QKV) {
      if (has_rows) {
        epi_bar();
        epilogue<AT, EPI, 128>(a, src, src_ld, mt * kSkM + r_lo, rows_per, 0, ntok, rstd_s, et);
      }
    } else {
      // partial sums of squares of this CTA's rows, per (head in the tile, token)
      const int D = a.qf.D;
      for (int i = et; i < 4 * kSkN; i += 128) sh->psq[i / kSkN][i % kSkN] = 0.f;
      epi_bar();
      if (has_rows) {
        const int h_lo = r_lo / D, h_n = rows_per >= D ? rows_per / D : 1;
        for (int i = et; i < h_n * ntok; i += 128) {
          const int hl = h_lo + i / ntok, t = i % ntok;
          const int a0 = max(hl * D, r_lo), a1 = min(hl * D + D, r_lo + rows_per);
          float ss = 0.f;
          for (int r = a0; r < a1; ++r) {
            const float y = src[t * src_ld + (r - r_lo)] * rstd_s[t];
            ss = fmaf(y, y, ss);
          }
          sh->psq[hl][t] = ss;
        }
      }
    }
  }
  if constexpr (EPI == EPI_QKV) {
    cluster_sync();  // every CTA's partial sums and reduced rows are visible
    const QkvFuse& f = a.qf;
    const int D = f.D, half = D / 2;
    if (warp >= 2 && has_rows) {
      const int et = threadIdx.x - 64;
      // per token: position and cache block; per (head of this CTA's rows, token): 1/rms
      for (int t = et; t < ntok; t += 128) {
        const int pos = f.meta.tok_pos[t];
        sh->tpos[t] = pos;
        sh->tblk[t] = qkv_block(f, t, pos);
      }
      const int h_lo = r_lo / D, h_n = rows_per >= D ? rows_per / D : 1;
      for (int i = et; i < h_n * ntok; i += 128) {
        const int hl = h_lo + i / ntok, t = i % ntok;
        float pv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (q < ks) pv[q] = ks > 1 ? dsmem_ld(dsmem_addr(&sh->psq[hl][t], (uint32_t)q)) : sh->psq[hl][t];
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (q < ks) ss += pv[q];
        sh->rn[hl][t] = 1.0f / sqrtf(ss / (float)D + a.eps);
      }
      epi_bar();
      for (int i = et; i < ntok * rows_per; i += 128) {
        const int t = i / rows_per, rr = i - t * rows_per;
        const int r = r_lo + rr, hl = r / D, j = r - hl * D;
        const int gh = (mt * kSkM + hl * D) / D;
        const float y = src[t * src_ld + rr] * rstd_s[t];
        float out = y;
        if (gh < f.H + f.Hkv) {
          const int rp = j < half ? r + half : r - half;
          const int zo = rp / rows_per;
          const float yp = zo == z ? src[t * src_ld + (rp - r_lo)]
                                   : dsmem_ld(dsmem_addr(red + t * kSkRedLd + (rp - zo * rows_per), (uint32_t)zo));
          out = qk_rope(f, gh, j, y, yp * rstd_s[t], sh->rn[hl][t], sh->tpos[t]);
        }
        qkv_store<__half>(f, t, gh, j, out, sh->tpos[t], sh->tblk[t]);
      }
    }
  }
  cluster_sync();  // no CTA leaves while another still reads its tile

  if (*abort_flag) {
    if (threadIdx.x == 0) {
      for (int j = sh->consumed; j < issued; ++j) {
        const uint64_t t0 = global_ns();
        while (!mbar_try(&sh->full[j % kSkStages], (j / kSkStages) & 1) && global_ns() - t0 < kWaitLimitNs) {
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kSkCols) : "memory");
  }
}

// Split factor: the smallest power of two giving at least 128 CTAs, at most 16
// and at most the number of 64-wide K blocks (which it must divide).
int skinny_splits(int rows, int K) {
  const int m_tiles = rows / kSkM, nkb = K / kSkK;
  int ks = 1;
  while (ks < 16 && m_tiles * ks < 128 && nkb % (2 * ks) == 0) ks *= 2;
  return ks;
}

bool tc_skinny_eligible(const GemvArgs& a) {
  return a.rows % kSkM == 0 && a.K % kSkK == 0 && a.T >= 1 && a.T <= kSkN && a.x_row == nullptr;
}

template <typename AT, int EPI>
static cudaError_t skinny_one(const GemvArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX, uint32_t* err,
                              bool pdl, cudaStream_t s) {
  static SmemOptIn opt;
  cudaError_t e = opt.ensure(k_gemm_tc_skinny<AT, EPI>, (int)kSkSmemBytes, /*nonportable_cluster=*/true);
  if (e != cudaSuccess) return e;
  const int ks = skinny_splits(a.rows, a.K);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.rows / kSkM) * ks, 1, 1);
  cfg.blockDim = dim3(kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = kSkSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = ks;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k_gemm_tc_skinny<AT, EPI>, *tmW, *tmX, a, ks, err);
}

cudaError_t launch_gemm_tc_skinny(const GemvArgs& a, int epi, const void* tmW, const void* tmX, uint32_t* err,
                                  bool pdl, cudaStream_t s) {
  const CUtensorMap* w = reinterpret_cast<const CUtensorMap*>(tmW);
  const CUtensorMap* x = reinterpret_cast<const CUtensorMap*>(tmX);
  switch (epi) {
    case EPI_QKV_RAW: return skinny_one<bf16, EPI_QKV_RAW>(a, w, x, err, pdl, s);
    case EPI_QKV: return skinny_one<bf16, EPI_QKV>(a, w, x, err, pdl, s);
    case EPI_RESID: return skinny_one<bf16, EPI_RESID>(a, w, x, err, pdl, s);
    case EPI_SWIGLU: return skinny_one<bf16, EPI_SWIGLU>(a, w, x, err, pdl, s);
    default: return skinny_one<bf16, EPI_LOGITS>(a, w, x, err, pdl, s);
  }
}

}  // namespace dec
