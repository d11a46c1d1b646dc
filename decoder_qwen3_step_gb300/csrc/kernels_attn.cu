// kernels_attn.cu - causal grouped-query attention over the paged KV cache.
//
// o_t = sum_{j <= pos(t)} softmax_j(q_t . k_j / sqrt(D)) v_j, query head h
// reading KV head floor(h * Hkv / H); each query attends over exactly its
// visible keys, no mask is stored (tinyllm L10.1 "Candle model runner ...",
// section 2.4 and its batch-invariance paragraph).  Keys live in pool blocks:
// position j of a sequence is slot j % B of block table[j / B].
//
// Decode (one query per sequence): split-K over fixed 64-key chunks (the split
// never depends on the batch), one warp per 16-key block, warp-shuffle softmax;
// each chunk's CTA writes its record, and the CTA that finishes a (sequence,
// KV head)'s count merges all of its chunk records in chunk order, in the
// same launch.
// Prefill: one CTA per (tile of queries, KV head) with the G query heads of
// the group stacked as rows; key tiles of 32 are staged in shared memory and
// folded in with an online softmax.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

template <typename KT, int N>
__device__ __forceinline__ void loadN(const KT* p, float* v) {
  if constexpr (N % 8 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 8) load8(p + i, v + i);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = to_f32(p[i]);
  }
}

// Raw storage of N cache elements in 32-bit registers, filled by the widest
// aligned vector loads (16, 8 or 4 bytes); converted to fp32 at use.
template <typename KT, int N>
struct Raw {
  static constexpr int kWords = N * (int)sizeof(KT) / 4;
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const KT* p) {
    constexpr int B = N * (int)sizeof(KT);
    if constexpr (B % 16 == 0) {
#pragma unroll
      for (int i = 0; i < B / 16; ++i) reinterpret_cast<uint4*>(w)[i] = reinterpret_cast<const uint4*>(p)[i];
    } else if constexpr (B % 8 == 0) {
#pragma unroll
      for (int i = 0; i < B / 8; ++i) reinterpret_cast<uint2*>(w)[i] = reinterpret_cast<const uint2*>(p)[i];
    } else {
#pragma unroll
      for (int i = 0; i < kWords; ++i) w[i] = reinterpret_cast<const uint32_t*>(p)[i];
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ float get(int i) const {
    if constexpr (sizeof(KT) == 4) {
      return __uint_as_float(w[i]);
    } else {
      return __half2float(reinterpret_cast<const __half*>(w)[i]);
    }
  }
};

// ---------------------------------------------------------------------------
// Decode attention, split-K.  grid (chunk, kv head, sequence), 4 warps.  Keys
// are cut into fixed 64-key chunks (4 blocks of 16; the cut depends only on
// the position, never on the batch), one chunk per CTA.  One thread issues
// bulk asynchronous copies of the chunk's K and V slabs (4 KB each per block
// and KV head at the serving shape) into shared memory on one mbarrier, so a
// whole chunk is in flight at once without holding registers.  Warp w then
// folds blocks w and w + 4 into an online softmax: lane l holds D/32 dims of
// the G queries, forms partial dots with 16 keys, and a 31-shuffle
// reduce-scatter leaves lane l with the full score of (head l/16, key l%16);
// the value rows are read one 256-byte row per instruction.  The 4 warps'
// states merge in warp order into one (max, sum, o[D]) record per chunk and
// query head; the last CTA of a (sequence, KV head) to finish merges all
// records in chunk order, writes the attention output and re-arms the counter.
// ---------------------------------------------------------------------------
constexpr int kDecWarps = 4;
constexpr int kDecBlocks = kDecodeChunk / 16;  // 4
constexpr int kMaxChunks = (kMaxPositions + kDecodeChunk - 1) / kDecodeChunk;

template <typename KT, int D>
__host__ __device__ constexpr size_t decode_smem_bytes() {
  return (size_t)2 * kDecBlocks * 16 * D * sizeof(KT);
}

// The score of lane (head lane/16, key lane%16) from 32 per-lane partials
// v[i*16 + k] (G = 2): reduce-scatter over the warp, 31 shuffles.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = up ? v[j] : v[j + w];
      const float keep = up ? v[j + w] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

template <typename KT, typename AT, int D, int G>
__global__ void __launch_bounds__(kDecWarps * 32) k_attn_decode(AttnArgs a) {
  pdl_launch_next();
  constexpr int kThreads = kDecWarps * 32, kDim = D / 32;
  const Dims& dm = a.dims;
  const int c = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int ctx = a.meta.seq_ctx[s];
  const int nch = (ctx + kDecodeChunk - 1) / kDecodeChunk;
  if (c >= nch) return;
  extern __shared__ __align__(128) uint8_t dsm[];
  KT* Ks = reinterpret_cast<KT*>(dsm);        // [4 blocks][16 keys][D]
  KT* Vs = Ks + kDecBlocks * 16 * D;          // [4 blocks][16 keys][D]
  __shared__ float qs[G][D];
  __shared__ float ms[kDecWarps][G], ls[kDecWarps][G];
  __shared__ float os[kDecWarps][G][D];
  __shared__ float fac[G][kMaxChunks];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int last_flag, abort_flag;
  const int t = a.meta.seq_start[s];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int keys_here = min(kDecodeChunk, ctx - c * kDecodeChunk);
  const int nblk = (keys_here + 15) / 16;
  constexpr uint32_t kSlab = 16 * D * sizeof(KT);

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // lane b looks up block b's pool id and issues its two copies: the table
  // reads are independent, so their latencies overlap
  auto issue = [&]() {
    if (lane == 0) mbar_expect_tx(&bar, 2 * kSlab * nblk);
    __syncwarp();
    if (lane < nblk) {
      const KT* kv = reinterpret_cast<const KT*>(a.kv);
      const int blk = table_block(a.meta.tables, s, c * kDecBlocks + lane, dm.max_blocks, dm.n_blocks, a.err);
      bulk_g2s(Ks + lane * 16 * D, kv + kv_offset(a.layer, blk, 0, g, 0, dm.n_blocks, dm.Hkv, 16, D), kSlab, &bar);
      bulk_g2s(Vs + lane * 16 * D, kv + kv_offset(a.layer, blk, 1, g, 0, dm.n_blocks, dm.Hkv, 16, D), kSlab, &bar);
    }
  };
  // Every key of a chunk before the last was written by an earlier step (a
  // decode step writes position ctx - 1 only) and the metadata before this
  // step's first kernel, so those copies start before the wait on the
  // previous kernel (programmatic dependent launch: they overlap its tail).
  // The last chunk holds this step's key: its copy waits; so does Q.
  const bool old_chunk = c < nch - 1;
  if (warp == 0 && old_chunk) issue();
  pdl_wait_prev();
  if (warp == 0 && !old_chunk) issue();
  for (int i = threadIdx.x; i < G * D; i += kThreads)
    qs[i / D][i % D] = a.Q[((size_t)t * dm.H + g * G + i / D) * D + i % D];
  __syncthreads();
  float q[G][kDim];
#pragma unroll
  for (int i = 0; i < G; ++i)
#pragma unroll
    for (int e = 0; e < kDim; ++e) q[i][e] = qs[i][lane * kDim + e];
  const bool ok = mbar_wait(&bar, 0, &abort_flag, a.err);

  float m[G], l[G], o[G][kDim];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < kDim; ++e) o[i][e] = 0.f;
  }
  if (ok) {
    for (int b = warp; b < nblk; b += kDecWarps) {
      const KT* Kb = Ks + b * 16 * D;
      const KT* Vb = Vs + b * 16 * D;
      const int nkeys = min(16, keys_here - b * 16);
      float sc[G];
      if constexpr (G == 2) {
        float v[32];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float kk[kDim];
#pragma unroll
          for (int e = 0; e < kDim; ++e) kk[e] = to_f32(Kb[k * D + lane * kDim + e]);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < kDim; ++e) acc = fmaf(q[i][e], kk[e], acc);
            v[i * 16 + k] = acc;
          }
        }
        const float full = reduce_scatter32(v, lane) * a.scale;  // lane = head*16 + key
        sc[0] = sc[1] = ((lane & 15) < nkeys) ? full : -INFINITY;
      } else {
        // general group size: one butterfly per (key, head); lane (i*16 + k) keeps its own
#pragma unroll
        for (int i = 0; i < G; ++i) sc[i] = -INFINITY;
        for (int k = 0; k < 16; ++k) {
          float kk[kDim];
#pragma unroll
          for (int e = 0; e < kDim; ++e) kk[e] = to_f32(Kb[k * D + lane * kDim + e]);
#pragma unroll
          for (int i = 0; i < G; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < kDim; ++e) acc = fmaf(q[i][e], kk[e], acc);
            acc = warp_sum(acc) * a.scale;
            if ((lane & 15) == k && k < nkeys) sc[i] = acc;
          }
        }
      }
      // per head: the block's max over its 16 keys, rescale the running state
      float p[G];
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const int owner = G == 2 ? i : 0;  // G == 2: lanes 16*i .. 16*i+15 hold head i
        float mx = sc[i];
#pragma unroll
        for (int o2 = 8; o2 >= 1; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float mb = __shfl_sync(0xffffffffu, mx, owner * 16);
        const float m_new = fmaxf(m[i], mb);
        const float corr = m[i] == -INFINITY ? 0.f : expf(m[i] - m_new);
        p[i] = sc[i] == -INFINITY ? 0.f : expf(sc[i] - m_new);
        float ps = p[i];
#pragma unroll
        for (int o2 = 8; o2 >= 1; o2 >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o2);
        ps = __shfl_sync(0xffffffffu, ps, owner * 16);
        l[i] = l[i] * corr + ps;
        m[i] = m_new;
#pragma unroll
        for (int e = 0; e < kDim; ++e) o[i][e] *= corr;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k >= nkeys) break;  // slots past the context may hold anything, even NaN
        float vv[kDim];
#pragma unroll
        for (int e = 0; e < kDim; ++e) vv[e] = to_f32(Vb[k * D + lane * kDim + e]);
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const float pk = __shfl_sync(0xffffffffu, p[i], (G == 2 ? i * 16 : 0) + k);
#pragma unroll
          for (int e = 0; e < kDim; ++e) o[i][e] = fmaf(pk, vv[e], o[i][e]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < G; ++i) {
    if (lane == 0) {
      ms[warp][i] = m[i];
      ls[warp][i] = l[i];
    }
#pragma unroll
    for (int e = 0; e < kDim; ++e) os[warp][i][lane * kDim + e] = o[i][e];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += kThreads) {
    const int h = i / D, dd = i % D;
    float M = ms[0][h];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) M = fmaxf(M, ms[w][h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float f = ms[w][h] == -INFINITY ? 0.f : expf(ms[w][h] - M);
      L = fmaf(ls[w][h], f, L);
      O = fmaf(os[w][h][dd], f, O);
    }
    float* part = a.part + (((size_t)s * dm.H + g * G + h) * a.nchunk_cap + c) * (D + 2);
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
  if (threadIdx.x == 0) last_flag = atomicAdd(a.counters + s * dm.Hkv + g, 1) == nch - 1;
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  const float* base = a.part + ((size_t)s * dm.H + g * G) * a.nchunk_cap * (D + 2);
  if (warp < G) {
    const float* ph = base + (size_t)warp * a.nchunk_cap * (D + 2);
    float mx = -INFINITY;
    for (int cc = lane; cc < nch; cc += 32) mx = fmaxf(mx, __ldcg(ph + cc * (D + 2)));
    mx = warp_max(mx);
    float sum = 0.f;
    for (int cc = lane; cc < nch; cc += 32) {
      const float f = expf(__ldcg(ph + cc * (D + 2)) - mx);
      fac[warp][cc] = f;
      sum = fmaf(__ldcg(ph + cc * (D + 2) + 1), f, sum);
    }
    sum = warp_sum(sum);
    if (lane == 0) ms[0][warp] = sum;
  }
  __syncthreads();
  AT* out = reinterpret_cast<AT*>(a.ATT);
  for (int i = threadIdx.x; i < G * D; i += kThreads) {
    const int h = i / D, dd = i % D;
    const float* ph = base + (size_t)h * a.nchunk_cap * (D + 2) + 2 + dd;
    float O = 0.f;
#pragma unroll 4
    for (int cc = 0; cc < nch; ++cc) O = fmaf(__ldcg(ph + cc * (D + 2)), fac[h][cc], O);
    out[((size_t)t * dm.H + g * G + h) * D + dd] = from_f32<AT>(O / ms[0][h]);
  }
  if (threadIdx.x == 0) a.counters[s * dm.Hkv + g] = 0;
}

// ---------------------------------------------------------------------------
// Prefill attention.  grid (work tile, kv head), 128 threads.  A tile is up to
// QT = 64/G consecutive new tokens of one sequence; its 64 query-head rows are
// row r = query * G + head-in-group.  Thread (ty, tx) = (tid / 8, tid % 8) owns
// rows 4ty..4ty+3; for scores it owns keys tx + 8i of the 32-key tile, for the
// output it owns dims tx*4 + 32i + (0..3).
// ---------------------------------------------------------------------------
constexpr int kPfRows = 64;
constexpr int kPfKeys = 32;

template <typename KT, typename AT, int D, int G>
__global__ void __launch_bounds__(128) k_attn_prefill(AttnArgs a) {
  pdl_launch_next();
  pdl_wait_prev();
  constexpr int LD = D + 4;  // padded row stride (floats)
  constexpr int kDimGroups = D / 32;
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm;                      // [64][LD]
  float* Ks = Qs + kPfRows * LD;       // [32][LD]
  float* Vs = Ks + kPfKeys * LD;       // [32][LD]
  float* Ps = Vs + kPfKeys * LD;       // [64][33]
  const Dims& dm = a.dims;
  const int* w = a.meta.work + blockIdx.x * 3;
  const int s = w[0], tok0 = w[1], ntok = w[2];
  const int g = blockIdx.y;
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
  const int p0 = a.meta.tok_pos[tok0];
  const int p_last = p0 + ntok - 1;
  const KT* kv = reinterpret_cast<const KT*>(a.kv);

  for (int i = tid; i < kPfRows * (D / 4); i += 128) {
    const int r = i / (D / 4), c4 = i % (D / 4);
    const int qi = r / G, hh = r % G;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (qi < ntok) v = *reinterpret_cast<const float4*>(a.Q + ((size_t)(tok0 + qi) * dm.H + g * G + hh) * D + c4 * 4);
    *reinterpret_cast<float4*>(Qs + r * LD + c4 * 4) = v;
  }
  float m[4], l[4], o[4][kDimGroups][4];
  int rpos[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
    rpos[i] = p0 + (ty * 4 + i) / G;
#pragma unroll
    for (int j = 0; j < kDimGroups; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][j][e] = 0.f;
  }
  const int ntiles = p_last / kPfKeys + 1;
  for (int kt = 0; kt < ntiles; ++kt) {
    const int j0 = kt * kPfKeys;
    __syncthreads();  // previous tile fully consumed
    for (int i = tid; i < kPfKeys * (D / 8); i += 128) {
      const int kk = i / (D / 8), c8 = (i % (D / 8)) * 8;
      const int j = j0 + kk;
      float kvv[8], vvv[8];
      if (j <= p_last) {
        const int blk = table_block(a.meta.tables, s, j / dm.B, dm.max_blocks, dm.n_blocks, a.err);
        const int slot = j % dm.B;
        load8(kv + kv_offset(a.layer, blk, 0, g, slot, dm.n_blocks, dm.Hkv, dm.B, D) + c8, kvv);
        load8(kv + kv_offset(a.layer, blk, 1, g, slot, dm.n_blocks, dm.Hkv, dm.B, D) + c8, vvv);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) kvv[e] = vvv[e] = 0.f;
      }
      *reinterpret_cast<float4*>(Ks + kk * LD + c8) = make_float4(kvv[0], kvv[1], kvv[2], kvv[3]);
      *reinterpret_cast<float4*>(Ks + kk * LD + c8 + 4) = make_float4(kvv[4], kvv[5], kvv[6], kvv[7]);
      *reinterpret_cast<float4*>(Vs + kk * LD + c8) = make_float4(vvv[0], vvv[1], vvv[2], vvv[3]);
      *reinterpret_cast<float4*>(Vs + kk * LD + c8 + 4) = make_float4(vvv[4], vvv[5], vvv[6], vvv[7]);
    }
    __syncthreads();
    // scores: 4 rows x 4 keys per thread
    float sc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[i][j] = 0.f;
#pragma unroll 4
    for (int d4 = 0; d4 < D; d4 += 4) {
      float4 q[4], k[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = *reinterpret_cast<const float4*>(Qs + (ty * 4 + i) * LD + d4);
#pragma unroll
      for (int j = 0; j < 4; ++j) k[j] = *reinterpret_cast<const float4*>(Ks + (tx + 8 * j) * LD + d4);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float acc = sc[i][j];
          acc = fmaf(q[i].x, k[j].x, acc);
          acc = fmaf(q[i].y, k[j].y, acc);
          acc = fmaf(q[i].z, k[j].z, acc);
          acc = fmaf(q[i].w, k[j].w, acc);
          sc[i][j] = acc;
        }
    }
    // online softmax per row over the 8 threads sharing ty
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = j0 + tx + 8 * j;
        sc[i][j] = key <= rpos[i] ? sc[i][j] * a.scale : -INFINITY;
        mx = fmaxf(mx, sc[i][j]);
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[i], mx);
      float corr = 1.f, rs = 0.f;
      if (m_new != -INFINITY) {
        corr = m[i] == -INFINITY ? 0.f : expf(m[i] - m_new);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p = sc[i][j] == -INFINITY ? 0.f : expf(sc[i][j] - m_new);
          Ps[(ty * 4 + i) * (kPfKeys + 1) + tx + 8 * j] = p;
          rs += p;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) Ps[(ty * 4 + i) * (kPfKeys + 1) + tx + 8 * j] = 0.f;
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      m[i] = m_new;
      l[i] = l[i] * corr + rs;
#pragma unroll
      for (int j = 0; j < kDimGroups; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][j][e] *= corr;
    }
    __syncthreads();
    // o += P V
#pragma unroll 4
    for (int kk = 0; kk < kPfKeys; ++kk) {
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = Ps[(ty * 4 + i) * (kPfKeys + 1) + kk];
#pragma unroll
      for (int j = 0; j < kDimGroups; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(Vs + kk * LD + tx * 4 + 32 * j);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[i][j][0] = fmaf(p[i], v.x, o[i][j][0]);
          o[i][j][1] = fmaf(p[i], v.y, o[i][j][1]);
          o[i][j][2] = fmaf(p[i], v.z, o[i][j][2]);
          o[i][j][3] = fmaf(p[i], v.w, o[i][j][3]);
        }
      }
    }
  }
  AT* out = reinterpret_cast<AT*>(a.ATT);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i, qi = r / G, hh = r % G;
    if (qi >= ntok) continue;
    const float inv = 1.0f / l[i];
    AT* dst = out + ((size_t)(tok0 + qi) * dm.H + g * G + hh) * D;
#pragma unroll
    for (int j = 0; j < kDimGroups; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[tx * 4 + 32 * j + e] = from_f32<AT>(o[i][j][e] * inv);
  }
}

int prefill_tile_queries(int G) { return kPfRows / G; }

// ---------------------------------------------------------------------------
// launchers: head_dim in {32, 64, 128}, group size in {1, 2, 4}
// ---------------------------------------------------------------------------
template <typename KT, typename AT, int D, int G>
static cudaError_t attn_decode_t(const AttnArgs& a, int nchunk, cudaStream_t s) {
  static SmemOptIn opt;
  constexpr size_t smem = decode_smem_bytes<KT, D>();
  cudaError_t e = opt.ensure(k_attn_decode<KT, AT, D, G>, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nchunk, a.dims.Hkv, a.S);
  cfg.blockDim = dim3(kDecWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // older chunks' copies overlap the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attn_decode<KT, AT, D, G>, a);
}

template <typename KT, typename AT, int D, int G>
static cudaError_t attn_prefill_t(const AttnArgs& a, int n_work, cudaStream_t s) {
  constexpr int LD = D + 4;
  const size_t smem = ((size_t)kPfRows * LD + 2 * kPfKeys * LD + kPfRows * (kPfKeys + 1)) * sizeof(float);
  static SmemOptIn opt;
  cudaError_t e = opt.ensure(k_attn_prefill<KT, AT, D, G>, (int)smem);
  if (e != cudaSuccess) return e;
  k_attn_prefill<KT, AT, D, G><<<dim3(n_work, a.dims.Hkv), 128, smem, s>>>(a);
  return cudaGetLastError();
}

#define DEC_DISPATCH_DG(FN, KT, AT, ...)                                         \
  do {                                                                          \
    const int D_ = a.dims.D, G_ = a.dims.H / a.dims.Hkv;                        \
    if (D_ == 128 && G_ == 2) return FN<KT, AT, 128, 2>(a, __VA_ARGS__);        \
    if (D_ == 128 && G_ == 1) return FN<KT, AT, 128, 1>(a, __VA_ARGS__);        \
    if (D_ == 128 && G_ == 4) return FN<KT, AT, 128, 4>(a, __VA_ARGS__);        \
    if (D_ == 64 && G_ == 2) return FN<KT, AT, 64, 2>(a, __VA_ARGS__);          \
    if (D_ == 64 && G_ == 1) return FN<KT, AT, 64, 1>(a, __VA_ARGS__);          \
    if (D_ == 64 && G_ == 4) return FN<KT, AT, 64, 4>(a, __VA_ARGS__);          \
    if (D_ == 32 && G_ == 2) return FN<KT, AT, 32, 2>(a, __VA_ARGS__);          \
    if (D_ == 32 && G_ == 1) return FN<KT, AT, 32, 1>(a, __VA_ARGS__);          \
    if (D_ == 32 && G_ == 4) return FN<KT, AT, 32, 4>(a, __VA_ARGS__);          \
    return cudaErrorInvalidValue;                                               \
  } while (0)

cudaError_t launch_attn_decode(const AttnArgs& a, int nchunk, bool wbf16, cudaStream_t s) {
  if (wbf16) DEC_DISPATCH_DG(attn_decode_t, __half, bf16, nchunk, s);
  DEC_DISPATCH_DG(attn_decode_t, float, float, nchunk, s);
}

cudaError_t launch_attn_prefill(const AttnArgs& a, int n_work, bool wbf16, cudaStream_t s) {
  if (wbf16) DEC_DISPATCH_DG(attn_prefill_t, __half, bf16, n_work, s);
  DEC_DISPATCH_DG(attn_prefill_t, float, float, n_work, s);
}

}  // namespace dec
