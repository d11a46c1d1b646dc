// kernels_attn_dec_tc.cu - decode attention of the serving mode (f16 KV
// cache, two query heads per KV head) on the warp-level tensor cores, with
// the QK-norm, RoPE and cache append of the new token fused in.
//
// o = sum_{j < ctx} softmax_j(q . k_j / sqrt(D)) v_j for the newest token of
// every sequence, query head h reading KV head h / 2 (tinyllm L10.1 "Candle
// model runner ...", section 2.4, at one token per sequence; QK-norm before
// split-half RoPE as octlm "A real model in our own decoder" switches them
// on).  Keys are cut into the same fixed 64-key chunks as the CUDA-core
// kernel (the cut depends only on the position), and the work items are the
// (sequence, KV head, chunk) triples, sequence-major.
//
// One persistent CTA per SM takes a contiguous range of items:
//   * a producer warp streams each item's K and V blocks by TMA (boxes of 16
//     rows, 128-byte swizzle) into a ring of six 32 KB slots; chunks older
//     than the step are copied before the wait on the previous kernel, a
//     sequence's last chunk after it;
//   * three groups of four consumer warps take the items in turn (group q
//     owns slots q and q + 3): warps 0 and 1 form the group's two queries
//     from the raw q|k|v row of the QKV product (RMSNorm over the head, then
//     RoPE at the token's position); in a sequence's last chunk warps 2 and 3
//     form the new key (normed and rotated) and value, store them to the
//     cache as f16 and patch the landed tile, value rows past the context
//     zeroed; warp w folds block w on the tensor cores (fold16) and the four
//     warps' states merge in warp order into one record per chunk and head;
//   * when its items are done the CTA adds its chunk counts to the
//     per-(sequence, KV head) counters, and the CTA that completes a count
//     merges that pair's records in chunk order and writes the attention
//     output.  Every reduction has one order fixed by the shapes, so the
//     output does not depend on the batch or the grid.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "attn_fold.cuh"
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

namespace {

constexpr int kBlocks = kDecodeChunk / 16;  // 16-key blocks per chunk
constexpr int kChunkCap = (kMaxPositions + kDecodeChunk - 1) / kDecodeChunk;

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

constexpr int kRingSlots = 6;
constexpr int kRingGroups = 3;
constexpr int kRingConsumers = kRingGroups * 128;
constexpr int kRingThreads = kRingConsumers + 32;
// Item k lands in slot k % kRingSlots and is folded by group k % kRingGroups:
// every slot must belong to one group, or a group running ahead could test a
// full-barrier parity that an earlier phase of the slot already completed.
static_assert(kRingSlots % kRingGroups == 0, "each ring slot is consumed by one group");
constexpr int kRingPairs = 32;  // (sequence, KV head) pairs counted and merged together at a CTA's end

template <int D>
struct RingSmem {
  static constexpr int kSlab = KvSlab<D>::kBytes;
  static constexpr int kSlot = 2 * kBlocks * kSlab;           // K blocks, then V blocks
  static constexpr int kGQ = 0;                               // per group: f16 [2][D] queries
  static constexpr int kGO = 2 * D * 2;                       //            float [4][2][D]
  static constexpr int kGM = kGO + 4 * 2 * D * 4;             //            float [4][2] max, [4][2] sum
  static constexpr int kGroup = (kGM + 2 * 4 * 2 * 4 + 127) / 128 * 128;
  static constexpr int kGroups = kRingSlots * kSlot;
  static constexpr int kF = kGroups + kRingGroups * kGroup;   // the end-of-CTA pair list and completion flags
                                                              // (4 x kRingPairs ints of the area used)
  static constexpr int kZ = (kF + (2 * kChunkCap + 2) * 4 + 127) / 128 * 128;  // f16 [D] zeros
  static constexpr int kBar = (kZ + D * 2 + 15) / 16 * 16;    // full[kRingSlots], empty[kRingSlots], flags
  static constexpr int kTotal = kBar + 2 * kRingSlots * 8 + 16 * 4;
  // TMA 128-byte swizzle wants 1024-byte slots; ldmatrix rows (queries, zeros) 16 bytes;
  // the fold's float2 stores 8; mbarriers 8
  static_assert(kSlot % 1024 == 0 && kGroups % 1024 == 0, "slot alignment");
  static_assert(kGroup % 16 == 0 && kGQ % 16 == 0 && kGO % 16 == 0 && kGM % 8 == 0, "group alignment");
  static_assert(kF % 16 == 0 && kZ % 16 == 0 && kBar % 16 == 0, "tail alignment");
};

__device__ __forceinline__ void ring_share(int units, int P, int b, int& u0, int& u1) {
  u0 = (int)(((long long)units * b) / P);
  u1 = (int)(((long long)units * (b + 1)) / P);
}

struct RingItem {
  int s, g, c, nch;
};
// The item at flat index i (item_start: the first item of every sequence).
__device__ __forceinline__ RingItem ring_item(const int32_t* item_start, const int32_t* seq_ctx, int S, int i) {
  int s = 0, hi = S - 1;  // the last sequence whose first item is <= i
  while (s < hi) {
    const int mid = (s + hi + 1) >> 1;
    if (__ldg(item_start + mid) <= i) s = mid;
    else hi = mid - 1;
  }
  const int nch = (__ldg(seq_ctx + s) + kDecodeChunk - 1) / kDecodeChunk;
  const int rem = i - __ldg(item_start + s);
  return {s, rem / nch, rem % nch, nch};
}
// The item after `it` in the flat order.
__device__ __forceinline__ void ring_next(RingItem& it, const int32_t* seq_ctx, int S, int Hkv) {
  if (++it.c < it.nch) return;
  it.c = 0;
  if (++it.g < Hkv) return;
  it.g = 0;
  if (++it.s < S) it.nch = (__ldg(seq_ctx + it.s) + kDecodeChunk - 1) / kDecodeChunk;
}

template <int D>
__global__ void __launch_bounds__(kRingThreads, 1) k_attn_decode_ring(const __grid_constant__ CUtensorMap tm_kv,
                                                                     const __grid_constant__ AttnDecTcArgs a,
                                                                     const int32_t* __restrict__ item_start) {
  pdl_launch_next();
  using SM = RingSmem<D>;
  constexpr int kDim = D / 32, kSlab = SM::kSlab, kB = KvSlab<D>::kBoxes;
  const Dims& dm = a.at.dims;
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + SM::kBar);
  uint64_t* empty = full + kRingSlots;
  int* flags = reinterpret_cast<int*>(empty + kRingSlots);  // [0] abort, [2..7] the end-of-CTA pair list header
  __half* zrow = reinterpret_cast<__half*>(dsm + SM::kZ);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.at.S, P = gridDim.x, b = blockIdx.x;
  const int* seq_ctx = a.at.meta.seq_ctx;
  const int n_items = __ldg(item_start + S);
  int i0, i1;
  ring_share(n_items, P, b, i0, i1);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);  // the four warps of the group that folded the slot
    }
    flags[0] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < D; i += kRingThreads) zrow[i] = __float2half_rn(0.f);
  __syncthreads();
  volatile int* abort_flag = flags;

  if (warp == kRingGroups * 4) {
    // ---- producer: the CTA's items in order, one slot each ----
    // lane L < 2 * kB * kBlocks copies box L % kB of block (L / kB) % kBlocks of K (or V)
    const int bx = lane % kB, j = (lane / kB) % kBlocks, is_v = lane / (kB * kBlocks);
    const int n = i1 - i0;
    bool waited = false;
    RingItem it = n > 0 ? ring_item(item_start, seq_ctx, S, i0) : RingItem{0, 0, 0, 1};
    // Table entries come in batches of 8 items, one batch ahead: lane L loads
    // block L % 4 of item base + L / 4 (-1 past the context), and the copying
    // lanes pick theirs by shuffle, so no copy waits on a table read.
    RingItem bit = it;  // the first item of the next batch to load
    auto batch = [&](int base) {
      RingItem x = bit;
      for (int q = 0; q < (lane >> 2); ++q) ring_next(x, seq_ctx, S, dm.Hkv);
      for (int q = 0; q < 8; ++q) ring_next(bit, seq_ctx, S, dm.Hkv);
      const int jb = x.c * kBlocks + (lane & 3);
      return base + (lane >> 2) < n && jb * 16 < __ldg(seq_ctx + min(x.s, S - 1))
                 ? table_block(a.at.meta.tables, x.s, jb, dm.max_blocks, dm.n_blocks, a.at.err)
                 : -1;
    };
    int tb_cur = batch(0), tb_next = batch(8);
    for (int k = 0; k < n; ++k) {
      const int slot = k % kRingSlots;
      if (k > 0 && (k & 7) == 0) {
        tb_cur = tb_next;
        tb_next = batch(k + 8);
      }
      const int blk = __shfl_sync(0xffffffffu, tb_cur, (k & 7) * 4 + j);
      bool ok = true;
      if (lane == 0 && k >= kRingSlots) ok = mbar_wait(&empty[slot], ((k / kRingSlots) - 1) & 1, abort_flag, a.at.err);
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
      // a sequence's last chunk holds the position this step writes: wait for the step's kernels before it
      if (it.c == it.nch - 1 && !waited) {
        pdl_wait_prev();
        waited = true;
      }
      const int ctx = __ldg(seq_ctx + it.s);
      const int nblk = (min(kDecodeChunk, ctx - it.c * kDecodeChunk) + 15) / 16;
      if (lane == 0) mbar_expect_tx(&full[slot], 2 * kSlab * nblk);
      __syncwarp();
      if (lane < 2 * kB * kBlocks && blk >= 0) {
        const int row = (((a.at.layer * dm.n_blocks + blk) * 2 + is_v) * dm.Hkv + it.g) * 16;
        tma_load_2d(dsm + slot * SM::kSlot + is_v * kBlocks * kSlab + j * kSlab + bx * KvSlab<D>::kBoxBytes, &tm_kv,
                    bx * KvSlab<D>::kBoxDims, row, &full[slot]);
      }
      __syncwarp();
      ring_next(it, seq_ctx, S, dm.Hkv);
    }
    if (!waited) pdl_wait_prev();
  } else {
    // ---- consumers: group gq takes the CTA's items gq, gq + kRingGroups, ... ----
    pdl_wait_prev();  // the raw q|k|v rows are the previous kernel's
    const int gq = warp >> 2, gw = warp & 3, ltid = threadIdx.x & 127;
    uint8_t* G = dsm + SM::kGroups + gq * SM::kGroup;
    __half* qs = reinterpret_cast<__half*>(G + SM::kGQ);
    float* os = reinterpret_cast<float*>(G + SM::kGO);
    float* ms = reinterpret_cast<float*>(G + SM::kGM);
    float* ls = ms + 8;
    int qs_s = -1, qs_g = -1;  // the (sequence, KV head) whose queries qs holds
    RingItem it = i0 + gq < i1 ? ring_item(item_start, seq_ctx, S, i0 + gq) : RingItem{0, 0, 0, 1};
    for (int k = gq; k < i1 - i0; k += kRingGroups) {
      const int slot = k % kRingSlots;
      const int ctx = __ldg(seq_ctx + it.s), pos = ctx - 1;
      const int t = __ldg(a.at.meta.seq_start + it.s);
      const int keys_here = min(kDecodeChunk, ctx - it.c * kDecodeChunk);
      const bool last = it.c == it.nch - 1;
      uint8_t* Ks = dsm + slot * SM::kSlot;
      uint8_t* Vs = Ks + kBlocks * kSlab;
      if (it.s != qs_s || it.g != qs_g) {  // the group's two queries: QK-norm, RoPE, f16
        if (gw < 2) {
          float v[kDim];
          head_row<D>(a, t, (2 * it.g + gw) * D, a.q_norm, pos, v);
#pragma unroll
          for (int e = 0; e < kDim; ++e) qs[gw * D + lane * kDim + e] = __float2half_rn(v[e]);
        }
        qs_s = it.s;
        qs_g = it.g;
      }
      __half hv[kDim];
      if (last && gw >= 2) {  // the new key (QK-norm, RoPE) and value: to the cache as f16
        const int is_v = gw == 3;
        float v[kDim];
        head_row<D>(a, t, (is_v ? dm.H + dm.Hkv + it.g : dm.H + it.g) * D, is_v ? nullptr : a.k_norm, pos, v);
        const int blk = table_block(a.at.meta.tables, it.s, pos / 16, dm.max_blocks, dm.n_blocks, a.at.err);
        __half* dst = const_cast<__half*>(reinterpret_cast<const __half*>(a.at.kv)) +
                      kv_offset(a.at.layer, blk, is_v, it.g, pos % 16, dm.n_blocks, dm.Hkv, 16, D);
#pragma unroll
        for (int e = 0; e < kDim; ++e) {
          hv[e] = __float2half_rn(v[e]);
          dst[lane * kDim + e] = hv[e];
        }
      }
      const bool ok = mbar_wait(&full[slot], (k / kRingSlots) & 1, abort_flag, a.at.err);
      if (last && gw >= 2 && ok) {
        const int kk = pos - it.c * kDecodeChunk;
        patch_row<D>((gw == 3 ? Vs : Ks) + (kk / 16) * kSlab, kk % 16, hv, gw == 3);
        // the slot is refilled by the async proxy later: order these stores before it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      asm volatile("bar.sync %0, 128;" ::"r"(1 + gq) : "memory");  // queries and patches visible to the group
      if (ok)
        fold16<D>(qs, qs + D, zrow, Ks + gw * kSlab, Vs + gw * kSlab, min(16, keys_here - gw * 16), a.at.scale,
                  os + gw * 2 * D, ms + gw * 2, ls + gw * 2);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the slot
      asm volatile("bar.sync %0, 128;" ::"r"(1 + gq) : "memory");
      // the chunk's record per query head: the four warps merged in warp order
      for (int i = ltid; i < 2 * D; i += 128) {
        const int h = i / D, dd = i % D;
        float M = -INFINITY, L = 0.f, O = 0.f;
        if (ok) {
#pragma unroll
          for (int w = 0; w < 4; ++w) M = fmaxf(M, ms[w * 2 + h]);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float f = ms[w * 2 + h] == -INFINITY ? 0.f : expf(ms[w * 2 + h] - M);
            L = fmaf(ls[w * 2 + h], f, L);
            O = fmaf(os[(w * 2 + h) * D + dd], f, O);
          }
        }
        float* part = a.at.part + (((size_t)it.s * dm.H + 2 * it.g + h) * a.at.nchunk_cap + it.c) * (D + 2);
        if (dd == 0) {
          part[0] = M;
          part[1] = L;
        }
        part[2 + dd] = O;
      }
      // os, ms and ls are rewritten by the next fold, qs perhaps by the next queries
      asm volatile("bar.sync %0, 128;" ::"r"(1 + gq) : "memory");
#pragma unroll
      for (int q = 0; q < kRingGroups; ++q) ring_next(it, seq_ctx, S, dm.Hkv);  // this group's next item
    }
  }
  // ---- count the CTA's chunks into their (sequence, KV head) pairs; merge the pairs it completes ----
  // Up to kRingPairs pairs at a time: thread 0 lists them, one thread per pair
  // adds its chunk count (the atomics overlap), and consumer group q merges
  // the completed pairs q, q + kRingGroups, ... in its own third of the idle
  // ring (records staged in one round trip, then the merge reads shared
  // memory; the arithmetic and its order are the same for every path).
  // The records go before the counts that publish them: the CTA barrier
  // orders every thread's records before the counting threads' atomics,
  // which release (and acquire: the merging side reads other CTAs' records).
  __syncthreads();
  if (i0 >= i1) return;
  int* pl = flags + 2;  // [kRingPairs] (sequence, KV head, chunks here) packed, then [kRingPairs] completed
  uint32_t* plist = reinterpret_cast<uint32_t*>(dsm + SM::kF);   // the factor area holds the list
  int* pdone = reinterpret_cast<int*>(plist + 3 * kRingPairs);
  RingItem it = ring_item(item_start, seq_ctx, S, i0);
  for (int i = i0; i < i1;) {
    if (threadIdx.x == 0) {  // the next pairs of the CTA's range
      int np = 0;
      while (i < i1 && np < kRingPairs) {
        const int here = min(i1 - i, it.nch - it.c);
        plist[3 * np] = it.s;
        plist[3 * np + 1] = it.g;
        plist[3 * np + 2] = here;
        ++np;
        i += here;
        it.c += here - 1;
        ring_next(it, seq_ctx, S, dm.Hkv);
      }
      pl[0] = np;
      pl[1] = i;
      pl[2] = it.s;
      pl[3] = it.g;
      pl[4] = it.c;
      pl[5] = it.nch;
    }
    __syncthreads();
    const int np = pl[0];
    if ((int)threadIdx.x < np) {
      const int s = plist[3 * threadIdx.x], g = plist[3 * threadIdx.x + 1], here = plist[3 * threadIdx.x + 2];
      const int nch = (__ldg(seq_ctx + s) + kDecodeChunk - 1) / kDecodeChunk;
      unsigned old;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                   : "=r"(old)
                   : "l"(a.at.counters + s * dm.Hkv + g), "r"((unsigned)here)
                   : "memory");
      pdone[threadIdx.x] = (int)old + here == nch;
    }
    __syncthreads();
    i = pl[1];
    it = RingItem{pl[2], pl[3], pl[4], pl[5]};
    if (warp < kRingGroups * 4) {
      const int gq = warp >> 2, ltid = threadIdx.x & 127, gwarp = warp & 3;
      constexpr int kPart = SM::kGroups / kRingGroups / 16 * 16;  // bytes of the ring per group
      float* stg = reinterpret_cast<float*>(dsm + gq * kPart);
      float* fac = stg + (kPart / 4 - 2 * kChunkCap - 2);  // [2][kChunkCap] factors, [2] sums at the part's end
      float* sums = fac + 2 * kChunkCap;
      for (int p = gq; p < np; p += kRingGroups) {
        if (!pdone[p]) continue;
        const int s = plist[3 * p], g = plist[3 * p + 1];
        const int nch = (__ldg(seq_ctx + s) + kDecodeChunk - 1) / kDecodeChunk;
        const int t = __ldg(a.at.meta.seq_start + s);
        const float* base = a.at.part + ((size_t)s * dm.H + 2 * g) * a.at.nchunk_cap * (D + 2);
        const int per_head = nch * (D + 2);
        const bool staged = 2 * per_head + 2 * kChunkCap + 2 <= kPart / 4 && !*abort_flag;
        if (staged) {
          // float2 pieces (per_head / 2 a head), kU loads in flight per thread before their stores
          // (one pass up to 23 chunks at D = 128, 31 below)
          constexpr int kU = D == 128 ? 24 : 16;
          for (int x0 = ltid; x0 < per_head; x0 += 128 * kU) {
            float2 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const int x = x0 + u * 128, h = x / (per_head / 2), r = x % (per_head / 2);
              if (x < per_head)
                v[u] = __ldcg(reinterpret_cast<const float2*>(base + (size_t)h * a.at.nchunk_cap * (D + 2)) + r);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const int x = x0 + u * 128, h = x / (per_head / 2), r = x % (per_head / 2);
              if (x < per_head) *reinterpret_cast<float2*>(stg + h * per_head + 2 * r) = v[u];
            }
          }
          asm volatile("bar.sync %0, 128;" ::"r"(1 + gq) : "memory");
        }
        auto rec = [&](int h, int cc, int off) -> float {
          return staged ? stg[h * per_head + cc * (D + 2) + off]
                        : __ldcg(base + (size_t)h * a.at.nchunk_cap * (D + 2) + cc * (D + 2) + off);
        };
        if (gwarp < 2) {
          float mx = -INFINITY;
          for (int cc = lane; cc < nch; cc += 32) mx = fmaxf(mx, rec(gwarp, cc, 0));
          mx = warp_max(mx);
          float sum = 0.f;
          for (int cc = lane; cc < nch; cc += 32) {
            const float f = expf(rec(gwarp, cc, 0) - mx);
            fac[gwarp * kChunkCap + cc] = f;
            sum = fmaf(rec(gwarp, cc, 1), f, sum);
          }
          sum = warp_sum(sum);
          if (lane == 0) sums[gwarp] = sum;
        }
        asm volatile("bar.sync %0, 128;" ::"r"(1 + gq) : "memory");
        bf16* out = reinterpret_cast<bf16*>(a.at.ATT);
        for (int x = ltid; x < 2 * D; x += 128) {
          const int h = x / D, dd = x % D;
          float O = 0.f;
#pragma unroll 4
          for (int cc = 0; cc < nch; ++cc) O = fmaf(rec(h, cc, 2 + dd), fac[h * kChunkCap + cc], O);
          out[((size_t)t * dm.H + 2 * g + h) * D + dd] = __float2bfloat16_rn(O / sums[h]);
        }
        if (ltid == 0) a.at.counters[s * dm.Hkv + g] = 0;  // re-armed for the next layer
        asm volatile("bar.sync %0, 128;" ::"r"(1 + gq) : "memory");  // stg, fac and sums are free again
      }
    }
    __syncthreads();  // the list is free again
  }
  // after an abort, let the copies still in flight land before the CTA exits
  if (threadIdx.x == 0 && *abort_flag) {
    const uint64_t t0 = global_ns();
    const int n = i1 - i0;
    for (int k = n > kRingSlots ? n - kRingSlots : 0; k < n; ++k)
      while (!mbar_try(&full[k % kRingSlots], (k / kRingSlots) & 1) && global_ns() - t0 < kWaitLimitNs) {
      }
  }
}

template <int D>
cudaError_t launch_ring(const AttnDecTcArgs& a, const CUtensorMap* tm, const int32_t* item_start, int grid,
                        cudaStream_t s) {
  static SmemOptIn opt;
  constexpr int smem = RingSmem<D>::kTotal;
  cudaError_t e = opt.ensure(k_attn_decode_ring<D>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRingThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // older chunks' copies overlap the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attn_decode_ring<D>, *tm, a, item_start);
}

}  // namespace

cudaError_t launch_attn_decode_ring(const AttnDecTcArgs& a, const void* tm_kv, const int32_t* item_start, int grid,
                                    cudaStream_t s) {
  const CUtensorMap* tm = reinterpret_cast<const CUtensorMap*>(tm_kv);
  switch (a.at.dims.D) {
    case 32: return launch_ring<32>(a, tm, item_start, grid, s);
    case 64: return launch_ring<64>(a, tm, item_start, grid, s);
    case 128: return launch_ring<128>(a, tm, item_start, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

bool attn_decode_tc_eligible(const Dims& dm) {
  return dm.H == 2 * dm.Hkv && (dm.D == 32 || dm.D == 64 || dm.D == 128) && dm.B == 16;
}

}  // namespace dec
