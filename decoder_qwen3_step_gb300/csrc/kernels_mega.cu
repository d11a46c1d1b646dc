// kernels_mega.cu - one serving-mode decode step (bf16 weights, f16 KV cache,
// at most 8 sequences, one new token each) as a single persistent kernel.
//
// The step is the decoder forward of tinyllm L10.1 "Candle model runner ...",
// section 2.4 (RMSNorm, Q/K/V, QK-norm, split-half RoPE, cache append, causal
// GQA attention, O projection and residual, RMSNorm, SwiGLU, down projection
// and residual; final RMSNorm, tied LM head, greedy argmax) at one token per
// sequence, with the Qwen3 switches of octlm "A real model in our own
// decoder".
//
// Why one kernel: at decode batch sizes each weight product streams a few
// megabytes, about a microsecond of HBM time, so a step of ~170 dependent
// launches is bound by launch and ramp latency.  Here one CTA per SM lives
// for the whole step.
//
// Weight and key streaming.  A loader warp walks the CTA's fixed schedule of
// weight tiles (up to 16 rows x 1024 k of bf16) and past-key tiles (64 cached
// keys and values of one KV head) and streams them with bulk asynchronous
// copies into a byte-addressed ring in shared memory: a tile takes exactly
// its bytes, so the loader can run as far ahead as the ring holds.  Weights
// and past keys never depend on the step, so the stream crosses stage
// boundaries freely.
//
// Hand-offs between CTAs.  A stage's output that other CTAs read (q|k|v
// rows, attention output, x * gain, SwiGLU output, sums of squares) goes to a
// plain buffer; after writing, each CTA adds one to a step-wide counter with
// release semantics, and a CTA starting the next stage has one thread wait
// (acquire) until every CTA has arrived, the others parked at a CTA barrier,
// then loads the whole input in one round trip.  Per-chunk attention records
// are counted per (sequence, KV head) instead, so only the CTA merging a pair
// waits for its chunks.  One polling thread per CTA keeps the waits from
// flooding L2, which the weight stream shares.  The two RMSNorm inputs of a
// layer use separate buffers.
//
// Products: warp-level bf16 MMA (m16n8k16, fp32 accumulation) with weight
// rows as M and tokens as N: a CTA owns about 27 rows of a 4096-row product,
// far below the 64/128-row tiles of tcgen05, and the step is bound by HBM and
// latency, not by MMA throughput.  Attention: each 64-key chunk is folded by
// four warps, 16 keys each, S = Q K^T and O = P V on the f16 tensor cores
// (queries and probabilities rounded to f16, the cache's own type), the
// softmax in fp32; every chunk leaves one record, and the CTA that folded a
// (sequence, KV head)'s last chunk merges its records in chunk order with all
// its threads.
//
// Every reduction runs in one order fixed by the shapes and the grid, so a
// sequence's logits are the same bits alone or in a batch.  The RMSNorm ahead
// of a product is split: the producer of x writes x * gain (bf16) and a
// per-CTA partial sum of x^2; the consumer forms 1/rms from the partials in
// CTA order and scales its output rows.  Layer 0's input is the embedding,
// which every CTA gathers itself.
#include <cuda_runtime.h>
#include <math.h>

#include "attn_fold.cuh"
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

namespace {

constexpr int kCW = kMegaComputeWarps;  // compute warps
constexpr int kCT = kCW * 32;           // compute threads
constexpr int kThreads = kCT + 32;      // + the loader warp
constexpr int kRows = 16;               // weight rows per tile (the MMA's M)
constexpr int kKS = kMegaKSlice;        // k elements per tile
constexpr int kKeys = kMegaKeys;        // keys per attention tile
constexpr int kNB = kMegaTiles;         // tile descriptors of the ring
constexpr int kGroups = kCW / 4;        // attention: groups of four warps
constexpr int kMaxT = kMegaMaxTokens;
constexpr int kSubStamps = 284;         // trace: first stamp of layer 1's sub-stage points (5 per stage)
constexpr int kLoadStamps = 310;        // trace: loader issue of layer 1's stages' first tiles, then layer 2's QKV

static_assert(kCW % 4 == 0 && kCT % 128 == 0, "attention groups are four warps; merges run parts of D threads");
static_assert(kMaxT <= 8, "the token rows form one 8-column MMA tile");

enum { P_QKV = 0, P_RESID = 1, P_SWIGLU = 2, P_LOGITS = 3 };

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }
// AND of a flag over the compute threads; every one gets the same answer.
__device__ __forceinline__ bool cbar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kCT)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void gbar(int g) { asm volatile("bar.sync %0, 128;" ::"r"(2 + g) : "memory"); }
__device__ __forceinline__ bool gbar_and(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(2 + g)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(x));
  const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  return lo | (hi << 16);
}
__device__ __forceinline__ uint32_t ld_acquire(const unsigned int* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// One thread waits until *p >= target (acquire).  Gives up, raising the
// CTA's abort flag, when any CTA of the launch gave up or after the wait
// limit (then also the launch's abort word and the device error word).
__device__ __forceinline__ bool wait_count(const unsigned int* p, unsigned int target, volatile int* abort_s,
                                        unsigned int* abort_g, uint32_t* err, uint64_t limit = kWaitLimitNs) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(p) >= target) return true;
    if ((it & 7) == 7) {
      if (*abort_s || *reinterpret_cast<volatile unsigned int*>(abort_g)) {
        *abort_s = 1;
        return false;
      }
      if (global_ns() - t0 > limit) {
        *abort_s = 1;
        atomicOr(abort_g, 1u);
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

// ---- warp-level MMA ---------------------------------------------------------------
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Units [u0, u1) of `units` that CTA b of P owns (contiguous, sizes differ by
// at most one).  The loader and the compute warps use the same split.
__device__ __forceinline__ void share(int units, int P, int b, int& u0, int& u1) {
  u0 = (int)(((long long)units * b) / P);
  u1 = (int)(((long long)units * (b + 1)) / P);
}

// Rows of the product stages: QKV rows one by one; the O and down
// projections by pairs of d (the same pairs, so each CTA owns the residual
// rows it updates, and a bf16 pair word has one writer); gate/up by groups
// of 16 interleaved rows (8 gate, 8 up).
constexpr int kGranQkv = 1, kGranResid = 2, kGranGu = 2 * kGuGroup, kGranHead = 1;

// Attention work item i of a layer: (sequence, KV head, 64-key chunk).  Items
// run sequence-major, then KV head, then chunk; CTA b takes a contiguous range.
struct Item {
  int s, g, c, nch;
};
__device__ __forceinline__ void next_item(const MegaArgs& a, Item& it) {
  if (++it.c < it.nch) return;
  it.c = 0;
  if (++it.g < a.Hkv) return;
  it.g = 0;
  if (++it.s < a.T) it.nch = (__ldg(a.seq_ctx + it.s) + kKeys - 1) / kKeys;
}
__device__ __forceinline__ Item item_of(const MegaArgs& a, int i) {
  int s = 0;
  while (s + 1 < a.T && __ldg(a.item_start + s + 1) <= i) ++s;
  const int nch = (__ldg(a.seq_ctx + s) + kKeys - 1) / kKeys;
  const int rem = i - __ldg(a.item_start + s);
  return {s, rem / nch, rem % nch, nch};
}
// The CTA's items cut into kGroups contiguous parts (one per group of four
// warps).  The loader issues the parts' tiles round robin, so every group has
// tiles in flight.  Part q of CTA b: items [first, first + len).
__device__ __forceinline__ void attn_part(int n_items, int P, int b, int q, int& first, int& len) {
  int i0, i1, j0, j1;
  share(n_items, P, b, i0, i1);
  share(i1 - i0, kGroups, q, j0, j1);
  first = i0 + j0;
  len = j1 - j0;
}
// Ring position (from the first attention tile) of the k-th item of part q,
// given every part's length.
__device__ __forceinline__ int attn_pos(const int* plen, int q, int k) {
  int p = 0;
#pragma unroll
  for (int r = 0; r < kGroups; ++r) p += min(plen[r], k) + (r < q && plen[r] > k ? 1 : 0);
  return p;
}

// Per attention group: roped queries, per-warp softmax states.
template <int D>
struct GroupScr {
  __half q[2][D];     // the group's two query heads, f16 (MMA rows 0 and 1)
  float m[4][2], l[4][2];
  float o[4][2][D];   // per warp, per head: probability-weighted values
};
template <int D>
__host__ __device__ constexpr int group_scr_bytes() {
  return (int)((sizeof(GroupScr<D>) + 127) / 128 * 128);
}
template <int D>
__host__ __device__ constexpr int scr_bytes() {
  const int attn = kGroups * group_scr_bytes<D>();
  const int prod = 2 * kCW * 128 * 4;                 // two halves of 16 partial tiles
  const int merge = (kCT * 4 + 2 * D) * 4;            // per-thread states, merged values
  return attn > prod ? (attn > merge ? attn : merge) : (prod > merge ? prod : merge);
}

// Shared memory of one CTA.
struct Smem {
  uint8_t* ring;
  uint8_t* stage;              // [T][K*2+16] the product's input rows (bf16)
  float* scr;                  // union: partial tiles | group scratch | merge scratch
  float* rstd;                 // [8]
  unsigned long long* best;    // [8]
  float* sq;                   // [8][16]
  int* flags;                  // [0] abort, [1] tiles issued (at the loader's end), [2] tiles claimed
  __half* zrow;                // [D] zeros (MMA rows 2..15 of the queries)
  uint64_t* full;              // [kNB]
  uint64_t* empty;             // [kNB]
  uint32_t* toff;              // [kNB] ring offset of each tile in flight
  uint32_t* vstart;            // [kNB] (loader) virtual ring position of each tile in flight
  Item* start;                 // [kGroups + 1] first item of each group, then of the CTA
  int* plen;                   // [kGroups + 1] items of each group, then of the CTA
};
constexpr int kSmallBytes = 32 + 64 + 512 + 64 + 256;  // rstd, best, sq, flags, zrow
constexpr int kBarBytes = kNB * (8 + 8 + 4 + 4) + (kGroups + 1) * ((int)sizeof(Item) + 4);

// A compute warp's wait for ring tile n.  A parity test only tells the
// barrier's current phase from the one before: while tile n - kNB (the
// previous use of the same barrier) is still landing, the test for tile n
// passes on the phase before that.  So after the wait, the loader's claim
// count must show tile n as claimed (its claim waited for the release of
// tile n - kNB); if not, wait for the claim and then for the tile again.
__device__ __noinline__ bool tile_rewait(const Smem& sm, uint32_t n, uint32_t* err) {  // the rare path, kept out of line
  volatile int* claimed = sm.flags + 2;
  const uint64_t t0 = global_ns();
  while ((uint32_t)*claimed <= n) {
    if (*(volatile int*)sm.flags) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *(volatile int*)sm.flags = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
  return mbar_wait(&sm.full[n % kNB], (n / kNB) & 1, sm.flags, err);
}
__device__ __forceinline__ bool tile_wait(const Smem& sm, uint32_t n, uint32_t* err) {
  if (!mbar_wait(&sm.full[n % kNB], (n / kNB) & 1, sm.flags, err)) return false;
  if ((uint32_t) * (volatile int*)(sm.flags + 2) > n) return true;
  return tile_rewait(sm, n, err);
}

// ---------------------------------------------------------------------------
// The loader warp: the CTA's tiles in the order the compute warps take them.
// ---------------------------------------------------------------------------
template <int D>
__device__ void loader(const MegaArgs& a, const Smem& sm, int b, int P) {
  const int lane = threadIdx.x & 31;
  const uint32_t R = (uint32_t)a.ring;
  volatile int* abort_s = sm.flags;
  uint32_t n = 0;              // tiles issued
  uint32_t k_old = 0;          // oldest tile not known to be released (lane 0)
  uint32_t vhead = 0;          // virtual ring position of the next tile (lane 0)
  // Reserve `foot` ring bytes for tile n, arm its barrier for `tx` bytes;
  // the ring offset, or -1 on abort (warp-uniform).
  auto claim = [&](uint32_t foot, uint32_t tx, uint32_t align) -> int {
    int off = -1;
    if (lane == 0) {
      uint32_t v = (vhead + align - 1) / align * align;
      if (v % R + foot > R) v = (v / R + 1) * R;  // never wrap inside a tile
      bool ok = true;
      while (k_old < n && (n - k_old >= (uint32_t)kNB || v + foot > sm.vstart[k_old % kNB] + R)) {
        if (!mbar_wait(&sm.empty[k_old % kNB], (k_old / kNB) & 1, abort_s, a.err)) {
          ok = false;
          break;
        }
        ++k_old;
      }
      if (ok) {
        sm.vstart[n % kNB] = v;
        vhead = v + foot;
        off = (int)(v % R);
        sm.toff[n % kNB] = (uint32_t)off;
        mbar_expect_tx(&sm.full[n % kNB], tx);
        *(volatile int*)(sm.flags + 2) = (int)(n + 1);  // tiles claimed (tile_wait)
      }
    }
    return __shfl_sync(0xffffffffu, off, 0);
  };
  // This CTA's rows of a product: contiguous in HBM (rows x K bf16).
  auto rows_of = [&](int K, int Rr, int gran, int& r0, int& nrows) {
    int u0, u1;
    share(Rr / gran, P, b, u0, u1);
    r0 = u0 * gran;
    nrows = (u1 - u0) * gran;
  };
  int ls = -1;  // trace: stamp slot for this product's first tile (layer 1 only)
  auto lstamp = [&](int k) {
    if (a.trace && lane == 0 && k >= 0) a.trace[(size_t)b * kMegaTraceStride + k] = global_ns();
  };
  auto product = [&](const bf16* W, int K, int Rr, int gran) -> bool {
    int r0, nrows;
    rows_of(K, Rr, gran, r0, nrows);
    lstamp(ls);
    const int mt = (nrows + kRows - 1) / kRows, nks = (K + kKS - 1) / kKS;
    for (int ks = 0; ks < nks; ++ks) {
      const int kslice = min(kKS, K - ks * kKS), rs = kslice * 2 + 16;
      for (int m = 0; m < mt; ++m) {
        const int rows_here = min(kRows, nrows - m * kRows);
        const int off = claim((uint32_t)((rows_here * rs + 127) & ~127), (uint32_t)(rows_here * kslice * 2), 128u);
        if (off < 0) return false;
        if (lane < rows_here)
          bulk_g2s(sm.ring + off + lane * rs, W + (size_t)(r0 + m * kRows + lane) * K + (size_t)ks * kKS,
                   (uint32_t)kslice * 2, &sm.full[n % kNB]);
        __syncwarp();
        ++n;
      }
    }
    return true;
  };
  const uint32_t slab = 16 * D * 2;  // bytes of one block's keys (or values) of one KV head
  int maxlen = 0;
#pragma unroll
  for (int q = 0; q < kGroups; ++q) maxlen = max(maxlen, sm.plen[q]);
  const int QR = (a.H + 2 * a.Hkv) * D;
  bool ok = true;
  for (int l = 0; l < a.n_layers && ok; ++l) {
    const char* Lb = a.layers + (size_t)l * a.layer_stride;
    ls = l == 1 ? kLoadStamps : l == 2 ? kLoadStamps + 5 : -1;
    ok = product(reinterpret_cast<const bf16*>(Lb + a.o_wqkv), a.d, QR, kGranQkv);
    lstamp(l == 1 ? kLoadStamps + 1 : -1);
    Item cur[kGroups];
#pragma unroll
    for (int q = 0; q < kGroups; ++q) cur[q] = sm.start[q];
    for (int k = 0; k < maxlen && ok; ++k) {
#pragma unroll
      for (int q = 0; q < kGroups; ++q) {
        if (!ok || k >= sm.plen[q]) continue;
        const Item it = cur[q];
        next_item(a, cur[q]);
        const int ctx = __ldg(a.seq_ctx + it.s);
        const int nb = (min(kKeys, ctx - it.c * kKeys) + 15) / 16;
        const int off = claim(2 * (kKeys / 16) * slab, 2 * nb * slab, 1024u);
        if (off < 0) {
          ok = false;
          continue;
        }
        // lane = (K or V, block, box): one 16-row box each
        constexpr int kB = KvSlab<D>::kBoxes;
        if (lane < 2 * nb * kB) {
          const int bx = lane % kB, j = (lane / kB) % nb, is_v = lane / (kB * nb);
          const int blk = table_block(a.tables, it.s, it.c * (kKeys / 16) + j, a.max_blocks, a.n_blocks, a.err);
          const int row = (((l * a.n_blocks + blk) * 2 + is_v) * a.Hkv + it.g) * 16;
          tma_load_2d(sm.ring + off + (is_v * (kKeys / 16) + j) * slab + bx * KvSlab<D>::kBoxBytes, &a.tm_kv,
                      bx * KvSlab<D>::kBoxDims, row, &sm.full[n % kNB]);
        }
        __syncwarp();
        ++n;
      }
    }
    if (!ok) break;
    ls = l == 1 ? kLoadStamps + 2 : -1;
    ok = product(reinterpret_cast<const bf16*>(Lb + a.o_wo), a.H * D, a.d, kGranResid);
    ls = l == 1 ? kLoadStamps + 3 : -1;
    ok = ok && product(reinterpret_cast<const bf16*>(Lb + a.o_wgu), a.d, 2 * a.F, kGranGu);
    ls = l == 1 ? kLoadStamps + 4 : -1;
    ok = ok && product(reinterpret_cast<const bf16*>(Lb + a.o_wd), a.F, a.d, kGranResid);
  }
  if (ok) product(a.embed, a.d, a.vocab, kGranHead);
  if (lane == 0) sm.flags[1] = (int)n;
  if (lane == 0 && a.trace) a.trace[(size_t)b * kMegaTraceStride + kMegaTraceStride - 1] = global_ns();
}

// ---------------------------------------------------------------------------
// The compute warps.
// ---------------------------------------------------------------------------
template <int D>
struct Flow {
  static constexpr int kDim = D / 32;  // head dims per lane
  const MegaArgs& a;
  const Smem& sm;
  int b, P, T;
  int ctid, warp, lane;
  uint32_t tile;   // next ring tile
  uint32_t nsync;  // sync points this CTA has arrived at
  int sub = -1;    // trace: first sub-stage stamp slot of this stage (layer 1 only), else -1

  __device__ Flow(const MegaArgs& a_, const Smem& sm_, int b_, int P_)
      : a(a_), sm(sm_), b(b_), P(P_), T(a_.T), ctid(threadIdx.x), warp(threadIdx.x >> 5), lane(threadIdx.x & 31),
        tile(0), nsync(0) {}

  __device__ void stamp(int k) const {
    if (a.trace && ctid == 0 && k < kMegaTraceStride - 1) a.trace[(size_t)b * kMegaTraceStride + k] = global_ns();
  }
  __device__ void substamp(int i) const {
    if (sub >= 0) stamp(sub + i);
  }

  // This CTA's outputs of the stage are written: count it in (every compute
  // thread calls this).
  __device__ void arrive() {
    cbar();
    if (ctid == 0) red_release(a.sync, 1u);
    ++nsync;
  }
  // Wait until every CTA has arrived at this CTA's latest sync point.  Every
  // compute thread returns the same answer (false: gave up).
  __device__ bool wait_all() const {
    bool ok = true;
    if (ctid == 0) ok = wait_count(a.sync, nsync * (uint32_t)P + a.wait_extra, sm.flags, a.abort, a.err, a.wait_limit);
    return cbar_and(ok);
  }

  // Wait for the previous stage, then stage a product's input: T rows of K
  // bf16 from src [T, K] into the staging rows (stride K*2+16 bytes), and,
  // when ssq is given, 1/rms of every row from the per-CTA partial sums
  // ssq [T, grid] (added lane-strided in CTA order, then across the warp).
  __device__ bool pull(const bf16* src, int K, const float* ssq) {
    if (!wait_all()) return false;
    const int SR = K * 2 + 16, nv = K / 8, nvec = T * nv;
    constexpr int kSk = kMegaMaxGrid / 32, kU = 4;
    if (ssq != nullptr && warp < T) {
      const float* row = ssq + (size_t)warp * kMegaMaxGrid;
      float v[kSk];
#pragma unroll
      for (int k = 0; k < kSk; ++k) v[k] = lane + 32 * k < P ? __ldcg(row + lane + 32 * k) : 0.f;
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < kSk; ++k) s += v[k];
      s = warp_sum(s);
      if (lane == 0) sm.rstd[warp] = 1.0f / sqrtf(s / (float)a.d + a.eps);
    }
    for (int v0 = 0; v0 < nvec; v0 += kCT * kU) {
      uint4 w[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = v0 + ctid + j * kCT;
        if (i < nvec) w[j] = __ldcg(reinterpret_cast<const uint4*>(src) + i);
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = v0 + ctid + j * kCT;
        if (i < nvec) {
          const int t = i / nv, vv = i - t * nv;
          *reinterpret_cast<uint4*>(sm.stage + (size_t)t * SR + vv * 16) = w[j];
        }
      }
    }
    cbar();
    return true;
  }

  // x = E[id] of every token, gathered by this CTA itself: the staging rows
  // get x * (first gain) in bf16, rstd the full sum of x^2 (lane-strided
  // chunks of 8, then across the warp), X the rows this CTA owns.
  __device__ void embed() {
    const int d = a.d, SR = d * 2 + 16;
    int u0, u1;
    share(d / kGranResid, P, b, u0, u1);
    const int e0 = u0 * kGranResid, e1 = u1 * kGranResid;
    if (warp < T) {
      const int t = warp;
      int id = __ldg(a.ids + t);
      if (id < 0 || id >= a.vocab) {
        if (lane == 0 && b == 0) atomicOr(a.err, kErrBadId);
        id = 0;
      }
      const bf16* E = a.embed + (size_t)id * d;
      float s = 0.f;
      for (int k = lane * 8; k < d; k += 256) {
        float x[8];
        load8(E + k, x);
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s = fmaf(x[i], x[i], s);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          pk[i] = pack_bf16(x[2 * i] * a.w_attn0[k + 2 * i], x[2 * i + 1] * a.w_attn0[k + 2 * i + 1]);
        *reinterpret_cast<uint4*>(sm.stage + (size_t)t * SR + k * 2) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (k + i >= e0 && k + i < e1) a.X[(size_t)t * d + k + i] = x[i];
      }
      s = warp_sum(s);
      if (lane == 0) sm.rstd[t] = 1.0f / sqrtf(s / (float)d + a.eps);
    }
    cbar();
  }

  // y of (tile q of the group, row r, token t): the group's k-range partials in order.
  __device__ float ysum(int half, int q, int krpt, int r, int t) const {
    const float* p = sm.scr + ((size_t)(half * kCW + q * krpt)) * 128 + r * 8 + t;
    float y = 0.f;
    for (int kr = 0; kr < krpt; ++kr) y += p[kr * 128];
    return y;
  }

  struct Out {
    void* y;                // P_QKV: raw (f32); P_RESID: x * next gain (bf16); P_SWIGLU: act (bf16)
    float* ssq;             // P_RESID: per-CTA partial sums (this CTA's column)
    const float* w_next;    // P_RESID: the next RMSNorm's gain
  };

  // One weight product over this CTA's rows, input staged, with its fused
  // epilogue.  Tiles go two at a time (half the warps each) or one at a
  // time; a warp takes one (tile, k range) and, for inputs wider than one
  // slice, the same range of every slice.  The epilogue adds a tile's k-range
  // partials in order, so a row's result does not depend on the number of
  // tokens.
  template <int EPI>
  __device__ bool product(const bf16* W, int K, int R, int gran, Out o) {
    int u0, u1;
    share(R / gran, P, b, u0, u1);
    const int r0 = u0 * gran, nrows = (u1 - u0) * gran;
    const int mt = (nrows + kRows - 1) / kRows, nks = (K + kKS - 1) / kKS;
    const int SR = K * 2 + 16;
    const uint32_t st_s = smem_u32(sm.stage);
    if (EPI == P_LOGITS && ctid < T) sm.best[ctid] = 0ull;
    // RESID: this thread's residual pair (fetched while the tiles land)
    float2 xres = make_float2(0.f, 0.f);
    if (EPI == P_RESID && ctid < 8 * T && 2 * (ctid & 7) < nrows)
      xres = *reinterpret_cast<const float2*>(a.X + (size_t)(ctid >> 3) * a.d + r0 + 2 * (ctid & 7));
    int half = 0;
    for (int m = 0; m < mt;) {
      const int tp = mt - m >= 2 ? 2 : 1, krpt = kCW / tp;
      const int q = warp / krpt, kr = warp - q * krpt;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      bool got = true;
      const int rows_here = min(kRows, nrows - (m + q) * kRows);
      int ar = lane & 15;
      if (ar >= rows_here) ar = 0;  // rows past the tile read row 0; their results are dropped
      int bt = lane & 7;
      if (bt >= T) bt = 0;          // token columns past T likewise
      for (int ks = 0; ks < nks; ++ks) {
        const int kslice = min(kKS, K - ks * kKS), rs = kslice * 2 + 16, nsteps = kslice / 16;
        const uint32_t n = tile + ks * mt + m + q;
        if (!tile_wait(sm, n, a.err)) {
          got = false;
          break;
        }
        if (m == 0 && ks == 0) substamp(0);
        const int st0 = kr * nsteps / krpt, st1 = (kr + 1) * nsteps / krpt;
        const uint32_t a_addr = smem_u32(sm.ring + sm.toff[n % kNB]) + ar * rs + (lane >> 4) * 16 + st0 * 32;
        const uint32_t b_addr = st_s + bt * SR + ((lane >> 3) & 1) * 16 + (ks * kKS + st0 * 16) * 2;
        // four k steps' fragments loaded together, their MMAs on four
        // accumulators (added in a fixed order at the end)
        const int cnt = st1 - st0;
        float c4[4][4] = {};
        int st = 0;
#pragma unroll 2
        for (; st + 4 <= cnt; st += 4) {
          uint32_t A[4][4], B[4][2];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            ldsm4(a_addr + (st + j) * 32, A[j]);
            ldsm2(b_addr + (st + j) * 32, B[j]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) mma_bf16(c4[j], A[j], B[j][0], B[j][1]);
        }
        for (; st < cnt; ++st) {
          uint32_t A[4], B[2];
          ldsm4(a_addr + st * 32, A);
          ldsm2(b_addr + st * 32, B);
          mma_bf16(c4[0], A, B[0], B[1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += (c4[0][e] + c4[1][e]) + (c4[2][e] + c4[3][e]);
      }
      if (m == 0) substamp(1);
      {
        float* red = sm.scr + (size_t)(half * kCW + warp) * 128;
        const int g = lane >> 2, c2 = (lane & 3) * 2;
        *reinterpret_cast<float2*>(red + g * 8 + c2) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2*>(red + (g + 8) * 8 + c2) = make_float2(acc[2], acc[3]);
      }
      if (!cbar_and(got)) return false;
      if (m == 0) substamp(2);
      if (ctid == 0)
        for (int ks = 0; ks < nks; ++ks)
          for (int qq = 0; qq < tp; ++qq) mbar_arrive(&sm.empty[(tile + ks * mt + m + qq) % kNB]);
      if (EPI == P_QKV) {
        float* y = reinterpret_cast<float*>(o.y);
        for (int i = ctid; i < tp * 16 * T; i += kCT) {
          const int r = i & 15, rest = i >> 4, t = rest % T, qq = rest / T;
          const int row = (m + qq) * kRows + r;
          if (row < nrows) y[(size_t)t * R + r0 + row] = ysum(half, qq, krpt, r, t) * sm.rstd[t];
        }
      } else if (EPI == P_RESID) {  // one tile (at most 16 rows), pairs of rows
        if (ctid < 8 * T) {
          const int pr = ctid & 7, t = ctid >> 3, r = 2 * pr;
          float x0 = 0.f, x1 = 0.f;
          if (r < nrows) {
            const size_t off = (size_t)t * a.d + r0 + r;
            x0 = xres.x + ysum(half, 0, krpt, r, t);
            x1 = xres.y + ysum(half, 0, krpt, r + 1, t);
            *reinterpret_cast<float2*>(a.X + off) = make_float2(x0, x1);
            *reinterpret_cast<uint32_t*>(reinterpret_cast<bf16*>(o.y) + off) =
                pack_bf16(x0 * o.w_next[r0 + r], x1 * o.w_next[r0 + r + 1]);
          }
          sm.sq[t * 16 + r] = x0 * x0;
          sm.sq[t * 16 + r + 1] = x1 * x1;
        }
      } else if (EPI == P_SWIGLU) {  // a tile is one group: 8 gate rows, then the 8 up rows
        bf16* y = reinterpret_cast<bf16*>(o.y);
        for (int i = ctid; i < tp * 4 * T; i += kCT) {
          const int pr = i & 3, rest = i >> 2, t = rest % T, qq = rest / T, j = 2 * pr;
          const float rs = sm.rstd[t];
          const float g0 = ysum(half, qq, krpt, j, t) * rs, g1 = ysum(half, qq, krpt, j + 1, t) * rs;
          const float v0 = ysum(half, qq, krpt, j + kGuGroup, t) * rs, v1 = ysum(half, qq, krpt, j + 1 + kGuGroup, t) * rs;
          const int grp = (r0 + (m + qq) * kRows) / (2 * kGuGroup);
          *reinterpret_cast<uint32_t*>(y + (size_t)t * a.F + grp * kGuGroup + j) = pack_bf16(silu(g0) * v0, silu(g1) * v1);
        }
      } else {  // P_LOGITS: 16 consecutive threads hold the 16 rows of one (tile, token)
        const int n_i = tp * 16 * T;
        for (int i0 = 0; i0 < n_i; i0 += kCT) {  // whole warps in every round (shuffles)
          const int i = i0 + ctid, r = i & 15, rest = i >> 4, t = rest % T, qq = rest / T;
          const int row = (m + qq) * kRows + r;
          unsigned long long key = 0ull;
          if (i < n_i && row < nrows) {
            const float v = ysum(half, qq, krpt, r, t) * sm.rstd[t];
            if (a.logits) a.logits[(size_t)t * a.vocab + r0 + row] = v;
            key = argmax_key(v, r0 + row);
          }
#pragma unroll
          for (int x = 8; x >= 1; x >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, x);
            key = other > key ? other : key;
          }
          if (i < n_i && r == 0 && key) atomicMax(&sm.best[t], key);
        }
      }
      if (m == 0) substamp(3);
      half ^= 1;
      m += tp;
    }
    tile += (uint32_t)(mt * nks);
    if (EPI == P_RESID) {
      // this CTA's partial sum of x^2 per token row (its rows in order; none: 0)
      cbar();
      if (ctid < T) {
        float s = 0.f;
        for (int r = 0; r < nrows; ++r) s += sm.sq[ctid * 16 + r];
        o.ssq[(size_t)ctid * kMegaMaxGrid + b] = s;
      }
    }
    if (EPI == P_LOGITS) {
      cbar();
      if (ctid < T && sm.best[ctid]) atomicMax(a.keys + ctid, sm.best[ctid]);
    }
    return true;
  }

  // ---- attention ------------------------------------------------------------
  __device__ GroupScr<D>* group_scr(int gq) const {
    return reinterpret_cast<GroupScr<D>*>(reinterpret_cast<uint8_t*>(sm.scr) + gq * group_scr_bytes<D>());
  }

  // Row `row` of token t's q|k|v (D values) after QK-norm and RoPE at
  // position pos (norm != null), else as written: this lane's kDim channels.
  // Whole warp.
  __device__ void head_row(int t, int row, const float* norm, int pos, float (&v)[kDim]) const {
    const int QR = (a.H + 2 * a.Hkv) * D, half = D / 2;
    const float* p = a.raw + (size_t)t * QR + row + lane * kDim;
    if constexpr (kDim == 4) {
      const float4 u = __ldcg(reinterpret_cast<const float4*>(p));
      v[0] = u.x;
      v[1] = u.y;
      v[2] = u.z;
      v[3] = u.w;
    } else if constexpr (kDim == 2) {
      const float2 u = __ldcg(reinterpret_cast<const float2*>(p));
      v[0] = u.x;
      v[1] = u.y;
    } else {
      v[0] = __ldcg(p);
    }
    if (norm) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < kDim; ++e) ss = fmaf(v[e], v[e], ss);
      const float rn = 1.0f / sqrtf(warp_sum(ss) / (float)D + a.eps);
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

  // Warp gw folds block gw (16 keys) of a tile for both query heads of its
  // group on the f16 tensor cores (fold16): (max, sum) and O per head to the
  // group scratch.
  __device__ void fold(GroupScr<D>* gs, const __half* Ks, const __half* Vs, int keys_here) {
    const int gw = warp & 3;
    fold16<D>(gs->q[0], gs->q[1], sm.zrow, reinterpret_cast<const uint8_t*>(Ks + gw * 16 * D),
              reinterpret_cast<const uint8_t*>(Vs + gw * 16 * D), min(16, keys_here - gw * 16), a.scale,
              &gs->o[gw][0][0], gs->m[gw], gs->l[gw]);
  }

  // The chunk's record: the four warps' states merged in warp order, per
  // head (max, sum, values).
  __device__ void write_record(GroupScr<D>* gs, int s, int g, int c) {
    const int ltid = ctid & 127, hp = (D + 2) / 2;
    float* rec = a.rec + ((size_t)(s * a.Hkv + g) * a.nch_cap + c) * (2 * (D + 2));
    for (int pidx = ltid; pidx < 2 * hp; pidx += 128) {
      const int h = pidx / hp, j = pidx - h * hp;
      float M = gs->m[0][h];
#pragma unroll
      for (int w = 1; w < 4; ++w) M = fmaxf(M, gs->m[w][h]);
      float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float f = gs->m[w][h] == -INFINITY ? 0.f : expf(gs->m[w][h] - M);
        L = fmaf(gs->l[w][h], f, L);
        if (j > 0) {
          o0 = fmaf(gs->o[w][h][2 * j - 2], f, o0);
          o1 = fmaf(gs->o[w][h][2 * j - 1], f, o1);
        }
      }
      *reinterpret_cast<float2*>(rec + h * (D + 2) + 2 * j) = j == 0 ? make_float2(M, L) : make_float2(o0, o1);
    }
  }

  // Merge every chunk record of (sequence s, KV head g) once all nch of this
  // layer's are counted, and write the two heads' attention output.  All
  // compute threads: thread = (part, head, dim); each part runs the online
  // softmax merge over chunks part, part + parts, ... in order, then the
  // parts are merged in order.
  __device__ bool merge(int s, int g, int nch, int l) {
    constexpr int kSlots = D, kParts = kCT / kSlots, kB = 8;  // slot = (head, pair of dims)
    bool ok = true;
    if (ctid == 0)
      ok = wait_count(a.acnt + s * a.Hkv + g, (uint32_t)((l + 1) * nch), sm.flags, a.abort, a.err);
    if (!cbar_and(ok)) return false;
    const int slot = ctid % kSlots, part = ctid / kSlots, h = slot / (D / 2), dd = 2 * (slot - h * (D / 2));
    const float* base = a.rec + ((size_t)(s * a.Hkv + g) * a.nch_cap) * (2 * (D + 2)) + h * (D + 2);
    float m = -INFINITY, ls = 0.f, o0 = 0.f, o1 = 0.f;
    for (int c0 = part; c0 < nch; c0 += kParts * kB) {
      float2 ml[kB], ov[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int c = c0 + kParts * j;
        if (c < nch) {
          const float* p = base + (size_t)c * (2 * (D + 2));
          ml[j] = __ldcg(reinterpret_cast<const float2*>(p));
          ov[j] = __ldcg(reinterpret_cast<const float2*>(p + 2 + dd));
        }
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int c = c0 + kParts * j;
        if (c < nch) {
          const float Mc = ml[j].x, Lc = ml[j].y;
          if (Mc > m) {
            const float f = expf(m - Mc);
            ls = fmaf(ls, f, Lc);
            o0 = fmaf(o0, f, ov[j].x);
            o1 = fmaf(o1, f, ov[j].y);
            m = Mc;
          } else {
            const float f = expf(Mc - m);
            ls = fmaf(Lc, f, ls);
            o0 = fmaf(ov[j].x, f, o0);
            o1 = fmaf(ov[j].y, f, o1);
          }
        }
      }
    }
    float* st = sm.scr;  // [kParts][kSlots][4], then the merged values [2 * kSlots]
    float* outv = sm.scr + kCT * 4;
    *reinterpret_cast<float4*>(st + (part * kSlots + slot) * 4) = make_float4(m, ls, o0, o1);
    cbar();
    if (ctid < kSlots) {
      float4 acc = *reinterpret_cast<const float4*>(st + ctid * 4);
      for (int pp = 1; pp < kParts; ++pp) {
        const float4 q = *reinterpret_cast<const float4*>(st + (pp * kSlots + ctid) * 4);
        if (q.y == 0.f) continue;  // a part with no chunks
        if (q.x > acc.x) {
          const float f = expf(acc.x - q.x);
          acc = make_float4(q.x, fmaf(acc.y, f, q.y), fmaf(acc.z, f, q.z), fmaf(acc.w, f, q.w));
        } else {
          const float f = expf(q.x - acc.x);
          acc = make_float4(acc.x, fmaf(q.y, f, acc.y), fmaf(q.z, f, acc.z), fmaf(q.w, f, acc.w));
        }
      }
      // features (2g + h) * D + dd, dd + 1 of the sequence's row
      const int hh = ctid / (D / 2), d2 = 2 * (ctid - hh * (D / 2));
      *reinterpret_cast<uint32_t*>(a.att + (size_t)s * (a.H * D) + (size_t)(2 * g + hh) * D + d2) =
          pack_bf16(acc.z / acc.y, acc.w / acc.y);
    }
    cbar();  // the scratch is read again by the next merge
    (void)outv;
    return true;
  }

  // Attention of layer l over this CTA's items.  Group gq of four warps takes
  // its part of the CTA's contiguous range of (sequence, KV head, 64-key
  // chunk) items.  Consecutive items of one (sequence, KV head) form a run:
  // the two queries are normed and rotated once per run, and the run's
  // records are counted in with one release-add.  The group holding a
  // sequence's last chunk also finishes the new key and value (QK-norm and
  // RoPE on the key), appends them to the cache and patches its tile.  Then
  // the CTA merges the pairs whose last chunk it folded.
  __device__ bool attention(int l) {
    const int gq = warp >> 2, gw = warp & 3, ltid = ctid & 127;
    if (!wait_all()) return false;  // every CTA's q|k|v rows are written
    const uint32_t tile0 = tile;
    const int mylen = sm.plen[gq], total = sm.plen[kGroups];
    GroupScr<D>* gs = group_scr(gq);
    const char* Lb = a.layers + (size_t)l * a.layer_stride;
    const float* q_norm = reinterpret_cast<const float*>(Lb + a.o_q_norm);
    const float* k_norm = reinterpret_cast<const float*>(Lb + a.o_k_norm);
    constexpr int kSlabElems = 16 * D;
    bool ok = true;
    int run = 0;  // chunks of the current run folded so far
    Item it = sm.start[gq];
    for (int k = 0; k < mylen; ++k, next_item(a, it)) {
      const uint32_t n = tile0 + attn_pos(sm.plen, gq, k);
      const int s = it.s, g = it.g, c = it.c;
      const int ctx = __ldg(a.seq_ctx + s), pos = ctx - 1;
      if ((k == 0 || c == 0) && gw < 2) {  // the run's queries
        float v[kDim];
        head_row(s, (2 * g + gw) * D, q_norm, pos, v);
#pragma unroll
        for (int e = 0; e < kDim; ++e) gs->q[gw][lane * kDim + e] = __float2half_rn(v[e]);
      }
      if (k == 0) substamp(0);
      bool wok = tile_wait(sm, n, a.err);
      if (k == 0) substamp(1);
      const int keys_here = min(kKeys, ctx - c * kKeys);
      __half* Ks = reinterpret_cast<__half*>(sm.ring + sm.toff[n % kNB]);
      __half* Vs = Ks + (kKeys / 16) * kSlabElems;
      if (c == it.nch - 1 && gw >= 2 && wok) {
        // the newest key (warp 2) and value (warp 3): append them to the cache
        // (f16, round to nearest even) and patch the tile
        const int is_v = gw == 3;
        float v[kDim];
        head_row(s, (is_v ? a.H + a.Hkv + g : a.H + g) * D, is_v ? nullptr : k_norm, pos, v);
        const int blk = table_block(a.tables, s, pos / 16, a.max_blocks, a.n_blocks, a.err);
        __half* dst = a.kv + kv_offset(l, blk, is_v, g, pos % 16, a.n_blocks, a.Hkv, 16, D);
        const int kk = pos - c * kKeys;
        __half hv[kDim];
#pragma unroll
        for (int e = 0; e < kDim; ++e) {
          hv[e] = __float2half_rn(v[e]);
          dst[lane * kDim + e] = hv[e];
        }
        // patch the tile; value rows past the context (the block's tail)
        // become zeros: P V must not meet NaN bits
        patch_row<D>(reinterpret_cast<uint8_t*>((is_v ? Vs : Ks) + (kk / 16) * kSlabElems), kk % 16, hv, is_v);
        // the slot is refilled by bulk copies later: order these stores before them
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      if (!gbar_and(gq, wok)) {
        ok = false;
        break;
      }
      fold(gs, Ks, Vs, keys_here);
      gbar(gq);
      if (k == 0) substamp(2);
      if (ltid == 0) mbar_arrive(&sm.empty[n % kNB]);  // the tile is no longer read
      write_record(gs, s, g, c);
      ++run;
      gbar(gq);  // the records are written; the scratch is free again
      if (k == 0) substamp(3);
      if (k + 1 == mylen || c + 1 == it.nch) {  // end of the run: count its chunks in
        if (ltid == 0) red_release(a.acnt + s * a.Hkv + g, (unsigned)run);
        run = 0;
      }
    }
    tile = tile0 + (uint32_t)total;
    if (!cbar_and(ok)) return false;
    // merges of the (sequence, KV head) pairs whose last chunk this CTA folded
    Item cur = sm.start[kGroups];
    for (int i = 0; i < total && ok; ++i, next_item(a, cur))
      if (cur.c == cur.nch - 1) ok = merge(cur.s, cur.g, cur.nch, l);
    substamp(4);
    return ok;
  }
};

// The compute warps' whole step.  Sync points per layer: q|k|v written,
// attention output written, O projection, gate/up, down projection.
template <int D>
__device__ void compute_main(const MegaArgs& a, const Smem& sm, int b, int P) {
  Flow<D> f(a, sm, b, P);
  const int L = a.n_layers, QR = (a.H + 2 * a.Hkv) * D, HD = a.H * D;
  using Out = typename Flow<D>::Out;
  f.stamp(0);
  f.embed();
  bool ok = true;
  for (int l = 0; l < L && ok; ++l) {
    const char* Lb = a.layers + (size_t)l * a.layer_stride;
    const float* w_next =
        l + 1 < L ? reinterpret_cast<const float*>(Lb + a.layer_stride + a.o_attn_norm) : a.final_norm;
    const int s0 = l * 5;
    auto sub = [&](int k) { f.sub = l == 1 ? kSubStamps + 5 * k : -1; };
    // RMSNorm + QKV (layer 0's input is the embedding this CTA gathered)
    if (l > 0) ok = f.pull(a.xa, a.d, a.sa);
    f.stamp(1 + 2 * s0);
    sub(0);
    ok = ok && f.template product<P_QKV>(reinterpret_cast<const bf16*>(Lb + a.o_wqkv), a.d, QR, kGranQkv,
                                         Out{a.raw, nullptr, nullptr});
    f.arrive();
    f.stamp(2 + 2 * s0);
    // attention
    f.stamp(3 + 2 * s0);
    sub(1);
    ok = ok && f.attention(l);
    f.arrive();
    f.stamp(4 + 2 * s0);
    // O projection + residual
    ok = ok && f.pull(a.att, HD, nullptr);
    f.stamp(5 + 2 * s0);
    sub(2);
    ok = ok && f.template product<P_RESID>(reinterpret_cast<const bf16*>(Lb + a.o_wo), HD, a.d, kGranResid,
                                           Out{a.xb, a.sb, reinterpret_cast<const float*>(Lb + a.o_mlp_norm)});
    f.arrive();
    f.stamp(6 + 2 * s0);
    // RMSNorm + gate/up + SiLU*mul
    ok = ok && f.pull(a.xb, a.d, a.sb);
    f.stamp(7 + 2 * s0);
    sub(3);
    ok = ok && f.template product<P_SWIGLU>(reinterpret_cast<const bf16*>(Lb + a.o_wgu), a.d, 2 * a.F, kGranGu,
                                            Out{a.act, nullptr, nullptr});
    f.arrive();
    f.stamp(8 + 2 * s0);
    // down projection + residual
    ok = ok && f.pull(a.act, a.F, nullptr);
    f.stamp(9 + 2 * s0);
    sub(4);
    ok = ok && f.template product<P_RESID>(reinterpret_cast<const bf16*>(Lb + a.o_wd), a.F, a.d, kGranResid,
                                           Out{a.xa, a.sa, w_next});
    f.arrive();
    f.stamp(10 + 2 * s0);
  }
  // final RMSNorm + tied LM head + argmax keys
  f.sub = -1;
  ok = ok && f.pull(a.xa, a.d, a.sa);
  f.stamp(1 + 2 * 5 * L);
  ok = ok && f.template product<P_LOGITS>(a.embed, a.d, a.vocab, kGranHead, Out{nullptr, nullptr, nullptr});
  f.stamp(2 + 2 * 5 * L);
  // the last CTA to finish turns the keys into ids
  cbar();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(a.done, 1u);
    if (prev == (unsigned)P - 1) {
      __threadfence();
      for (int t = 0; t < a.T; ++t) {
        const unsigned long long key = *reinterpret_cast<volatile unsigned long long*>(a.keys + t);
        a.argmax[t] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_decode_mega(const __grid_constant__ MegaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Smem sm;
  sm.ring = smem;
  sm.stage = smem + a.o_stage;
  sm.scr = reinterpret_cast<float*>(smem + a.o_scr);
  uint8_t* small = smem + a.o_small;
  sm.rstd = reinterpret_cast<float*>(small);
  sm.best = reinterpret_cast<unsigned long long*>(small + 32);
  sm.sq = reinterpret_cast<float*>(small + 96);
  sm.flags = reinterpret_cast<int*>(small + 608);
  sm.zrow = reinterpret_cast<__half*>(small + 672);
  uint8_t* bars = smem + a.o_bars;
  sm.full = reinterpret_cast<uint64_t*>(bars);
  sm.empty = sm.full + kNB;
  sm.toff = reinterpret_cast<uint32_t*>(sm.empty + kNB);
  sm.vstart = sm.toff + kNB;
  sm.start = reinterpret_cast<Item*>(sm.vstart + kNB);
  const int b = blockIdx.x, P = gridDim.x;
  sm.plen = reinterpret_cast<int*>(sm.start + kGroups + 1);
  if (threadIdx.x <= kGroups) {  // first attention item and item count of each group, then of the CTA
    const int n_items = __ldg(a.item_start + a.T), q = threadIdx.x;
    int first, len;
    if (q < kGroups) {
      attn_part(n_items, P, b, q, first, len);
    } else {
      int i1;
      share(n_items, P, b, first, i1);
      len = i1 - first;
    }
    sm.start[q] = len > 0 ? item_of(a, first) : Item{0, 0, 0, 1};
    sm.plen[q] = len;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNB; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 16; ++i) sm.flags[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < D; i += kThreads) sm.zrow[i] = __float2half_rn(0.f);
  __syncthreads();
  if (threadIdx.x >= kCT) {
    loader<D>(a, sm, b, P);
  } else {
    compute_main<D>(a, sm, b, P);
  }
  __syncthreads();
  // after an abort, let the copies still in flight land before the CTA
  // exits: the last kNB tiles issued are the only ones that can be
  if (threadIdx.x == 0) {
    const uint32_t issued = (uint32_t)sm.flags[1];
    const uint64_t t0 = global_ns();
    for (uint32_t n = issued > (uint32_t)kNB ? issued - kNB : 0u; n < issued; ++n)
      while (!mbar_try(&sm.full[n % kNB], (n / kNB) & 1) && global_ns() - t0 < kWaitLimitNs) {
      }
  }
}

template <int D>
cudaError_t configure(int smem) {
  static SmemOptIn opt;
  return opt.ensure(k_decode_mega<D>, smem);
}

template <int D>
cudaError_t launch_d(const MegaArgs& a, int grid, int smem, cudaStream_t s) {
  cudaError_t e = configure<D>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_mega<D>, a);
}

template <int D>
int scr_bytes_of() {
  return scr_bytes<D>();
}

}  // namespace

MegaSmem mega_smem(int T, int kmax, int D, int smem_limit) {
  MegaSmem s{};
  const int scr = D == 32 ? scr_bytes_of<32>() : D == 64 ? scr_bytes_of<64>() : scr_bytes_of<128>();
  const int rest = ((T * (kmax * 2 + 16) + 127) & ~127) + ((scr + 127) & ~127) + kSmallBytes + kBarBytes + 256;
  int ring = (smem_limit - rest) & ~1023;
  if (ring < kMegaMinRing) return s;
  s.ring = ring;
  int off = ring;
  s.o_stage = off;
  off += (T * (kmax * 2 + 16) + 127) & ~127;
  s.o_scr = off;
  off += (scr + 127) & ~127;
  s.o_small = off;
  off += (kSmallBytes + 127) & ~127;
  s.o_bars = off;
  off += kBarBytes;
  s.total = off;
  return s.total <= smem_limit ? s : MegaSmem{};
}

cudaError_t launch_decode_mega(const MegaArgs& a, int grid, int smem, cudaStream_t s) {
  switch (a.D) {
    case 32: return launch_d<32>(a, grid, smem, s);
    case 64: return launch_d<64>(a, grid, smem, s);
    case 128: return launch_d<128>(a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

int mega_threads() { return kThreads; }

bool mega_fits(int D, int smem) {
  int blocks = 0;
  cudaError_t e;
  switch (D) {
    case 32:
      e = configure<32>(smem);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_decode_mega<32>, kThreads, smem);
      break;
    case 64:
      e = configure<64>(smem);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_decode_mega<64>, kThreads, smem);
      break;
    case 128:
      e = configure<128>(smem);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_decode_mega<128>, kThreads, smem);
      break;
    default: return false;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return blocks >= 1;
}

}  // namespace dec
