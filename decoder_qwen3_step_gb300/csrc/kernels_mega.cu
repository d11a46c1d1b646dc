// kernels_mega.cu - one serving-mode decode step (bf16 weights, f16 KV cache,
// at most 32 sequences, one new token each) as a single persistent kernel.
//
// The step is the decoder forward of tinyllm L10.1 "Candle model runner ...",
// section 2.4 (RMSNorm, Q/K/V, QK-norm, split-half RoPE, cache append, causal
// GQA attention, O projection and residual, RMSNorm, SwiGLU, down projection
// and residual; final RMSNorm, tied LM head, greedy argmax) at one token per
// sequence.
//
// Why one kernel: at decode batch sizes each weight product streams a few
// megabytes, about a microsecond of HBM time, so a step of ~170 dependent
// launches is bound by launch and ramp latency rather than by HBM.  Here one
// CTA per SM lives for the whole step.  A loader warp walks the CTA's fixed
// schedule of weight tiles (16 rows x up to 1024 k of bf16) and past-key tiles
// (64 cached keys and values of one KV head) and streams them with bulk
// asynchronous copies into a ring of shared-memory slots.  Weights and past
// keys never depend on the step, so the loader runs ahead across stage
// boundaries while sixteen compute warps run the stages in order, with a
// grid-wide barrier between dependent stages:
//   embedding | per layer: RMSNorm + QKV | attention (QK-norm, RoPE, cache
//   append, split-K over 64-key chunks, in-order merge) | O-proj + residual |
//   RMSNorm + gate/up + SiLU*mul | down-proj + residual | final RMSNorm +
//   LM head + argmax.
// The weight products use the warp-level bf16 tensor-core MMA (m16n8k16,
// fp32 accumulation): a CTA owns about 27 rows of a 4096-row product, far
// below the 64/128-row tiles of tcgen05, and the step is bound by HBM, not by
// the MMA rate.  Every reduction runs in one fixed order that does not depend
// on the batch, so a sequence's logits are the same in any batch.
//
// The RMSNorm ahead of a product is split as in the layered kernels: the
// producer of x writes x * gain (bf16) as the product's input and per-CTA
// partial sums of x^2; the consumer turns the partials into 1/rms (fixed
// order) and scales its output rows.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace dec {

namespace {

constexpr int kCW = kMegaComputeWarps;  // compute warps
constexpr int kCT = kCW * 32;           // compute threads (512)
constexpr int kThreads = kCT + 32;      // + the loader warp
constexpr int kRows = 16;               // weight rows per tile (the MMA's M)
constexpr int kKS = kMegaKSlice;        // k elements per tile
constexpr int kRS = kMegaRowStride;     // bytes between tile rows in shared memory
constexpr int kSlot = kMegaSlotBytes;
constexpr int kKeys = kMegaKeys;        // keys per attention tile
constexpr int kKR = 8;                  // k ranges a tile's product is split into (fixed)
constexpr int kGroups = kCW / 4;        // attention: groups of four warps
constexpr int kMaxItems = 4 * kKR / kCW;  // (tile, token tile, k range) items a warp may take: 32 a phase at most

static_assert(kCT == 512, "the named barriers below count 512 compute threads");

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// AND of a flag over the compute threads; every one gets the same answer.
__device__ __forceinline__ bool cbar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 512, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
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

__device__ __forceinline__ uint32_t ld_acquire(const unsigned int* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- warp-level MMA, bf16 x bf16 -> fp32 ---------------------------------------
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// N consecutive f16 values (N = 1, 2 or 4; 2N-byte aligned) as fp32, one load.
template <int N>
__device__ __forceinline__ void ld_halves(const __half* p, float (&f)[N]) {
  if constexpr (N == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    f[0] = x.x;
    f[1] = x.y;
    f[2] = y.x;
    f[3] = y.y;
  } else if constexpr (N == 2) {
    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(p));
    f[0] = x.x;
    f[1] = x.y;
  } else {
    f[0] = __half2float(*p);
  }
}

// Units [u0, u1) of `units` that CTA b of P owns (contiguous, sizes differ by
// at most one).  The loader and the compute warps use the same split.
__device__ __forceinline__ void share(int units, int P, int b, int& u0, int& u1) {
  u0 = (int)(((long long)units * b) / P);
  u1 = (int)(((long long)units * (b + 1)) / P);
}

// Attention work item i of a layer: (sequence, KV head, 64-key chunk).  Items
// run sequence-major, then KV head, then chunk; CTA b takes items b, b+P, ...
struct Item {
  int s, g, c, nch;
};
// The item after `it` in the flat order.
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
// Attention items of CTA b: a contiguous range, cut into four contiguous parts
// (one per group of four warps).  The loader issues the parts' tiles round
// robin, so every group has tiles in flight; ring position of the k-th item
// of part q, counted from the first attention tile:
struct AttnSplit {
  int first[kGroups], len[kGroups];
  __device__ AttnSplit(int n_items, int P, int b) {
    int i0, i1;
    share(n_items, P, b, i0, i1);
    for (int q = 0; q < kGroups; ++q) {
      int j0, j1;
      share(i1 - i0, kGroups, q, j0, j1);
      first[q] = i0 + j0;
      len[q] = j1 - j0;
    }
  }
  __device__ int total() const {
    int n = 0;
    for (int q = 0; q < kGroups; ++q) n += len[q];
    return n;
  }
  __device__ int pos(int q, int k) const {
    int p = 0;
    for (int r = 0; r < kGroups; ++r) p += min(len[r], k) + (r < q && len[r] > k ? 1 : 0);
    return p;
  }
};

// Shared memory of one CTA (offsets from the dynamic base).
struct Smem {
  uint8_t* ring;                // [nslots][kSlot]
  uint8_t* act;                 // [8 * nt][kRS]: one k slice of the product's input rows (bf16)
  float* scr;                   // products: [nt * kKR][128] partial tiles; attention: per-group scratch
  float* rstd;                  // [32]
  unsigned long long* best;     // [32]
  float* sq;                    // [32][16]
  uint64_t* full;               // [nslots]
  uint64_t* empty;              // [nslots]
  int* flags;                   // [0] abort, [1] tiles issued, [2] tiles consumed, [4..8) group flags
  Item* start;                  // [kGroups] first attention item of each group (the same in every layer)
};

// Per attention group: roped queries, per-warp states, merge results.
template <int D>
struct GroupScr {
  float qs[2][D];
  float os[4][2][D];
  float ms[4][2], ls[4][2];
  float ML[2][2];
};

template <int D>
__host__ __device__ constexpr size_t scr_bytes(int nt) {
  const size_t prod = (size_t)(nt == 1 ? 2 : 1) * nt * kKR * 128 * 4;  // partial tiles of one phase
  const size_t attn = kGroups * ((sizeof(GroupScr<D>) + 127) / 128 * 128);
  return prod > attn ? prod : attn;
}

__host__ __device__ constexpr size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

template <int D>
__host__ __device__ size_t smem_layout(int nslots, int nt, size_t* o_act, size_t* o_scr, size_t* o_small,
                                       size_t* o_bars) {
  size_t off = (size_t)nslots * kSlot;
  *o_act = off;
  off = align128(off + (size_t)8 * nt * kRS);
  *o_scr = off;
  off = align128(off + scr_bytes<D>(nt));
  *o_small = off;
  off = align128(off + 32 * 4 + 32 * 8 + 32 * 16 * 4 + 16 * 4);
  *o_bars = off;
  off += (size_t)2 * nslots * 8 + kGroups * sizeof(Item);
  return off;
}

// ---------------------------------------------------------------------------
// The loader warp: the CTA's tiles in the order the compute warps take them.
// ---------------------------------------------------------------------------
template <int D>
__device__ void loader(const MegaArgs& a, const Smem& sm, int b, int P) {
  const int lane = threadIdx.x & 31;
  const int ns = a.nslots;
  volatile int* abort_s = sm.flags;
  uint32_t n = 0;
  // Claim the next slot and arm it for `bytes`; false (warp-uniform) on abort.
  auto begin = [&](uint32_t bytes) -> bool {
    const uint32_t slot = n % ns;
    int ok = 1;
    if (lane == 0) {
      if (n >= (uint32_t)ns) ok = mbar_wait(&sm.empty[slot], ((n / ns) - 1) & 1, abort_s, a.err);
      if (ok) mbar_expect_tx(&sm.full[slot], bytes);
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  auto product = [&](const bf16* W, int K, int R, int gran) -> bool {
    int u0, u1;
    share(R / gran, P, b, u0, u1);
    const int r0 = u0 * gran, nrows = (u1 - u0) * gran;
    const int mt = (nrows + kRows - 1) / kRows, nks = (K + kKS - 1) / kKS;
    for (int ks = 0; ks < nks; ++ks) {
      const int kslice = min(kKS, K - ks * kKS);
      for (int m = 0; m < mt; ++m) {
        const int rows_here = min(kRows, nrows - m * kRows);
        if (!begin((uint32_t)(rows_here * kslice * 2))) return false;
        uint8_t* dst = sm.ring + (size_t)(n % ns) * kSlot;
        if (lane < rows_here)
          bulk_g2s(dst + lane * kRS, W + (size_t)(r0 + m * kRows + lane) * K + (size_t)ks * kKS,
                   (uint32_t)kslice * 2, &sm.full[n % ns]);
        __syncwarp();
        ++n;
      }
    }
    return true;
  };
  const __half* kv = a.kv;
  const uint32_t slab = 16 * D * 2;  // bytes of one block's keys (or values) of one KV head
  const AttnSplit split(__ldg(a.item_start + a.T), P, b);
  int maxlen = 0;
  for (int q = 0; q < kGroups; ++q) maxlen = max(maxlen, split.len[q]);
  bool ok = true;
  for (int l = 0; l < a.n_layers && ok; ++l) {
    const char* Lb = a.layers + (size_t)l * a.layer_stride;
    const int QR = (a.H + 2 * a.Hkv) * D;
    ok = product(reinterpret_cast<const bf16*>(Lb + a.o_wqkv), a.d, QR, 1);
    Item cur[kGroups];
    for (int q = 0; q < kGroups; ++q) cur[q] = sm.start[q];
    for (int k = 0; k < maxlen && ok; ++k)
      for (int q = 0; q < kGroups && ok; ++q) {
        if (k >= split.len[q]) continue;
        const Item it = cur[q];
        next_item(a, cur[q]);
        const int ctx = __ldg(a.seq_ctx + it.s);
        const int nb = (min(kKeys, ctx - it.c * kKeys) + 15) / 16;
        if (!begin(2 * nb * slab)) {
          ok = false;
          break;
        }
        uint8_t* dst = sm.ring + (size_t)(n % ns) * kSlot;
        if (lane < nb) {
          const int blk = __ldg(a.tables + (size_t)it.s * a.max_blocks + it.c * (kKeys / 16) + lane);
          bulk_g2s(dst + lane * slab, kv + kv_offset(l, blk, 0, it.g, 0, a.n_blocks, a.Hkv, 16, D), slab,
                   &sm.full[n % ns]);
          bulk_g2s(dst + (kKeys / 16 + lane) * slab, kv + kv_offset(l, blk, 1, it.g, 0, a.n_blocks, a.Hkv, 16, D),
                   slab, &sm.full[n % ns]);
        }
        __syncwarp();
        ++n;
      }
    if (!ok) break;
    ok = product(reinterpret_cast<const bf16*>(Lb + a.o_wo), a.H * D, a.d, 1) &&
         product(reinterpret_cast<const bf16*>(Lb + a.o_wgu), a.d, 2 * a.F, 2 * kGuGroup) &&
         product(reinterpret_cast<const bf16*>(Lb + a.o_wd), a.F, a.d, 1);
  }
  if (ok) product(a.embed, a.d, a.vocab, 1);
  if (lane == 0) sm.flags[1] = (int)n;
  if (lane == 0 && a.trace) a.trace[(size_t)b * kMegaTraceStride + kMegaTraceStride - 1] = global_ns();
}

// ---------------------------------------------------------------------------
// The compute warps.
// ---------------------------------------------------------------------------
enum { P_QKV = 0, P_RESID = 1, P_SWIGLU = 2, P_LOGITS = 3 };

// Grid-wide barrier of the compute warps of every CTA (the loader never waits
// on one).  Returns false, on every compute thread, if this or any CTA gave up.
__device__ bool grid_sync(const MegaArgs& a, const Smem& sm, int P, uint32_t& gen, bool ok) {
  const int ctid = threadIdx.x;
  ok = cbar_and(ok);
  if (!ok) {
    if (ctid == 0) sm.flags[0] = 1;
    return false;
  }
  int res = 1;
  if (ctid == 0) {
    // the CTA barrier above orders every compute thread's writes before this release
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.bar) : "memory");
    const unsigned target = (gen + 1) * (unsigned)P;
    const uint64_t t0 = global_ns();
    while (ld_acquire(a.bar) < target) {
      if (*reinterpret_cast<volatile uint32_t*>(a.err) & kErrTimeout) {
        res = 0;
        break;
      }
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(a.err, kErrTimeout);
        res = 0;
        break;
      }
    }
    if (!res) sm.flags[0] = 1;
  }
  ++gen;
  return cbar_and(ctid == 0 ? res != 0 : true);
}

// The compute warps' view of one stage; every stage builds its own, so no
// value stays live from one stage to the next but the ring position.
template <int D>
struct Compute {
  const MegaArgs& a;
  const Smem& sm;
  int b, P, nt, ns;
  int ctid, warp, lane;
  uint32_t tile;  // next ring tile

  int sub = -1;   // trace: first stamp slot of this stage (layer 1 only), else -1
  int nsub = 0;
  __device__ Compute(const MegaArgs& a_, const Smem& sm_, int b_, int P_, uint32_t tile_)
      : a(a_), sm(sm_), b(b_), P(P_), nt((a_.T + 7) / 8), ns(a_.nslots), ctid(threadIdx.x), warp(threadIdx.x >> 5),
        lane(threadIdx.x & 31), tile(tile_) {}
  // trace: the timer at points inside one stage of layer 1 (thread 0, up to 6 stamps a stage)
  __device__ void stamp() {
    if (sub >= 0 && ctid == 0 && nsub < 6) a.trace[(size_t)b * kMegaTraceStride + sub + nsub] = global_ns();
    ++nsub;
  }

  // 1 / rms of every token row from the per-CTA partial sums, in one order.
  __device__ void compute_rstd() {
#pragma unroll 2
    for (int t = warp; t < a.T; t += kCW) {
      float v[kMegaMaxGrid / 32];
#pragma unroll
      for (int k = 0; k < kMegaMaxGrid / 32; ++k) {
        const int p = lane + 32 * k;
        v[k] = p < P ? __ldcg(a.SSQP + (size_t)t * P + p) : 0.f;
      }
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < kMegaMaxGrid / 32; ++k) s += v[k];
      s = warp_sum(s);
      if (lane == 0) sm.rstd[t] = 1.0f / sqrtf(s / (float)a.d + a.eps);
    }
  }

  // Copy k slice ks of the token rows of X (bf16 [T, ldx]) into the staging rows.
  // Copy k slice ks of the token rows of X (bf16 [T, ldx]) into the staging
  // rows with 16-byte asynchronous copies (cached in L2 only: the data was
  // written by other CTAs this step), all in flight together.  The caller
  // waits with cp_wait() before the CTA barrier.
  __device__ void stage_act(const bf16* X, int ldx, int ks, int kslice) {
    const int nv = kslice / 8;
    for (int i = ctid; i < a.T * nv; i += kCT) {
      const int t = i / nv, v = i - t * nv;
      const uint32_t dst = smem_u32(sm.act + (size_t)t * kRS + v * 16);
      const bf16* src = X + (size_t)t * ldx + (size_t)ks * kKS + v * 8;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  __device__ void cp_wait() const { asm volatile("cp.async.wait_all;" ::: "memory"); }

  // y of (row r, token t) of tile ml of the phase: the k-range partials in order.
  __device__ float ysum(int ml, int r, int t) const {
    const float* p = sm.scr + (size_t)((ml * nt + (t >> 3)) * kKR) * 128 + r * 8 + (t & 7);
    float y = 0.f;
#pragma unroll
    for (int kr = 0; kr < kKR; ++kr) y += p[kr * 128];
    return y;
  }

  struct Out {
    float* f32;          // P_QKV: raw q|k|v [T, rows]; P_LOGITS: logits [T, rows] (may be null)
    const float* w_next; // P_RESID: the next RMSNorm's gain
  };

  // One weight product over this CTA's rows with its fused epilogue.  Tiles
  // go two at a time while the token rows fit one 8-row MMA tile, else one
  // at a time.  A warp takes (tile, token tile, k range) items; the epilogue
  // adds a tile's eight k-range partials in order, so the result of a row
  // does not depend on how many tiles or tokens share the phase.
  template <int EPI>
  __device__ bool product(const bf16* W, int K, int R, int gran, const bf16* X, int ldx, Out o) {
    int u0, u1;
    share(R / gran, P, b, u0, u1);
    const int r0 = u0 * gran, nrows = (u1 - u0) * gran;
    const int mt = (nrows + kRows - 1) / kRows, nks = (K + kKS - 1) / kKS;
    const int T = a.T;
    const int TP = nt == 1 ? 2 : 1;
    if (EPI != P_RESID) compute_rstd();
    if (EPI == P_LOGITS && ctid < T) sm.best[ctid] = 0ull;
    // RESID: this thread's residual values (row i & 15, token i >> 4 for
    // i = ctid, ctid + 256), fetched while the input is staged
    float xres[2] = {0.f, 0.f};
    if (EPI == P_RESID)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = ctid + u * kCT;
        if ((i >> 4) < T && (i & 15) < nrows) xres[u] = __ldcg(a.X + (size_t)(i >> 4) * a.d + r0 + (i & 15));
      }
    float acc[kMaxItems][4];
    const uint32_t act_s = smem_u32(sm.act);
    for (int ks = 0; ks < (mt > 0 ? nks : 0); ++ks) {
      const int kslice = min(kKS, K - ks * kKS), nsteps = kslice / 16;
      stage_act(X, ldx, ks, kslice);  // the previous slice's readers passed the barrier after its products
      cp_wait();
      cbar();
      if (ks == 0) stamp();  // input staged
      for (int mb = 0; mb < mt; mb += TP) {
        const int tp = min(TP, mt - mb);
        bool got = true;
        for (int q = 0; q < tp; ++q)
          got = mbar_wait(&sm.full[(tile + q) % ns], ((tile + q) / ns) & 1, sm.flags, a.err) && got;
        if (!cbar_and(got)) return false;
        if (mb == 0 && ks == nks - 1) stamp();  // first tile of the last slice in shared memory
        const int per_tile = nt * kKR, nitems = tp * per_tile;
        if (ks == 0) {
#pragma unroll
          for (int q = 0; q < kMaxItems; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
        }
        // this warp's items advance one k step at a time, side by side
        uint32_t a_addr[kMaxItems], b_addr[kMaxItems];
        int cnt[kMaxItems], maxc = 0;
#pragma unroll
        for (int q = 0; q < kMaxItems; ++q) {
          const int it = warp + q * kCW;
          cnt[q] = 0;
          a_addr[q] = b_addr[q] = 0u;
          if (it < nitems) {
            const int ml = it / per_tile, rem = it - ml * per_tile, nn = rem / kKR, kr = rem % kKR;
            const int st0 = kr * nsteps / kKR, st1 = (kr + 1) * nsteps / kKR;
            const uint32_t slot_s = smem_u32(sm.ring + (size_t)((tile + ml) % ns) * kSlot);
            a_addr[q] = slot_s + ((lane & 7) + ((lane >> 3) & 1) * 8) * kRS + (lane >> 4) * 16 + st0 * 32;
            b_addr[q] = act_s + (nn * 8 + (lane & 7)) * kRS + ((lane >> 3) & 1) * 16 + st0 * 32;
            cnt[q] = st1 - st0;
            maxc = max(maxc, cnt[q]);
          }
        }
#pragma unroll 2
        for (int st = 0; st < maxc; ++st) {
#pragma unroll
          for (int q = 0; q < kMaxItems; ++q) {
            if (st < cnt[q]) {
              uint32_t A[4], B[2];
              ldsm4(a_addr[q] + st * 32, A);
              ldsm2(b_addr[q] + st * 32, B);
              mma16816(acc[q], A, B);
            }
          }
        }
        const bool last = ks == nks - 1;
        if (last) {
#pragma unroll
          for (int q = 0; q < kMaxItems; ++q) {
            const int it = warp + q * kCW;
            if (it < nitems) {
              float* red = sm.scr + (size_t)it * 128;
              const int g = lane >> 2, c2 = (lane & 3) * 2;
              *reinterpret_cast<float2*>(red + g * 8 + c2) = make_float2(acc[q][0], acc[q][1]);
              *reinterpret_cast<float2*>(red + (g + 8) * 8 + c2) = make_float2(acc[q][2], acc[q][3]);
            }
          }
        }
        cbar();
        if (mb == 0 && last) stamp();  // first products done
        if (ctid == 0)
          for (int q = 0; q < tp; ++q) mbar_arrive(&sm.empty[(tile + q) % ns]);
        tile += tp;
        if (!last) continue;
        if (EPI == P_QKV) {
          for (int i = ctid; i < tp * 16 * T; i += kCT) {
            const int r = i & 15, rest = i >> 4, t = rest % T, ml = rest / T;
            if (r < min(kRows, nrows - (mb + ml) * kRows))
              o.f32[(size_t)t * R + r0 + (mb + ml) * kRows + r] = ysum(ml, r, t) * sm.rstd[t];
          }
        } else if (EPI == P_RESID) {  // one tile (at most 16 rows per CTA)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int i = ctid + u * kCT, r = i & 15, t = i >> 4;
            float xn = 0.f;
            if (t < T && r < nrows) {
              const size_t off = (size_t)t * a.d + r0 + r;
              xn = xres[u] + ysum(0, r, t);
              a.X[off] = xn;
              a.XN[off] = __float2bfloat16_rn(xn * o.w_next[r0 + r]);
            }
            if (t < T) sm.sq[t * 16 + r] = xn * xn;
          }
        } else if (EPI == P_SWIGLU) {
          for (int i = ctid; i < tp * 8 * T; i += kCT) {
            const int j = i & 7, rest = i >> 3, t = rest % T, ml = rest / T;
            const float rs = sm.rstd[t];
            const float gte = ysum(ml, j, t) * rs, up = ysum(ml, j + kGuGroup, t) * rs;
            const int rbase = r0 + (mb + ml) * kRows;
            a.ACT[(size_t)t * a.F + (rbase / (2 * kGuGroup)) * kGuGroup + j] = __float2bfloat16_rn(silu(gte) * up);
          }
        } else {  // P_LOGITS: 16 consecutive threads hold the 16 rows of one (tile, token)
          const int n_i = tp * 16 * T;
          for (int i0 = 0; i0 < n_i; i0 += kCT) {  // whole warps in every round (shuffles)
            const int i = i0 + ctid, r = i & 15, rest = i >> 4, t = rest % T, ml = rest / T;
            const int rbase = r0 + (mb + ml) * kRows;
            unsigned long long key = 0ull;
            if (i < n_i && r < min(kRows, nrows - (mb + ml) * kRows)) {
              const float v = ysum(ml, r, t) * sm.rstd[t];
              if (o.f32) o.f32[(size_t)t * R + rbase + r] = v;
              key = argmax_key(v, rbase + r);
            }
#pragma unroll
            for (int x = 8; x >= 1; x >>= 1) {
              const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, x);
              key = other > key ? other : key;
            }
            if (i < n_i && r == 0 && key) atomicMax(&sm.best[t], key);
          }
        }
        cbar();
      }
    }
    if (EPI == P_RESID) {
      // this CTA's partial sum of x^2 per token row (rows in order; none: 0)
      if (mt == 0)
        for (int i = ctid; i < T * 16; i += kCT) sm.sq[i] = 0.f;
      cbar();
      if (ctid < T) {
        float s = 0.f;
        for (int r = 0; r < 16; ++r) s += sm.sq[ctid * 16 + r];
        a.SSQP[(size_t)ctid * P + b] = s;
      }
    }
    if (EPI == P_LOGITS) {
      cbar();
      if (ctid < T && sm.best[ctid]) atomicMax(a.keys + ctid, sm.best[ctid]);
    }
    return true;
  }

  // x = E[id] for this CTA's features of every token, x * (first gain), partials.
  __device__ void embed() {
    int e0, e1;
    share(a.d, P, b, e0, e1);
    const int nr = e1 - e0;
    for (int i = ctid; i < a.T * 16; i += kCT) {
      const int r = i & 15, t = i >> 4;
      float x = 0.f;
      if (r < nr) {
        int id = __ldg(a.ids + t);
        if (id < 0 || id >= a.vocab) {
          atomicOr(a.err, kErrBadId);
          id = 0;
        }
        const size_t off = (size_t)t * a.d + e0 + r;
        x = __bfloat162float(a.embed[(size_t)id * a.d + e0 + r]);
        a.X[off] = x;
        a.XN[off] = __float2bfloat16_rn(x * a.w_attn0[e0 + r]);
      }
      sm.sq[t * 16 + r] = x * x;
    }
    cbar();
    if (ctid < a.T) {
      float s = 0.f;
      for (int rr = 0; rr < 16; ++rr) s += sm.sq[ctid * 16 + rr];
      a.SSQP[(size_t)ctid * P + b] = s;
    }
  }


  // Warp gw folds block gw (16 keys) of a tile for both query heads of its
  // group into (max, sum, weighted values) in the group scratch.
  __device__ void fold(GroupScr<D>* gs, const __half* Ks, const __half* Vs, int keys_here, int nb) {
    constexpr int kDim = D / 32;
    constexpr int kSlabElems = 16 * D;
    const int gw = warp & 3;
    float q[2][kDim];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < kDim; ++e) q[i][e] = gs->qs[i][lane * kDim + e];
    float mw[2] = {-INFINITY, -INFINITY}, lw[2] = {0.f, 0.f}, ow[2][kDim];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < kDim; ++e) ow[i][e] = 0.f;
    if (gw < nb) {
      const __half* Kb = Ks + gw * kSlabElems;
      const __half* Vb = Vs + gw * kSlabElems;
      const int nkeys = min(16, keys_here - gw * 16);
      float v[32];
#pragma unroll
      for (int kx = 0; kx < 16; ++kx) {
        float kf[kDim];
        asm volatile("" ::: "memory");  // one key's loads at a time (register pressure)
        ld_halves<kDim>(Kb + kx * D + lane * kDim, kf);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < kDim; ++e) acc = fmaf(q[i][e], kf[e], acc);
          v[i * 16 + kx] = acc;
        }
      }
      // reduce-scatter: lane (head lane/16, key lane%16) ends with its full score
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int jx = 0; jx < w; ++jx) {
          const float send = up ? v[jx] : v[jx + w];
          const float keep = up ? v[jx + w] : v[jx];
          v[jx] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
      }
      const float sc = ((lane & 15) < nkeys) ? v[0] * a.scale : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int x = 8; x >= 1; x >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
      const float p = sc == -INFINITY ? 0.f : expf(sc - mx);  // each 16-lane half: its head's max
      float ps = p;
#pragma unroll
      for (int x = 8; x >= 1; x >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, x);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mw[i] = __shfl_sync(0xffffffffu, mx, i * 16);
        lw[i] = __shfl_sync(0xffffffffu, ps, i * 16);
      }
#pragma unroll
      for (int kx = 0; kx < 16; ++kx) {
        if (kx >= nkeys) break;  // slots past the context may hold anything
        float vf[kDim];
        ld_halves<kDim>(Vb + kx * D + lane * kDim, vf);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float pk = __shfl_sync(0xffffffffu, p, i * 16 + kx);
#pragma unroll
          for (int e = 0; e < kDim; ++e) ow[i][e] = fmaf(pk, vf[e], ow[i][e]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (lane == 0) {
        gs->ms[gw][i] = mw[i];
        gs->ls[gw][i] = lw[i];
      }
#pragma unroll
      for (int e = 0; e < kDim; ++e) gs->os[gw][i][lane * kDim + e] = ow[i][e];
    }
  }

  // Merge every chunk record of (sequence s, KV head g) in a fixed order and
  // write the two heads' attention output; re-arm the counter.
  __device__ void merge(GroupScr<D>* gs, int s, int g, int nch, int gq) {
    constexpr int kDim = D / 32;
    const int gw = warp & 3, ltid = ctid & 127, t = s;
    __threadfence();
    const float* recs = a.PART + ((size_t)s * a.H + 2 * g) * a.nch_cap * (D + 2);
    const size_t hstride = (size_t)a.nch_cap * (D + 2);
    if (gw < 2) {  // per head: the maximum and the weighted sum of the chunk records' sums
      const float* rec = recs + gw * hstride;
      float mx = -INFINITY;
      for (int cc = lane; cc < nch; cc += 32) mx = fmaxf(mx, __ldcg(rec + (size_t)cc * (D + 2)));
      mx = warp_max(mx);
      float sum = 0.f;
      for (int cc = lane; cc < nch; cc += 32)
        sum = fmaf(__ldcg(rec + (size_t)cc * (D + 2) + 1), expf(__ldcg(rec + (size_t)cc * (D + 2)) - mx), sum);
      sum = warp_sum(sum);
      if (lane == 0) {
        gs->ML[gw][0] = mx;
        gs->ML[gw][1] = sum;
      }
    }
    gbar(gq);
    {  // warp gw sums chunks gw, gw+4, ... of both heads over its lanes' dims
      float o[2][kDim];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < kDim; ++e) o[i][e] = 0.f;
      const float M0 = gs->ML[0][0], M1 = gs->ML[1][0];
      int cc = gw;
      for (; cc + 12 < nch; cc += 16) {  // four chunks per pass, their loads together
        float mv[2][4], ov[2][4][kDim];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float* r = recs + i * hstride + (size_t)(cc + 4 * u) * (D + 2);
            mv[i][u] = __ldcg(r);
#pragma unroll
            for (int e = 0; e < kDim; ++e) ov[i][u][e] = __ldcg(r + 2 + lane * kDim + e);
          }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float f = expf(mv[i][u] - (i ? M1 : M0));
#pragma unroll
            for (int e = 0; e < kDim; ++e) o[i][e] = fmaf(ov[i][u][e], f, o[i][e]);
          }
      }
      for (; cc < nch; cc += 4)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float* r = recs + i * hstride + (size_t)cc * (D + 2);
          const float f = expf(__ldcg(r) - (i ? M1 : M0));
#pragma unroll
          for (int e = 0; e < kDim; ++e) o[i][e] = fmaf(__ldcg(r + 2 + lane * kDim + e), f, o[i][e]);
        }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < kDim; ++e) gs->os[gw][i][lane * kDim + e] = o[i][e];
    }
    gbar(gq);
    for (int idx = ltid; idx < 2 * D; idx += 128) {
      const int i = idx / D, dd = idx - i * D;
      const float O = ((gs->os[0][i][dd] + gs->os[1][i][dd]) + gs->os[2][i][dd]) + gs->os[3][i][dd];
      a.ATT[(size_t)t * a.H * D + (2 * g + i) * D + dd] = __float2bfloat16_rn(O / gs->ML[i][1]);
    }
    if (ltid == 0) a.acnt[s * a.Hkv + g] = 0;
  }

  // Attention of layer l over this CTA's items.  Group gq of four warps takes
  // its part of the CTA's contiguous range of (sequence, KV head, 64-key
  // chunk) items.  Consecutive items of one (sequence, KV head) form a run:
  // the two queries are normed and rotated once per run, every chunk leaves
  // its own record (the four warps' blocks merged in warp order), and the run
  // counts its chunks into the (sequence, KV head) counter with one atomic.
  // The group that completes the count merges every chunk record in a fixed
  // order, so the output does not depend on how the chunks were shared out.
  __device__ bool attention(int l) {
    constexpr int kDim = D / 32;
    const int gq = warp >> 2, gw = warp & 3, ltid = ctid & 127;
    const AttnSplit split(__ldg(a.item_start + a.T), P, b);
    const uint32_t tile0 = tile;
    GroupScr<D>* gs = reinterpret_cast<GroupScr<D>*>(
        reinterpret_cast<uint8_t*>(sm.scr) + gq * ((sizeof(GroupScr<D>) + 127) / 128 * 128));
    const int QR = (a.H + 2 * a.Hkv) * D, half = D / 2;
    const char* Lb = a.layers + (size_t)l * a.layer_stride;
    const float* q_norm = reinterpret_cast<const float*>(Lb + a.o_q_norm);
    const float* k_norm = reinterpret_cast<const float*>(Lb + a.o_k_norm);
    constexpr int kSlabElems = 16 * D;
    bool ok = true;
    int run = 0;  // chunks of the current run done so far
    Item it = sm.start[gq];
    for (int k = 0; k < split.len[gq]; ++k, next_item(a, it)) {
      const uint32_t n = tile0 + split.pos(gq, k);
      const int s = it.s, g = it.g, c = it.c, t = s;
      const int ctx = __ldg(a.seq_ctx + s), pos = ctx - 1;
      if ((k == 0 || c == 0) && gw < 2) {
        // the run's queries: QK-norm over the head, then split-half RoPE at the token's position
        const int row = (2 * g + gw) * D;
        float v[kDim], y[kDim];
#pragma unroll
        for (int e = 0; e < kDim; ++e) v[e] = __ldcg(a.RAW + (size_t)t * QR + row + lane * kDim + e);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < kDim; ++e) ss = fmaf(v[e], v[e], ss);
        const float rn = 1.0f / sqrtf(warp_sum(ss) / (float)D + a.eps);
#pragma unroll
        for (int e = 0; e < kDim; ++e) y[e] = v[e] * rn * q_norm[lane * kDim + e];
#pragma unroll
        for (int e = 0; e < kDim; ++e) {
          const float yp = __shfl_xor_sync(0xffffffffu, y[e], 16);  // channel j +- D/2
          const int jd = lane * kDim + e, jj = jd < half ? jd : jd - half;
          const float cs = a.rope[((size_t)pos * half + jj) * 2], sn = a.rope[((size_t)pos * half + jj) * 2 + 1];
          gs->qs[gw][jd] = jd < half ? y[e] * cs - yp * sn : y[e] * cs + yp * sn;
        }
      }
      if (gq == 0 && k == 0) stamp();  // queries (first run)
      const bool got = mbar_wait(&sm.full[n % ns], (n / ns) & 1, sm.flags, a.err);
      if (!gbar_and(gq, got)) {
        ok = false;
        break;
      }
      const int keys_here = min(kKeys, ctx - c * kKeys), nb = (keys_here + 15) / 16;
      __half* Ks = reinterpret_cast<__half*>(sm.ring + (size_t)(n % ns) * kSlot);
      __half* Vs = Ks + (kKeys / 16) * kSlabElems;
      if (c == it.nch - 1 && gw >= 2) {
        // the newest key (warp 2, QK-norm + RoPE) and value (warp 3): append
        // them to the cache (f16, round to nearest even) and patch the tile
        const int is_v = gw == 3;
        const int row = is_v ? (a.H + a.Hkv + g) * D : (a.H + g) * D;
        float v[kDim];
#pragma unroll
        for (int e = 0; e < kDim; ++e) v[e] = __ldcg(a.RAW + (size_t)t * QR + row + lane * kDim + e);
        if (!is_v) {
          float ss = 0.f;
#pragma unroll
          for (int e = 0; e < kDim; ++e) ss = fmaf(v[e], v[e], ss);
          const float rn = 1.0f / sqrtf(warp_sum(ss) / (float)D + a.eps);
          float y[kDim];
#pragma unroll
          for (int e = 0; e < kDim; ++e) y[e] = v[e] * rn * k_norm[lane * kDim + e];
#pragma unroll
          for (int e = 0; e < kDim; ++e) {
            const float yp = __shfl_xor_sync(0xffffffffu, y[e], 16);
            const int jd = lane * kDim + e, jj = jd < half ? jd : jd - half;
            const float cs = a.rope[((size_t)pos * half + jj) * 2], sn = a.rope[((size_t)pos * half + jj) * 2 + 1];
            v[e] = jd < half ? y[e] * cs - yp * sn : y[e] * cs + yp * sn;
          }
        }
        const int blk = __ldg(a.tables + (size_t)s * a.max_blocks + pos / 16);
        __half* dst = a.kv + kv_offset(l, blk, is_v, g, pos % 16, a.n_blocks, a.Hkv, 16, D);
        const int kk = pos - c * kKeys;
        __half* st = (is_v ? Vs : Ks) + (kk / 16) * kSlabElems + (kk % 16) * D;
#pragma unroll
        for (int e = 0; e < kDim; ++e) {
          const __half h = __float2half_rn(v[e]);
          dst[lane * kDim + e] = h;
          st[lane * kDim + e] = h;
        }
        // the slot is refilled by bulk copies later: order these stores before them
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      gbar(gq);
      if (gq == 0 && k == 0) stamp();  // first tile in shared memory
      fold(gs, Ks, Vs, keys_here, nb);
      if (gq == 0 && k == 0) stamp();  // first tile folded
      gbar(gq);
      if (ltid == 0) mbar_arrive(&sm.empty[n % ns]);  // the tile is no longer read
      // the chunk's record per query head: the four warps merged in warp order
      for (int idx = ltid; idx < 2 * D; idx += 128) {
        const int i = idx / D, dd = idx - i * D;
        float M = gs->ms[0][i];
#pragma unroll
        for (int w = 1; w < 4; ++w) M = fmaxf(M, gs->ms[w][i]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float f = gs->ms[w][i] == -INFINITY ? 0.f : expf(gs->ms[w][i] - M);
          L = fmaf(gs->ls[w][i], f, L);
          O = fmaf(gs->os[w][i][dd], f, O);
        }
        float* rec = a.PART + (((size_t)s * a.H + 2 * g + i) * a.nch_cap + c) * (D + 2);
        if (dd == 0) {
          rec[0] = M;
          rec[1] = L;
        }
        rec[2 + dd] = O;
      }
      ++run;
      if (k + 1 < split.len[gq] && c + 1 < it.nch) continue;  // the run goes on
      // end of the run: count its chunks; the group that completes the count merges
      gbar(gq);
      if (ltid == 0) {
        __threadfence();
        sm.flags[4 + gq] = atomicAdd(a.acnt + s * a.Hkv + g, run) + run == it.nch;
      }
      run = 0;
      gbar(gq);
      if (gq == 0) stamp();  // run counted
      if (sm.flags[4 + gq]) merge(gs, s, g, it.nch, gq);
      if (gq == 0) stamp();  // merged (if last)
      gbar(gq);  // the group's scratch is free again
    }
    tile = ok ? tile0 + split.total() : tile0;  // after an abort, count none of them consumed
    return ok;
  }

};

// One product stage / one attention stage, each its own function.  They
// return the next ring position, with the top bit set if the stage gave up.
template <int D, int EPI>
__device__ __forceinline__ uint32_t product_stage(const MegaArgs& a, const Smem& sm, int b, int P, uint32_t tile,
                                               const bf16* W, int K, int R, int gran, const bf16* X, int ldx,
                                               float* f32, const float* w_next, int trace_slot) {
  Compute<D> c(a, sm, b, P, tile);
  if (a.trace && trace_slot >= 0) c.sub = trace_slot;
  c.stamp();  // entered
  const bool ok = c.template product<EPI>(W, K, R, gran, X, ldx, typename Compute<D>::Out{f32, w_next});
  return ok ? c.tile : (c.tile | 0x80000000u);
}

template <int D>
__device__ __forceinline__ uint32_t attention_stage(const MegaArgs& a, const Smem& sm, int b, int P, uint32_t tile,
                                                 int l, int trace_slot) {
  Compute<D> c(a, sm, b, P, tile);
  if (a.trace && trace_slot >= 0) c.sub = trace_slot;
  c.stamp();  // entered
  const bool ok = c.attention(l);
  return ok ? c.tile : (c.tile | 0x80000000u);
}

// The compute warps' whole step.
template <int D>
__device__ void compute_main(const MegaArgs& a, const Smem& sm, int b, int P) {
  const int ctid = threadIdx.x;
  const int QR = (a.H + 2 * a.Hkv) * D;
  uint32_t tile = 0, gen = 0;
  int mk = 0;
  // optional trace: compute thread 0 of every CTA stamps the global timer when
  // a stage's work is done and when its grid barrier releases
  auto mark = [&](int k) {
    if (a.trace && ctid == 0 && k < kMegaTraceStride) a.trace[(size_t)b * kMegaTraceStride + k] = global_ns();
  };
  auto sync = [&](bool ok) {
    mark(++mk);
    ok = grid_sync(a, sm, P, gen, ok);
    mark(++mk);
    return ok;
  };
  auto take = [&](uint32_t r) {
    tile = r & 0x7FFFFFFFu;
    return (r >> 31) == 0;
  };
  mark(0);
  {
    Compute<D> c(a, sm, b, P, 0);
    c.embed();
  }
  bool ok = sync(true);
  for (int l = 0; l < a.n_layers && ok; ++l) {
    const char* Lb = a.layers + (size_t)l * a.layer_stride;
    const float* w_next =
        l + 1 < a.n_layers ? reinterpret_cast<const float*>(Lb + a.layer_stride + a.o_attn_norm) : a.final_norm;
    ok = sync(take(product_stage<D, P_QKV>(a, sm, b, P, tile, reinterpret_cast<const bf16*>(Lb + a.o_wqkv), a.d, QR,
                                           1, a.XN, a.d, a.RAW, nullptr, l == 1 ? 290 : -1)));
    if (ok) ok = sync(take(attention_stage<D>(a, sm, b, P, tile, l, l == 1 ? 296 : -1)));
    if (ok)
      ok = sync(take(product_stage<D, P_RESID>(a, sm, b, P, tile, reinterpret_cast<const bf16*>(Lb + a.o_wo),
                                               a.H * D, a.d, 1, a.ATT, a.H * D, nullptr,
                                               reinterpret_cast<const float*>(Lb + a.o_mlp_norm), l == 1 ? 302 : -1)));
    if (ok)
      ok = sync(take(product_stage<D, P_SWIGLU>(a, sm, b, P, tile, reinterpret_cast<const bf16*>(Lb + a.o_wgu), a.d,
                                                2 * a.F, 2 * kGuGroup, a.XN, a.d, nullptr, nullptr, l == 1 ? 308 : -1)));
    if (ok)
      ok = sync(take(product_stage<D, P_RESID>(a, sm, b, P, tile, reinterpret_cast<const bf16*>(Lb + a.o_wd), a.F,
                                               a.d, 1, a.ACT, a.F, nullptr, w_next, -1)));
  }
  if (ok)
    ok = sync(take(product_stage<D, P_LOGITS>(a, sm, b, P, tile, a.embed, a.d, a.vocab, 1, a.XN, a.d, a.logits,
                                              nullptr, -1)));
  if (ok && b == 0 && ctid < a.T)
    a.argmax[ctid] = (int32_t)(0xFFFFFFFFu - (uint32_t)(__ldcg(a.keys + ctid) & 0xFFFFFFFFull));
  if (ctid == 0) sm.flags[2] = (int)tile;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_decode_mega(const __grid_constant__ MegaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int nt = (a.T + 7) / 8;
  size_t o_act, o_scr, o_small, o_bars;
  smem_layout<D>(a.nslots, nt, &o_act, &o_scr, &o_small, &o_bars);
  Smem sm;
  sm.ring = smem;
  sm.act = smem + o_act;
  sm.scr = reinterpret_cast<float*>(smem + o_scr);
  sm.rstd = reinterpret_cast<float*>(smem + o_small);
  sm.best = reinterpret_cast<unsigned long long*>(smem + o_small + 128);
  sm.sq = reinterpret_cast<float*>(smem + o_small + 128 + 256);
  sm.flags = reinterpret_cast<int*>(smem + o_small + 128 + 256 + 2048);
  sm.full = reinterpret_cast<uint64_t*>(smem + o_bars);
  sm.empty = sm.full + a.nslots;
  sm.start = reinterpret_cast<Item*>(sm.empty + a.nslots);
  const int b = blockIdx.x, P = gridDim.x;
  if (threadIdx.x < kGroups) {  // first attention item of each group
    const AttnSplit split(__ldg(a.item_start + a.T), P, b);
    sm.start[threadIdx.x] = split.len[threadIdx.x] > 0 ? item_of(a, split.first[threadIdx.x]) : Item{0, 0, 0, 1};
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nslots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 16; ++i) sm.flags[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // token rows of the staging buffer past T stay zero
  for (int i = threadIdx.x; i < 8 * nt * kRS / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm.act)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (threadIdx.x >= kCT) {
    loader<D>(a, sm, b, P);
  } else {
    compute_main<D>(a, sm, b, P);
  }
  __syncthreads();
  // after an abort, let the copies still in flight land before the CTA exits
  if (threadIdx.x == 0) {
    const uint32_t issued = (uint32_t)sm.flags[1], consumed = (uint32_t)sm.flags[2];
    const uint64_t t0 = global_ns();
    const uint32_t first = issued > (uint32_t)a.nslots && issued - a.nslots > consumed ? issued - a.nslots : consumed;
    for (uint32_t n = first; n < issued; ++n)
      while (!mbar_try(&sm.full[n % a.nslots], (n / a.nslots) & 1) && global_ns() - t0 < kWaitLimitNs) {
      }
  }
}

// Allow the kernel the current device's whole opt-in shared memory, once per
// head size and device (the occupancy check counts on that limit).
template <int D>
cudaError_t configure() {
  static SmemOptIn opt;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = opt.ensure(k_decode_mega<D>, optin);
  return e;
}

template <int D>
cudaError_t launch_d(const MegaArgs& a, int grid, cudaStream_t s) {
  const size_t smem = mega_smem_bytes(a.T, a.nslots, D);
  cudaError_t e = configure<D>();
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

}  // namespace

size_t mega_smem_bytes(int T, int nslots, int D) {
  size_t o_act, o_scr, o_small, o_bars;
  const int nt = (T + 7) / 8;
  switch (D) {
    case 32: return smem_layout<32>(nslots, nt, &o_act, &o_scr, &o_small, &o_bars);
    case 64: return smem_layout<64>(nslots, nt, &o_act, &o_scr, &o_small, &o_bars);
    default: return smem_layout<128>(nslots, nt, &o_act, &o_scr, &o_small, &o_bars);
  }
}

int mega_slots(int T, int D, size_t smem_limit) {
  int ns = 0;
  while (ns < kMegaMaxSlots && mega_smem_bytes(T, ns + 1, D) <= smem_limit) ++ns;
  return ns;
}

cudaError_t launch_decode_mega(const MegaArgs& a, int grid, cudaStream_t s) {
  switch (a.D) {
    case 32: return launch_d<32>(a, grid, s);
    case 64: return launch_d<64>(a, grid, s);
    case 128: return launch_d<128>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

int mega_threads() { return kThreads; }

bool mega_fits(int T, int D, int nslots) {
  const size_t smem = mega_smem_bytes(T, nslots, D);
  int blocks = 0;
  cudaError_t e;
  switch (D) {
    case 32:
      e = configure<32>();
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_decode_mega<32>, kThreads, smem);
      break;
    case 64:
      e = configure<64>();
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_decode_mega<64>, kThreads, smem);
      break;
    case 128:
      e = configure<128>();
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
