// sampler.cu - the sampling step after the LM head, on the device, in f64.
//
// tinyllm L10.1 "Candle model runner (Llama + bigram, int4), Rust KV cache,
// sampler and PCG32", section 2.6 "The sampler and PCG32": widen the logits to
// f64; repetition penalty over the distinct ids of prompt and output (divide
// a positive logit, multiply the others); presence and frequency over the
// output only (subtract frequency * count + presence); the logprob is the
// log-softmax at that point; T = 0 is the argmax, ties to the lowest id, with
// no draw; otherwise divide by T, keep the top k in (logit desc, id asc)
// order, keep the nucleus up to and including the id whose running sum
// reaches p, keep ids whose probability is at least min_p times the largest,
// softmax over the kept ids, draw one uniform and walk the cumulative sum in
// ascending id order to the first id with u < c.  The generator is PCG32
// (O'Neill's XSH RR 64/32) seeded per request by child_seed(seed, 4) =
// mix64(seed + 4 * 0x9E3779B97F4A7C15) on sequence 4; mix64 is read as
// SplitMix64's finaliser (the worked example of section 3 pins that reading).
//
// The device plan (per sequence; every kept set is a prefix of the
// (logit desc, id asc) order, cut further by the min-p bound):
//   k_mark      scatter the history into a per-sequence mark word per id:
//               bit 0 set by the prompt, bits 1.. the output count; a
//               non-zero word means the id was seen
//   k_scan1     multi-CTA: penalised maximum (lowest id) and finite minimum
//   k_scan2     multi-CTA, f64: e = exp(l - M) summed for the log-partition;
//               when sampling, l/T, e' = exp(l/T - M/T), a linear bucket of
//               l/T between its minimum and maximum (2048 buckets, bucket 0
//               the top), bucket counts and fixed-point masses
//   k_pick      one CTA: greedy ends here; otherwise the bucket histogram
//               finds the bucket where the top-k count or the nucleus mass
//               is reached, the candidates of the buckets up to there (or of
//               that bucket alone, with an exact sum of the mass above it)
//               are gathered into shared memory and sorted exactly; the
//               nucleus and min-p cuts are taken there, and when the whole
//               kept set is in shared memory the final softmax and CDF walk
//               too.  Buckets too crowded to gather are split further by an
//               8-bit radix on the (order key, id) pair.
//   k_final_*   when the kept set is larger than shared memory: per-chunk
//               sums of the kept e' (multi-CTA), then one CTA finds the chunk
//               and the id where the cumulative sum passes u.
//   k_mark      clears the marks it set.
// All sums are fixed trees, so the result is the same bits alone or in a
// batch.  The sums run in another order than the plain left-to-right loops
// of the definition, so a token can differ from it only where u or a filter
// threshold sits within rounding of a cumulative sum.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "../../include/dec.h"
#include "internal.h"

namespace {

constexpr int kChunk = 1024;       // elements per scan CTA (and per final chunk)
constexpr int kScanThreads = 256;  // 4 elements per thread
constexpr int kBins = 2048;        // linear buckets of l/T
constexpr int kCap = 4096;         // candidates held in shared memory
constexpr int kPick = 1024;        // threads of the one-CTA kernels
constexpr int kMaxChunks = 1024;   // chunks per sequence: vocab <= 2^20
constexpr double kFix = 35184372088832.0;       // 2^45: fixed-point scale of bucket masses
constexpr double kFixTol = 33554432.0;          // 2^25 = 2^-20 in e' units: slack on mass buckets
constexpr uint64_t kPcgMult = 6364136223846793005ull;
constexpr int kStage = 4;

struct SeqParam {  // 64 bytes, one per sequence
  double T, top_p, min_p, rep, pres, freq;
  int32_t top_k, hist_off, n_hist, n_prompt;
};

struct Part1 {
  double mx, mn;
  int32_t arg, pad;
  double pad2;
};

struct Part2 {
  double se, se2;
};

struct PickState {  // hand-off from k_pick to the final kernels
  int32_t mode;     // 0 done; 1 kept = order prefix up to `last` (if has_last) with e' >= emin
  int32_t has_last;
  int32_t last_id;
  int32_t pad;
  uint64_t last_key;
  uint64_t emin_bits;
  double M, lse;
};

struct Layout {
  size_t seqs, marks, W, E, bins, part1, part2, hcnt, hmass, state, fsum, status, total;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

Layout layout_of(int V, int S) {
  const size_t NB = (size_t)(V + kChunk - 1) / kChunk;
  Layout L;
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    size_t at = o;
    o += al256(bytes);
    return at;
  };
  L.seqs = take((size_t)S * sizeof(SeqParam));
  L.marks = take((size_t)S * V * 4);
  L.W = take((size_t)S * V * 8);
  L.E = take((size_t)S * V * 8);
  L.bins = take((size_t)S * V * 2);
  L.part1 = take((size_t)S * NB * sizeof(Part1));
  L.part2 = take((size_t)S * NB * sizeof(Part2));
  L.hcnt = take((size_t)S * kBins * 4);
  L.hmass = take((size_t)S * kBins * 8);
  L.state = take((size_t)S * sizeof(PickState));
  L.fsum = take((size_t)S * NB * 8);
  L.status = take(256);
  L.total = o;
  return L;
}

// ---- shared device helpers ------------------------------------------------------

__device__ __forceinline__ float load_logit(const float* x, int i, bool& bad) {
  float v = x[i];
  if (!(v < INFINITY)) {  // NaN or +inf: flagged, read as -inf
    bad = true;
    v = -INFINITY;
  }
  return v;
}

// the penalties, with the rounding steps of the definition (no contraction)
__device__ __forceinline__ double penalize(float x, int32_t mk, const SeqParam& q) {
  double l = (double)x;
  if (mk != 0) {
    l = l > 0.0 ? __ddiv_rn(l, q.rep) : __dmul_rn(l, q.rep);
    const int c = mk >> 1;
    if (c > 0) l = __dsub_rn(l, __dadd_rn(__dmul_rn(q.freq, (double)c), q.pres));
  }
  return l;
}

// order key: larger key = earlier in (value desc); -0 and +0 share one key
__device__ __forceinline__ uint64_t okey(double x) {
  uint64_t b = (uint64_t)__double_as_longlong(x);
  if (b == 0x8000000000000000ull) b = 0;
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

// (key, id) a comes before (key, id) b in (value desc, id asc) order
__device__ __forceinline__ bool before(uint64_t ka, int32_t ia, uint64_t kb, int32_t ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ unsigned __int128 ckey(uint64_t k, int32_t id) {
  return ((unsigned __int128)k << 32) | (uint32_t)(~(uint32_t)id);
}

__device__ __forceinline__ uint32_t pcg_next(uint64_t& state, uint64_t inc) {
  const uint64_t old = state;
  state = old * kPcgMult + inc;
  const uint32_t xs = (uint32_t)(((old >> 18) ^ old) >> 27);
  const uint32_t rot = (uint32_t)(old >> 59);
  return (xs >> rot) | (xs << ((32u - rot) & 31u));
}

__device__ __forceinline__ double pcg_uniform(uint64_t& state, uint64_t inc) {
  const uint32_t a = pcg_next(state, inc);
  const uint32_t b = pcg_next(state, inc);
  return (double)(((uint64_t)(a >> 5) << 26) + (b >> 6)) * 0x1p-53;
}

// (max, lowest id) pair: a beats b
__device__ __forceinline__ bool better(double va, int ia, double vb, int ib) { return va > vb || (va == vb && ia < ib); }


// deterministic block sum of one double per thread (fixed butterfly tree)
template <int NT>
__device__ double block_sum(double v, double* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  double t = l < NT / 32 ? red[l] : 0.0;
#pragma unroll
  for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;  // every thread holds the total
}

template <int NT>
__device__ void block_argmax(double& v, int& id, double* redv, int* redi) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const double ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, id, o);
    if (better(ov, oi, v, id)) v = ov, id = oi;
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) redv[w] = v, redi[w] = id;
  __syncthreads();
  v = l < NT / 32 ? redv[l] : -INFINITY;
  id = l < NT / 32 ? redi[l] : 0x7fffffff;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const double ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, id, o);
    if (better(ov, oi, v, id)) v = ov, id = oi;
  }
}

template <int NT>
__device__ double block_min(double v, double* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmin(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  double t = l < NT / 32 ? red[l] : INFINITY;
#pragma unroll
  for (int o = 16; o; o >>= 1) t = fmin(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

// inclusive scan of one value per thread (1024 threads), deterministic
template <typename U>
__device__ U block_scan(U v, U* red, U& total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const U n = __shfl_up_sync(0xffffffffu, v, o);
    if (l >= o) v += n;
  }
  __syncthreads();
  if (l == 31) red[w] = v;
  __syncthreads();
  if (w == 0) {
    U t = red[l];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const U n = __shfl_up_sync(0xffffffffu, t, o);
      if (l >= o) t += n;
    }
    red[l] = t;
  }
  __syncthreads();
  // every lane reads one warp prefix; the offset comes by shuffle (no red[w - 1]
  // load, which the compiler may hoist above its w > 0 guard)
  const U x = red[l];
  total = __shfl_sync(0xffffffffu, x, 31);
  U off = __shfl_sync(0xffffffffu, x, (w + 31) & 31);
  if (w == 0) off = U(0);
  __syncthreads();
  return v + off;
}

// ---- history marks ----------------------------------------------------------------

__global__ void k_mark(const SeqParam* __restrict__ sp, const int32_t* __restrict__ hist, int32_t* marks, int V,
                       int set, uint32_t* status) {
  const int s = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const SeqParam q = sp[s];
  if (j >= q.n_hist) return;
  const int id = hist[q.hist_off + j];
  if (id < 0 || id >= V) {
    if (set) atomicOr(status, (uint32_t)DEC_SAMPLE_BAD_ID);
    return;
  }
  int32_t* m = marks + (size_t)s * V + id;
  if (!set)
    *m = 0;
  else if (j < q.n_prompt)
    atomicOr(m, 1);  // seen
  else
    atomicAdd(m, 2);  // one more output count (a non-zero word is "seen")
}

// ---- scans over the vocabulary ----------------------------------------------------------

__global__ void __launch_bounds__(kScanThreads) k_scan1(const float* __restrict__ logits, int64_t ld,
                                                         const int32_t* __restrict__ marks,
                                                         const SeqParam* __restrict__ sp, int V, int NB,
                                                         Part1* __restrict__ part, uint32_t* status) {
  __shared__ double redv[32];
  __shared__ int redi[32];
  const int s = blockIdx.y, b = blockIdx.x, t = threadIdx.x;
  const SeqParam q = sp[s];
  const float* x = logits + (size_t)s * ld;
  const int32_t* mk = marks + (size_t)s * V;
  float fmx = -INFINITY, fmn = INFINITY;
  int fa = 0x7fffffff;
  double dmx = -INFINITY, dmn = INFINITY;
  int da = 0x7fffffff;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kChunk / kScanThreads; ++j) {
    const int i = b * kChunk + j * kScanThreads + t;
    if (i < V) {
      const float v = load_logit(x, i, bad);
      const int32_t m = mk[i];
      if (m == 0) {  // unpenalised: compare in f32 (the widening is exact)
        if (v > fmx) fmx = v, fa = i;
        if (v > -INFINITY && v < fmn) fmn = v;
      } else {
        const double l = penalize(v, m, q);
        if (l > dmx) dmx = l, da = i;
        if (l > -INFINITY && l < dmn) dmn = l;
      }
    }
  }
  if (bad) atomicOr(status, (uint32_t)DEC_SAMPLE_BAD_LOGIT);
  double mx = (double)fmx;
  int arg = fa;
  if (better(dmx, da, mx, arg)) mx = dmx, arg = da;
  const double mn = fmin((double)fmn, dmn);
  block_argmax<kScanThreads>(mx, arg, redv, redi);
  const double mnb = block_min<kScanThreads>(mn, redv);
  if (t == 0) {
    Part1 p;
    p.mx = mx;
    p.mn = mnb;
    p.arg = arg;
    p.pad = 0;
    p.pad2 = 0;
    part[(size_t)s * NB + b] = p;
  }
}

// every CTA reduces the per-chunk maxima in the same way: M, its lowest id, the finite minimum
template <int NT>
__device__ void reduce_part1(const Part1* p, int NB, double& M, int& arg, double& mn, double* redv, int* redi) {
  double v = -INFINITY, m = INFINITY;
  int id = 0x7fffffff;
  for (int c = threadIdx.x; c < NB; c += NT) {
    const Part1 e = p[c];
    if (better(e.mx, e.arg, v, id)) v = e.mx, id = e.arg;
    m = fmin(m, e.mn);
  }
  block_argmax<NT>(v, id, redv, redi);
  mn = block_min<NT>(m, redv);
  M = v;
  arg = id;
}

__global__ void __launch_bounds__(kScanThreads) k_scan2(const float* __restrict__ logits, int64_t ld,
                                                         const int32_t* __restrict__ marks,
                                                         const SeqParam* __restrict__ sp, int V, int NB,
                                                         const Part1* __restrict__ part1, Part2* __restrict__ part2,
                                                         double* __restrict__ W, double* __restrict__ E,
                                                         uint16_t* __restrict__ bins, uint32_t* __restrict__ hcnt,
                                                         unsigned long long* __restrict__ hmass, uint32_t* status) {
  __shared__ double redv[32];
  __shared__ int redi[32];
  __shared__ uint32_t sc[kBins];
  __shared__ unsigned long long sm[kBins];
  const int s = blockIdx.y, b = blockIdx.x, t = threadIdx.x;
  const SeqParam q = sp[s];
  double M, mn;
  int arg;
  reduce_part1<kScanThreads>(part1 + (size_t)s * NB, NB, M, arg, mn, redv, redi);
  if (!(M > -INFINITY)) {  // no finite logit
    if (t == 0 && b == 0) atomicOr(status, (uint32_t)DEC_SAMPLE_NO_FINITE);
    return;
  }
  const bool sampling = q.T > 0.0;
  const bool unit = q.T == 1.0;
  const double Mt = unit ? M : __ddiv_rn(M, q.T);
  const double mtn = unit ? mn : __ddiv_rn(mn, q.T);
  const double R = Mt - mtn;
  double scale = R > 0.0 ? (double)kBins / R : 0.0;
  if (!(scale < 1e300)) scale = 0.0;
  if (sampling) {
    for (int i = t; i < kBins; i += kScanThreads) sc[i] = 0, sm[i] = 0;
    __syncthreads();
  }
  const float* x = logits + (size_t)s * ld;
  const int32_t* mk = marks + (size_t)s * V;
  const size_t row = (size_t)s * V;
  double se = 0.0, se2 = 0.0;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kChunk / kScanThreads; ++j) {
    const int i = b * kChunk + j * kScanThreads + t;
    if (i < V) {
      const double l = penalize(load_logit(x, i, bad), mk[i], q);
      const double e = exp(l - M);
      se += e;
      if (sampling) {
        const double lt = unit ? l : __ddiv_rn(l, q.T);
        const double et = unit ? e : exp(lt - Mt);
        se2 += et;
        W[row + i] = lt;
        E[row + i] = et;
        const int bin = scale > 0.0 ? (int)fmin((Mt - lt) * scale, (double)(kBins - 1)) : 0;
        bins[row + i] = (uint16_t)bin;
        atomicAdd(&sc[bin], 1u);
        atomicAdd(&sm[bin], (unsigned long long)__double2ull_rn(et * kFix));
      }
    }
  }
  (void)bad;  // k_scan1 already flagged it
  se = block_sum<kScanThreads>(se, redv);
  se2 = block_sum<kScanThreads>(se2, redv);
  if (t == 0) part2[(size_t)s * NB + b] = Part2{se, se2};
  if (sampling) {
    __syncthreads();
    for (int i = t; i < kBins; i += kScanThreads)
      if (sc[i]) {
        atomicAdd(&hcnt[(size_t)s * kBins + i], sc[i]);
        atomicAdd(&hmass[(size_t)s * kBins + i], sm[i]);
      }
  }
}

// ---- the one-CTA pick ---------------------------------------------------------------------

struct PickSmem {
  uint64_t ck[kCap];   // order keys of the candidates
  double ce[kCap];     // their e'
  int32_t cid[kCap];   // their ids
  uint32_t hc[kBins];  // bucket (or digit) counts
  unsigned long long hm[kBins];
  double redd[32];
  int redi[32];
  unsigned long long redu[32];
  int n;           // candidates gathered
  int flag;
};

struct Frame {     // where a gathered list sits in the order
  long long above;   // elements of the restricted set before the list
  double m_above;    // their e' sum
};

enum { kCount = 0, kMass = 1 };

struct Lim {          // restriction to the order prefix ending at (key, id), bucket `bin`
  int on;
  uint64_t key;
  int32_t id;
  int bin;
};

__device__ __forceinline__ bool in_lim(const Lim& L, int bin, uint64_t k, int32_t id) {
  if (!L.on || bin < L.bin) return true;
  if (bin > L.bin) return false;
  return !before(L.key, L.id, k, id);  // (k, id) at or before the limit
}

// bitonic sort of sm.ck/ce/cid[0..n) in (key desc, id asc) order (by_id: id asc)
__device__ void sort_list(PickSmem& sm, int n, bool by_id) {
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + threadIdx.x; i < P; i += kPick) sm.ck[i] = 0, sm.ce[i] = 0.0, sm.cid[i] = 0x7fffffff;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += kPick) {
        const int p = i ^ j;
        if (p > i) {
          const bool up = (i & k) == 0;
          bool first_is_i;
          if (by_id)
            first_is_i = sm.cid[i] < sm.cid[p];
          else
            first_is_i = before(sm.ck[i], sm.cid[i], sm.ck[p], sm.cid[p]);
          if (first_is_i != up) {
            const uint64_t tk = sm.ck[i];
            sm.ck[i] = sm.ck[p];
            sm.ck[p] = tk;
            const double te = sm.ce[i];
            sm.ce[i] = sm.ce[p];
            sm.ce[p] = te;
            const int32_t ti = sm.cid[i];
            sm.cid[i] = sm.cid[p];
            sm.cid[p] = ti;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Gather, into shared memory and sorted, the stretch of the order where a
// cumulative target is reached: count target `tc` elements, or e' mass `tm`,
// over the elements allowed by `lim`.  Level 0 uses the bucket histogram in
// sm.hc/hm (already restricted).  Returns the frame of the list.
__device__ Frame gather(PickSmem& sm, int kind, long long tc, double tm, const Lim& lim, const uint16_t* bins,
                        const double* W, const double* E, int V, uint32_t* status) {
  const int t = threadIdx.x;
  __shared__ int s_lo, s_hi;
  __shared__ long long s_cnt_hi, s_cnt_before;
  __shared__ unsigned long long s_m_before;
  // ---- level 0: cumulative bucket counts and masses, two buckets per thread
  {
    const uint32_t c0 = sm.hc[2 * t], c1 = sm.hc[2 * t + 1];
    const unsigned long long m0 = sm.hm[2 * t], m1 = sm.hm[2 * t + 1];
    unsigned long long ctot, mtot;
    const unsigned long long cinc = block_scan<unsigned long long>((unsigned long long)c0 + c1, sm.redu, ctot);
    const unsigned long long minc = block_scan<unsigned long long>(m0 + m1, sm.redu, mtot);
    const unsigned long long cb0 = cinc - c0 - c1, mb0 = minc - m0 - m1;  // before bucket 2t
    const unsigned long long ca0 = cb0 + c0, ma0 = mb0 + m0;              // through bucket 2t
    if (t == 0) s_lo = kBins - 1, s_hi = kBins - 1;
    __syncthreads();
    if (kind == kCount) {
      if (ca0 >= (unsigned long long)tc && cb0 < (unsigned long long)tc) atomicMin(&s_lo, 2 * t);
      if (cinc >= (unsigned long long)tc && ca0 < (unsigned long long)tc) atomicMin(&s_lo, 2 * t + 1);
    } else {
      const double lo_t = tm * kFix - kFixTol, hi_t = tm * kFix + kFixTol;
      if ((double)ma0 >= lo_t) atomicMin(&s_lo, 2 * t);
      else if ((double)minc >= lo_t) atomicMin(&s_lo, 2 * t + 1);
      if ((double)ma0 >= hi_t) atomicMin(&s_hi, 2 * t);
      else if ((double)minc >= hi_t) atomicMin(&s_hi, 2 * t + 1);
    }
    __syncthreads();
    if (kind == kCount && t == 0) s_hi = s_lo;
    __syncthreads();
    const int lo = s_lo, hi = s_hi;
    if (2 * t == lo) s_cnt_before = (long long)cb0, s_m_before = mb0;
    if (2 * t + 1 == lo) s_cnt_before = (long long)ca0, s_m_before = ma0;
    if (2 * t == hi) s_cnt_hi = (long long)ca0;
    if (2 * t + 1 == hi) s_cnt_hi = (long long)cinc;
    __syncthreads();
  }
  const int lo = s_lo, hi = s_hi;
  const long long cnt_before = s_cnt_before, cnt_through = s_cnt_hi;
  int mode;  // 0 whole prefix through `hi`, 1 buckets lo..hi, 2 radix inside lo..hi
  if (cnt_through <= kCap)
    mode = 0;
  else if (cnt_through - cnt_before <= kCap)
    mode = 1;
  else
    mode = 2;

  // ---- radix refinement inside buckets lo..hi on the 96-bit (order key, ~id)
  int shift = 96;
  unsigned __int128 pre = 0;
  long long r_above = cnt_before;
  unsigned long long r_mabove = s_m_before;
  if (mode == 2) {
    while (true) {
      for (int i = t; i < 256; i += kPick) sm.hc[i] = 0, sm.hm[i] = 0;
      __syncthreads();
      for (int i = t; i < V; i += kPick) {
        const int bn = bins[i];
        if (bn < lo || bn > hi) continue;
        const uint64_t k = okey(W[i]);
        if (!in_lim(lim, bn, k, i)) continue;
        const unsigned __int128 K = ckey(k, i);
        if (shift < 96 && (K >> shift) != pre) continue;
        const int d = (int)((K >> (shift - 8)) & 255);
        atomicAdd(&sm.hc[d], 1u);
        if (kind == kMass) atomicAdd(&sm.hm[d], (unsigned long long)__double2ull_rn(E[i] * kFix));
      }
      __syncthreads();
      // walk digits from 255 (earliest) down: one thread, 256 steps
      __shared__ int s_d;
      __shared__ long long s_above;
      __shared__ unsigned long long s_mabove;
      if (t == 0) {
        long long c = r_above;
        unsigned long long m = r_mabove;
        int pick = -1, last = -1;
        for (int d = 255; d >= 0; --d) {
          if (!sm.hc[d]) continue;
          last = d;
          const long long c2 = c + sm.hc[d];
          const unsigned long long m2 = m + sm.hm[d];
          const bool hit = kind == kCount ? c2 >= tc : (double)m2 >= tm * kFix;
          if (hit) {
            pick = d;
            break;
          }
          c = c2;
          m = m2;
        }
        if (pick < 0 && last >= 0) {  // target beyond the set (rounding): the last digit holds the end
          pick = last;
          c -= sm.hc[last];
          m -= sm.hm[last];
        }
        if (pick < 0) {  // no element matched (cannot happen: the digit was non-empty)
          atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW);
          pick = 0;
        }
        s_d = pick;
        s_above = c;
        s_mabove = m;
      }
      __syncthreads();
      const int d = s_d;
      const uint32_t cd = sm.hc[d];
      r_above = s_above;
      r_mabove = s_mabove;
      pre = (pre << 8) | (unsigned __int128)d;
      shift -= 8;
      __syncthreads();
      if (cd <= (uint32_t)kCap || shift == 0) break;
    }
  }

  // ---- gather
  if (t == 0) sm.n = 0;
  __syncthreads();
  double msum = 0.0;
  for (int i = t; i < V; i += kPick) {
    const int bn = bins[i];
    if (bn > hi) continue;
    bool take;
    if (mode == 0) {
      if (lim.on && bn == lim.bin) {
        const uint64_t k = okey(W[i]);
        take = in_lim(lim, bn, k, i);
        if (take) {
          const int slot = atomicAdd(&sm.n, 1);
          if (slot < kCap) sm.ck[slot] = k, sm.ce[slot] = E[i], sm.cid[slot] = i;
        }
        continue;
      }
      take = in_lim(lim, bn, 0, i);
    } else if (bn < lo) {
      if (in_lim(lim, bn, 0, i)) msum += E[i];  // wholly before the list
      continue;
    } else {
      const uint64_t k = okey(W[i]);
      if (!in_lim(lim, bn, k, i)) continue;
      if (mode == 2) {
        const unsigned __int128 K = ckey(k, i);
        const unsigned __int128 top = K >> shift;
        if (top > pre) {
          msum += E[i];  // inside the buckets, before the list
          continue;
        }
        if (top < pre) continue;
      }
      const int slot = atomicAdd(&sm.n, 1);
      if (slot < kCap) sm.ck[slot] = k, sm.ce[slot] = E[i], sm.cid[slot] = i;
      continue;
    }
    if (take) {
      const int slot = atomicAdd(&sm.n, 1);
      if (slot < kCap) sm.ck[slot] = okey(W[i]), sm.ce[slot] = E[i], sm.cid[slot] = i;
    }
  }
  const double m_above = block_sum<kPick>(msum, sm.redd);
  __syncthreads();
  if (sm.n > kCap) {
    if (t == 0) atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW);
    __syncthreads();
    if (t == 0) sm.n = kCap;
    __syncthreads();
  }
  sort_list(sm, sm.n, false);
  Frame f;
  f.above = mode == 0 ? 0 : (mode == 1 ? cnt_before : r_above);
  f.m_above = mode == 0 ? 0.0 : m_above;
  return f;
}

// first list index j (< n) where above/Z + sum_{i<=j} ce_i/Z >= p; n-1 if never
__device__ int walk_mass(PickSmem& sm, int n, double Z, double start, double p) {
  const int t = threadIdx.x;
  double v[4];
  double run = 0.0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = 4 * t + r;
    const double qv = j < n ? sm.ce[j] / Z : 0.0;
    run += qv;
    v[r] = run;
  }
  double total;
  const double inc = block_scan<double>(run, sm.redd, total);
  const double base = start + (inc - run);
  __shared__ int s_first;
  if (t == 0) s_first = n - 1;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = 4 * t + r;
    if (j < n && base + v[r] >= p) {
      atomicMin(&s_first, j);
      break;
    }
  }
  __syncthreads();
  const int f = s_first;
  __syncthreads();
  return f;
}

// sum of ce[0..n) (fixed tree)
__device__ double list_sum(PickSmem& sm, int n) {
  double v = 0.0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = 4 * threadIdx.x + r;
    if (j < n) v += sm.ce[j];
  }
  return block_sum<kPick>(v, sm.redd);
}

__device__ double logprob_of(const float* x, const int32_t* mk, int id, const SeqParam& q, double M, double lse) {
  bool bad = false;
  return (penalize(load_logit(x, id, bad), mk[id], q) - M) - lse;
}

// the bucket histogram of one sequence, restricted to the order prefix `lim` allows
__device__ void load_hist(PickSmem& sm, const Lim& lim, const uint32_t* hc, const unsigned long long* hm,
                          const uint16_t* bins, const double* W, const double* E, int V) {
  const int t = threadIdx.x;
  for (int i = t; i < kBins; i += kPick) {
    const bool cut = lim.on && i > lim.bin;
    sm.hc[i] = cut ? 0u : hc[i];
    sm.hm[i] = cut ? 0ull : hm[i];
  }
  __syncthreads();
  if (!lim.on) return;
  // the limit's own bucket: only the elements at or before the limit
  __shared__ unsigned int s_c;
  __shared__ unsigned long long s_m;
  if (t == 0) s_c = 0, s_m = 0;
  __syncthreads();
  unsigned int c = 0;
  unsigned long long m = 0;
  for (int i = t; i < V; i += kPick) {
    if (bins[i] != lim.bin) continue;
    if (in_lim(lim, lim.bin, okey(W[i]), i)) ++c, m += __double2ull_rn(E[i] * kFix);
  }
  atomicAdd(&s_c, c);
  atomicAdd(&s_m, m);
  __syncthreads();
  if (t == 0) sm.hc[lim.bin] = s_c, sm.hm[lim.bin] = s_m;
  __syncthreads();
}

__global__ void __launch_bounds__(kPick, 1) k_pick(const float* __restrict__ logits, int64_t ld,
                                                    const int32_t* __restrict__ marks,
                                                    const SeqParam* __restrict__ sp, int V, int NB,
                                                    const Part1* __restrict__ part1, const Part2* __restrict__ part2,
                                                    const double* __restrict__ Wall, const double* __restrict__ Eall,
                                                    const uint16_t* __restrict__ ball, const uint32_t* __restrict__ hcnt,
                                                    const unsigned long long* __restrict__ hmass,
                                                    PickState* __restrict__ state, dec_rng* __restrict__ rng,
                                                    int32_t* __restrict__ tokens, double* __restrict__ logprobs,
                                                    uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PickSmem& sm = *reinterpret_cast<PickSmem*>(smem_raw);
  const int s = blockIdx.x, t = threadIdx.x;
  const SeqParam q = sp[s];
  const float* x = logits + (size_t)s * ld;
  const int32_t* mk = marks + (size_t)s * V;
  const size_t row = (size_t)s * V;
  const double* W = Wall + row;
  const double* E = Eall + row;
  const uint16_t* bins = ball + row;

  double M, mn;
  int arg;
  reduce_part1<kPick>(part1 + (size_t)s * NB, NB, M, arg, mn, sm.redd, sm.redi);
  PickState st;
  st.mode = 0;
  st.has_last = 0;
  st.last_id = 0;
  st.pad = 0;
  st.last_key = 0;
  st.emin_bits = 0;
  if (!(M > -INFINITY)) {  // flagged by k_scan2
    if (t == 0) {
      tokens[s] = -1;
      logprobs[s] = -INFINITY;
      state[s] = st;
    }
    return;
  }
  const Part2 pz = t < NB ? part2[(size_t)s * NB + t] : Part2{0.0, 0.0};
  const double Z = block_sum<kPick>(pz.se, sm.redd);
  const double Zall = block_sum<kPick>(pz.se2, sm.redd);
  const double lse = log(Z);
  st.M = M;
  st.lse = lse;
  if (q.T == 0.0) {  // greedy: no draw
    if (t == 0) {
      tokens[s] = arg;
      logprobs[s] = (M - M) - lse;
      state[s] = st;
    }
    return;
  }
  const long long kk = (q.top_k > 0 && q.top_k < V) ? q.top_k : V;
  const bool p_on = q.top_p < 1.0;
  const bool m_on = q.min_p > 0.0;

  // the list: (has_list) sm holds n sorted elements starting `above` into the order;
  // the kept prefix ends at list index `end` (or, without a list, at the set's end)
  bool has_list = false;
  int n = 0, end = -1;
  Frame fr{0, 0.0};
  double Zk = Zall;
  Lim none{0, 0, 0, 0};

  // ---- top-k
  Lim klim = none;
  if (kk < V) {
    load_hist(sm, none, hcnt + (size_t)s * kBins, hmass + (size_t)s * kBins, bins, W, E, V);
    fr = gather(sm, kCount, kk, 0.0, none, bins, W, E, V, status);
    has_list = true;
    n = sm.n;
    if (n == 0) {  // cannot happen: the bucket walk found the k-th element
      if (t == 0) atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW), tokens[s] = arg, logprobs[s] = -lse, state[s] = st;
      return;
    }
    end = (int)(kk - fr.above - 1);
    if (end >= n) end = n - 1;  // cannot happen unless capacity overflowed
    if (end < 0) end = 0;
    // Zk: e' over the top-k set
    const double in_list = list_sum(sm, end + 1);
    Zk = fr.m_above + in_list;
    klim.on = 1;
    klim.key = sm.ck[end];
    klim.id = sm.cid[end];
    klim.bin = bins[klim.id];
    __syncthreads();
  }

  // ---- nucleus
  if (p_on) {
    if (has_list && fr.above == 0) {
      end = walk_mass(sm, end + 1, Zk, 0.0, q.top_p);
    } else {
      load_hist(sm, klim, hcnt + (size_t)s * kBins, hmass + (size_t)s * kBins, bins, W, E, V);
      fr = gather(sm, kMass, 0, q.top_p * Zk, klim, bins, W, E, V, status);
      has_list = true;
      n = sm.n;
      if (n == 0) {  // cannot happen: the restricted set holds at least the top
        if (t == 0) atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW), tokens[s] = arg, logprobs[s] = -lse, state[s] = st;
        return;
      }
      end = walk_mass(sm, n, Zk, fr.m_above / Zk, q.top_p);
    }
  }

  // ---- min-p: q_i >= min_p * q_top, q_top = e'_top / Zk = 1 / Zk; as a bound on e'
  double emin = 0.0;
  if (m_on) {
    const double bound = q.min_p * (1.0 / Zk);
    double e = bound * Zk;
    if (e > 1.0) e = 1.0;
    for (int it = 0; it < 64 && e > 0.0 && nextafter(e, 0.0) / Zk >= bound; ++it) e = nextafter(e, 0.0);
    for (int it = 0; it < 64 && e / Zk < bound; ++it) e = nextafter(e, 2.0);
    emin = e;
  }

  // ---- final: in shared memory when the whole kept set is the list's head
  const bool whole = has_list && fr.above == 0;
  if (whole) {
    int nf = end + 1;
    if (m_on) {
      __shared__ int s_nf;
      if (t == 0) s_nf = 0;
      __syncthreads();
      for (int j = t; j < nf; j += kPick)
        if (sm.ce[j] >= emin) atomicMax(&s_nf, j + 1);
      __syncthreads();
      nf = s_nf;
      __syncthreads();
    }
    sort_list(sm, nf, true);  // ascending ids
    const double Zf = list_sum(sm, nf);
    __shared__ double s_u;
    __shared__ uint64_t s_state;
    if (t == 0) {
      dec_rng r = rng[s];
      uint64_t stt = r.state;
      s_u = pcg_uniform(stt, r.inc);
      s_state = stt;
    }
    __syncthreads();
    const double u = s_u;
    // CDF in ascending id order: first j with u < c_j
    double v[4];
    double run = 0.0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = 4 * t + r;
      run += j < nf ? sm.ce[j] / Zf : 0.0;
      v[r] = run;
    }
    double total;
    const double inc = block_scan<double>(run, sm.redd, total);
    const double base = inc - run;
    __shared__ int s_tok;
    if (t == 0) s_tok = nf - 1;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = 4 * t + r;
      if (j < nf && u < base + v[r]) {
        atomicMin(&s_tok, j);
        break;
      }
    }
    __syncthreads();
    if (t == 0) {
      const int tok = sm.cid[s_tok];
      tokens[s] = tok;
      logprobs[s] = logprob_of(x, mk, tok, q, M, lse);
      rng[s].state = s_state;
      state[s] = st;
    }
    return;
  }
  // ---- hand-off: the kept set is the order prefix through `last` with e' >= emin
  if (t == 0) {
    st.mode = 1;
    st.has_last = has_list ? 1 : 0;
    if (has_list) st.last_key = sm.ck[end], st.last_id = sm.cid[end];
    st.emin_bits = (uint64_t)__double_as_longlong(emin);
    state[s] = st;
  }
}

__device__ __forceinline__ bool kept_by(const PickState& st, double w, double e, int i) {
  if (st.has_last && before(st.last_key, st.last_id, okey(w), i)) return false;
  return (uint64_t)__double_as_longlong(e) >= st.emin_bits;  // e' >= 0: bit order is value order
}

__global__ void __launch_bounds__(kScanThreads) k_final_sum(const PickState* __restrict__ state, int V, int NB,
                                                             const double* __restrict__ Wall,
                                                             const double* __restrict__ Eall,
                                                             double* __restrict__ fsum) {
  __shared__ double red[32];
  const int s = blockIdx.y, b = blockIdx.x, t = threadIdx.x;
  const PickState st = state[s];
  if (st.mode == 0) return;
  const size_t row = (size_t)s * V;
  double v = 0.0;
#pragma unroll
  for (int j = 0; j < kChunk / kScanThreads; ++j) {
    const int i = b * kChunk + j * kScanThreads + t;
    if (i < V) {
      const double e = Eall[row + i];
      if (kept_by(st, Wall[row + i], e, i)) v += e;
    }
  }
  v = block_sum<kScanThreads>(v, red);
  if (t == 0) fsum[(size_t)s * NB + b] = v;
}

__global__ void __launch_bounds__(kPick, 1) k_final_pick(const float* __restrict__ logits, int64_t ld,
                                                          const int32_t* __restrict__ marks,
                                                          const SeqParam* __restrict__ sp,
                                                          const PickState* __restrict__ state, int V, int NB,
                                                          const double* __restrict__ Wall,
                                                          const double* __restrict__ Eall,
                                                          const double* __restrict__ fsum, dec_rng* __restrict__ rng,
                                                          int32_t* __restrict__ tokens, double* __restrict__ logprobs) {
  __shared__ double redd[32];
  __shared__ double s_u;
  __shared__ uint64_t s_state;
  __shared__ int s_chunk, s_tok, s_last;
  const int s = blockIdx.x, t = threadIdx.x;
  const PickState st = state[s];
  if (st.mode == 0) return;
  const SeqParam q = sp[s];
  const size_t row = (size_t)s * V;
  const double fs = t < NB ? fsum[(size_t)s * NB + t] : 0.0;
  const double Zf = block_sum<kPick>(fs, redd);
  double tot;
  const double cinc = block_scan<double>(t < NB ? fs / Zf : 0.0, redd, tot);
  if (t == 0) {
    dec_rng r = rng[s];
    uint64_t stt = r.state;
    s_u = pcg_uniform(stt, r.inc);
    s_state = stt;
    s_chunk = NB;
    s_last = -1;
    s_tok = 0x7fffffff;
  }
  __syncthreads();
  const double u = s_u;
  if (t < NB && u < cinc) atomicMin(&s_chunk, t);
  if (t < NB && fs > 0.0) atomicMax(&s_last, t);
  __syncthreads();
  int c = s_chunk;
  const bool past_end = c >= NB;  // rounding left the total at or below u
  if (past_end) c = s_last;
  // the chunk: one element per thread, in ascending ids
  const int i = c * kChunk + t;
  double p = 0.0;
  bool kept = false;
  if (i < V) {
    const double e = Eall[row + i];
    kept = kept_by(st, Wall[row + i], e, i);
    if (kept) p = e / Zf;
  }
  __shared__ double s_base;
  __shared__ int s_lastid;
  if (t == c) s_base = cinc - (fs / Zf);  // cumulative before chunk c
  if (t == 0) s_lastid = -1;
  __syncthreads();
  const double base = s_base;
  double ctot;
  const double cin = block_scan<double>(p, redd, ctot);
  if (!past_end && kept && u < base + cin) atomicMin(&s_tok, i);
  if (kept) atomicMax(&s_lastid, i);
  __syncthreads();
  if (t == 0) {
    // nothing passed u in the chunk (rounding): its last kept id
    const int tok = s_tok != 0x7fffffff ? s_tok : s_lastid;
    tokens[s] = tok;
    logprobs[s] = tok >= 0 ? logprob_of(logits + (size_t)s * ld, marks + row, tok, q, st.M, st.lse) : -INFINITY;
    rng[s].state = s_state;
  }
}

}  // namespace

// ---- host side ------------------------------------------------------------------------------

struct dec_sampler {
  int device;
  int V, S, NB;
  Layout L;
  unsigned char* ws;
  SeqParam* stage[kStage];
  cudaEvent_t stage_ev[kStage];
  int stage_next;
};

namespace {

int sfail(int code, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  return dec::set_error(code, buf);
}

#define S_CUDA(call)                                                                       \
  do {                                                                                     \
    cudaError_t e_ = (call);                                                               \
    if (e_ != cudaSuccess) return sfail(DEC_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

int check_params(const dec_sampling& p) {
  if (!(p.temperature >= 0.0) || !std::isfinite(p.temperature)) return sfail(DEC_EINVAL, "temperature must be finite and >= 0");
  if (p.top_k < 0) return sfail(DEC_EINVAL, "top_k must be >= 0");
  if (!(p.top_p >= 0.0 && p.top_p <= 1.0)) return sfail(DEC_EINVAL, "top_p must lie in [0, 1]");
  if (!(p.min_p >= 0.0 && p.min_p <= 1.0)) return sfail(DEC_EINVAL, "min_p must lie in [0, 1]");
  if (!(p.repetition_penalty > 0.0) || !std::isfinite(p.repetition_penalty))
    return sfail(DEC_EINVAL, "repetition_penalty must be finite and > 0");
  if (!std::isfinite(p.presence_penalty) || !std::isfinite(p.frequency_penalty))
    return sfail(DEC_EINVAL, "presence and frequency penalties must be finite");
  return DEC_OK;
}

}  // namespace

extern "C" {

uint64_t dec_child_seed(uint64_t seed, uint64_t purpose) { return mix64(seed + purpose * 0x9E3779B97F4A7C15ull); }

uint32_t dec_rng_next_u32(dec_rng* r) {
  const uint64_t old = r->state;
  r->state = old * kPcgMult + r->inc;
  const uint32_t xs = (uint32_t)(((old >> 18) ^ old) >> 27);
  const uint32_t rot = (uint32_t)(old >> 59);
  return (xs >> rot) | (xs << ((32u - rot) & 31u));
}

double dec_rng_uniform(dec_rng* r) {
  const uint32_t a = dec_rng_next_u32(r);
  const uint32_t b = dec_rng_next_u32(r);
  return (double)(((uint64_t)(a >> 5) << 26) + (b >> 6)) * 0x1p-53;
}

void dec_rng_stream(uint64_t seed, uint64_t purpose, dec_rng* out) {
  if (!out) return;
  out->state = 0;
  out->inc = (purpose << 1) | 1u;
  dec_rng_next_u32(out);
  out->state += dec_child_seed(seed, purpose);
  dec_rng_next_u32(out);
}

int dec_sampler_workspace_bytes(int32_t vocab, int32_t max_seqs, size_t* bytes) {
  if (!bytes) return sfail(DEC_EINVAL, "bytes is NULL");
  if (vocab < 1 || vocab > kChunk * kMaxChunks) return sfail(DEC_EINVAL, "vocab must lie in [1, %d]", kChunk * kMaxChunks);
  if (max_seqs < 1 || max_seqs > 65535) return sfail(DEC_EINVAL, "max_seqs must lie in [1, 65535]");
  *bytes = layout_of(vocab, max_seqs).total;
  return DEC_OK;
}

int dec_sampler_create(int32_t vocab, int32_t max_seqs, void* workspace, size_t bytes, dec_sampler** out) {
  if (!out) return sfail(DEC_EINVAL, "out is NULL");
  *out = nullptr;
  size_t need = 0;
  int rc = dec_sampler_workspace_bytes(vocab, max_seqs, &need);
  if (rc) return rc;
  if (!workspace || bytes < need) return sfail(DEC_EINVAL, "workspace too small: %zu bytes needed", need);
  if ((uintptr_t)workspace % 256) return sfail(DEC_EINVAL, "workspace must be 256-byte aligned");
  dec_sampler* s = new dec_sampler();
  S_CUDA(cudaGetDevice(&s->device));
  s->V = vocab;
  s->S = max_seqs;
  s->NB = (vocab + kChunk - 1) / kChunk;
  s->L = layout_of(vocab, max_seqs);
  s->ws = (unsigned char*)workspace;
  s->stage_next = 0;
  for (int i = 0; i < kStage; ++i) s->stage[i] = nullptr, s->stage_ev[i] = nullptr;
  for (int i = 0; i < kStage; ++i) {
    if (cudaHostAlloc((void**)&s->stage[i], (size_t)max_seqs * sizeof(SeqParam), cudaHostAllocDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&s->stage_ev[i], cudaEventDisableTiming) != cudaSuccess) {
      dec_sampler_destroy(s);
      return sfail(DEC_ECUDA, "pinned staging allocation failed");
    }
  }
  // marks start (and stay, between calls) zero; the status word starts clear
  if (cudaMemset(s->ws + s->L.marks, 0, (size_t)max_seqs * vocab * 4) != cudaSuccess ||
      cudaMemset(s->ws + s->L.status, 0, 256) != cudaSuccess) {
    dec_sampler_destroy(s);
    return sfail(DEC_ECUDA, "workspace clear failed");
  }
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_pick, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(PickSmem)) != cudaSuccess) {
      dec_sampler_destroy(s);
      return sfail(DEC_ECUDA, "cannot reserve %zu bytes of shared memory for the pick kernel", sizeof(PickSmem));
    }
    attr_set = true;
  }
  *out = s;
  return DEC_OK;
}

void dec_sampler_destroy(dec_sampler* s) {
  if (!s) return;
  for (int i = 0; i < kStage; ++i) {
    if (s->stage_ev[i]) {
      cudaEventSynchronize(s->stage_ev[i]);
      cudaEventDestroy(s->stage_ev[i]);
    }
    if (s->stage[i]) cudaFreeHost(s->stage[i]);
  }
  delete s;
}

int dec_sampler_status(dec_sampler* s, uint32_t* flags) {
  if (!s || !flags) return sfail(DEC_EINVAL, "NULL argument");
  S_CUDA(cudaMemcpy(flags, s->ws + s->L.status, 4, cudaMemcpyDeviceToHost));
  return DEC_OK;
}

int dec_sample(dec_sampler* s, const float* logits, int64_t ld, int32_t n, const dec_sampling* params,
               const int32_t* history, const int32_t* history_offsets, const int32_t* n_prompt, dec_rng* rng,
               int32_t* tokens, double* logprobs, void* stream) {
  if (!s) return sfail(DEC_EINVAL, "sampler is NULL");
  if (n < 0 || n > s->S) return sfail(DEC_EINVAL, "n_seqs %d outside 0 .. max_seqs (%d)", n, s->S);
  if (n == 0) return DEC_OK;
  if (!logits || !params || !rng || !tokens || !logprobs) return sfail(DEC_EINVAL, "NULL argument");
  if (ld < s->V) return sfail(DEC_EINVAL, "ld %lld below vocab %d", (long long)ld, s->V);
  int max_hist = 0;
  for (int i = 0; i < n; ++i) {
    int rc = check_params(params[i]);
    if (rc) return rc;
    const int h0 = history_offsets ? history_offsets[i] : 0, h1 = history_offsets ? history_offsets[i + 1] : 0;
    const int np = n_prompt ? n_prompt[i] : 0;
    if (h1 < h0 || h0 < 0) return sfail(DEC_EINVAL, "history offsets must be non-decreasing from 0 (sequence %d)", i);
    if (np < 0 || np > h1 - h0) return sfail(DEC_EINVAL, "n_prompt of sequence %d outside its history", i);
    if (h1 > h0 && !history) return sfail(DEC_EINVAL, "history is NULL");
    if (h1 - h0 > max_hist) max_hist = h1 - h0;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const int slot = s->stage_next;
  s->stage_next = (s->stage_next + 1) % kStage;
  S_CUDA(cudaEventSynchronize(s->stage_ev[slot]));
  SeqParam* H = s->stage[slot];
  for (int i = 0; i < n; ++i) {
    const dec_sampling& p = params[i];
    SeqParam& q = H[i];
    q.T = p.temperature;
    q.top_p = p.top_p;
    q.min_p = p.min_p;
    q.rep = p.repetition_penalty;
    q.pres = p.presence_penalty;
    q.freq = p.frequency_penalty;
    q.top_k = p.top_k;
    q.hist_off = history_offsets ? history_offsets[i] : 0;
    q.n_hist = history_offsets ? history_offsets[i + 1] - history_offsets[i] : 0;
    q.n_prompt = n_prompt ? n_prompt[i] : 0;
  }
  unsigned char* w = s->ws;
  SeqParam* dsp = (SeqParam*)(w + s->L.seqs);
  S_CUDA(cudaMemcpyAsync(dsp, H, (size_t)n * sizeof(SeqParam), cudaMemcpyHostToDevice, st));
  S_CUDA(cudaEventRecord(s->stage_ev[slot], st));
  S_CUDA(cudaMemsetAsync(w + s->L.hcnt, 0, (size_t)n * kBins * 4, st));
  S_CUDA(cudaMemsetAsync(w + s->L.hmass, 0, (size_t)n * kBins * 8, st));
  int32_t* marks = (int32_t*)(w + s->L.marks);
  uint32_t* status = (uint32_t*)(w + s->L.status);
  const int V = s->V, NB = s->NB;
  Part1* p1 = (Part1*)(w + s->L.part1);
  Part2* p2 = (Part2*)(w + s->L.part2);
  double* W = (double*)(w + s->L.W);
  double* E = (double*)(w + s->L.E);
  uint16_t* bins = (uint16_t*)(w + s->L.bins);
  uint32_t* hc = (uint32_t*)(w + s->L.hcnt);
  unsigned long long* hm = (unsigned long long*)(w + s->L.hmass);
  PickState* ps = (PickState*)(w + s->L.state);
  double* fsum = (double*)(w + s->L.fsum);
  const dim3 hgrid((max_hist + 255) / 256, n);
  if (max_hist > 0) k_mark<<<hgrid, 256, 0, st>>>(dsp, history, marks, V, 1, status);
  const dim3 grid(NB, n);
  k_scan1<<<grid, kScanThreads, 0, st>>>(logits, ld, marks, dsp, V, NB, p1, status);
  k_scan2<<<grid, kScanThreads, 0, st>>>(logits, ld, marks, dsp, V, NB, p1, p2, W, E, bins, hc, hm, status);
  k_pick<<<n, kPick, sizeof(PickSmem), st>>>(logits, ld, marks, dsp, V, NB, p1, p2, W, E, bins, hc, hm, ps, rng, tokens,
                                             logprobs, status);
  k_final_sum<<<grid, kScanThreads, 0, st>>>(ps, V, NB, W, E, fsum);
  k_final_pick<<<n, kPick, 0, st>>>(logits, ld, marks, dsp, ps, V, NB, W, E, fsum, rng, tokens, logprobs);
  if (max_hist > 0) k_mark<<<hgrid, 256, 0, st>>>(dsp, history, marks, V, 0, status);
  S_CUDA(cudaGetLastError());
  return DEC_OK;
}

}  // extern "C"
