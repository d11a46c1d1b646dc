// sampler.cu - the sampling step after the LM head, on the device.
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
// Arithmetic.  This GPU issues f64 at about 1/64 of its f32 rate, so the
// per-id work avoids the f64 pipe: the penalised logit is exact f64 (an f32
// widened, or one f64 penalty step for the few ids of the history); order
// comparisons use integer keys of those f64 values; exponentials, sums and
// thresholds run in double-f32 arithmetic (a float head plus a float tail,
// Dekker's and Knuth's error-free sums and products) with a table-driven
// exponential (Tang's method: exp(x) = 2^n * 2^(j/64) * exp(r), |r| <=
// ln2/128, r reduced with a four-piece ln2/64 and exp(r) from its Taylor
// polynomial of degree 5), accurate to about 2^-46.  The log-partition
// takes one f64 logarithm per sequence.  Results agree with the plain f64
// definition to about 1e-13 relative; a token can differ from it only where
// u or a filter threshold sits within that of a cumulative sum.
//
// The device plan (per sequence; every kept set is a prefix of the
// (logit desc, id asc) order, cut further by the min-p bound):
//   k_mark      scatter the history into a per-sequence mark word per id:
//               bit 0 set by the prompt, bits 1.. the output count; a
//               non-zero word means the id was seen
//   k_scan1     multi-CTA: penalised maximum (lowest id) and finite minimum
//   k_scan2     multi-CTA: e = exp(l - M) summed for the log-partition;
//               when sampling, e' = exp((l - M)/T), the order key, a linear
//               bucket of l between its minimum and maximum (2048 buckets,
//               bucket 0 the top), bucket counts and fixed-point masses
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
// batch.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "../../include/dec.h"
#include "internal.h"
#include "optin.h"

namespace {

constexpr int kChunk1 = 2048;      // elements per CTA of the maximum scan
constexpr int kChunk = 1024;       // elements per CTA of the exp scan (and per final chunk)
constexpr int kScanThreads = 256;  // 4 elements per thread
constexpr int kBins = 2048;        // linear buckets of the logit
constexpr int kCap = 4096;         // candidates held in shared memory
constexpr int kPick = 1024;        // threads of the one-CTA kernels
constexpr int kMaxChunks = 1024;   // chunks per sequence: vocab <= 2^20
// bucket masses are exact fixed point: an integer word in units of 2^-45 and a
// fraction word in units of 2^-90 (integer sums: the same bits in any order)
constexpr int kFixBits = 45;
constexpr float kFixF = 35184372088832.0f;  // 2^45
constexpr double kFix = 35184372088832.0;
constexpr double kFixSlack = 4096.0;        // bucket-walk slack, in 2^-45 units
constexpr uint64_t kPcgMult = 6364136223846793005ull;
constexpr int kStage = 4;
enum { kSampling = 1, kUnitT = 2, kTopP = 4, kMinP = 8 };
static_assert(kBins == 2 * kPick, "the bucket scan takes two buckets per thread");
static_assert(kCap == 4 * kPick, "list scans take four candidates per thread");

struct SeqParam {  // 96 bytes, one per sequence
  double T, top_p, min_p, rep, pres, freq;
  float rTh, rTl;  // 1/T as head + tail
  float pph, ppl;  // top_p
  float mph, mpl;  // min_p
  int32_t top_k;
  int32_t flags;   // kSampling | kUnitT | kTopP | kMinP, set on the host: no f64 compare on the device
  int32_t hist_off, n_hist, n_prompt, pad1;
};

struct Part1 {
  uint64_t key;
  float mn;
  int32_t arg;
};

struct Stats {  // per sequence: the penalised maximum and the finite minimum
  uint64_t key;
  double M;
  float mn, Mh, Ml;
  int32_t arg;
};

struct Part2 {
  float zh, zl, z2h, z2l;
};

struct PickState {  // hand-off from k_pick to the final kernels
  int32_t mode;     // 0 done; 1 kept = order prefix up to `last` (if has_last) with e' >= min_p
  int32_t has_last;
  int32_t last_id;
  int32_t pad;
  uint64_t last_key;
  double M, lse;
};

struct Layout {
  size_t seqs, marks, K, E, bins, part1, stats, part2, hcnt, hmh, hml, state, fsum, status, total;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// rows of the per-id arrays are padded to 8 ids (16-byte loads of the buckets)
int padded(int V) { return (V + 7) & ~7; }

Layout layout_of(int V, int S) {
  const size_t NB = (size_t)(V + kChunk - 1) / kChunk;
  const size_t NB1 = (size_t)(V + kChunk1 - 1) / kChunk1;
  const size_t Vp = (size_t)padded(V);
  Layout L;
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    size_t at = o;
    o += al256(bytes);
    return at;
  };
  L.seqs = take((size_t)S * sizeof(SeqParam));
  L.marks = take((size_t)S * V * 4);
  L.K = take((size_t)S * Vp * 8);
  L.E = take((size_t)S * Vp * 8);
  L.bins = take((size_t)S * Vp * 2);
  L.part1 = take((size_t)S * NB1 * sizeof(Part1));
  L.stats = take((size_t)S * sizeof(Stats));
  L.part2 = take((size_t)S * NB * sizeof(Part2));
  L.hcnt = take((size_t)S * kBins * 4);
  L.hmh = take((size_t)S * kBins * 8);
  L.hml = take((size_t)S * kBins * 8);
  L.state = take((size_t)S * sizeof(PickState));
  L.fsum = take((size_t)S * NB * sizeof(float2));
  L.status = take(256);
  L.total = o;
  return L;
}

// ---- double-f32 arithmetic --------------------------------------------------------

struct df {
  float h, l;
};

__device__ __forceinline__ df mk(float h, float l) {
  df r;
  r.h = h;
  r.l = l;
  return r;
}

// Knuth's two-sum: s + e == a + b exactly
__device__ __forceinline__ df two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  return mk(s, e);
}

// Dekker's fast two-sum, |a| >= |b| (or a == 0)
__device__ __forceinline__ df quick_two_sum(float a, float b) {
  const float s = a + b;
  return mk(s, b - (s - a));
}

// p + e == a * b exactly (one fused multiply-add)
__device__ __forceinline__ df two_prod(float a, float b) {
  const float p = a * b;
  return mk(p, fmaf(a, b, -p));
}

__device__ __forceinline__ df df_add(df a, df b) {
  df s = two_sum(a.h, b.h);
  const df t = two_sum(a.l, b.l);
  s.l += t.h;
  s = quick_two_sum(s.h, s.l);
  s.l += t.l;
  return quick_two_sum(s.h, s.l);
}

// a + b where no leading digits cancel (same signs, or |b| far below |a|):
// Dekker's shorter sum, error about 2^-47 relative
__device__ __forceinline__ df df_add_fast(df a, df b) {
  df s = two_sum(a.h, b.h);
  s.l += a.l + b.l;
  return quick_two_sum(s.h, s.l);
}

__device__ __forceinline__ df df_add_f(df a, float b) {  // a + b, b a float
  df s = two_sum(a.h, b);
  s.l += a.l;
  return quick_two_sum(s.h, s.l);
}

__device__ __forceinline__ df df_mul(df a, df b) {
  df p = two_prod(a.h, b.h);
  p.l = fmaf(a.h, b.l, fmaf(a.l, b.h, p.l));
  return quick_two_sum(p.h, p.l);
}

__device__ __forceinline__ bool df_ge(df a, df b) { return a.h > b.h || (a.h == b.h && a.l >= b.l); }
__device__ __forceinline__ bool df_gt(df a, df b) { return a.h > b.h || (a.h == b.h && a.l > b.l); }

__device__ __forceinline__ df df_of(double x) {
  const float h = __double2float_rn(x);
  return mk(h, __double2float_rn(x - (double)h));
}

__device__ __forceinline__ double dbl_of(df x) { return (double)x.h + (double)x.l; }

// Rounding without conversion instructions (they issue on the f64 pipe here):
// adding 1.5 * 2^23 rounds a float below 2^22 in magnitude to the nearest
// integer, which then sits in the low mantissa bits.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kMagicBits = 0x4B400000;

// nearest integer (ties to even) of |x| < 2^22, as a float and an int
__device__ __forceinline__ int round_i(float x, float& r) {
  const float y = x + kMagic;
  r = y - kMagic;
  return __float_as_int(y) - kMagicBits;
}

// floor of |x| < 2^22, as a float and an int
__device__ __forceinline__ int floor_i(float x, float& f) {
  float y = x + kMagic;
  f = y - kMagic;
  int i = __float_as_int(y) - kMagicBits;
  if (f > x) f -= 1.0f, --i;
  return i;
}

// floor of 0 <= x < 2^23 (adding 2^23 leaves the integer part in the mantissa)
__device__ __forceinline__ uint32_t floor_u(float x, float& f) {
  float y = x + 8388608.0f;
  f = y - 8388608.0f;
  if (f > x) f -= 1.0f, y -= 1.0f;
  return __float_as_uint(y) & 0x7FFFFFu;
}

// 2^(j/64) = head + tail, j = 0..63 (gen_exp_tables.py)
__device__ const float2 kExp2Tab[64] = {
  {0x1.0000000000000p+0f, 0x0.0p+0f},
  {0x1.02c9a40000000p+0f, -0x1.887fa00000000p-28f},
  {0x1.059b0e0000000p+0f, -0x1.9d4f520000000p-25f},
  {0x1.0874520000000p+0f, -0x1.e2990e0000000p-26f},
  {0x1.0b55860000000p+0f, 0x1.9f31220000000p-25f},
  {0x1.0e3ec40000000p+0f, -0x1.a585cc0000000p-25f},
  {0x1.11301e0000000p+0f, -0x1.fdb4960000000p-25f},
  {0x1.1429aa0000000p+0f, 0x1.d525bc0000000p-25f},
  {0x1.172b840000000p+0f, -0x1.c157420000000p-27f},
  {0x1.1a35be0000000p+0f, 0x1.6df96e0000000p-25f},
  {0x1.1d48740000000p+0f, -0x1.d2e8ca0000000p-25f},
  {0x1.2063b80000000p+0f, 0x1.0c519a0000000p-25f},
  {0x1.2387a60000000p+0f, 0x1.ceac480000000p-25f},
  {0x1.26b4560000000p+0f, 0x1.789f380000000p-26f},
  {0x1.29e9e00000000p+0f, -0x1.5c04240000000p-25f},
  {0x1.2d285a0000000p+0f, 0x1.b900c20000000p-26f},
  {0x1.306fe00000000p+0f, 0x1.4636e20000000p-25f},
  {0x1.33c08c0000000p+0f, -0x1.b37d200000000p-25f},
  {0x1.371a740000000p+0f, -0x1.18aac60000000p-25f},
  {0x1.3a7db40000000p+0f, -0x1.634c020000000p-25f},
  {0x1.3dea640000000p+0f, 0x1.8246840000000p-25f},
  {0x1.4160a20000000p+0f, 0x1.f72e2a0000000p-28f},
  {0x1.44e0860000000p+0f, 0x1.8624b40000000p-30f},
  {0x1.486a2c0000000p+0f, -0x1.47d8660000000p-25f},
  {0x1.4bfdae0000000p+0f, -0x1.593abc0000000p-25f},
  {0x1.4f9b280000000p+0f, -0x1.2c5a6c0000000p-25f},
  {0x1.5342b60000000p+0f, -0x1.2c56100000000p-25f},
  {0x1.56f4740000000p+0f, -0x1.295b040000000p-25f},
  {0x1.5ab07e0000000p+0f, -0x1.5bd5ec0000000p-27f},
  {0x1.5e76f20000000p+0f, -0x1.4a5bd60000000p-25f},
  {0x1.6247ec0000000p+0f, -0x1.f8b5500000000p-25f},
  {0x1.6623880000000p+0f, 0x1.2a91120000000p-27f},
  {0x1.6a09e60000000p+0f, 0x1.9fcef40000000p-26f},
  {0x1.6dfb240000000p+0f, -0x1.cd72e80000000p-27f},
  {0x1.71f75e0000000p+0f, 0x1.1d8bee0000000p-25f},
  {0x1.75feb60000000p+0f, -0x1.37b3060000000p-25f},
  {0x1.7a11480000000p+0f, -0x1.829fd00000000p-25f},
  {0x1.7e2f340000000p+0f, -0x1.2616340000000p-25f},
  {0x1.82589a0000000p+0f, -0x1.accc7c0000000p-26f},
  {0x1.868d9a0000000p+0f, -0x1.2edb440000000p-26f},
  {0x1.8ace540000000p+0f, 0x1.15506e0000000p-27f},
  {0x1.8f1aea0000000p+0f, -0x1.baa2320000000p-26f},
  {0x1.93737c0000000p+0f, -0x1.e647440000000p-25f},
  {0x1.97d82a0000000p+0f, -0x1.0d8d840000000p-31f},
  {0x1.9c49180000000p+0f, 0x1.51f8480000000p-27f},
  {0x1.a0c6680000000p+0f, -0x1.2886a60000000p-26f},
  {0x1.a5503c0000000p+0f, -0x1.b83b540000000p-25f},
  {0x1.a9e6b60000000p+0f, -0x1.50c0480000000p-25f},
  {0x1.ae89fa0000000p+0f, -0x1.a94b140000000p-26f},
  {0x1.b33a2c0000000p+0f, -0x1.ec3a820000000p-26f},
  {0x1.b7f7700000000p+0f, -0x1.a094380000000p-25f},
  {0x1.bcc1ea0000000p+0f, -0x1.f687c60000000p-25f},
  {0x1.c199be0000000p+0f, -0x1.3d56b20000000p-27f},
  {0x1.c67f120000000p+0f, 0x1.cafa2a0000000p-25f},
  {0x1.cb720e0000000p+0f, -0x1.8837cc0000000p-27f},
  {0x1.d072d40000000p+0f, 0x1.40f1300000000p-25f},
  {0x1.d5818e0000000p+0f, -0x1.822dbc0000000p-27f},
  {0x1.da9e600000000p+0f, 0x1.ed99420000000p-27f},
  {0x1.dfc9740000000p+0f, -0x1.908c940000000p-25f},
  {0x1.e502ee0000000p+0f, 0x1.e2cffe0000000p-26f},
  {0x1.ea4afa0000000p+0f, 0x1.52486c0000000p-27f},
  {0x1.efa1be0000000p+0f, 0x1.cc2b440000000p-25f},
  {0x1.f507660000000p+0f, -0x1.246eb00000000p-26f},
  {0x1.fa7c180000000p+0f, 0x1.9e90d80000000p-28f},
};

// ln2/64 = L1 + L2 + L3 + L4; L1..L3 have 11 significant bits, so k * Li is exact for |k| < 2^13
constexpr float kL1 = 0x1.62c0000000000p-7f;
constexpr float kL2 = 0x1.2140000000000p-18f;
constexpr float kL3 = 0x1.fbc0000000000p-29f;
constexpr float kL4 = 0x1.473de60000000p-40f;
constexpr float k64OverLn2 = 0x1.7154760000000p+6f;

// exp(x) for x <= 0 in double-f32 (Tang's table-driven method); 0 below -87
__device__ __forceinline__ df df_exp(df x) {
  if (!(x.h > -87.0f)) return mk(0.0f, 0.0f);
  float kf;
  const int k = round_i(x.h * k64OverLn2, kf);
  const float r0 = fmaf(-kf, kL1, x.h);  // exact: the two are within a factor of two
  df r = two_sum(r0, -kf * kL2);
  r = df_add_f(r, -kf * kL3);
  r = df_add_f(r, -kf * kL4);
  r = df_add_f(r, x.l);
  // exp(r) = 1 + r + r^2/2 + (r^3/6 + r^4/24 + r^5/120); |r^2/2| <= |r|/360 and the
  // bracket is below 3e-8, so no sum below cancels leading digits
  const df r2 = df_mul(r, r);
  const float rh = r.h;
  const float c = rh * rh * rh * (0.16666667f + rh * (0.041666668f + rh * 0.0083333338f));
  df s = df_add_fast(r, mk(0.5f * r2.h, 0.5f * r2.l));
  s = df_add_f(s, c);
  df e = quick_two_sum(1.0f, s.h);
  e.l += s.l;
  e = quick_two_sum(e.h, e.l);
  const float2 t = kExp2Tab[k & 63];
  e = df_mul(e, mk(t.x, t.y));
  const float sc = __int_as_float(((k >> 6) + 127) << 23);  // 2^n, n >= -126
  return mk(e.h * sc, e.l * sc);
}

// ---- keys, penalties, generator -------------------------------------------------------

__device__ __forceinline__ float load_logit(const float* x, int i, bool& bad) {
  float v = x[i];
  if (!(v < INFINITY)) {  // NaN or +inf: flagged, read as -inf
    bad = true;
    v = -INFINITY;
  }
  return v;
}

// the penalties in f64, with the rounding steps of the definition (no contraction)
__device__ __forceinline__ double penalize(float x, int32_t mk_, const SeqParam& q) {
  double l = (double)x;
  if (mk_ != 0) {
    l = l > 0.0 ? __ddiv_rn(l, q.rep) : __dmul_rn(l, q.rep);
    const int c = mk_ >> 1;
    if (c > 0) l = __dsub_rn(l, __dadd_rn(__dmul_rn(q.freq, (double)c), q.pres));
  }
  return l;
}

// order key of an f64 value: larger key = larger value; -0 and +0 share one key
__device__ __forceinline__ uint64_t okey_bits(uint64_t b) {
  if (b == 0x8000000000000000ull) b = 0;
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}
__device__ __forceinline__ uint64_t okey(double x) { return okey_bits((uint64_t)__double_as_longlong(x)); }

// okey((double)x) from the float's bits with integer operations
__device__ __forceinline__ uint64_t okey_f32(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t e = (u >> 23) & 0xFFu, m = u & 0x7FFFFFu;
  uint64_t b;
  if (e == 0) {
    if (m == 0) return 0x8000000000000000ull;  // +-0
    // subnormal m * 2^-149: the top bit p of m sets the f64 exponent p - 149
    const uint32_t pbit = 31u - (uint32_t)__clz(m);
    b = ((uint64_t)(u >> 31) << 63) | ((uint64_t)(pbit + 874u) << 52) | ((uint64_t)(m ^ (1u << pbit)) << (52u - pbit));
  } else if (e == 0xFFu) {
    b = ((uint64_t)(u >> 31) << 63) | 0x7FF0000000000000ull | ((uint64_t)m << 29);
  } else {
    b = ((uint64_t)(u >> 31) << 63) | ((uint64_t)(e + 896u) << 52) | ((uint64_t)m << 29);
  }
  return okey_bits(b);
}

__device__ __forceinline__ double key_value(uint64_t k) {
  const uint64_t b = (k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
  return __longlong_as_double((long long)b);
}

// (key, id) a comes before (key, id) b in (value desc, id asc) order
__device__ __forceinline__ bool before(uint64_t ka, int32_t ia, uint64_t kb, int32_t ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ unsigned __int128 ckey(uint64_t k, int32_t id) {
  return ((unsigned __int128)k << 32) | (uint32_t)(~(uint32_t)id);
}

struct Fix {
  unsigned long long h, l;
};

// a float in [0, 2^45] as floor (an integer, from two 22/23-bit pieces) and its
// exact fraction, with no conversion instructions
__device__ __forceinline__ unsigned long long floor45(float x, float& frac) {
  if (x >= 0x1p45f) {  // e' = 1 exactly
    frac = 0.0f;
    return 1ull << 45;
  }
  float a;
  const uint32_t ai = floor_u(x * 0x1p-22f, a);  // < 2^23
  const float r = fmaf(-a, 0x1p22f, x);           // exact, in [0, 2^22)
  float b;
  const uint32_t bi = floor_u(r, b);
  frac = r - b;                                   // exact, in [0, 1)
  return ((unsigned long long)ai << 22) + bi;
}

// a fraction f in [0, 1) in units of 2^-45, rounded: the same two-piece split
__device__ __forceinline__ unsigned long long frac45(float f) {
  float c;
  const uint32_t ci = floor_u(f * 0x1p23f, c);  // < 2^23
  const float r = fmaf(-c, 0x1p-23f, f);         // exact, in [0, 2^-23)
  float rr;
  const int ri = round_i(r * 0x1p45f, rr);       // <= 2^22
  return ((unsigned long long)ci << 22) + (uint32_t)ri;
}

// e' (head + tail, >= 0) as fixed point: h units of 2^-45 plus l units of 2^-90
__device__ __forceinline__ Fix fix_of(float2 e) {
  const float xh = e.x * kFixF, xl = e.y * kFixF;  // exact scalings; |xl| <= 2^21
  float fh, il;
  const unsigned long long ih = floor45(xh, fh);
  const int ili = floor_i(xl, il);
  const float fl = xl - il;                        // exact, in [0, 1)
  Fix f;
  f.h = ih + (unsigned long long)(long long)ili;
  f.l = frac45(fh) + frac45(fl);
  return f;
}

__device__ __forceinline__ df u64_df(unsigned long long x) {  // x < 2^63
  const float h = __ull2float_rn(x);
  return mk(h, __ll2float_rn((long long)(x - (unsigned long long)h)));
}

// h * 2^-45 + l * 2^-90 as double-f32
__device__ __forceinline__ df fix_df(unsigned long long h, unsigned long long l) {
  h += l >> kFixBits;
  l &= (1ull << kFixBits) - 1;
  const df a = u64_df(h);
  const float s = 1.0f / kFixF;
  return df_add(mk(a.h * s, a.l * s), mk(__ull2float_rn(l) * (s * s), 0.0f));
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

// ---- block reductions (fixed trees) ------------------------------------------------------

__device__ __forceinline__ df shfl_xor_df(df v, int o) {
  return mk(__shfl_xor_sync(0xffffffffu, v.h, o), __shfl_xor_sync(0xffffffffu, v.l, o));
}

template <int NT>
__device__ df block_sum_df(df v, float2* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = make_float2(v.h, v.l);
  __syncthreads();
  const float2 r = red[l & (NT / 32 - 1)];
  df t = l < NT / 32 ? mk(r.x, r.y) : mk(0.0f, 0.0f);
#pragma unroll
  for (int o = 16; o; o >>= 1) t = df_add(t, shfl_xor_df(t, o));
  return t;  // every thread holds the total
}

// the largest key, lowest id on ties
template <int NT>
__device__ void block_maxkey(uint64_t& k, int& id, unsigned long long* redk, int* redi) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint64_t ok = __shfl_xor_sync(0xffffffffu, (unsigned long long)k, o);
    const int oi = __shfl_xor_sync(0xffffffffu, id, o);
    if (before(ok, oi, k, id)) k = ok, id = oi;
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) redk[w] = k, redi[w] = id;
  __syncthreads();
  const int src = l & (NT / 32 - 1);
  k = l < NT / 32 ? redk[src] : 0ull;
  id = l < NT / 32 ? redi[src] : 0x7fffffff;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint64_t ok = __shfl_xor_sync(0xffffffffu, (unsigned long long)k, o);
    const int oi = __shfl_xor_sync(0xffffffffu, id, o);
    if (before(ok, oi, k, id)) k = ok, id = oi;
  }
}

template <int NT>
__device__ float block_minf(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = l < NT / 32 ? red[l & (NT / 32 - 1)] : INFINITY;
#pragma unroll
  for (int o = 16; o; o >>= 1) t = fminf(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

// inclusive scan of one value per thread over 1024 threads (fixed tree)
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

// the same for double-f32 values
__device__ df block_scan_df(df v, float2* red, df& total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const df n = mk(__shfl_up_sync(0xffffffffu, v.h, o), __shfl_up_sync(0xffffffffu, v.l, o));
    if (l >= o) v = df_add(v, n);
  }
  __syncthreads();
  if (l == 31) red[w] = make_float2(v.h, v.l);
  __syncthreads();
  if (w == 0) {
    const float2 r = red[l];
    df t = mk(r.x, r.y);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const df n = mk(__shfl_up_sync(0xffffffffu, t.h, o), __shfl_up_sync(0xffffffffu, t.l, o));
      if (l >= o) t = df_add(t, n);
    }
    red[l] = make_float2(t.h, t.l);
  }
  __syncthreads();
  const float2 x = red[l];
  total = mk(__shfl_sync(0xffffffffu, x.x, 31), __shfl_sync(0xffffffffu, x.y, 31));
  df off = mk(__shfl_sync(0xffffffffu, x.x, (w + 31) & 31), __shfl_sync(0xffffffffu, x.y, (w + 31) & 31));
  if (w == 0) off = mk(0.0f, 0.0f);
  __syncthreads();
  return df_add(v, off);
}

struct Pen {
  uint64_t key;
  float h, l;
};

// a penalised id (a rare branch: kept out of line so that its f64 work is
// never issued, predicated off, for the other ids)
__device__ __noinline__ Pen penalized_logit(float v, int32_t m, const SeqParam& q) {
  const double d = penalize(v, m, q);
  const df l = df_of(d);
  Pen r;
  r.key = okey(d);
  r.h = l.h;
  r.l = l.l;
  return r;
}

// the penalised logit as a double-f32 pair, its order key and its float
__device__ __forceinline__ void logit_of(float v, int32_t m, const SeqParam& q, df& l, uint64_t& key, float& lf) {
  if (m == 0) {
    l = mk(v, 0.0f);
    key = okey_f32(v);
    lf = v;
  } else {
    const Pen r = penalized_logit(v, m, q);
    l = mk(r.h, r.l);
    key = r.key;
    lf = r.h;
  }
}

// ---- history marks ----------------------------------------------------------------

__global__ void k_mark(const SeqParam* __restrict__ sp, const int32_t* __restrict__ hist, int32_t* marks, int V,
                       int set, uint32_t* status) {
  const int s = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const SeqParam& q = sp[s];
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
  __shared__ unsigned long long redk[32];
  __shared__ int redi[32];
  __shared__ float redf[32];
  const int s = blockIdx.y, b = blockIdx.x, t = threadIdx.x;
  const SeqParam& q = sp[s];
  const float* x = logits + (size_t)s * ld;
  const int32_t* mkv = marks + (size_t)s * V;
  uint64_t bk = 0;
  int ba = 0x7fffffff;
  float mn = INFINITY;
  bool bad = false;
  constexpr int kPer = kChunk1 / kScanThreads;
  float xv[kPer];
  int32_t mv[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {  // every load first, then the work
    const int i = b * kChunk1 + j * kScanThreads + t;
    xv[j] = i < V ? x[i] : -INFINITY;
    mv[j] = i < V ? mkv[i] : 0;
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = b * kChunk1 + j * kScanThreads + t;
    if (i < V) {
      float v = xv[j];
      if (!(v < INFINITY)) bad = true, v = -INFINITY;  // NaN or +inf: flagged, read as -inf
      const int32_t m = mv[j];
      df l;
      uint64_t key;
      float lf;
      logit_of(v, m, q, l, key, lf);
      if (key > bk) bk = key, ba = i;  // ids rise: ties keep the lowest
      if (lf > -INFINITY && lf < mn) mn = lf;
    }
  }
  if (bad) atomicOr(status, (uint32_t)DEC_SAMPLE_BAD_LOGIT);
  block_maxkey<kScanThreads>(bk, ba, redk, redi);
  const float mnb = block_minf<kScanThreads>(mn, redf);
  if (t == 0) {
    Part1 p;
    p.key = bk;
    p.mn = mnb;
    p.arg = ba;
    part[(size_t)s * NB + b] = p;
  }
}

// every CTA reduces the per-chunk maxima the same way: the top key, its lowest id, the finite minimum
template <int NT>
__device__ void reduce_part1(const Part1* p, int NB, uint64_t& M, int& arg, float& mn, unsigned long long* redk,
                             int* redi, float* redf) {
  uint64_t k = 0;
  int id = 0x7fffffff;
  float m = INFINITY;
  for (int c = threadIdx.x; c < NB; c += NT) {
    const Part1 e = p[c];
    if (before(e.key, e.arg, k, id)) k = e.key, id = e.arg;
    m = fminf(m, e.mn);
  }
  block_maxkey<NT>(k, id, redk, redi);
  mn = block_minf<NT>(m, redf);
  M = k;
  arg = id;
}

// one CTA per sequence: the maximum and minimum over the per-chunk partials
__global__ void __launch_bounds__(kScanThreads) k_stats(const Part1* __restrict__ part1, int NB1,
                                                         Stats* __restrict__ stats, uint32_t* status) {
  __shared__ unsigned long long redk[32];
  __shared__ int redi[32];
  __shared__ float redf[32];
  const int s = blockIdx.x;
  uint64_t Mk;
  int arg;
  float mn;
  reduce_part1<kScanThreads>(part1 + (size_t)s * NB1, NB1, Mk, arg, mn, redk, redi, redf);
  if (threadIdx.x == 0) {
    Stats st;
    st.key = Mk;
    st.M = key_value(Mk);
    const df Md = df_of(st.M);
    st.Mh = Md.h;
    st.Ml = Md.l;
    st.mn = mn;
    st.arg = arg;
    if (!(st.M > -INFINITY)) {  // no finite logit
      atomicOr(status, (uint32_t)DEC_SAMPLE_NO_FINITE);
      st.Mh = -INFINITY;
      st.Ml = 0.0f;
    }
    stats[s] = st;
  }
}


__global__ void __launch_bounds__(kScanThreads) k_scan2(const float* __restrict__ logits, int64_t ld,
                                                         const int32_t* __restrict__ marks,
                                                         const SeqParam* __restrict__ sp, int V, int Vp, int NB,
                                                         const Stats* __restrict__ stats, Part2* __restrict__ part2,
                                                         uint64_t* __restrict__ K, float2* __restrict__ E,
                                                         uint16_t* __restrict__ bins, uint32_t* __restrict__ hcnt,
                                                         unsigned long long* __restrict__ hmh,
                                                         unsigned long long* __restrict__ hml) {
  __shared__ float2 redd[32];
  __shared__ uint32_t sc[kBins];
  __shared__ unsigned long long sh[kBins], sl[kBins];
  const int s = blockIdx.y, b = blockIdx.x, t = threadIdx.x;
  const SeqParam& q = sp[s];
  const Stats stt = stats[s];
  const float Mh = stt.Mh, Ml = stt.Ml, mn = stt.mn;
  if (!(Mh > -INFINITY)) return;  // no finite logit (flagged by k_stats)
  const int flags = q.flags;
  const bool sampling = flags & kSampling;
  const bool unit = flags & kUnitT;
  const df rT = mk(q.rTh, q.rTl);
  const float R = Mh - mn;
  float scale = R > 0.0f ? (float)kBins / R : 0.0f;
  if (!(scale < 1e30f)) scale = 0.0f;
  if (sampling) {
    for (int i = t; i < kBins; i += kScanThreads) sc[i] = 0, sh[i] = 0, sl[i] = 0;
    __syncthreads();
  }
  const float* x = logits + (size_t)s * ld;
  const int32_t* mkv = marks + (size_t)s * V;
  const size_t row = (size_t)s * Vp;
  df z = mk(0.0f, 0.0f), z2 = mk(0.0f, 0.0f);
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kChunk / kScanThreads; ++j) {
    const int i = b * kChunk + j * kScanThreads + t;
    if (i < V) {
      df l;
      uint64_t key;
      float lf;
      logit_of(load_logit(x, i, bad), mkv[i], q, l, key, lf);
      df e = mk(0.0f, 0.0f), e2 = mk(0.0f, 0.0f);
      if (lf > -INFINITY) {
        df d = two_sum(l.h, -Mh);
        if (l.l != 0.0f || Ml != 0.0f) d = df_add(d, mk(l.l - Ml, 0.0f));
        e = df_exp(d);
        if (sampling) e2 = unit ? e : df_exp(df_mul(d, rT));
      }
      z = df_add_fast(z, e);
      if (sampling) {
        z2 = df_add_fast(z2, e2);
        K[row + i] = key;
        E[row + i] = make_float2(e2.h, e2.l);
        float bf;
        const int bin = scale > 0.0f ? (int)floor_u(fminf((Mh - lf) * scale, (float)(kBins - 1)), bf) : 0;
        bins[row + i] = (uint16_t)bin;
        atomicAdd(&sc[bin], 1u);
        const Fix f = fix_of(make_float2(e2.h, e2.l));
        atomicAdd(&sh[bin], f.h);
        atomicAdd(&sl[bin], f.l);
      }
    }
  }
  (void)bad;  // k_scan1 already flagged it
  z = block_sum_df<kScanThreads>(z, redd);
  z2 = block_sum_df<kScanThreads>(z2, redd);
  if (t == 0) {
    Part2 p;
    p.zh = z.h;
    p.zl = z.l;
    p.z2h = z2.h;
    p.z2l = z2.l;
    part2[(size_t)s * NB + b] = p;
  }
  if (sampling) {
    __syncthreads();
    for (int i = t; i < kBins; i += kScanThreads)
      if (sc[i]) {
        atomicAdd(&hcnt[(size_t)s * kBins + i], sc[i]);
        atomicAdd(&hmh[(size_t)s * kBins + i], sh[i]);
        atomicAdd(&hml[(size_t)s * kBins + i], sl[i]);
      }
  }
}

// ---- the one-CTA pick ---------------------------------------------------------------------

struct PickSmem {
  uint64_t ck[kCap];   // order keys of the candidates
  float2 ce[kCap];     // their e' (head, tail)
  int32_t cid[kCap];   // their ids
  uint32_t hc[kBins];  // bucket (or digit) counts
  unsigned long long hmh[kBins], hml[kBins];  // bucket masses: integer and fraction words
  float2 redd[32];
  unsigned long long redk[32];
  int redi[32];
  float redf[32];
  int n;
  int flag;
};

struct Frame {      // where a gathered list sits in the order
  long long above;  // elements of the restricted set before the list
  df m_above;       // their e' sum
};

enum { kCount = 0, kMass = 1 };

struct Lim {  // restriction to the order prefix ending at (key, id), bucket `bin`
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

__device__ __forceinline__ df ce_of(const PickSmem& sm, int j) { return mk(sm.ce[j].x, sm.ce[j].y); }

// bitonic sort of sm.ck/ce/cid[0..n) in (key desc, id asc) order (by_id: id asc)
__device__ void sort_list(PickSmem& sm, int n, bool by_id) {
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + threadIdx.x; i < P; i += kPick) sm.ck[i] = 0, sm.ce[i] = make_float2(0.f, 0.f), sm.cid[i] = 0x7fffffff;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += kPick) {
        const int p = i ^ j;
        if (p > i) {
          const bool up = (i & k) == 0;
          const bool first_is_i = by_id ? sm.cid[i] < sm.cid[p] : before(sm.ck[i], sm.cid[i], sm.ck[p], sm.cid[p]);
          if (first_is_i != up) {
            const uint64_t tk = sm.ck[i];
            sm.ck[i] = sm.ck[p];
            sm.ck[p] = tk;
            const float2 te = sm.ce[i];
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

// a mass target in the integer word's units (2^-45), floored, with `slack` units either side
__device__ __forceinline__ unsigned long long fix_target(df tm, double slack) {
  const double v = dbl_of(tm) * kFix + slack;
  return v <= 0.0 ? 0ull : (v >= 1.8e19 ? ~0ull : (unsigned long long)v);
}

// Gather, into shared memory and sorted, the stretch of the order where a
// cumulative target is reached: count target `tc` elements, or e' mass `tm`,
// over the elements allowed by `lim`.  Level 0 uses the bucket histogram in
// sm.hc/hmh/hml (already restricted).  Returns the frame of the list.
__device__ Frame gather(PickSmem& sm, int kind, long long tc, df tm, const Lim& lim, const uint16_t* bins,
                        const uint64_t* K, const float2* E, int V, uint32_t* status) {
  const int t = threadIdx.x;
  __shared__ int s_lo, s_hi;
  __shared__ long long s_cnt_hi, s_cnt_before;
  __shared__ unsigned long long s_mh_before, s_ml_before;
  const unsigned long long lo_u = kind == kMass ? fix_target(tm, -kFixSlack) : 0ull;
  const unsigned long long hi_u = kind == kMass ? fix_target(tm, kFixSlack) : 0ull;
  const unsigned long long mid_u = kind == kMass ? fix_target(tm, 0.0) : 0ull;
  // ---- level 0: cumulative bucket counts and masses, two buckets per thread
  {
    const uint32_t c0 = sm.hc[2 * t], c1 = sm.hc[2 * t + 1];
    const unsigned long long h0 = sm.hmh[2 * t], h1 = sm.hmh[2 * t + 1];
    const unsigned long long l0 = sm.hml[2 * t], l1 = sm.hml[2 * t + 1];
    // the walk compares integer words with the fraction words' carries folded in
    const unsigned long long m0 = h0 + (l0 >> kFixBits), m1 = h1 + (l1 >> kFixBits);
    unsigned long long ctot, mtot, htot, ltot;
    const unsigned long long cinc = block_scan<unsigned long long>((unsigned long long)c0 + c1, sm.redk, ctot);
    const unsigned long long minc = block_scan<unsigned long long>(m0 + m1, sm.redk, mtot);
    const unsigned long long hinc = block_scan<unsigned long long>(h0 + h1, sm.redk, htot);
    const unsigned long long linc = block_scan<unsigned long long>(l0 + l1, sm.redk, ltot);
    const unsigned long long cb0 = cinc - c0 - c1, mb0 = minc - m0 - m1;  // before bucket 2t
    const unsigned long long ca0 = cb0 + c0, ma0 = mb0 + m0;              // through bucket 2t
    const unsigned long long hb0 = hinc - h0 - h1, lb0 = linc - l0 - l1;
    if (t == 0) s_lo = kBins - 1, s_hi = kBins - 1;
    __syncthreads();
    if (kind == kCount) {
      const unsigned long long tcu = (unsigned long long)tc;
      if (ca0 >= tcu && cb0 < tcu) atomicMin(&s_lo, 2 * t);
      if (cinc >= tcu && ca0 < tcu) atomicMin(&s_lo, 2 * t + 1);
    } else {
      if (ma0 >= lo_u)
        atomicMin(&s_lo, 2 * t);
      else if (minc >= lo_u)
        atomicMin(&s_lo, 2 * t + 1);
      if (ma0 >= hi_u)
        atomicMin(&s_hi, 2 * t);
      else if (minc >= hi_u)
        atomicMin(&s_hi, 2 * t + 1);
    }
    __syncthreads();
    if (kind == kCount && t == 0) s_hi = s_lo;
    __syncthreads();
    const int lo = s_lo, hi = s_hi;
    if (2 * t == lo) s_cnt_before = (long long)cb0, s_mh_before = hb0, s_ml_before = lb0;
    if (2 * t + 1 == lo) s_cnt_before = (long long)ca0, s_mh_before = hb0 + h0, s_ml_before = lb0 + l0;
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
  unsigned long long r_h = s_mh_before, r_l = s_ml_before;
  if (mode == 2) {
    __shared__ int s_d;
    __shared__ long long s_above;
    __shared__ unsigned long long s_h, s_l;
    while (true) {
      for (int i = t; i < 256; i += kPick) sm.hc[i] = 0, sm.hmh[i] = 0, sm.hml[i] = 0;
      __syncthreads();
      for (int i = t; i < V; i += kPick) {
        const int bn = bins[i];
        if (bn < lo || bn > hi) continue;
        const uint64_t k = K[i];
        if (!in_lim(lim, bn, k, i)) continue;
        const unsigned __int128 Kc = ckey(k, i);
        if (shift < 96 && (Kc >> shift) != pre) continue;
        const int d = (int)((Kc >> (shift - 8)) & 255);
        atomicAdd(&sm.hc[d], 1u);
        const Fix f = fix_of(E[i]);
        atomicAdd(&sm.hmh[d], f.h);
        atomicAdd(&sm.hml[d], f.l);
      }
      __syncthreads();
      // walk digits from 255 (earliest) down: one thread, 256 steps
      if (t == 0) {
        long long c = r_above;
        unsigned long long h = r_h, l = r_l;
        int pick = -1, last = -1;
        for (int d = 255; d >= 0; --d) {
          if (!sm.hc[d]) continue;
          last = d;
          const long long c2 = c + sm.hc[d];
          const unsigned long long h2 = h + sm.hmh[d], l2 = l + sm.hml[d];
          const bool hit = kind == kCount ? c2 >= tc : h2 + (l2 >> kFixBits) >= mid_u;
          if (hit) {
            pick = d;
            break;
          }
          c = c2;
          h = h2;
          l = l2;
        }
        if (pick < 0 && last >= 0) {  // target beyond the set (rounding): the last digit holds the end
          pick = last;
          c -= sm.hc[last];
          h -= sm.hmh[last];
          l -= sm.hml[last];
        }
        if (pick < 0) {  // no element matched (cannot happen: the digit was non-empty)
          atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW);
          pick = 0;
        }
        s_d = pick;
        s_above = c;
        s_h = h;
        s_l = l;
      }
      __syncthreads();
      const int d = s_d;
      const uint32_t cd = sm.hc[d];
      r_above = s_above;
      r_h = s_h;
      r_l = s_l;
      pre = (pre << 8) | (unsigned __int128)d;
      shift -= 8;
      __syncthreads();
      if (cd <= (uint32_t)kCap || shift == 0) break;
    }
  }

  // ---- gather: eight buckets per 16-byte load
  if (t == 0) sm.n = 0;
  __syncthreads();
  const uint4* b4 = reinterpret_cast<const uint4*>(bins);
  const int n8 = (V + 7) >> 3;
  for (int g = t; g < n8; g += kPick) {
    const uint4 w = b4[g];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 8 * g + q;
      const int bn = (int)((ws[q >> 1] >> ((q & 1) * 16)) & 0xFFFFu);
      if (i >= V || bn > hi || (mode != 0 && bn < lo)) continue;
      const uint64_t k = K[i];
      if (!in_lim(lim, bn, k, i)) continue;
      if (mode == 2 && (ckey(k, i) >> shift) != pre) continue;
      const int slot = atomicAdd(&sm.n, 1);
      if (slot < kCap) sm.ck[slot] = k, sm.ce[slot] = E[i], sm.cid[slot] = i;
    }
  }
  __syncthreads();
  if (sm.n > kCap) {
    if (t == 0) atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW);
    __syncthreads();
    if (t == 0) sm.n = kCap;
    __syncthreads();
  }
  sort_list(sm, sm.n, false);
  Frame f;
  f.above = mode == 0 ? 0 : r_above;
  f.m_above = mode == 0 ? mk(0.0f, 0.0f) : fix_df(r_h, r_l);
  return f;
}

// first list index j (< n) where start + sum_{i<=j} ce_i >= target; n-1 if never
__device__ int walk_mass(PickSmem& sm, int n, df start, df target) {
  const int t = threadIdx.x;
  df v[4];
  df run = mk(0.0f, 0.0f);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = 4 * t + r;
    if (j < n) run = df_add(run, ce_of(sm, j));
    v[r] = run;
  }
  df total;
  const df inc = block_scan_df(run, sm.redd, total);
  const df base = df_add(start, df_add(inc, mk(-run.h, -run.l)));  // start + exclusive prefix
  __shared__ int s_first;
  if (t == 0) s_first = n - 1;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = 4 * t + r;
    if (j < n && df_ge(df_add(base, v[r]), target)) {
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
__device__ df list_sum(PickSmem& sm, int n) {
  df v = mk(0.0f, 0.0f);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = 4 * threadIdx.x + r;
    if (j < n) v = df_add(v, ce_of(sm, j));
  }
  return block_sum_df<kPick>(v, sm.redd);
}

__device__ double logprob_of(const float* x, const int32_t* mkv, int id, const SeqParam& q, double M, double lse) {
  bool bad = false;
  return (penalize(load_logit(x, id, bad), mkv[id], q) - M) - lse;
}

// the bucket histogram of one sequence, restricted to the order prefix `lim` allows
__device__ void load_hist(PickSmem& sm, const Lim& lim, const uint32_t* hc, const unsigned long long* hh,
                          const unsigned long long* hl, const uint16_t* bins, const uint64_t* K, const float2* E,
                          int V) {
  const int t = threadIdx.x;
  for (int i = t; i < kBins; i += kPick) {
    const bool cut = lim.on && i > lim.bin;
    sm.hc[i] = cut ? 0u : hc[i];
    sm.hmh[i] = cut ? 0ull : hh[i];
    sm.hml[i] = cut ? 0ull : hl[i];
  }
  __syncthreads();
  if (!lim.on) return;
  // the limit's own bucket: only the elements at or before the limit
  __shared__ unsigned int s_c;
  __shared__ unsigned long long s_h, s_l;
  if (t == 0) s_c = 0, s_h = 0, s_l = 0;
  __syncthreads();
  unsigned int c = 0;
  unsigned long long h = 0, l = 0;
  for (int i = t; i < V; i += kPick) {
    if (bins[i] != lim.bin) continue;
    if (in_lim(lim, lim.bin, K[i], i)) {
      const Fix f = fix_of(E[i]);
      ++c, h += f.h, l += f.l;
    }
  }
  atomicAdd(&s_c, c);
  atomicAdd(&s_h, h);
  atomicAdd(&s_l, l);
  __syncthreads();
  if (t == 0) sm.hc[lim.bin] = s_c, sm.hmh[lim.bin] = s_h, sm.hml[lim.bin] = s_l;
  __syncthreads();
}

__global__ void __launch_bounds__(kPick, 1) k_pick(const float* __restrict__ logits, int64_t ld,
                                                    const int32_t* __restrict__ marks,
                                                    const SeqParam* __restrict__ sp, int V, int Vp, int NB,
                                                    const Stats* __restrict__ stats, const Part2* __restrict__ part2,
                                                    const uint64_t* __restrict__ Kall, const float2* __restrict__ Eall,
                                                    const uint16_t* __restrict__ ball, const uint32_t* __restrict__ hcnt,
                                                    const unsigned long long* __restrict__ hmh,
                                                    const unsigned long long* __restrict__ hml,
                                                    PickState* __restrict__ state, dec_rng* __restrict__ rng,
                                                    int32_t* __restrict__ tokens, double* __restrict__ logprobs,
                                                    uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PickSmem& sm = *reinterpret_cast<PickSmem*>(smem_raw);
  __shared__ double s_lse;
  const int s = blockIdx.x, t = threadIdx.x;
  const SeqParam& q = sp[s];
  const Stats stt = stats[s];
  const float* x = logits + (size_t)s * ld;
  const int32_t* mkv = marks + (size_t)s * V;
  const size_t row = (size_t)s * Vp;
  const uint64_t* K = Kall + row;
  const float2* E = Eall + row;
  const uint16_t* bins = ball + row;
  const size_t hrow = (size_t)s * kBins;

  const double M = stt.M;
  const int arg = stt.arg;
  Part2 pz;
  pz.zh = pz.zl = pz.z2h = pz.z2l = 0.0f;
  if (t < NB) pz = part2[(size_t)s * NB + t];
  const df Z = block_sum_df<kPick>(mk(pz.zh, pz.zl), sm.redd);
  const df Zall = block_sum_df<kPick>(mk(pz.z2h, pz.z2l), sm.redd);
  if (t == 0) s_lse = log(dbl_of(Z));  // the only f64 transcendental: one logarithm per sequence
  __syncthreads();
  const double lse = s_lse;
  PickState st;
  st.mode = 0;
  st.has_last = 0;
  st.last_id = 0;
  st.pad = 0;
  st.last_key = 0;
  st.M = M;
  st.lse = lse;
  if (!(M > -INFINITY)) {  // flagged by k_stats
    if (t == 0) {
      tokens[s] = -1;
      logprobs[s] = -INFINITY;
      state[s] = st;
    }
    return;
  }
  const int flags = q.flags;
  if (!(flags & kSampling)) {  // greedy: no draw
    if (t == 0) {
      tokens[s] = arg;
      logprobs[s] = (M - M) - lse;
      state[s] = st;
    }
    return;
  }
  const long long kk = (q.top_k > 0 && q.top_k < V) ? q.top_k : V;
  const bool p_on = flags & kTopP;
  const bool m_on = flags & kMinP;
  const df minp = mk(q.mph, q.mpl);

  // the list: (has_list) sm holds n sorted elements starting `above` into the order;
  // the kept prefix ends at list index `end`
  bool has_list = false;
  int n = 0, end = -1;
  Frame fr;
  fr.above = 0;
  fr.m_above = mk(0.0f, 0.0f);
  df Zk = Zall;
  Lim none;
  none.on = 0;
  none.key = 0;
  none.id = 0;
  none.bin = 0;

  // ---- top-k
  Lim klim = none;
  if (kk < V) {
    load_hist(sm, none, hcnt + hrow, hmh + hrow, hml + hrow, bins, K, E, V);
    fr = gather(sm, kCount, kk, mk(0.0f, 0.0f), none, bins, K, E, V, status);
    has_list = true;
    n = sm.n;
    if (n == 0) {  // cannot happen: the bucket walk found the k-th element
      if (t == 0) atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW), tokens[s] = arg, logprobs[s] = -lse, state[s] = st;
      return;
    }
    end = (int)(kk - fr.above - 1);
    if (end >= n) end = n - 1;  // cannot happen unless capacity overflowed
    if (end < 0) end = 0;
    Zk = df_add(fr.m_above, list_sum(sm, end + 1));
    klim.on = 1;
    klim.key = sm.ck[end];
    klim.id = sm.cid[end];
    klim.bin = bins[klim.id];
    __syncthreads();
  }

  // ---- nucleus: the running e' sum reaches p * Zk
  if (p_on) {
    const df target = df_mul(mk(q.pph, q.ppl), Zk);
    if (has_list && fr.above == 0) {
      end = walk_mass(sm, end + 1, mk(0.0f, 0.0f), target);
    } else {
      load_hist(sm, klim, hcnt + hrow, hmh + hrow, hml + hrow, bins, K, E, V);
      fr = gather(sm, kMass, 0, target, klim, bins, K, E, V, status);
      has_list = true;
      n = sm.n;
      if (n == 0) {  // cannot happen: the restricted set holds at least the top
        if (t == 0) atomicOr(status, (uint32_t)DEC_SAMPLE_OVERFLOW), tokens[s] = arg, logprobs[s] = -lse, state[s] = st;
        return;
      }
      end = walk_mass(sm, n, fr.m_above, target);
    }
  }

  // ---- final: in shared memory when the whole kept set is the list's head.
  // min-p keeps e' >= min_p (e' of the top id is exactly 1)
  const bool whole = has_list && fr.above == 0;
  if (whole) {
    int nf = end + 1;
    if (m_on) {
      __shared__ int s_nf;
      if (t == 0) s_nf = 1;
      __syncthreads();
      for (int j = t; j < nf; j += kPick)
        if (df_ge(ce_of(sm, j), minp)) atomicMax(&s_nf, j + 1);
      __syncthreads();
      nf = s_nf;
      __syncthreads();
    }
    sort_list(sm, nf, true);  // ascending ids
    const df Zf = list_sum(sm, nf);
    __shared__ double s_u;
    __shared__ uint64_t s_state;
    if (t == 0) {
      const dec_rng r = rng[s];
      uint64_t g = r.state;
      s_u = pcg_uniform(g, r.inc);
      s_state = g;
    }
    __syncthreads();
    const df target = df_mul(df_of(s_u), Zf);  // u < c_j  <=>  u * Zf < running e' sum
    df v[4];
    df run = mk(0.0f, 0.0f);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = 4 * t + r;
      if (j < nf) run = df_add(run, ce_of(sm, j));
      v[r] = run;
    }
    df total;
    const df inc = block_scan_df(run, sm.redd, total);
    const df base = df_add(inc, mk(-run.h, -run.l));
    __shared__ int s_tok;
    if (t == 0) s_tok = nf - 1;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = 4 * t + r;
      if (j < nf && df_gt(df_add(base, v[r]), target)) {
        atomicMin(&s_tok, j);
        break;
      }
    }
    __syncthreads();
    if (t == 0) {
      const int tok = sm.cid[s_tok];
      tokens[s] = tok;
      logprobs[s] = logprob_of(x, mkv, tok, q, M, lse);
      rng[s].state = s_state;
      state[s] = st;
    }
    return;
  }
  // ---- hand-off: the kept set is the order prefix through `last` with e' >= min_p
  if (t == 0) {
    st.mode = 1;
    st.has_last = has_list ? 1 : 0;
    if (has_list) st.last_key = sm.ck[end], st.last_id = sm.cid[end];
    state[s] = st;
  }
}

__device__ __forceinline__ bool kept_by(const PickState& st, const SeqParam& q, uint64_t k, float2 e, int i) {
  if (st.has_last && before(st.last_key, st.last_id, k, i)) return false;
  return !(q.flags & kMinP) || df_ge(mk(e.x, e.y), mk(q.mph, q.mpl));
}

__global__ void __launch_bounds__(kScanThreads) k_final_sum(const SeqParam* __restrict__ sp,
                                                             const PickState* __restrict__ state, int V, int Vp,
                                                             int NB, const uint64_t* __restrict__ Kall,
                                                             const float2* __restrict__ Eall,
                                                             float2* __restrict__ fsum) {
  __shared__ float2 red[32];
  const int s = blockIdx.y, b = blockIdx.x, t = threadIdx.x;
  const PickState st = state[s];
  if (st.mode == 0) return;
  const SeqParam& q = sp[s];
  const size_t row = (size_t)s * Vp;
  df v = mk(0.0f, 0.0f);
#pragma unroll
  for (int j = 0; j < kChunk / kScanThreads; ++j) {
    const int i = b * kChunk + j * kScanThreads + t;
    if (i < V) {
      const float2 e = Eall[row + i];
      if (kept_by(st, q, st.has_last ? Kall[row + i] : 0ull, e, i)) v = df_add(v, mk(e.x, e.y));
    }
  }
  v = block_sum_df<kScanThreads>(v, red);
  if (t == 0) fsum[(size_t)s * NB + b] = make_float2(v.h, v.l);
}

__global__ void __launch_bounds__(kPick, 1) k_final_pick(const float* __restrict__ logits, int64_t ld,
                                                          const int32_t* __restrict__ marks,
                                                          const SeqParam* __restrict__ sp,
                                                          const PickState* __restrict__ state, int V, int Vp, int NB,
                                                          const uint64_t* __restrict__ Kall,
                                                          const float2* __restrict__ Eall,
                                                          const float2* __restrict__ fsum, dec_rng* __restrict__ rng,
                                                          int32_t* __restrict__ tokens, double* __restrict__ logprobs) {
  __shared__ float2 redd[32];
  __shared__ double s_u;
  __shared__ uint64_t s_state;
  __shared__ int s_chunk, s_tok, s_last, s_lastid;
  __shared__ float2 s_base;
  const int s = blockIdx.x, t = threadIdx.x;
  const PickState st = state[s];
  if (st.mode == 0) return;
  const SeqParam& q = sp[s];
  const size_t row = (size_t)s * Vp;
  float2 f2 = make_float2(0.f, 0.f);
  if (t < NB) f2 = fsum[(size_t)s * NB + t];
  const df fs = mk(f2.x, f2.y);
  const df Zf = block_sum_df<kPick>(fs, redd);
  df tot;
  const df cinc = block_scan_df(fs, redd, tot);
  if (t == 0) {
    const dec_rng r = rng[s];
    uint64_t g = r.state;
    s_u = pcg_uniform(g, r.inc);
    s_state = g;
    s_chunk = NB;
    s_last = -1;
    s_tok = 0x7fffffff;
    s_lastid = -1;
  }
  __syncthreads();
  const df target = df_mul(df_of(s_u), Zf);  // u < c  <=>  u * Zf < running e' sum
  if (t < NB && df_gt(cinc, target)) atomicMin(&s_chunk, t);
  if (t < NB && fs.h > 0.0f) atomicMax(&s_last, t);
  __syncthreads();
  int c = s_chunk;
  const bool past_end = c >= NB;  // rounding left the total at or below u * Zf
  if (past_end) c = s_last;
  if (t == c) {
    const df b0 = df_add(cinc, mk(-fs.h, -fs.l));  // running sum before chunk c
    s_base = make_float2(b0.h, b0.l);
  }
  __syncthreads();
  const df base = mk(s_base.x, s_base.y);
  // the chunk: one element per thread, in ascending ids
  const int i = c * kChunk + t;
  df p = mk(0.0f, 0.0f);
  bool kept = false;
  if (i < V) {
    const float2 e = Eall[row + i];
    kept = kept_by(st, q, Kall[row + i], e, i);
    if (kept) p = mk(e.x, e.y);
  }
  df ctot;
  const df cin = block_scan_df(p, redd, ctot);
  if (!past_end && kept && df_gt(df_add(base, cin), target)) atomicMin(&s_tok, i);
  if (kept) atomicMax(&s_lastid, i);
  __syncthreads();
  if (t == 0) {
    // nothing passed u here (rounding): the chunk's last kept id
    const int tok = s_tok != 0x7fffffff ? s_tok : s_lastid;
    tokens[s] = tok;
    logprobs[s] = tok >= 0 ? logprob_of(logits + (size_t)s * ld, marks + (size_t)s * V, tok, q, st.M, st.lse)
                           : -INFINITY;
    rng[s].state = s_state;
  }
}

// ---- test hook: the double-f32 exponential on n device values --------------------------------

__global__ void k_df_exp(const double* __restrict__ x, double* __restrict__ y, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = dbl_of(df_exp(df_of(x[i])));
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
  static dec::SmemOptIn pick_optin;
  if (pick_optin.ensure(k_pick, (int)sizeof(PickSmem)) != cudaSuccess) {
    dec_sampler_destroy(s);
    return sfail(DEC_ECUDA, "cannot reserve %zu bytes of shared memory for the pick kernel", sizeof(PickSmem));
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
    q.pad1 = 0;
    q.flags = (p.temperature > 0.0 ? kSampling : 0) | (p.temperature == 1.0 ? kUnitT : 0) | (p.top_p < 1.0 ? kTopP : 0) |
              (p.min_p > 0.0 ? kMinP : 0);
    // 1/T, top_p and min_p as float head + tail (long double division where the host has it)
    const long double rT = p.temperature > 0.0 ? 1.0L / (long double)p.temperature : 0.0L;
    q.rTh = (float)rT;
    q.rTl = (float)(rT - (long double)q.rTh);
    q.pph = (float)p.top_p;
    q.ppl = (float)(p.top_p - (double)q.pph);
    q.mph = (float)p.min_p;
    q.mpl = (float)(p.min_p - (double)q.mph);
    q.hist_off = history_offsets ? history_offsets[i] : 0;
    q.n_hist = history_offsets ? history_offsets[i + 1] - history_offsets[i] : 0;
    q.n_prompt = n_prompt ? n_prompt[i] : 0;
  }
  unsigned char* w = s->ws;
  SeqParam* dsp = (SeqParam*)(w + s->L.seqs);
  S_CUDA(cudaMemcpyAsync(dsp, H, (size_t)n * sizeof(SeqParam), cudaMemcpyHostToDevice, st));
  S_CUDA(cudaEventRecord(s->stage_ev[slot], st));
  S_CUDA(cudaMemsetAsync(w + s->L.hcnt, 0, (size_t)n * kBins * 4, st));
  S_CUDA(cudaMemsetAsync(w + s->L.hmh, 0, (size_t)n * kBins * 8, st));
  S_CUDA(cudaMemsetAsync(w + s->L.hml, 0, (size_t)n * kBins * 8, st));
  int32_t* marks = (int32_t*)(w + s->L.marks);
  uint32_t* status = (uint32_t*)(w + s->L.status);
  const int V = s->V, NB = s->NB;
  Part1* p1 = (Part1*)(w + s->L.part1);
  Part2* p2 = (Part2*)(w + s->L.part2);
  uint64_t* K = (uint64_t*)(w + s->L.K);
  float2* E = (float2*)(w + s->L.E);
  uint16_t* bins = (uint16_t*)(w + s->L.bins);
  uint32_t* hc = (uint32_t*)(w + s->L.hcnt);
  unsigned long long* hh = (unsigned long long*)(w + s->L.hmh);
  unsigned long long* hl = (unsigned long long*)(w + s->L.hml);
  Stats* stats = (Stats*)(w + s->L.stats);
  const int Vp = padded(s->V), NB1 = (s->V + kChunk1 - 1) / kChunk1;
  PickState* ps = (PickState*)(w + s->L.state);
  float2* fsum = (float2*)(w + s->L.fsum);
  const dim3 hgrid((max_hist + 255) / 256, n);
  if (max_hist > 0) k_mark<<<hgrid, 256, 0, st>>>(dsp, history, marks, V, 1, status);
  const dim3 grid(NB, n), grid1(NB1, n);
  k_scan1<<<grid1, kScanThreads, 0, st>>>(logits, ld, marks, dsp, V, NB1, p1, status);
  k_stats<<<n, kScanThreads, 0, st>>>(p1, NB1, stats, status);
  k_scan2<<<grid, kScanThreads, 0, st>>>(logits, ld, marks, dsp, V, Vp, NB, stats, p2, K, E, bins, hc, hh, hl);
  k_pick<<<n, kPick, sizeof(PickSmem), st>>>(logits, ld, marks, dsp, V, Vp, NB, stats, p2, K, E, bins, hc, hh, hl, ps,
                                             rng, tokens, logprobs, status);
  k_final_sum<<<grid, kScanThreads, 0, st>>>(dsp, ps, V, Vp, NB, K, E, fsum);
  k_final_pick<<<n, kPick, 0, st>>>(logits, ld, marks, dsp, ps, V, Vp, NB, K, E, fsum, rng, tokens, logprobs);
  if (max_hist > 0) k_mark<<<hgrid, 256, 0, st>>>(dsp, history, marks, V, 0, status);
  S_CUDA(cudaGetLastError());
  return DEC_OK;
}

int dec_debug_df_exp(const double* x, double* y, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return sfail(DEC_EINVAL, "bad arguments");
  if (n == 0) return DEC_OK;
  k_df_exp<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(x, y, n);
  S_CUDA(cudaGetLastError());
  return DEC_OK;
}

}  // extern "C"
