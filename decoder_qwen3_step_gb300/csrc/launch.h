// launch.h - host-side launchers of the decoder kernels (internal to libdec).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "optin.h"

namespace dec {

enum Epi { EPI_QKV_RAW = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3, EPI_QKV = 4 };

// What the fused QKV epilogue (EPI_QKV) needs: QK-norm gains, the RoPE table,
// the query buffer and the KV pool with the step's positions and tables.
struct QkvFuse {
  const float* q_norm;
  const float* k_norm;
  const float* rope;  // [max_positions, D/2, 2] (cos, sin)
  float* Q;           // [T, H, D]
  void* kv;           // pool slabs
  int layer;
  StepMeta meta;
  int H, Hkv, D, B, n_blocks, max_blocks;
  uint32_t* err;  // device error word
};

// Token rows up to which the weight-streaming kernel runs a product.
constexpr int kGemvMaxTokens = 32;
constexpr int kQkvFuseMaxSkinny = 16;  // decode-size QKV products fuse their epilogue up to this many token rows
// weight-streaming products: rows per CTA (two per warp), token rows per pass, threads
constexpr int kGemvRows = 16;
constexpr int kGemvTok = 8;
constexpr int kGemvThreads = 256;
constexpr int kInt4MaxK = 4096;  // int4 products stage 16 rows of codes and 8 token rows in shared memory (25 bytes per input column)

// One weight-streaming product Y[t, r] = sum_k X[row(t), k] W[r, k] with a
// fused epilogue.  W is [rows, K] (fp32 or bf16), X is [*, K] (act type).
struct GemvArgs {
  const void* W;
  int rows, K;
  const void* X;
  const int32_t* x_row;   // activation row of token-row t (null: t)
  int T;                  // token rows
  const float* ssq;       // RMSNorm partials of the activation rows (null: no row scale)
  int d;
  float eps;
  float* out_f32;         // QKV_RAW [T, rows]; LOGITS [T, rows] (may be null)
  float* X_res;           // RESID residual [T, d]
  void* XN;               // RESID next GEMM input [T, d]
  float* SSQ_out;         // RESID partials [T, d/16]
  const float* w_next;    // RESID next RMSNorm gain [d]
  void* act_out;          // SWIGLU output [T, F]
  int F;
  unsigned long long* keys; // LOGITS argmax keys [T]
  QkvFuse qf;             // EPI_QKV
};

struct EmbedArgs {
  const void* E;  // [vocab, d] weight type
  const int32_t* ids;
  int T, d, vocab, R;
  const float* w0;  // first RMSNorm gain
  float* X;
  void* XN;
  float* SSQ;
  unsigned long long* keys;
  uint32_t* err;
};

struct QkvPostArgs {
  const float* raw;  // [T, (H+2Hkv)*D]
  const float* q_norm;
  const float* k_norm;
  const float* rope;  // [max_positions, D/2, 2] (cos, sin)
  float* Q;           // [T, H, D]
  void* kv;           // pool slabs
  int layer;
  StepMeta meta;
  Dims dims;
  uint32_t* err;  // device error word
};

struct AttnArgs {
  const float* Q;   // [T, H, D]
  const void* kv;   // pool slabs
  int layer;
  StepMeta meta;
  Dims dims;
  void* ATT;        // [T, H*D] act type
  float* part;      // decode partials [S, H, nchunk_cap, D+2]
  int nchunk_cap;
  int S;
  float scale;      // 1/sqrt(D)
  int* counters;    // decode: finished CTAs per (sequence, kv head), zero between launches
  uint32_t* err;    // device error word
};

// Launchers; `wbf16` selects bf16 weights / activations / f16 KV (serving
// mode) versus fp32 everywhere (parity mode).  Return cudaGetLastError().
cudaError_t launch_embed(const EmbedArgs& a, bool wbf16, cudaStream_t s);
cudaError_t launch_gemv(const GemvArgs& a, int epi, bool wbf16, cudaStream_t s);
cudaError_t launch_qkv_post(const QkvPostArgs& a, int T, bool wbf16, cudaStream_t s);
cudaError_t launch_argmax_finalize(const unsigned long long* keys, int32_t* ids, int R, cudaStream_t s);
cudaError_t launch_attn_decode(const AttnArgs& a, int nchunk, bool wbf16, cudaStream_t s);
cudaError_t launch_attn_prefill(const AttnArgs& a, int n_work, bool wbf16, cudaStream_t s);
// Packing: dst row map modes.
enum PackMode { PACK_IDENTITY = 0, PACK_GATE = 1, PACK_UP = 2 };
cudaError_t launch_pack(void* dst, const float* src, int rows, int cols, int mode, bool wbf16, cudaStream_t s);
// int4 projections (kernels_int4.cu): the product reads codes then scales (rows * K/2 bytes,
// then rows * K/32 f16 values) at GemvArgs::W; the quantizer writes one source matrix
// (rows x K f32, row mapping as launch_pack) into such a layout's codes and scales.
cudaError_t launch_gemv_i4(const GemvArgs& a, int epi, cudaStream_t s);
cudaError_t launch_quant_i4(void* nib, void* scl, const float* src, int rows, int K, int mode, cudaStream_t s);
cudaError_t launch_f32_to_f16(const float* in, uint16_t* out, int64_t n, cudaStream_t s);

// tcgen05 products (bf16 weights and activations): eligible shapes and launch.
// tmW / tmX point at host copies of CUtensorMap (weights [rows, K] and
// activations [T, K], bf16, box 64 x 128, 128-byte swizzle).
bool tc_eligible(const GemvArgs& a);
cudaError_t launch_gemm_tc(const GemvArgs& a, int epi, const void* tmW, const void* tmX, int num_sms, uint32_t* err,
                           cudaStream_t s);

// tcgen05 products of decode steps (1..32 token rows; activation maps with a
// 32-row box), cluster split-K; pdl launches with programmatic serialisation.
bool tc_skinny_eligible(const GemvArgs& a);
int skinny_splits(int rows, int K);
cudaError_t launch_gemm_tc_skinny(const GemvArgs& a, int epi, const void* tmW, const void* tmX, uint32_t* err,
                                  bool pdl, cudaStream_t s);

// Serving-mode decode attention (f16 KV cache, two query heads per KV head)
// on the warp-level tensor cores, with QK-norm, RoPE and the cache append of
// the step's token fused in: it reads the QKV product's raw rows instead of
// Q.  tm_kv points at a host copy of the pool's CUtensorMap ([rows, D] f16,
// box 16 x min(D, 64), 128-byte swizzle when D >= 64).
struct AttnDecTcArgs {
  AttnArgs at;            // Q is not read
  const float* raw;       // [T, (H+2Hkv)*D] q|k|v before QK-norm and RoPE
  const float* q_norm;    // [D] QK-norm gains of the layer
  const float* k_norm;
  const float* rope;      // [max_positions, D/2, 2] (cos, sin)
};
bool attn_decode_tc_eligible(const Dims& dm);
// One persistent CTA per SM (grid CTAs) streaming its share of the
// (sequence, KV head, 64-key chunk) items through a TMA ring; item_start
// [S+1] (device) is the first item of every sequence (Hkv * chunks each).
cudaError_t launch_attn_decode_ring(const AttnDecTcArgs& a, const void* tm_kv, const int32_t* item_start, int grid,
                                    cudaStream_t s);

// Query rows of one prefill attention tile (query-head rows / group size).
int prefill_tile_queries(int G);

// Serving-mode prefill attention on the warp-level tensor cores (f16 K/V,
// f16 queries and probabilities, fp32 accumulation); same work tiles.
bool attn_prefill_tc_eligible(const AttnArgs& a);
cudaError_t launch_attn_prefill_tc(const AttnArgs& a, int n_work, cudaStream_t s);

// ---- the whole decode step in one persistent kernel (serving mode) -----------
constexpr int kMegaComputeWarps = 8;                  // + one loader warp
constexpr int kMegaKSlice = 1024;                     // k elements per weight tile
constexpr int kMegaKeys = 64;                         // cached keys per attention tile
constexpr int kMegaTiles = 32;                        // ring tiles in flight at most (mbarrier pairs)
constexpr int kMegaMaxTokens = 8;                     // sequences per step the kernel supports
// Steps of at most this many sequences take the one-kernel path by default.
constexpr int kMegaAutoTokens = 8;
constexpr int kMegaMaxGrid = 256;                     // CTAs (one per SM) the partial sums are sized for
constexpr int kMegaTraceStride = 320;                 // trace stamps per CTA (the last: the loader's end)
constexpr int kMegaMinRing = 128 * 1024;              // smallest weight/KV ring worth running with

struct MegaArgs {
  // the KV pool as a 2-D f16 tensor [layers * blocks * 2 * Hkv * 16 rows, D]:
  // boxes of 16 rows x min(D, 64) columns, 128-byte swizzle when D >= 64
  CUtensorMap tm_kv;
  // packed weights: layer 0 at `layers`, then every layer_stride bytes
  const char* layers;
  size_t layer_stride;
  size_t o_attn_norm, o_mlp_norm, o_q_norm, o_k_norm, o_wqkv, o_wo, o_wgu, o_wd;
  const bf16* embed;        // [vocab, d], also the LM head
  const float* final_norm;  // [d]
  const float* w_attn0;     // layer 0's attention RMSNorm gain [d]
  const float* rope;        // [max_positions, D/2, 2] (cos, sin)
  __half* kv;               // pool slabs
  int n_blocks;
  int vocab, d, n_layers, H, Hkv, D, F, max_blocks;
  float eps, scale;
  // the step: T sequences of one new token each
  int T;
  const int32_t* ids;         // [T]
  const int32_t* seq_ctx;     // [T] context length after this token
  const int32_t* tables;      // [T, max_blocks]
  const int32_t* item_start;  // [T+1] first attention item of each sequence (Hkv * 64-key chunks each)
  float* X;                   // [T, d] residual; each CTA reads and writes only the rows it owns
  // buffers other CTAs read (each written once per stage, read after a sync)
  bf16* xa;                   // [T, d]  x * next gain after the down projection (QKV and LM-head input)
  bf16* xb;                   // [T, d]  the same after the O projection (gate/up input)
  float* sa;                  // [T, kMegaMaxGrid] per-CTA sums of x^2 paired with xa
  float* sb;                  // [T, kMegaMaxGrid] paired with xb
  float* raw;                 // [T, (H+2Hkv)*D] q|k|v before QK-norm/RoPE
  bf16* att;                  // [T, H*D] attention output
  bf16* act;                  // [T, F] silu(gate)*up
  float* rec;                 // [T, Hkv, nch_cap, 2*(D+2)] per-chunk records: per head max, sum, values
  int nch_cap;
  unsigned int* sync;         // CTAs arrived, summed over the step's sync points; zero at launch
  unsigned int* acnt;         // [T, Hkv] chunks recorded, summed over layers; zero at launch
  unsigned int* done;         // CTAs finished; zero at launch
  unsigned int* abort;        // set by a CTA that gave up; zero at launch
  unsigned long long* keys;   // [T] argmax keys, zero at launch
  float* logits;              // [T, vocab] or null
  int32_t* argmax;            // [T]
  uint32_t* err;
  // test hook: every CTA hand-off wait expects wait_extra more arrivals than
  // will come and gives up after wait_limit ns (normally 0 and 1 s)
  unsigned int wait_extra;
  unsigned long long wait_limit;
  // dynamic shared memory: ring of `ring` bytes at 0, then the other regions
  int ring, o_stage, o_scr, o_small, o_bars;
  unsigned long long* trace;  // null, or [grid, kMegaTraceStride] global-timer stamps
};

// Shared-memory plan of the kernel for T tokens, product inputs up to kmax
// wide and head size D: the largest ring (a multiple of 1 KB) that fits in
// `smem_limit` bytes.  total == 0 if not even kMegaMinRing fits.
struct MegaSmem {
  int ring, o_stage, o_scr, o_small, o_bars, total;
};
MegaSmem mega_smem(int T, int kmax, int D, int smem_limit);
int mega_threads();
// Whether one CTA of the kernel for head size D fits on an SM with `smem` bytes.
bool mega_fits(int D, int smem);
cudaError_t launch_decode_mega(const MegaArgs& a, int grid, int smem, cudaStream_t s);

}  // namespace dec
