// launch.h - host-side launchers of the decoder kernels (internal to libdec).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

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
};

// Token rows up to which the weight-streaming kernel runs a product.
constexpr int kGemvMaxTokens = 32;

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

// Query rows of one prefill attention tile (query-head rows / group size).
int prefill_tile_queries(int G);

}  // namespace dec
