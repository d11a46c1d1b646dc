// api.cu - the C ABI of libdec (declared in include/dec.h): config checks,
// weight packing, the paged KV pool's host allocator, batch validation,
// per-step metadata staging and the launch sequence of one decoder step.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dec.h"
#include "common.cuh"
#include "internal.h"
#include "launch.h"

using namespace dec;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

}  // namespace

int dec::set_error(int code, const char* msg) {
  g_err = msg;
  return code;
}

namespace {

#define DEC_CUDA(call)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess) return fail(DEC_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int act_bytes(const dec_config& c) { return c.mode == DEC_FP32 ? 4 : 2; }
int kv_bytes(const dec_config& c) { return c.mode == DEC_FP32 ? 4 : 2; }
int qkv_rows(const dec_config& c) { return (c.n_heads + 2 * c.n_kv_heads) * c.head_dim; }
bool serving(const dec_config& c) { return c.mode != DEC_FP32; }       // bf16 GEMM inputs, f16 KV
bool int4_proj(const dec_config& c) { return c.mode == DEC_INT4_F16KV; } // int4 projections
// bytes of one projection matrix in the packed buffer: elements, or int4 codes then f16 group scales
size_t mat_bytes(const dec_config& c, size_t rows, size_t K) {
  if (int4_proj(c)) return rows * K / 2 + rows * (K / 32) * 2;
  return rows * K * (c.mode == DEC_FP32 ? 4 : 2);
}
int max_blocks_of(const dec_config& c) { return (c.max_positions + c.block_tokens - 1) / c.block_tokens; }
int max_chunks_of(const dec_config& c) { return (c.max_positions + kDecodeChunk - 1) / kDecodeChunk; }

int check_config(const dec_config* c) {
  if (!c) return fail(DEC_EINVAL, "config is NULL");
  if (c->mode != DEC_FP32 && c->mode != DEC_BF16_F16KV && c->mode != DEC_INT4_F16KV)
    return fail(DEC_EINVAL, "unknown mode %d", c->mode);
  if (c->rope_scaling) return fail(DEC_EINVAL, "unsupported: scaled RoPE");
  if (c->sliding_window) return fail(DEC_EINVAL, "unsupported: sliding-window attention");
  if (c->attention_bias) return fail(DEC_EINVAL, "unsupported: attention biases");
  if (c->qk_norm != 1 || c->rope_split != 1 || c->tied != 1)
    return fail(DEC_EINVAL, "unsupported: qk_norm, rope_split and tied must all be 1");
  if (c->vocab <= 0 || c->d_model <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
      c->head_dim <= 0 || c->ff_hidden <= 0 || c->max_positions <= 0)
    return fail(DEC_EINVAL, "dimensions must be positive");
  if (c->n_heads % c->n_kv_heads) return fail(DEC_EINVAL, "n_heads must be a multiple of n_kv_heads");
  const int G = c->n_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4) return fail(DEC_EINVAL, "query heads per KV head must be 1, 2 or 4");
  if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
    return fail(DEC_EINVAL, "head_dim must be 32, 64 or 128");
  if (c->d_model % 32) return fail(DEC_EINVAL, "d_model must be a multiple of 32");
  if (c->ff_hidden % 16) return fail(DEC_EINVAL, "ff_hidden must be a multiple of 16");
  if (c->vocab % 16) return fail(DEC_EINVAL, "vocab must be a multiple of 16");
  if (c->block_tokens != 16) return fail(DEC_EINVAL, "block_tokens must be 16");
  if (!(c->rope_base > 1.0) || !(c->rms_eps > 0.0)) return fail(DEC_EINVAL, "rope_base must be > 1, rms_eps > 0");
  if (c->max_positions > kMaxPositions) return fail(DEC_EINVAL, "max_positions above %d", kMaxPositions);
  if (c->mode == DEC_INT4_F16KV && (c->ff_hidden % 32 || (c->n_heads * c->head_dim) % 32))
    return fail(DEC_EINVAL, "int4 weights need every input width (d_model, n_heads*head_dim, ff_hidden) a multiple of 32");
  if (c->mode == DEC_INT4_F16KV &&
      (c->d_model > kInt4MaxK || c->ff_hidden > kInt4MaxK || c->n_heads * c->head_dim > kInt4MaxK))
    return fail(DEC_EINVAL, "int4 weights: input widths above %d are not supported", kInt4MaxK);
  return DEC_OK;
}

// Packed weight buffer: RoPE table, embedding, final gain, then per layer
// gains and the fused matrices [Wq;Wk;Wv], Wo, gate/up interleaved by 8 rows, Wd.
struct PackedLayout {
  size_t rope, embed, final_norm;
  size_t attn_norm, mlp_norm, q_norm, k_norm, wqkv, wo, wgu, wd;  // offsets within a layer
  size_t layer0, layer_stride, total;
};

PackedLayout packed_layout(const dec_config& c) {
  PackedLayout L{};
  const size_t wb = c.mode == DEC_FP32 ? 4 : 2;  // the embedding: f32, else bf16
  const size_t d = c.d_model, D = c.head_dim, F = c.ff_hidden, HD = (size_t)c.n_heads * D;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  L.rope = take((size_t)c.max_positions * (D / 2) * 2 * sizeof(float));
  L.embed = take((size_t)c.vocab * d * wb);
  L.final_norm = take(d * sizeof(float));
  L.layer0 = off;
  size_t lo = 0;
  auto ltake = [&](size_t bytes) { size_t o = lo; lo = align256(lo + bytes); return o; };
  L.attn_norm = ltake(d * 4);
  L.mlp_norm = ltake(d * 4);
  L.q_norm = ltake(D * 4);
  L.k_norm = ltake(D * 4);
  L.wqkv = ltake(mat_bytes(c, qkv_rows(c), d));
  L.wo = ltake(mat_bytes(c, d, HD));
  L.wgu = ltake(mat_bytes(c, 2 * F, d));
  L.wd = ltake(mat_bytes(c, d, F));
  L.layer_stride = lo;
  L.total = L.layer0 + (size_t)c.n_layers * lo;
  return L;
}

struct WsLayout {
  size_t X, XN, SSQ, RAW, Q, ATT, ACT, PART, ACNT, META, KEYS, ERR, MSYNC, FLOW, total;
  size_t meta_ints;
  size_t msync_bytes;
  // the one-kernel decode step's hand-over buffers (offsets within FLOW)
  size_t f_xa, f_xb, f_sa, f_sb, f_raw, f_att, f_act, f_rec, flow_bytes;
};

// 64-key chunks of the longest context (the one-kernel decode step's split).
int max_chunks64_of(const dec_config& c) { return (c.max_positions + kMegaKeys - 1) / kMegaKeys; }

WsLayout ws_layout(const dec_config& c, int T, int S) {
  WsLayout L{};
  const size_t a = act_bytes(c), d = c.d_model, HD = (size_t)c.n_heads * c.head_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  L.X = take((size_t)T * d * 4);
  L.XN = take((size_t)T * d * a);
  L.SSQ = take((size_t)T * (d / kSsqChunk) * 4);
  L.RAW = take((size_t)T * qkv_rows(c) * 4);
  L.Q = take((size_t)T * HD * 4);
  L.ATT = take((size_t)T * HD * a);
  L.ACT = take((size_t)T * c.ff_hidden * a);
  L.PART = take((size_t)S * max_chunks_of(c) * c.n_heads * (c.head_dim + 2) * 4);
  L.ACNT = take((size_t)S * c.n_kv_heads * 4);
  // ids, tok_pos, tok_seq, row_tok [T]; seq_start [S+1]; seq_ctx [S]; tables [S*MB]; then either the
  // prefill tiles [3*(T+S)] or the decode work list [1 + 2*S*chunks]
  L.meta_ints = 4 * (size_t)T + 2 * (size_t)S + 1 + (size_t)S * max_blocks_of(c) +
                std::max(3 * ((size_t)T + S), 1 + 2 * (size_t)S * max_chunks_of(c));
  L.META = take(L.meta_ints * 4);
  L.KEYS = take((size_t)T * 8);
  L.ERR = take(64);
  // one-kernel decode step: one block cleared before every launch (sync
  // counter | finished CTAs | abort word | argmax keys | chunk counters),
  // then the buffers its CTAs hand over to each other
  const size_t Tm = (size_t)std::min(T, kMegaMaxTokens);
  L.msync_bytes = 256 + align256(Tm * 8) + align256(Tm * c.n_kv_heads * 4);
  L.MSYNC = take(L.msync_bytes);
  size_t fo = 0;
  auto ftake = [&](size_t bytes) { size_t o = fo; fo = align256(fo + bytes); return o; };
  const size_t D = c.head_dim;
  L.f_xa = ftake(Tm * d * 2);
  L.f_xb = ftake(Tm * d * 2);
  L.f_sa = ftake(Tm * kMegaMaxGrid * 4);
  L.f_sb = ftake(Tm * kMegaMaxGrid * 4);
  L.f_raw = ftake(Tm * qkv_rows(c) * 4);
  L.f_att = ftake(Tm * HD * 2);
  L.f_act = ftake(Tm * c.ff_hidden * 2);
  L.f_rec = ftake(Tm * c.n_kv_heads * max_chunks64_of(c) * 2 * (D + 2) * 4);
  L.flow_bytes = fo;
  L.FLOW = take(L.flow_bytes);
  L.total = off;
  return L;
}

constexpr int kStageSlots = 4;
constexpr size_t kMaxGraphs = 8;

// The two event-record nodes a captured step holds around one launch of a
// profiled kernel class.
struct ProfNode {
  cudaGraphNode_t a, b;
  int cls;
};

struct GraphEntry {
  int S;
  int slots;
  const void* logits;
  const void* argmax;
  const void* slabs;
  int n_blocks;        // the pool's size (its tensor map is a kernel argument in the graph)
  uint32_t prof_mask;  // kernel classes profiled when the step was captured
  cudaGraph_t graph;   // kept while it has profiling nodes: their handles address the executable graph's nodes
  cudaGraphExec_t exec;
  std::vector<ProfNode> pnodes;
  int64_t n_launch;
  uint64_t last_use;
};

}  // namespace


struct dec_model {
  dec_config cfg;
  PackedLayout pl;
  WsLayout wl;
  char* packed;
  char* ws;
  int Tmax, Smax, MB, NCH;
  int device;
  int32_t* stage[kStageSlots];
  cudaEvent_t stage_ev[kStageSlots];
  int stage_next;
  float* dump;
  size_t dump_floats;
  cudaStream_t last_stream;
  // profiling: event pairs around the launches of enabled kernel classes
  struct ProfRec { cudaEvent_t a, b; int cls; };
  bool prof_on[DEC_K_COUNT];
  std::vector<ProfRec> prof_pending;
  std::vector<cudaEvent_t> ev_free;
  double prof_ms[DEC_K_COUNT];
  int64_t prof_n[DEC_K_COUNT];
  int64_t launches;
  int num_sms;
  // tcgen05 products: tensor maps of every bf16 weight matrix and activation buffer
  bool tc_on;
  bool tc_ready;
  std::vector<CUtensorMap> tm_qkv, tm_o, tm_gu, tm_d;
  CUtensorMap tm_embed, tm_xn, tm_att, tm_act;
  CUtensorMap tm_xn32, tm_att32, tm_act32;  // 32-row boxes for decode products
  // the one-kernel decode step
  bool mega_on;
  bool mega_shape;  // the shape and device allow it
  uint32_t wait_extra;         // test hook of the one-kernel step's hand-off waits
  uint64_t wait_limit;
  int32_t poison[3];           // debug builds: (sequence, column, value) for the next step's device table; seq -1: none
  const void* kvmap_slabs;  // the pool the one-kernel step's KV tensor map was made for
  int kvmap_blocks;
  CUtensorMap kvmap;
  unsigned long long* trace;  // per-stage timer stamps of the one-kernel step (or null)
  size_t trace_n;
  int smem_optin;
  // captured decode steps
  bool graphs_on;
  cudaStream_t cap_stream;
  std::vector<GraphEntry> graphs;
  uint64_t graph_clock;
  bool capturing;                   // a decode step is being captured on cap_stream
  std::vector<ProfRec> cap_recs;    // the profiling events that capture turned into graph nodes
};

namespace {

cudaEvent_t take_event(dec_model* m) {
  if (!m->ev_free.empty()) {
    cudaEvent_t e = m->ev_free.back();
    m->ev_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Record a profiling event; inside a capture it becomes an event-record node
// of the graph, which replays re-point at fresh events.
cudaError_t record_event(dec_model* m, cudaEvent_t e, cudaStream_t st) {
  if (!e) return cudaErrorMemoryAllocation;
  return m->capturing ? cudaEventRecordWithFlags(e, st, cudaEventRecordExternal) : cudaEventRecord(e, st);
}

// Launch one kernel (expr returns cudaError_t) of class cls on stream st,
// bracketed by CUDA events when that class is being profiled.
template <typename F>
int timed_launch(dec_model* m, int cls, cudaStream_t st, F&& fn, const char* what) {
  cudaEvent_t a = nullptr;
  if (m->prof_on[cls]) {
    a = take_event(m);
    cudaError_t e = record_event(m, a, st);
    if (e != cudaSuccess) {
      if (a) m->ev_free.push_back(a);
      return fail(DEC_ECUDA, "profiling event: %s", cudaGetErrorString(e));
    }
  }
  cudaError_t e = fn();
  if (e != cudaSuccess) {
    if (a) m->ev_free.push_back(a);
    return fail(DEC_ECUDA, "%s: %s", what, cudaGetErrorString(e));
  }
  if (a) {
    cudaEvent_t b = take_event(m);
    e = record_event(m, b, st);
    if (e != cudaSuccess) {
      m->ev_free.push_back(a);
      if (b) m->ev_free.push_back(b);
      return fail(DEC_ECUDA, "profiling event: %s", cudaGetErrorString(e));
    }
    (m->capturing ? m->cap_recs : m->prof_pending).push_back({a, b, cls});
  }
  ++m->launches;
  return DEC_OK;
}

}  // namespace

#define DEC_LAUNCH(cls, expr)                                                   \
  do {                                                                          \
    int rc_ = timed_launch(m, cls, st, [&]() { return (expr); }, #expr);        \
    if (rc_) return rc_;                                                        \
  } while (0)

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once per process (the static's
// initialisation is thread-safe); NULL when the driver does not export it.
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// 2-D bf16 tensor map of a row-major [rows, cols] matrix, box 64 x 128, 128-byte swizzle.
bool bf16_map(CUtensorMap* out, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D f16 tensor map of the KV pool as [rows, D] (a row: one slot of one KV
// head of one block of one layer, K or V), box 16 rows x min(D, 64) columns;
// 128-byte swizzle when a box row is 128 bytes.
bool kv_map(CUtensorMap* out, const void* slabs, uint64_t rows, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint32_t bd = D >= 64 ? 64u : (uint32_t)D;
  cuuint64_t dims[2] = {(cuuint64_t)D, rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {bd, 16};
  cuuint32_t estr[2] = {1, 1};
  return fn(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(slabs), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, bd == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps for the tcgen05 products (serving mode only); false leaves the
// CUDA-core products in charge.
bool build_tensor_maps(dec_model* m) {
  const dec_config& c = m->cfg;
  if (c.mode != DEC_BF16_F16KV) return false;
  const int d = c.d_model, HD = c.n_heads * c.head_dim, F = c.ff_hidden;
  char* P = m->packed;
  m->tm_qkv.resize(c.n_layers);
  m->tm_o.resize(c.n_layers);
  m->tm_gu.resize(c.n_layers);
  m->tm_d.resize(c.n_layers);
  bool ok = true;
  for (int l = 0; l < c.n_layers; ++l) {
    char* Lb = P + m->pl.layer0 + (size_t)l * m->pl.layer_stride;
    ok &= bf16_map(&m->tm_qkv[l], Lb + m->pl.wqkv, qkv_rows(c), d);
    ok &= bf16_map(&m->tm_o[l], Lb + m->pl.wo, d, HD);
    ok &= bf16_map(&m->tm_gu[l], Lb + m->pl.wgu, 2 * F, d);
    ok &= bf16_map(&m->tm_d[l], Lb + m->pl.wd, d, F);
  }
  ok &= bf16_map(&m->tm_embed, P + m->pl.embed, c.vocab, d);
  ok &= bf16_map(&m->tm_xn, m->ws + m->wl.XN, m->Tmax, d);
  ok &= bf16_map(&m->tm_att, m->ws + m->wl.ATT, m->Tmax, HD);
  ok &= bf16_map(&m->tm_act, m->ws + m->wl.ACT, m->Tmax, F);
  ok &= bf16_map(&m->tm_xn32, m->ws + m->wl.XN, m->Tmax, d, 32);
  ok &= bf16_map(&m->tm_att32, m->ws + m->wl.ATT, m->Tmax, HD, 32);
  ok &= bf16_map(&m->tm_act32, m->ws + m->wl.ACT, m->Tmax, F, 32);
  return ok;
}

}  // namespace

extern "C" {

const char* dec_last_error(void) { return g_err.c_str(); }
const char* dec_version(void) { return "libdec 0.1 (sm_103a)"; }

int dec_config_check(const dec_config* cfg) { return check_config(cfg); }

int dec_weights_bytes(const dec_config* cfg, size_t* bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!bytes) return fail(DEC_EINVAL, "bytes is NULL");
  *bytes = packed_layout(*cfg).total;
  return DEC_OK;
}

int dec_workspace_bytes(const dec_config* cfg, int32_t max_tokens, int32_t max_seqs, size_t* bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!bytes) return fail(DEC_EINVAL, "bytes is NULL");
  if (max_tokens < 1 || max_seqs < 1 || max_seqs > max_tokens)
    return fail(DEC_EINVAL, "need 1 <= max_seqs <= max_tokens");
  *bytes = ws_layout(*cfg, max_tokens, max_seqs).total;
  return DEC_OK;
}

int dec_create(const dec_config* cfg, const dec_weights* w, void* packed_buf, size_t packed_bytes, void* workspace,
               size_t workspace_bytes, int32_t max_tokens, int32_t max_seqs, void* stream, dec_model** out) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!w || !packed_buf || !workspace || !out) return fail(DEC_EINVAL, "NULL argument");
  if (max_tokens < 1 || max_seqs < 1 || max_seqs > max_tokens)
    return fail(DEC_EINVAL, "need 1 <= max_seqs <= max_tokens");
  const dec_config& c = *cfg;
  PackedLayout pl = packed_layout(c);
  WsLayout wl = ws_layout(c, max_tokens, max_seqs);
  if (packed_bytes < pl.total) return fail(DEC_EINVAL, "packed buffer too small: %zu < %zu", packed_bytes, pl.total);
  if (workspace_bytes < wl.total) return fail(DEC_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, wl.total);
  if (((uintptr_t)packed_buf | (uintptr_t)workspace) & 255) return fail(DEC_EINVAL, "buffers must be 256-byte aligned");
  if (!w->embed || !w->final_norm || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->q_norm || !w->k_norm ||
      !w->wo || !w->mlp_norm || !w->w_gate || !w->w_up || !w->w_down)
    return fail(DEC_EINVAL, "missing weight pointer");
  for (int l = 0; l < c.n_layers; ++l)
    if (!w->attn_norm[l] || !w->wq[l] || !w->wk[l] || !w->wv[l] || !w->q_norm[l] || !w->k_norm[l] || !w->wo[l] ||
        !w->mlp_norm[l] || !w->w_gate[l] || !w->w_up[l] || !w->w_down[l])
      return fail(DEC_EINVAL, "missing weight pointer in layer %d", l);

  cudaStream_t s = (cudaStream_t)stream;
  const bool bf = serving(c);
  const bool i4 = int4_proj(c);
  char* P = (char*)packed_buf;
  const int d = c.d_model, D = c.head_dim, F = c.ff_hidden, H = c.n_heads, Hkv = c.n_kv_heads;
  const size_t wb = bf ? 2 : 4;

  // RoPE table in double precision, rounded once to fp32: phi = pos * base^(-2j/D)
  // (1bit-MONSTER "Byte-identical", "The rope table that was too accurate").
  {
    std::vector<float> tab((size_t)c.max_positions * (D / 2) * 2);
    std::vector<double> theta(D / 2);
    for (int j = 0; j < D / 2; ++j) theta[j] = std::pow(c.rope_base, -2.0 * j / D);
    for (int p = 0; p < c.max_positions; ++p)
      for (int j = 0; j < D / 2; ++j) {
        const double phi = (double)p * theta[j];
        tab[((size_t)p * (D / 2) + j) * 2] = (float)std::cos(phi);
        tab[((size_t)p * (D / 2) + j) * 2 + 1] = (float)std::sin(phi);
      }
    DEC_CUDA(cudaMemcpyAsync(P + pl.rope, tab.data(), tab.size() * sizeof(float), cudaMemcpyHostToDevice, s));
    DEC_CUDA(cudaStreamSynchronize(s));
  }
  DEC_CUDA(launch_pack(P + pl.embed, w->embed, c.vocab, d, PACK_IDENTITY, bf, s));
  DEC_CUDA(cudaMemcpyAsync(P + pl.final_norm, w->final_norm, d * 4, cudaMemcpyDeviceToDevice, s));
  for (int l = 0; l < c.n_layers; ++l) {
    char* Lb = P + pl.layer0 + (size_t)l * pl.layer_stride;
    DEC_CUDA(cudaMemcpyAsync(Lb + pl.attn_norm, w->attn_norm[l], d * 4, cudaMemcpyDeviceToDevice, s));
    DEC_CUDA(cudaMemcpyAsync(Lb + pl.mlp_norm, w->mlp_norm[l], d * 4, cudaMemcpyDeviceToDevice, s));
    DEC_CUDA(cudaMemcpyAsync(Lb + pl.q_norm, w->q_norm[l], D * 4, cudaMemcpyDeviceToDevice, s));
    DEC_CUDA(cudaMemcpyAsync(Lb + pl.k_norm, w->k_norm[l], D * 4, cudaMemcpyDeviceToDevice, s));
    char* qkv = Lb + pl.wqkv;
    if (i4) {  // quantize at load: codes, then the scales of the whole matrix
      const size_t R = qkv_rows(c), dG = d / 32;
      char* qs = qkv + R * d / 2;
      DEC_CUDA(launch_quant_i4(qkv, qs, w->wq[l], H * D, d, PACK_IDENTITY, s));
      DEC_CUDA(launch_quant_i4(qkv + (size_t)H * D * d / 2, qs + (size_t)H * D * dG * 2, w->wk[l], Hkv * D, d,
                               PACK_IDENTITY, s));
      DEC_CUDA(launch_quant_i4(qkv + (size_t)(H + Hkv) * D * d / 2, qs + (size_t)(H + Hkv) * D * dG * 2, w->wv[l],
                               Hkv * D, d, PACK_IDENTITY, s));
      DEC_CUDA(launch_quant_i4(Lb + pl.wo, Lb + pl.wo + (size_t)d * H * D / 2, w->wo[l], d, H * D, PACK_IDENTITY, s));
      char* gu = Lb + pl.wgu;
      DEC_CUDA(launch_quant_i4(gu, gu + (size_t)2 * F * d / 2, w->w_gate[l], F, d, PACK_GATE, s));
      DEC_CUDA(launch_quant_i4(gu, gu + (size_t)2 * F * d / 2, w->w_up[l], F, d, PACK_UP, s));
      DEC_CUDA(launch_quant_i4(Lb + pl.wd, Lb + pl.wd + (size_t)d * F / 2, w->w_down[l], d, F, PACK_IDENTITY, s));
      continue;
    }
    DEC_CUDA(launch_pack(qkv, w->wq[l], H * D, d, PACK_IDENTITY, bf, s));
    DEC_CUDA(launch_pack(qkv + (size_t)H * D * d * wb, w->wk[l], Hkv * D, d, PACK_IDENTITY, bf, s));
    DEC_CUDA(launch_pack(qkv + (size_t)(H + Hkv) * D * d * wb, w->wv[l], Hkv * D, d, PACK_IDENTITY, bf, s));
    DEC_CUDA(launch_pack(Lb + pl.wo, w->wo[l], d, H * D, PACK_IDENTITY, bf, s));
    DEC_CUDA(launch_pack(Lb + pl.wgu, w->w_gate[l], F, d, PACK_GATE, bf, s));
    DEC_CUDA(launch_pack(Lb + pl.wgu, w->w_up[l], F, d, PACK_UP, bf, s));
    DEC_CUDA(launch_pack(Lb + pl.wd, w->w_down[l], d, F, PACK_IDENTITY, bf, s));
  }
  DEC_CUDA(cudaMemsetAsync((char*)workspace + wl.ERR, 0, 64, s));
  DEC_CUDA(cudaMemsetAsync((char*)workspace + wl.ACNT, 0, (size_t)max_seqs * c.n_kv_heads * 4, s));
  DEC_CUDA(cudaStreamSynchronize(s));
  int device = 0, num_sms = 0, smem_optin = 0, coop = 0;
  DEC_CUDA(cudaGetDevice(&device));
  DEC_CUDA(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device));
  DEC_CUDA(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device));
  DEC_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device));

  dec_model* m = new dec_model();
  m->cfg = c;
  m->pl = pl;
  m->wl = wl;
  m->packed = P;
  m->ws = (char*)workspace;
  m->Tmax = max_tokens;
  m->Smax = max_seqs;
  m->MB = max_blocks_of(c);
  m->NCH = max_chunks_of(c);
  m->device = device;
  m->stage_next = 0;
  m->dump = nullptr;
  m->dump_floats = 0;
  m->last_stream = s;
  for (int i = 0; i < DEC_K_COUNT; ++i) {
    m->prof_on[i] = false;
    m->prof_ms[i] = 0.0;
    m->prof_n[i] = 0;
  }
  m->launches = 0;
  m->num_sms = num_sms;
  m->graphs_on = true;
  m->mega_on = true;
  m->kvmap_slabs = nullptr;
  m->wait_extra = 0;
  m->wait_limit = 1000000000ull;
  m->poison[0] = -1;
  m->kvmap_blocks = 0;
  m->trace = nullptr;
  m->trace_n = 0;
  m->smem_optin = smem_optin;
  {
    const int P = m->num_sms;
    const int kmax = std::max(d, std::max(H * D, F));
    const MegaSmem ms = mega_smem(kMegaMaxTokens, kmax, D, m->smem_optin);
    // every product's tiles of one group must fit in the ring together: two
    // 16-row tiles, or one tile of each 1024-wide slice of the widest input
    const int slice_foot = 16 * (kMegaKSlice * 2 + 16);
    const int nks_max = (std::max(H * D, F) + kMegaKSlice - 1) / kMegaKSlice;
    m->mega_shape = c.mode == DEC_BF16_F16KV && coop && P <= kMegaMaxGrid && c.n_heads == 2 * c.n_kv_heads &&
                    (D == 32 || D == 64 || D == 128) && c.block_tokens == 16 && d <= kMegaKSlice && d % 64 == 0 &&
                    (H * D) % 64 == 0 && F % 64 == 0 && d <= 16 * P && 5 * c.n_layers <= 255 && ms.total > 0 &&
                    ms.ring >= std::max(2, nks_max) * slice_foot + 1024 && mega_fits(D, ms.total);
  }
  m->tc_on = true;
  m->tc_ready = build_tensor_maps(m);
  // dec_attend_noalloc's array on this device: resolved here, so that its
  // later calls on the device do no set-up (the first resolution loads the
  // module that holds the array, which allocates it under lazy loading)
  if (noalloc_prepare() != DEC_OK) {
    dec_destroy(m);
    return fail(DEC_ECUDA, "the no-allocation attention array could not be resolved");
  }
  m->cap_stream = nullptr;
  m->graph_clock = 0;
  for (int i = 0; i < kStageSlots; ++i) {
    m->stage[i] = nullptr;
    m->stage_ev[i] = nullptr;
  }
  for (int i = 0; i < kStageSlots; ++i) {
    cudaError_t e1 = cudaHostAlloc((void**)&m->stage[i], wl.meta_ints * 4, cudaHostAllocDefault);
    cudaError_t e2 = cudaEventCreateWithFlags(&m->stage_ev[i], cudaEventDisableTiming);
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
      dec_destroy(m);
      return fail(DEC_ECUDA, "pinned staging allocation failed");
    }
  }
  *out = m;
  return DEC_OK;
}

void dec_destroy(dec_model* m) {
  if (!m) return;
  for (int i = 0; i < kStageSlots; ++i) {
    if (m->stage_ev[i]) {
      cudaEventSynchronize(m->stage_ev[i]);
      cudaEventDestroy(m->stage_ev[i]);
    }
    if (m->stage[i]) cudaFreeHost(m->stage[i]);
  }
  for (auto& g : m->graphs) {  // graphs first: their nodes name profiling events
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
  }
  for (auto& r : m->prof_pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : m->ev_free) cudaEventDestroy(e);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  delete m;
}

int dec_device_status(dec_model* m, uint32_t* flags) {
  if (!m || !flags) return fail(DEC_EINVAL, "NULL argument");
  DEC_CUDA(cudaStreamSynchronize(m->last_stream));
  uint32_t v = 0;
  DEC_CUDA(cudaMemcpy(&v, m->ws + m->wl.ERR, 4, cudaMemcpyDeviceToHost));
  DEC_CUDA(cudaMemset(m->ws + m->wl.ERR, 0, 4));
  *flags = v;
  return DEC_OK;
}

int dec_profile_enable(dec_model* m, int32_t kernel_class, int32_t on) {
  if (!m || kernel_class < 0 || kernel_class >= DEC_K_COUNT) return fail(DEC_EINVAL, "bad model or kernel class");
  m->prof_on[kernel_class] = on != 0;
  return DEC_OK;
}

int dec_profile_read(dec_model* m, int32_t kernel_class, double* total_ms, int64_t* launches) {
  if (!m || !total_ms || !launches || kernel_class < 0 || kernel_class >= DEC_K_COUNT)
    return fail(DEC_EINVAL, "bad arguments");
  for (auto& r : m->prof_pending) {
    DEC_CUDA(cudaEventSynchronize(r.b));
    float ms = 0.f;
    DEC_CUDA(cudaEventElapsedTime(&ms, r.a, r.b));
    m->prof_ms[r.cls] += ms;
    m->prof_n[r.cls] += 1;
    m->ev_free.push_back(r.a);
    m->ev_free.push_back(r.b);
  }
  m->prof_pending.clear();
  *total_ms = m->prof_ms[kernel_class];
  *launches = m->prof_n[kernel_class];
  m->prof_ms[kernel_class] = 0.0;
  m->prof_n[kernel_class] = 0;
  return DEC_OK;
}

int dec_set_tensor_cores(dec_model* m, int32_t on) {
  if (!m) return fail(DEC_EINVAL, "model is NULL");
  m->tc_on = on != 0;
  return DEC_OK;
}

int dec_set_megakernel(dec_model* m, int32_t on) {
  if (!m) return fail(DEC_EINVAL, "NULL model");
  m->mega_on = on != 0;
  return DEC_OK;
}

int dec_set_step_trace(dec_model* m, uint64_t* stamps, size_t n) {
  if (!m) return fail(DEC_EINVAL, "NULL model");
  if (stamps && n < (size_t)m->num_sms * kMegaTraceStride)
    return fail(DEC_EINVAL, "the trace needs %zu stamps", (size_t)m->num_sms * kMegaTraceStride);
  m->trace = (unsigned long long*)stamps;
  m->trace_n = stamps ? n : 0;
  return DEC_OK;
}

int dec_debug_wait_timeout(dec_model* m, uint32_t extra, uint64_t limit_ns) {
  if (!m) return fail(DEC_EINVAL, "NULL model");
  if (extra && (limit_ns < 1000 || limit_ns > 1000000000ull))
    return fail(DEC_EINVAL, "the test limit must lie between 1 us and 1 s");
  m->wait_extra = extra;
  m->wait_limit = extra ? limit_ns : 1000000000ull;
  return DEC_OK;
}

uint32_t dec_build_flags(void) {
#ifdef DEC_DEBUG
  return DEC_BUILD_DEBUG;
#else
  return 0;
#endif
}

int dec_debug_poison_table(dec_model* m, int32_t seq, int32_t col, int32_t value) {
  if (!m) return fail(DEC_EINVAL, "NULL model");
#ifdef DEC_DEBUG
  if (seq < 0 || col < 0) return fail(DEC_EINVAL, "sequence and column must be >= 0");
  m->poison[0] = seq;
  m->poison[1] = col;
  m->poison[2] = value;
  return DEC_OK;
#else
  (void)seq;
  (void)col;
  (void)value;
  return fail(DEC_EINVAL, "dec_debug_poison_table needs a DEC_DEBUG build");
#endif
}

int dec_megakernel_available(const dec_model* m, int32_t* available) {
  if (!m || !available) return fail(DEC_EINVAL, "NULL argument");
  *available = m->mega_shape ? 1 : 0;
  return DEC_OK;
}

int dec_set_graphs(dec_model* m, int32_t on) {
  if (!m) return fail(DEC_EINVAL, "model is NULL");
  m->graphs_on = on != 0;
  return DEC_OK;
}

int dec_launch_count(dec_model* m, int64_t* launches) {
  if (!m || !launches) return fail(DEC_EINVAL, "bad arguments");
  *launches = m->launches;
  m->launches = 0;
  return DEC_OK;
}

int dec_set_dump(dec_model* m, float* dump, size_t dump_floats) {
  if (!m) return fail(DEC_EINVAL, "model is NULL");
  m->dump = dump;
  m->dump_floats = dump ? dump_floats : 0;
  return DEC_OK;
}

// ---- pool -------------------------------------------------------------------

int dec_pool_bytes(const dec_config* cfg, int32_t n_blocks, size_t* bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!bytes) return fail(DEC_EINVAL, "bytes is NULL");
  if (n_blocks <= 0) return fail(DEC_EINVAL, "a pool needs at least one block");
  *bytes = (size_t)n_blocks * cfg->n_layers * 2 * cfg->n_kv_heads * cfg->block_tokens * cfg->head_dim * kv_bytes(*cfg);
  return DEC_OK;
}

int dec_pool_create(const dec_config* cfg, int32_t n_blocks, void* slabs, size_t bytes, dec_pool** out) {
  size_t need = 0;
  int rc = dec_pool_bytes(cfg, n_blocks, &need);
  if (rc) return rc;
  if (!slabs || !out) return fail(DEC_EINVAL, "NULL argument");
  if (bytes < need) return fail(DEC_EINVAL, "slab buffer too small: %zu < %zu", bytes, need);
  if ((uintptr_t)slabs & 255) return fail(DEC_EINVAL, "slab buffer must be 256-byte aligned");
  dec_pool* p = new dec_pool();
  p->cfg = *cfg;
  p->n_blocks = n_blocks;
  p->slabs = slabs;
  p->refs.assign(n_blocks, 0);
  p->fill.assign(n_blocks, 0);
  p->registered.assign(n_blocks, 0);
  p->key.assign(n_blocks, 0);
  p->lru_pos.assign(n_blocks, p->lru.end());
  p->free_list.resize(n_blocks);
  for (int i = 0; i < n_blocks; ++i) p->free_list[i] = n_blocks - 1 - i;
  *out = p;
  return DEC_OK;
}

void dec_pool_destroy(dec_pool* p) { delete p; }

int dec_pool_alloc(dec_pool* p, int32_t n, int32_t* ids) {
  if (!p || (!ids && n > 0)) return fail(DEC_EINVAL, "NULL argument");
  if (n < 0) return fail(DEC_EINVAL, "negative block count");
  if ((size_t)n > p->free_list.size() + p->lru.size())
    return fail(DEC_ECAPACITY, "pool exhausted: %d blocks asked, %zu free, %zu cached", n, p->free_list.size(),
                p->lru.size());
  // free blocks first, then the cached prefix blocks released longest ago
  while (p->free_list.size() < (size_t)n) {
    const int32_t id = p->lru.front();
    p->lru.pop_front();
    p->lru_pos[id] = p->lru.end();
    p->index.erase(p->key[id]);
    p->registered[id] = 0;
    p->free_list.insert(p->free_list.begin(), id);
  }
  for (int i = 0; i < n; ++i) {
    ids[i] = p->free_list.back();
    p->free_list.pop_back();
    p->refs[ids[i]] = 1;
    p->fill[ids[i]] = 0;
  }
  return DEC_OK;
}

int dec_pool_retain(dec_pool* p, int32_t id) {
  if (!p) return fail(DEC_EINVAL, "pool is NULL");
  if (id < 0 || id >= p->n_blocks || p->refs[id] <= 0) return fail(DEC_EBLOCK, "block %d is not allocated", id);
  ++p->refs[id];
  return DEC_OK;
}

int dec_pool_release(dec_pool* p, int32_t id) {
  if (!p) return fail(DEC_EINVAL, "pool is NULL");
  if (id < 0 || id >= p->n_blocks || p->refs[id] <= 0) return fail(DEC_EBLOCK, "block %d is not allocated", id);
  if (--p->refs[id] == 0) {
    if (p->registered[id]) {  // keep its keys: a later lookup of the same prefix reacquires it
      p->lru.push_back(id);
      p->lru_pos[id] = std::prev(p->lru.end());
    } else {
      p->free_list.push_back(id);
    }
  }
  return DEC_OK;
}

int dec_pool_free_blocks(const dec_pool* p, int32_t* n) {
  if (!p || !n) return fail(DEC_EINVAL, "NULL argument");
  *n = (int32_t)p->free_list.size();
  return DEC_OK;
}

int dec_pool_refcount(const dec_pool* p, int32_t id, int32_t* refs) {
  if (!p || !refs) return fail(DEC_EINVAL, "NULL argument");
  if (id < 0 || id >= p->n_blocks) return fail(DEC_EBLOCK, "block %d outside the pool", id);
  *refs = p->refs[id];
  return DEC_OK;
}

int dec_kv_offset(const dec_pool* p, const int32_t* table, int32_t n_table, int32_t pos, int32_t layer,
                  int32_t kv_head, int32_t is_v, int64_t* offset) {
  if (!p || !table || !offset) return fail(DEC_EINVAL, "NULL argument");
  const dec_config& c = p->cfg;
  if (pos < 0 || layer < 0 || layer >= c.n_layers || kv_head < 0 || kv_head >= c.n_kv_heads || (is_v != 0 && is_v != 1))
    return fail(DEC_EINVAL, "bad position, layer, head or slab");
  const int bi = pos / c.block_tokens;
  if (bi >= n_table) return fail(DEC_ERANGE, "block table too short for position %d", pos);
  const int blk = table[bi];
  if (blk < 0 || blk >= p->n_blocks) return fail(DEC_EBLOCK, "block id %d outside the pool", blk);
  *offset = kv_offset(layer, blk, is_v, kv_head, pos % c.block_tokens, p->n_blocks, c.n_kv_heads, c.block_tokens,
                      c.head_dim);
  return DEC_OK;
}

// ---- the step ------------------------------------------------------------------

static bool same_shape(const dec_config& a, const dec_config& b) {
  return a.n_layers == b.n_layers && a.n_kv_heads == b.n_kv_heads && a.head_dim == b.head_dim &&
         a.block_tokens == b.block_tokens && a.mode == b.mode;
}

// Everything one step's kernels need, fixed before the first launch.
struct StepPlan {
  StepMeta meta;
  Dims dm;
  int N, S, R;
  bool decode;
  int n_work;
  int slots;  // decode attention CTAs per (sequence, kv head)
  bool rows_all;
  void* slabs;
  float* logits;
  int32_t* argmax;
};

// Serving-mode decode steps run attention on the tensor cores with the
// QK-norm, RoPE and cache append fused in (a persistent kernel whose launch
// does not depend on the contexts).
static bool decode_tc_attn(const dec_model* m, const StepPlan& sp) {
  return sp.decode && serving(m->cfg) && !int4_proj(m->cfg) && m->tc_on && m->tc_ready &&
         attn_decode_tc_eligible(sp.dm);
}

// The KV pool's tensor map (TMA boxes of 16 slots), made once per pool.
static int ensure_kvmap(dec_model* m, const StepPlan& sp) {
  const dec_config& c = m->cfg;
  if (m->kvmap_slabs != sp.slabs || m->kvmap_blocks != sp.dm.n_blocks) {
    const uint64_t rows = (uint64_t)c.n_layers * sp.dm.n_blocks * 2 * c.n_kv_heads * c.block_tokens;
    if (!kv_map(&m->kvmap, sp.slabs, rows, c.head_dim)) return fail(DEC_ECUDA, "tensor map of the KV pool failed");
    m->kvmap_slabs = sp.slabs;
    m->kvmap_blocks = sp.dm.n_blocks;
  }
  return DEC_OK;
}

// Queue the kernels of one step on `st` (eager, or into a capture).
static int enqueue_step(dec_model* m, const StepPlan& sp, cudaStream_t st) {
  const dec_config& c = m->cfg;
  const bool bf = serving(c);
  const bool i4 = int4_proj(c);
  char* P = m->packed;
  char* ws = m->ws;
  const PackedLayout& pl = m->pl;
  const WsLayout& wl = m->wl;
  float* X = (float*)(ws + wl.X);
  void* XN = ws + wl.XN;
  float* SSQ = (float*)(ws + wl.SSQ);
  float* RAW = (float*)(ws + wl.RAW);
  float* Q = (float*)(ws + wl.Q);
  void* ATT = ws + wl.ATT;
  void* ACT = ws + wl.ACT;
  float* PART = (float*)(ws + wl.PART);
  unsigned long long* KEYS = (unsigned long long*)(ws + wl.KEYS);
  uint32_t* ERR = (uint32_t*)(ws + wl.ERR);
  const int d = c.d_model, N = sp.N, R = sp.R;
  const Dims& dm = sp.dm;
  auto layer = [&](int l) { return P + pl.layer0 + (size_t)l * pl.layer_stride; };
  const bool dumping = m->dump && m->dump_floats >= (size_t)(c.n_layers + 1) * N * d;
  // many-token products go to the tensor cores in the serving mode
  auto product = [&](const GemvArgs& g, int epi, const CUtensorMap* tw, const CUtensorMap* tx,
                     const CUtensorMap* tx32, bool proj = true) -> cudaError_t {
    if (i4 && proj) return launch_gemv_i4(g, epi, st);  // int4 projections: dequantized in registers
    if (bf && m->tc_on && m->tc_ready && g.T > kGemvMaxTokens && tc_eligible(g))
      return launch_gemm_tc(g, epi, tw, tx, m->num_sms, ERR, st);
    if (bf && m->tc_on && m->tc_ready && tc_skinny_eligible(g))
      return launch_gemm_tc_skinny(g, epi, tw, tx32, ERR, true, st);
    return launch_gemv(g, epi, bf, st);
  };

  // serving-mode decode steps: attention on the tensor cores with the QK-norm,
  // RoPE and cache append fused in
  const bool dec_tc_attn = decode_tc_attn(m, sp);
  if (dec_tc_attn) {
    int rc = ensure_kvmap(m, sp);
    if (rc) return rc;
  }
  EmbedArgs ea{P + pl.embed, sp.meta.ids, N, d, c.vocab, R, (const float*)(layer(0) + pl.attn_norm), X, XN, SSQ, KEYS,
               ERR};
  DEC_LAUNCH(DEC_K_EMBED, launch_embed(ea, bf, st));
  if (dumping) DEC_CUDA(cudaMemcpyAsync(m->dump, X, (size_t)N * d * 4, cudaMemcpyDeviceToDevice, st));

  for (int l = 0; l < c.n_layers; ++l) {
    char* Lb = layer(l);
    GemvArgs g{};
    g.d = d;
    g.eps = dm.eps;
    g.F = c.ff_hidden;
    // RMSNorm + [Wq;Wk;Wv]
    g.W = Lb + pl.wqkv; g.rows = qkv_rows(c); g.K = d; g.X = XN; g.x_row = nullptr; g.T = N; g.ssq = SSQ;
    g.out_f32 = RAW;
    // decode steps of the serving mode: raw q|k|v, then the tensor-core
    // attention that also norms, rotates and appends (no launch in between);
    // otherwise the skinny product fuses QK-norm/RoPE/cache write up to 16
    // token rows, and from 17 to 32 its raw output and k_qkv_post measure faster
    const bool tc_qkv = bf && m->tc_on && m->tc_ready && !dec_tc_attn &&
                        ((N > kGemvMaxTokens && tc_eligible(g)) || (N <= kQkvFuseMaxSkinny && tc_skinny_eligible(g)));
    if (dec_tc_attn) {
      DEC_LAUNCH(DEC_K_QKV, product(g, EPI_QKV_RAW, &m->tm_qkv[l], &m->tm_xn, &m->tm_xn32));
    } else if (tc_qkv) {
      // tensor-core product with QK-norm, RoPE and the cache write in its epilogue
      g.qf = QkvFuse{(const float*)(Lb + pl.q_norm), (const float*)(Lb + pl.k_norm), (const float*)(P + pl.rope), Q,
                     sp.slabs, l, sp.meta, c.n_heads, c.n_kv_heads, c.head_dim, dm.B, dm.n_blocks, dm.max_blocks, ERR};
      DEC_LAUNCH(DEC_K_QKV, product(g, EPI_QKV, &m->tm_qkv[l], &m->tm_xn, &m->tm_xn32));
    } else {
      DEC_LAUNCH(DEC_K_QKV, product(g, EPI_QKV_RAW, bf ? &m->tm_qkv[l] : nullptr, &m->tm_xn, &m->tm_xn32));
      QkvPostArgs qa{RAW, (const float*)(Lb + pl.q_norm), (const float*)(Lb + pl.k_norm),
                     (const float*)(P + pl.rope), Q, sp.slabs, l, sp.meta, dm, ERR};
      DEC_LAUNCH(DEC_K_QKV_POST, launch_qkv_post(qa, N, bf, st));
    }
    // attention
    AttnArgs aa{Q, sp.slabs, l, sp.meta, dm, ATT, PART, m->NCH, sp.S, 1.0f / std::sqrt((float)c.head_dim),
                (int*)(ws + wl.ACNT), ERR};
    if (dec_tc_attn) {
      AttnDecTcArgs ta{aa, RAW, (const float*)(Lb + pl.q_norm), (const float*)(Lb + pl.k_norm),
                       (const float*)(P + pl.rope)};
      DEC_LAUNCH(DEC_K_ATTN, launch_attn_decode_ring(ta, &m->kvmap, sp.meta.work, m->num_sms, st));
    } else if (sp.decode) {
      DEC_LAUNCH(DEC_K_ATTN, launch_attn_decode(aa, sp.slots, bf, st));
    } else if (bf && m->tc_on && attn_prefill_tc_eligible(aa)) {
      DEC_LAUNCH(DEC_K_ATTN, launch_attn_prefill_tc(aa, sp.n_work, st));
    } else {
      DEC_LAUNCH(DEC_K_ATTN, launch_attn_prefill(aa, sp.n_work, bf, st));
    }
    // O projection + residual; next GEMM input x * w_mlp
    GemvArgs go{};
    go.d = d; go.eps = dm.eps; go.F = c.ff_hidden;
    go.W = Lb + pl.wo; go.rows = d; go.K = c.n_heads * c.head_dim; go.X = ATT; go.T = N; go.ssq = nullptr;
    go.X_res = X; go.XN = XN; go.SSQ_out = SSQ; go.w_next = (const float*)(Lb + pl.mlp_norm);
    DEC_LAUNCH(DEC_K_OPROJ, product(go, EPI_RESID, bf ? &m->tm_o[l] : nullptr, &m->tm_att, &m->tm_att32));
    // RMSNorm + gate/up + SiLU*mul
    GemvArgs gu{};
    gu.d = d; gu.eps = dm.eps; gu.F = c.ff_hidden;
    gu.W = Lb + pl.wgu; gu.rows = 2 * c.ff_hidden; gu.K = d; gu.X = XN; gu.T = N; gu.ssq = SSQ; gu.act_out = ACT;
    DEC_LAUNCH(DEC_K_GATEUP, product(gu, EPI_SWIGLU, bf ? &m->tm_gu[l] : nullptr, &m->tm_xn, &m->tm_xn32));
    // down projection + residual; next GEMM input x * (next attention gain | final gain)
    GemvArgs gd{};
    gd.d = d; gd.eps = dm.eps; gd.F = c.ff_hidden;
    gd.W = Lb + pl.wd; gd.rows = d; gd.K = c.ff_hidden; gd.X = ACT; gd.T = N; gd.ssq = nullptr;
    gd.X_res = X; gd.XN = XN; gd.SSQ_out = SSQ;
    gd.w_next = l + 1 < c.n_layers ? (const float*)(layer(l + 1) + pl.attn_norm) : (const float*)(P + pl.final_norm);
    DEC_LAUNCH(DEC_K_DOWN, product(gd, EPI_RESID, bf ? &m->tm_d[l] : nullptr, &m->tm_act, &m->tm_act32));
    if (dumping)
      DEC_CUDA(cudaMemcpyAsync(m->dump + (size_t)(l + 1) * N * d, X, (size_t)N * d * 4, cudaMemcpyDeviceToDevice, st));
  }
  // final RMSNorm + tied LM head + argmax
  GemvArgs gl{};
  gl.d = d; gl.eps = dm.eps; gl.F = c.ff_hidden;
  // every-row logits read the activations in place (no row indirection)
  gl.W = P + pl.embed; gl.rows = c.vocab; gl.K = d; gl.X = XN; gl.x_row = (sp.rows_all || sp.decode) ? nullptr : sp.meta.row_tok;
  gl.T = R; gl.ssq = SSQ;
  gl.out_f32 = sp.logits; gl.keys = KEYS;
  DEC_LAUNCH(DEC_K_LMHEAD, product(gl, EPI_LOGITS, &m->tm_embed, &m->tm_xn, &m->tm_xn32, false));
  DEC_LAUNCH(DEC_K_ARGMAX, launch_argmax_finalize(KEYS, sp.argmax, R, st));
  return DEC_OK;
}

// The whole decode step as one persistent kernel (serving mode, <= 32 sequences).
static int enqueue_mega(dec_model* m, const StepPlan& sp, cudaStream_t st) {
  const dec_config& c = m->cfg;
  char* ws = m->ws;
  const WsLayout& wl = m->wl;
  const PackedLayout& pl = m->pl;
  DEC_CUDA(cudaMemsetAsync(ws + wl.MSYNC, 0, wl.msync_bytes, st));
  MegaArgs a{};
  a.layers = m->packed + pl.layer0;
  a.layer_stride = pl.layer_stride;
  a.o_attn_norm = pl.attn_norm;
  a.o_mlp_norm = pl.mlp_norm;
  a.o_q_norm = pl.q_norm;
  a.o_k_norm = pl.k_norm;
  a.o_wqkv = pl.wqkv;
  a.o_wo = pl.wo;
  a.o_wgu = pl.wgu;
  a.o_wd = pl.wd;
  a.embed = (const bf16*)(m->packed + pl.embed);
  a.final_norm = (const float*)(m->packed + pl.final_norm);
  a.w_attn0 = (const float*)(m->packed + pl.layer0 + pl.attn_norm);
  a.rope = (const float*)(m->packed + pl.rope);
  a.kv = (__half*)sp.slabs;
  a.n_blocks = sp.dm.n_blocks;
  a.vocab = c.vocab;
  a.d = c.d_model;
  a.n_layers = c.n_layers;
  a.H = c.n_heads;
  a.Hkv = c.n_kv_heads;
  a.D = c.head_dim;
  a.F = c.ff_hidden;
  a.max_blocks = sp.dm.max_blocks;
  a.eps = sp.dm.eps;
  a.scale = 1.0f / std::sqrt((float)c.head_dim);
  a.T = sp.N;
  a.ids = sp.meta.ids;
  a.seq_ctx = sp.meta.seq_ctx;
  a.tables = sp.meta.tables;
  a.item_start = sp.meta.work;
  a.X = (float*)(ws + wl.X);
  char* fl = ws + wl.FLOW;
  a.xa = (bf16*)(fl + wl.f_xa);
  a.xb = (bf16*)(fl + wl.f_xb);
  a.sa = (float*)(fl + wl.f_sa);
  a.sb = (float*)(fl + wl.f_sb);
  a.raw = (float*)(fl + wl.f_raw);
  a.att = (bf16*)(fl + wl.f_att);
  a.act = (bf16*)(fl + wl.f_act);
  a.rec = (float*)(fl + wl.f_rec);
  a.nch_cap = max_chunks64_of(c);
  const size_t Tm = (size_t)std::min(m->Tmax, kMegaMaxTokens);
  char* ms0 = ws + wl.MSYNC;
  a.sync = (unsigned int*)ms0;
  a.done = (unsigned int*)(ms0 + 64);
  a.abort = (unsigned int*)(ms0 + 128);
  a.keys = (unsigned long long*)(ms0 + 256);
  a.acnt = (unsigned int*)(ms0 + 256 + align256(Tm * 8));
  a.logits = sp.logits;
  a.argmax = sp.argmax;
  a.err = (uint32_t*)(ws + wl.ERR);
  const int kmax = std::max(c.d_model, std::max(c.n_heads * c.head_dim, c.ff_hidden));
  const MegaSmem ms = mega_smem(sp.N, kmax, c.head_dim, m->smem_optin);
  if (!ms.total) return fail(DEC_ECUDA, "the one-kernel step does not fit in shared memory");
  a.ring = ms.ring;
  a.o_stage = ms.o_stage;
  a.o_scr = ms.o_scr;
  a.o_small = ms.o_small;
  a.o_bars = ms.o_bars;
  a.trace = m->trace && m->trace_n >= (size_t)m->num_sms * kMegaTraceStride ? m->trace : nullptr;
  int rc = ensure_kvmap(m, sp);
  if (rc) return rc;
  a.tm_kv = m->kvmap;
  a.wait_extra = m->wait_extra;
  a.wait_limit = m->wait_limit;
  DEC_LAUNCH(DEC_K_STEP, launch_decode_mega(a, m->num_sms, ms.total, st));
  return DEC_OK;
}

static uint32_t prof_mask(const dec_model* m) {
  uint32_t mask = 0;
  for (int i = 0; i < DEC_K_COUNT; ++i)
    if (m->prof_on[i]) mask |= 1u << i;
  return mask;
}

// The event-record nodes that capture made of the profiling events in recs,
// paired per launch (the graph's node list has no capture order, so nodes are
// matched by the event they record).
static int find_prof_nodes(cudaGraph_t g, const std::vector<dec_model::ProfRec>& recs, std::vector<ProfNode>* out) {
  size_t n = 0;
  DEC_CUDA(cudaGraphGetNodes(g, nullptr, &n));
  std::vector<cudaGraphNode_t> nodes(n);
  if (n) DEC_CUDA(cudaGraphGetNodes(g, nodes.data(), &n));
  std::unordered_map<cudaEvent_t, std::pair<size_t, int>> where;  // event -> (record, 0 = a / 1 = b)
  for (size_t i = 0; i < recs.size(); ++i) {
    where[recs[i].a] = {i, 0};
    where[recs[i].b] = {i, 1};
  }
  out->assign(recs.size(), ProfNode{nullptr, nullptr, 0});
  for (size_t i = 0; i < recs.size(); ++i) (*out)[i].cls = recs[i].cls;
  for (cudaGraphNode_t nd : nodes) {
    cudaGraphNodeType t;
    DEC_CUDA(cudaGraphNodeGetType(nd, &t));
    if (t != cudaGraphNodeTypeEventRecord) continue;
    cudaEvent_t ev = nullptr;
    DEC_CUDA(cudaGraphEventRecordNodeGetEvent(nd, &ev));
    auto it = where.find(ev);
    if (it == where.end()) continue;
    ProfNode& p = (*out)[it->second.first];
    (it->second.second ? p.b : p.a) = nd;
  }
  for (const ProfNode& p : *out)
    if (!p.a || !p.b) return fail(DEC_ECUDA, "a profiling event has no node in the captured step");
  return DEC_OK;
}

// Launch a captured step.  Its profiling nodes (if any) first move to fresh
// events, so each replay's launches are timed like eager ones; launches
// already queued keep the events they had.
static int replay_graph(dec_model* m, GraphEntry* g, cudaStream_t st) {
  for (const ProfNode& p : g->pnodes) {
    cudaEvent_t a = take_event(m), b = take_event(m);
    cudaError_t e = (a && b) ? cudaGraphExecEventRecordNodeSetEvent(g->exec, p.a, a) : cudaErrorMemoryAllocation;
    if (e == cudaSuccess) e = cudaGraphExecEventRecordNodeSetEvent(g->exec, p.b, b);
    if (e != cudaSuccess) {
      if (a) m->ev_free.push_back(a);
      if (b) m->ev_free.push_back(b);
      return fail(DEC_ECUDA, "profiling node: %s", cudaGetErrorString(e));
    }
    m->prof_pending.push_back({a, b, p.cls});
  }
  DEC_CUDA(cudaGraphLaunch(g->exec, st));
  m->launches += g->n_launch;
  return DEC_OK;
}

static void drop_graph(GraphEntry& g) {
  if (g.exec) cudaGraphExecDestroy(g.exec);
  if (g.graph) cudaGraphDestroy(g.graph);
  g.exec = nullptr;
  g.graph = nullptr;
}

// Decode steps of one shape replay a captured CUDA graph: the per-step
// metadata lives at fixed device addresses (one host->device copy before the
// replay), so (S, attention grid, logits, argmax, pool and its size, profiled
// classes) key a graph.  A key's first step runs eagerly; its second captures.
static int launch_decode_graph(dec_model* m, const StepPlan& sp, cudaStream_t st) {
  const uint32_t mask = prof_mask(m);
  GraphEntry* hit = nullptr;
  for (auto& e : m->graphs)
    if (e.S == sp.S && e.slots == sp.slots && e.logits == sp.logits && e.argmax == sp.argmax &&
        e.slabs == sp.slabs && e.n_blocks == sp.dm.n_blocks && e.prof_mask == mask)
      hit = &e;
  ++m->graph_clock;
  if (hit && hit->exec) {
    hit->last_use = m->graph_clock;
    return replay_graph(m, hit, st);
  }
  if (!hit) {  // first sighting: run eagerly, remember the key
    if (m->graphs.size() >= kMaxGraphs) {
      size_t victim = 0;
      for (size_t i = 1; i < m->graphs.size(); ++i)
        if (m->graphs[i].last_use < m->graphs[victim].last_use) victim = i;
      drop_graph(m->graphs[victim]);
      m->graphs.erase(m->graphs.begin() + victim);
    }
    GraphEntry e{};
    e.S = sp.S;
    e.slots = sp.slots;
    e.logits = sp.logits;
    e.argmax = sp.argmax;
    e.slabs = sp.slabs;
    e.n_blocks = sp.dm.n_blocks;
    e.prof_mask = mask;
    e.last_use = m->graph_clock;
    m->graphs.push_back(e);
    return enqueue_step(m, sp, st);
  }
  // second sighting: capture on the model's private stream, then replay on st
  if (!m->cap_stream) DEC_CUDA(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
  const int64_t before = m->launches;
  DEC_CUDA(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
  m->capturing = true;
  m->cap_recs.clear();
  int rc = enqueue_step(m, sp, m->cap_stream);
  m->capturing = false;
  std::vector<dec_model::ProfRec> recs;
  recs.swap(m->cap_recs);
  cudaGraph_t graph = nullptr;
  cudaError_t ec = cudaStreamEndCapture(m->cap_stream, &graph);
  std::vector<ProfNode> pnodes;
  if (!rc && ec == cudaSuccess && !recs.empty()) rc = find_prof_nodes(graph, recs, &pnodes);
  for (auto& r : recs) {  // the capture's own events never record anything
    m->ev_free.push_back(r.a);
    m->ev_free.push_back(r.b);
  }
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (ec != cudaSuccess) return fail(DEC_ECUDA, "graph capture: %s", cudaGetErrorString(ec));
  cudaGraphExec_t exec = nullptr;
  ec = cudaGraphInstantiate(&exec, graph, 0);
  if (ec != cudaSuccess) {
    cudaGraphDestroy(graph);
    return fail(DEC_ECUDA, "graph instantiate: %s", cudaGetErrorString(ec));
  }
  if (pnodes.empty()) {
    cudaGraphDestroy(graph);
    graph = nullptr;
  }
  hit->exec = exec;
  hit->graph = graph;
  hit->pnodes = std::move(pnodes);
  hit->n_launch = m->launches - before;
  m->launches = before;
  hit->last_use = m->graph_clock;
  return replay_graph(m, hit, st);
}

// Every check a step makes before it launches anything, host data only
// (tinyllm L10.1 section 4, forward_refuses_bad_batches: a scheduler's
// mistake surfaces as an error instead of corrupting the cache).  The blocks
// a sequence writes (positions p0 .. its last new position) must belong to it
// alone: refcount 1, not indexed in the prefix cache, and named by no other
// written position of the batch.
static int check_batch(const dec_config& c, const dec_pool* pool, const dec_batch* b, bool decode) {
  if (!b) return fail(DEC_EINVAL, "NULL argument");
  const int S = b->n_seqs, N = b->n_tokens;
  if (S < 1 || N < 1) return fail(DEC_EINVAL, "empty step: %d sequences, %d tokens", S, N);
  if (decode && N != S) return fail(DEC_EINVAL, "decode takes exactly one token per sequence");
  if (!b->seq_start || !b->positions || !b->block_table || (!b->ids && !b->ids_device))
    return fail(DEC_EINVAL, "NULL batch array");
  if (b->seq_start[0] != 0 || b->seq_start[S] != N) return fail(DEC_EINVAL, "seq_start must run from 0 to n_tokens");
  const int B = c.block_tokens;
  std::vector<int32_t> written;
  for (int s = 0; s < S; ++s) {
    const int a0 = b->seq_start[s], a1 = b->seq_start[s + 1];
    if (a1 <= a0) return fail(DEC_EINVAL, "sequence %d has no new tokens", s);
    const int p0 = b->positions[a0];
    if (p0 < 0) return fail(DEC_ERANGE, "negative position in sequence %d", s);
    for (int t = a0; t < a1; ++t) {
      if (b->positions[t] != p0 + (t - a0))
        return fail(DEC_ERANGE, "positions of sequence %d are not consecutive", s);
      if (b->ids && !b->ids_device && (b->ids[t] < 0 || b->ids[t] >= c.vocab))
        return fail(DEC_EVOCAB, "token id %d outside the vocabulary (%d)", b->ids[t], c.vocab);
    }
    const int last = p0 + (a1 - a0) - 1;
    if (last >= c.max_positions) return fail(DEC_ERANGE, "position %d past the context (%d)", last, c.max_positions);
    const int nb = last / B + 1;
    if (nb > b->max_blocks) return fail(DEC_ERANGE, "block table of sequence %d too short for position %d", s, last);
    for (int i = 0; i < nb; ++i) {
      const int id = b->block_table[(size_t)s * b->max_blocks + i];
      if (id < 0 || id >= pool->n_blocks || pool->refs[id] <= 0)
        return fail(DEC_EBLOCK, "sequence %d names block %d which is not allocated", s, id);
      if (i >= p0 / B) {  // this step writes K/V into block i
        if (pool->refs[id] != 1 || pool->registered[id])
          return fail(DEC_EBLOCK, "sequence %d would write block %d, which is shared (refcount %d) or in the prefix cache",
                      s, id, pool->refs[id]);
        written.push_back(id);
      }
    }
  }
  std::sort(written.begin(), written.end());
  const auto dup = std::adjacent_find(written.begin(), written.end());
  if (dup != written.end()) return fail(DEC_EBLOCK, "block %d would be written for two positions of the step", *dup);
  return DEC_OK;
}

static int run_step(dec_model* m, dec_pool* pool, const dec_batch* b, int rows_mode, float* logits, int32_t* argmax,
                    cudaStream_t st, bool decode) {
  if (!m || !pool || !b || !argmax) return fail(DEC_EINVAL, "NULL argument");
  const dec_config& c = m->cfg;
  if (!same_shape(c, pool->cfg)) return fail(DEC_EINVAL, "pool was made for another decoder shape or mode");
  if (rows_mode != DEC_ROWS_ALL && rows_mode != DEC_ROWS_LAST) return fail(DEC_EINVAL, "bad rows mode");
  const int S = b->n_seqs, N = b->n_tokens;
  if (S > m->Smax || N > m->Tmax)
    return fail(DEC_ERANGE, "step of %d tokens / %d sequences exceeds the workspace (%d / %d)", N, S, m->Tmax, m->Smax);
  int rc = check_batch(c, pool, b, decode);
  if (rc) return rc;
  const int B = c.block_tokens;
  const int R = rows_mode == DEC_ROWS_ALL ? N : S;
  int max_ctx = 0;
  for (int s = 0; s < S; ++s) max_ctx = std::max(max_ctx, b->positions[b->seq_start[s + 1] - 1] + 1);

  // ---- metadata: assemble, stage in pinned memory, one host->device copy ----
  const int MB = m->MB;
  const int G = c.n_heads / c.n_kv_heads;
  const int QT = prefill_tile_queries(G);
  const int slot = m->stage_next;
  m->stage_next = (m->stage_next + 1) % kStageSlots;
  DEC_CUDA(cudaEventSynchronize(m->stage_ev[slot]));  // the copy that last used this slot has run
  int32_t* H = m->stage[slot];
  size_t o = 0;
  const size_t o_ids = o; o += N;
  const size_t o_pos = o; o += N;
  const size_t o_seq = o; o += N;
  const size_t o_start = o; o += S + 1;
  const size_t o_ctx = o; o += S;
  const size_t o_row = o; o += R;
  const size_t o_tab = o; o += (size_t)S * MB;
  const size_t o_work = o;
  for (int s = 0; s < S; ++s) {
    const int a0 = b->seq_start[s], a1 = b->seq_start[s + 1];
    for (int t = a0; t < a1; ++t) {
      H[o_ids + t] = b->ids ? b->ids[t] : 0;
      H[o_pos + t] = b->positions[t];
      H[o_seq + t] = s;
    }
    H[o_start + s] = a0;
    H[o_ctx + s] = b->positions[a1 - 1] + 1;
    const int nb = b->positions[a1 - 1] / B + 1;
    for (int i = 0; i < MB; ++i) H[o_tab + (size_t)s * MB + i] = i < nb ? b->block_table[(size_t)s * b->max_blocks + i] : 0;
  }
  H[o_start + S] = N;
#ifdef DEC_DEBUG
  if (m->poison[0] >= 0) {  // test hook: a bad entry in the device copy only (the host used the real table)
    if (m->poison[0] < S && m->poison[1] < MB) H[o_tab + (size_t)m->poison[0] * MB + m->poison[1]] = m->poison[2];
    m->poison[0] = -1;
  }
#endif
  if (rows_mode == DEC_ROWS_ALL)
    for (int t = 0; t < N; ++t) H[o_row + t] = t;
  else
    for (int s = 0; s < S; ++s) H[o_row + s] = b->seq_start[s + 1] - 1;
  // prefill attention tiles, the ones reaching furthest first
  std::vector<std::array<int, 3>> work;
  if (!decode) {
    for (int s = 0; s < S; ++s)
      for (int t = b->seq_start[s]; t < b->seq_start[s + 1]; t += QT)
        work.push_back({s, t, std::min(QT, b->seq_start[s + 1] - t)});
    std::stable_sort(work.begin(), work.end(), [&](const std::array<int, 3>& x, const std::array<int, 3>& y) {
      return b->positions[x[1] + x[2] - 1] > b->positions[y[1] + y[2] - 1];
    });
  }
  for (size_t i = 0; i < work.size(); ++i)
    for (int k = 0; k < 3; ++k) H[o_work + 3 * i + k] = work[i][k];
  o += 3 * work.size();
  const bool mega = decode && m->mega_on && m->mega_shape && N <= kMegaAutoTokens && !m->dump;
  static_assert(kMegaKeys == kDecodeChunk, "one attention item layout for both decode paths");
  if (decode) {
    // decode attention items, sequence-major: the first of every sequence (KV heads x 64-key chunks each)
    int first = 0;
    for (int s = 0; s < S; ++s) {
      H[o_work + s] = first;
      first += c.n_kv_heads * ((b->positions[b->seq_start[s + 1] - 1] + kDecodeChunk) / kDecodeChunk);
    }
    H[o_work + S] = first;
    o += S + 1;
  }
  if (o > m->wl.meta_ints) return fail(DEC_ERANGE, "step metadata exceeds the workspace");

  int32_t* dmeta = (int32_t*)(m->ws + m->wl.META);
  DEC_CUDA(cudaMemcpyAsync(dmeta, H, o * 4, cudaMemcpyHostToDevice, st));
  DEC_CUDA(cudaEventRecord(m->stage_ev[slot], st));
  m->last_stream = st;

  const bool graph = decode && m->graphs_on && !m->dump;
  if (graph && b->ids_device)  // graphs read ids from the metadata block
    DEC_CUDA(cudaMemcpyAsync(dmeta + o_ids, b->ids_device, (size_t)N * 4, cudaMemcpyDeviceToDevice, st));

  StepPlan sp;
  sp.meta.ids = (b->ids_device && !graph) ? b->ids_device : dmeta + o_ids;
  sp.meta.tok_pos = dmeta + o_pos;
  sp.meta.tok_seq = dmeta + o_seq;
  sp.meta.seq_start = dmeta + o_start;
  sp.meta.seq_ctx = dmeta + o_ctx;
  sp.meta.row_tok = dmeta + o_row;
  sp.meta.tables = dmeta + o_tab;
  sp.meta.work = dmeta + o_work;
  sp.dm.vocab = c.vocab; sp.dm.d = c.d_model; sp.dm.n_layers = c.n_layers; sp.dm.H = c.n_heads;
  sp.dm.Hkv = c.n_kv_heads; sp.dm.D = c.head_dim; sp.dm.F = c.ff_hidden; sp.dm.B = B;
  sp.dm.n_blocks = pool->n_blocks; sp.dm.max_blocks = MB; sp.dm.eps = (float)c.rms_eps;
  sp.N = N;
  sp.S = S;
  sp.R = R;
  sp.decode = decode;
  sp.rows_all = rows_mode == DEC_ROWS_ALL;
  sp.n_work = (int)work.size();
  // decode attention grid: one CTA per 64-key chunk of the longest sequence, rounded
  // up to a multiple of 4 chunks so a captured graph serves 256 positions of growth
  sp.slots = std::min(m->NCH, ((max_ctx + kDecodeChunk - 1) / kDecodeChunk + 3) / 4 * 4);
  if (decode_tc_attn(m, sp)) sp.slots = 0;  // unused there: one captured graph serves every context
  sp.slabs = pool->slabs;
  sp.logits = logits;
  sp.argmax = argmax;
  if (mega) return enqueue_mega(m, sp, st);
  if (graph) return launch_decode_graph(m, sp, st);
  return enqueue_step(m, sp, st);
}

int dec_batch_check(const dec_pool* pool, const dec_batch* b, int32_t decode) {
  if (!pool) return fail(DEC_EINVAL, "NULL argument");
  return check_batch(pool->cfg, pool, b, decode != 0);
}

int dec_prefill(dec_model* m, dec_pool* pool, const dec_batch* b, int32_t rows, float* logits, int32_t* argmax,
                void* stream) {
  return run_step(m, pool, b, rows, logits, argmax, (cudaStream_t)stream, false);
}

int dec_decode(dec_model* m, dec_pool* pool, const dec_batch* b, float* logits, int32_t* argmax, void* stream) {
  return run_step(m, pool, b, DEC_ROWS_LAST, logits, argmax, (cudaStream_t)stream, true);
}

int dec_debug_product(dec_model* m, int32_t which, int32_t layer, const void* X, int32_t T, float* Y, int32_t path,
                      void* stream) {
  if (!m || !X || !Y || T < 1 || which < 0 || which > 4 || path < 0 || path > 2)
    return fail(DEC_EINVAL, "bad arguments");
  const dec_config& c = m->cfg;
  if (which < 4 && (layer < 0 || layer >= c.n_layers)) return fail(DEC_EINVAL, "bad layer");
  const bool bf = c.mode == DEC_BF16_F16KV;
  const bool i4 = int4_proj(c) && which < 4;
  const int d = c.d_model, HD = c.n_heads * c.head_dim, F = c.ff_hidden;
  char* Lb = m->packed + m->pl.layer0 + (size_t)(which < 4 ? layer : 0) * m->pl.layer_stride;
  GemvArgs g{};
  g.d = d;
  g.eps = (float)c.rms_eps;
  g.F = F;
  g.X = X;
  g.T = T;
  g.out_f32 = Y;
  const CUtensorMap* tw = nullptr;
  switch (which) {
    case 0: g.W = Lb + m->pl.wqkv; g.rows = qkv_rows(c); g.K = d; if (bf) tw = &m->tm_qkv[layer]; break;
    case 1: g.W = Lb + m->pl.wo; g.rows = d; g.K = HD; if (bf) tw = &m->tm_o[layer]; break;
    case 2: g.W = Lb + m->pl.wgu; g.rows = 2 * F; g.K = d; if (bf) tw = &m->tm_gu[layer]; break;
    case 3: g.W = Lb + m->pl.wd; g.rows = d; g.K = F; if (bf) tw = &m->tm_d[layer]; break;
    default: g.W = m->packed + m->pl.embed; g.rows = c.vocab; g.K = d; if (bf) tw = &m->tm_embed; break;
  }
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t* ERR = (uint32_t*)(m->ws + m->wl.ERR);
  if (path == 2) {
    if (!bf || !m->tc_ready || !tc_skinny_eligible(g))
      return fail(DEC_EINVAL, "the decode tensor-core path needs the serving mode, T <= 32 and a 128-row multiple");
    CUtensorMap tx;
    if (!bf16_map(&tx, X, T, g.K, 32)) return fail(DEC_ECUDA, "tensor map for X failed");
    DEC_CUDA(launch_gemm_tc_skinny(g, EPI_QKV_RAW, tw, &tx, ERR, false, st));
  } else if (path == 1) {
    if (!bf || !m->tc_ready || T <= kGemvMaxTokens || !tc_eligible(g))
      return fail(DEC_EINVAL, "the tensor-core path needs the serving mode, T > %d and a 128-row multiple",
                  kGemvMaxTokens);
    CUtensorMap tx;
    if (!bf16_map(&tx, X, T, g.K)) return fail(DEC_ECUDA, "tensor map for X failed");
    DEC_CUDA(launch_gemm_tc(g, EPI_QKV_RAW, tw, &tx, m->num_sms, ERR, st));
  } else if (i4) {
    DEC_CUDA(launch_gemv_i4(g, EPI_QKV_RAW, st));
  } else {
    DEC_CUDA(launch_gemv(g, EPI_QKV_RAW, serving(c), st));
  }
  m->last_stream = st;
  return DEC_OK;
}

int dec_quantize_int4(const float* W, int32_t rows, int32_t K, void* codes, void* scales, void* stream) {
  if (!W || !codes || !scales || rows < 1 || K < 32 || K % 32) return fail(DEC_EINVAL, "bad arguments");
  if (((uintptr_t)codes & 15) || ((uintptr_t)scales & 1)) return fail(DEC_EINVAL, "codes need 16-byte alignment");
  DEC_CUDA(launch_quant_i4(codes, scales, W, rows, K, PACK_IDENTITY, (cudaStream_t)stream));
  return DEC_OK;
}

int dec_f32_to_f16(const float* in, uint16_t* out, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return fail(DEC_EINVAL, "bad arguments");
  DEC_CUDA(launch_f32_to_f16(in, out, n, (cudaStream_t)stream));
  return DEC_OK;
}

}  // extern "C"
