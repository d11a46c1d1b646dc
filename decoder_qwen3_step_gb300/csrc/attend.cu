// attend.cu - decode attention on its own, through the C ABI: one query per
// sequence attends over its keys in the paged KV pool with the split-K kernel
// that dec_decode runs (tinyllm L10.1 "Candle model runner ...", section 2.4:
// o = sum_{j < ctx} softmax_j(q . k_j / sqrt(D)) v_j; query head h reads KV
// head floor(h * Hkv / H)).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <mutex>

#include "../../include/dec.h"
#include "common.cuh"
#include "internal.h"
#include "launch.h"

using namespace dec;

namespace {

int fail_msg(int code, const char* what) { return set_error(code, what); }

// Scratch layout (bytes from the start, 256-byte aligned pieces):
//   [0, 256)            error word (uint32) + padding
//   counters            int32 [S * Hkv], zero at every launch
//   meta                int32: seq_start [S+1] | ctx [S] | tables [S * max_blocks]
//   partials            fp32 [S, H, chunks, D+2]
struct AttendLayout {
  size_t counters, meta, part, total;
  int chunks;
};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

AttendLayout attend_layout(const dec_config& c, int S, int max_ctx, int max_blocks) {
  AttendLayout L{};
  L.chunks = (max_ctx + kDecodeChunk - 1) / kDecodeChunk;
  L.counters = 256;
  L.meta = up256(L.counters + (size_t)S * c.n_kv_heads * 4);
  L.part = up256(L.meta + ((size_t)2 * S + 1 + (size_t)S * max_blocks) * 4);
  L.total = up256(L.part + (size_t)S * c.n_heads * L.chunks * (c.head_dim + 2) * 4);
  return L;
}

// Host checks shared by both entry points; fills max_ctx.
int attend_check(const dec_pool* pool, int32_t layer, int32_t n_seqs, const float* q, const int32_t* ctx,
                 const int32_t* block_table, int32_t max_blocks, const void* out, int* max_ctx) {
  if (!pool || !q || !ctx || !block_table || !out) return fail_msg(DEC_EINVAL, "NULL argument");
  const dec_config& c = pool->cfg;
  if (layer < 0 || layer >= c.n_layers) return fail_msg(DEC_EINVAL, "layer outside the model");
  if (n_seqs < 1) return fail_msg(DEC_EINVAL, "n_seqs must be at least 1");
  if (max_blocks < 1) return fail_msg(DEC_EINVAL, "max_blocks must be at least 1");
  int mc = 0;
  for (int s = 0; s < n_seqs; ++s) {
    if (ctx[s] < 1 || ctx[s] > c.max_positions) return fail_msg(DEC_ERANGE, "context length outside 1 .. max_positions");
    const int nb = (ctx[s] + c.block_tokens - 1) / c.block_tokens;
    if (nb > max_blocks) return fail_msg(DEC_ERANGE, "block table too short for a context length");
    for (int i = 0; i < nb; ++i) {
      const int id = block_table[(size_t)s * max_blocks + i];
      if (id < 0 || id >= pool->n_blocks || pool->refs[id] <= 0)
        return fail_msg(DEC_EBLOCK, "a block table names a block that is not allocated");
    }
    mc = ctx[s] > mc ? ctx[s] : mc;
  }
  *max_ctx = mc;
  return DEC_OK;
}

// Upload the metadata into `scratch`, clear the counters and the error word,
// and launch the split-K kernel.
int attend_launch(const dec_pool* pool, int32_t layer, int32_t n_seqs, const float* q, const int32_t* ctx,
                  const int32_t* block_table, int32_t max_blocks, void* out, char* scratch, const AttendLayout& L,
                  const int32_t* seq_start_host, cudaStream_t st) {
  const dec_config& c = pool->cfg;
  const int S = n_seqs;
  int32_t* meta = reinterpret_cast<int32_t*>(scratch + L.meta);
  cudaError_t e = cudaMemsetAsync(scratch, 0, L.meta, st);  // error word and counters
  if (e == cudaSuccess) e = cudaMemcpyAsync(meta, seq_start_host, (size_t)(S + 1) * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(meta + S + 1, ctx, (size_t)S * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(meta + 2 * S + 1, block_table, (size_t)S * max_blocks * 4, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail_msg(DEC_ECUDA, cudaGetErrorString(e));
  AttnArgs a{};
  a.Q = q;
  a.kv = pool->slabs;
  a.layer = layer;
  a.meta.seq_start = meta;
  a.meta.seq_ctx = meta + S + 1;
  a.meta.tables = meta + 2 * S + 1;
  a.dims.vocab = c.vocab;
  a.dims.d = c.d_model;
  a.dims.n_layers = c.n_layers;
  a.dims.H = c.n_heads;
  a.dims.Hkv = c.n_kv_heads;
  a.dims.D = c.head_dim;
  a.dims.F = c.ff_hidden;
  a.dims.B = c.block_tokens;
  a.dims.n_blocks = pool->n_blocks;
  a.dims.max_blocks = max_blocks;
  a.dims.eps = (float)c.rms_eps;
  a.ATT = out;
  a.part = reinterpret_cast<float*>(scratch + L.part);
  a.nchunk_cap = L.chunks;
  a.S = S;
  a.scale = 1.0f / std::sqrt((float)c.head_dim);
  a.counters = reinterpret_cast<int*>(scratch + L.counters);
  a.err = reinterpret_cast<uint32_t*>(scratch);
  e = launch_attn_decode(a, L.chunks, c.mode != DEC_FP32, st);
  if (e != cudaSuccess) return fail_msg(DEC_ECUDA, cudaGetErrorString(e));
  return DEC_OK;
}

// ---- scratch that needs no allocation --------------------------------------
// Some callers cannot allocate device memory when they want attention: code
// embedded in a host framework that owns every device allocation and hands
// out only the tensors it manages, plug-ins whose memory budget was fixed
// when they were loaded, or latency-critical loops that must not pay for the
// allocator (cudaMalloc and cudaFree can synchronise the device).  For them
// dec_attend_noalloc keeps its scratch in the library's own device array,
// which every GPU that loads the library holds until the process exits.
constexpr size_t kNoAllocBytes = 4u << 20;  // 4 MiB
constexpr int kNoAllocMaxSeqs = 256;
constexpr int kMaxDevices = 64;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];

// The array's device address on the current device, looked up once per
// device (the host-side name of the array is not a device address).
int noalloc_scratch(char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_msg(DEC_ECUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail_msg(DEC_EINVAL, "device index beyond the scratch table");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return fail_msg(DEC_ECUDA, "cudaGetSymbolAddress of the scratch array failed");
    g_noalloc_ptr[dev] = p;
  }
  *out = static_cast<char*>(g_noalloc_ptr[dev]);
  return DEC_OK;
}

}  // namespace

// Resolve the no-allocation array's address on the current device now (the
// first resolution on a device loads the module that holds the array).
int dec::noalloc_prepare() {
  char* p = nullptr;
  return noalloc_scratch(&p);
}

extern "C" {

int dec_attend_scratch_bytes(const dec_config* cfg, int32_t n_seqs, int32_t max_ctx, int32_t max_blocks,
                             size_t* bytes) {
  if (!cfg || !bytes || n_seqs < 1 || max_ctx < 1 || max_blocks < 1) return fail_msg(DEC_EINVAL, "bad arguments");
  *bytes = attend_layout(*cfg, n_seqs, max_ctx, max_blocks).total;
  return DEC_OK;
}

int dec_attend(const dec_pool* pool, int32_t layer, int32_t n_seqs, const float* q, const int32_t* ctx,
               const int32_t* block_table, int32_t max_blocks, void* out, void* scratch, size_t scratch_bytes,
               void* stream) {
  int max_ctx = 0;
  int rc = attend_check(pool, layer, n_seqs, q, ctx, block_table, max_blocks, out, &max_ctx);
  if (rc) return rc;
  if (!scratch || ((uintptr_t)scratch & 255)) return fail_msg(DEC_EINVAL, "scratch must be 256-byte aligned device memory");
  const AttendLayout L = attend_layout(pool->cfg, n_seqs, max_ctx, max_blocks);
  if (scratch_bytes < L.total) return fail_msg(DEC_EINVAL, "scratch smaller than dec_attend_scratch_bytes");
  std::vector<int32_t> seq_start(n_seqs + 1);
  for (int s = 0; s <= n_seqs; ++s) seq_start[s] = s;
  return attend_launch(pool, layer, n_seqs, q, ctx, block_table, max_blocks, out, (char*)scratch, L,
                       seq_start.data(), (cudaStream_t)stream);
}

int dec_attend_noalloc_status(void* stream, uint32_t* flags) {
  if (!flags) return fail_msg(DEC_EINVAL, "NULL argument");
  char* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t v = 0;
  // the error word is the array's first word (the layout dec_attend uses)
  cudaError_t e = cudaMemcpyAsync(&v, scratch, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, 4, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_msg(DEC_ECUDA, cudaGetErrorString(e));
  *flags = v;
  return DEC_OK;
}

int dec_attend_noalloc(const dec_pool* pool, int32_t layer, int32_t n_seqs, const float* q, const int32_t* ctx,
                       const int32_t* block_table, int32_t max_blocks, void* out, void* stream) {
  int max_ctx = 0;
  int rc = attend_check(pool, layer, n_seqs, q, ctx, block_table, max_blocks, out, &max_ctx);
  if (rc) return rc;
  if (n_seqs > kNoAllocMaxSeqs) return fail_msg(DEC_ERANGE, "dec_attend_noalloc takes at most 256 sequences");
  const AttendLayout L = attend_layout(pool->cfg, n_seqs, max_ctx, max_blocks);
  if (L.total > kNoAllocBytes) {
    char msg[160];
    snprintf(msg, sizeof msg, "dec_attend_noalloc needs %zu bytes of scratch, more than its fixed %zu; use dec_attend",
             L.total, kNoAllocBytes);
    return fail_msg(DEC_ERANGE, msg);
  }
  char* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  thread_local int32_t seq_start[kNoAllocMaxSeqs + 1];
  for (int s = 0; s <= n_seqs; ++s) seq_start[s] = s;
  return attend_launch(pool, layer, n_seqs, q, ctx, block_table, max_blocks, out, scratch, L, seq_start,
                       (cudaStream_t)stream);
}

}  // extern "C"
