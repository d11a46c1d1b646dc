/*
 * dec.h - C ABI of libdec: one forward step of a Qwen3-style pre-norm decoder
 * with a paged KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * The step computed (tinyllm L10.1 "Candle model runner (Llama + bigram,
 * int4), Rust KV cache, sampler and PCG32", section 2.4 "The Llama forward,
 * one step"; octlm "A real model in our own decoder", the five switches):
 *
 *   x = E[id]
 *   per layer: h = RMSNorm(x) ; q,k,v = h W^T ; q,k <- per-head RMSNorm
 *              (QK-norm) ; q,k <- split-half RoPE at pos(t), base rope_base ;
 *              K/V of every new token -> its sequence's KV blocks ;
 *              o_t = sum_{j <= pos(t)} softmax_j(q_t . k_j / sqrt(D)) v_j
 *              (grouped-query: query head h reads KV head floor(h*Hkv/H)) ;
 *              x += o W_o^T ; x += (silu(h2 W_g^T) * (h2 W_u^T)) W_d^T,
 *              h2 = RMSNorm(x)
 *   logits = RMSNorm(x) E^T (tied embedding) ; greedy id = argmax, lowest
 *   id on ties (tinyllm L10.1 section 2.6).
 *
 * Conventions for every entry point:
 *  - Return value: DEC_OK (0) or one of the DEC_E* codes below;
 *    dec_last_error() then returns a message (thread-local, valid until the
 *    next call on the same thread).  All argument and batch checks run on the
 *    host BEFORE any device work is queued, so a refused call leaves the KV
 *    cache and every output untouched (tinyllm L10.1 section 4,
 *    forward_refuses_bad_batches).
 *  - Memory: the caller allocates every device buffer (weights, the packed
 *    weight buffer, the workspace, the KV slabs, logits, ids).  The library
 *    never calls cudaMalloc; it owns only host metadata (block refcounts and
 *    free list, descriptors, a small pinned staging ring for per-step
 *    metadata, captured CUDA graphs).
 *  - Streams: device work is queued on the caller's stream (a cudaStream_t
 *    passed as void*; NULL = the legacy default stream) and is asynchronous;
 *    outputs are valid once that stream has synchronised.
 *  - Devices: one GPU per model; all pointers given to a model live on the
 *    device that was current when dec_create ran.
 */
#ifndef DEC_H
#define DEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define DEC_OK        0
#define DEC_EINVAL    1 /* bad argument or unsupported config (scaled RoPE, sliding window, biases...) */
#define DEC_ECAPACITY 2 /* pool has fewer free blocks than asked (allocation is all-or-nothing) */
#define DEC_EBLOCK    3 /* block id outside the pool or not currently allocated */
#define DEC_ERANGE    4 /* position past max_positions, short block table, or too many tokens */
#define DEC_EVOCAB    5 /* token id outside [0, vocab) */
#define DEC_ECUDA     6 /* a CUDA runtime call failed */
#define DEC_EDEVICE   7 /* a kernel raised its device error word (see dec_device_status) */

/* ---- numeric modes -------------------------------------------------------- */
#define DEC_FP32       0 /* fp32 weights, fp32 activations, fp32 KV: parity mode, true fp32 (no TF32) */
#define DEC_BF16_F16KV 1 /* bf16 weights and GEMM inputs, fp32 accumulation and residual, f16 KV */
/* int4 projections and bf16 embedding, bf16 GEMM inputs, fp32 accumulation and
 * residual, f16 KV (tinyllm L10.1 section 2.5 "Int4 weights"): dec_create
 * quantizes the seven projections of every layer at load, per group of 32
 * input columns: s = f16(max|W| / 7) (f32 division, one rounding to f16),
 * q = clamp(rint(W / s), -8, 7) (ties to even), effective weight q * s; two
 * codes a byte, even column in the low nibble.  Each quantized matrix is its
 * codes (rows x K/2 bytes) followed by its scales (rows x K/32 f16).  Every
 * input width must be a multiple of 32 and at most 4096.  Products run on CUDA cores with the
 * codes dequantized in registers; the one-kernel decode step and the tensor-
 * core products are bf16-only. */
#define DEC_INT4_F16KV 2

/* which rows of a prefill get logits */
#define DEC_ROWS_ALL  0 /* every new token (octlm "Proving it's the same model": every position) */
#define DEC_ROWS_LAST 1 /* last new token of each sequence (tinyllm L10.1 section 2.4) */

/* Decoder shape and switches (octlm "A real model in our own decoder",
 * qwen_config).  Everything the decoder cannot run is refused with
 * DEC_EINVAL, never served wrong (tinyllm L10.1 section 2.3). */
typedef struct dec_config {
    int32_t vocab, d_model, n_layers, n_heads, n_kv_heads, head_dim, ff_hidden;
    int32_t max_positions; /* positions 0 .. max_positions-1 are valid; at most 40,960 */
    int32_t block_tokens;  /* KV block size B; 16 */
    int32_t mode;          /* DEC_FP32, DEC_BF16_F16KV or DEC_INT4_F16KV */
    double rope_base;      /* 1e6 for Qwen3 */
    double rms_eps;        /* 1e-6; inside the square root */
    int32_t qk_norm;       /* must be 1 */
    int32_t rope_split;    /* must be 1: channel j pairs with j + head_dim/2 */
    int32_t tied;          /* must be 1: the LM head is the embedding */
    int32_t rope_scaling;  /* must be 0 */
    int32_t sliding_window;/* must be 0 */
    int32_t attention_bias;/* must be 0 */
} dec_config;

/* Raw fp32 weights, DEVICE pointers, row-major [out, in] (y = x W^T).
 * Per-layer fields are HOST arrays of n_layers device pointers.  Read only
 * during dec_create; the caller may free them afterwards. */
typedef struct dec_weights {
    const float* embed;       /* [vocab, d_model] */
    const float* final_norm;  /* [d_model] */
    const float* const* attn_norm; /* [d_model] */
    const float* const* wq;   /* [n_heads*head_dim, d_model] */
    const float* const* wk;   /* [n_kv_heads*head_dim, d_model] */
    const float* const* wv;   /* [n_kv_heads*head_dim, d_model] */
    const float* const* q_norm; /* [head_dim], shared by all query heads */
    const float* const* k_norm; /* [head_dim], shared by all key heads */
    const float* const* wo;   /* [d_model, n_heads*head_dim] */
    const float* const* mlp_norm; /* [d_model] */
    const float* const* w_gate; /* [ff_hidden, d_model] */
    const float* const* w_up;   /* [ff_hidden, d_model] */
    const float* const* w_down; /* [d_model, ff_hidden] */
} dec_weights;

typedef struct dec_model dec_model; /* opaque */
typedef struct dec_pool dec_pool;   /* opaque */

/* One step: S sequences, each a run of new tokens at absolute positions
 * (tinyllm L10.1 section 2.4, ForwardSeq / ForwardBatch in section 4).
 * All arrays are HOST memory, read during the call only. */
typedef struct dec_batch {
    int32_t n_seqs;             /* S >= 1 */
    int32_t n_tokens;           /* N = total new tokens >= 1 */
    const int32_t* ids;         /* [N] token ids, sequences back to back; may be NULL if ids_device is set */
    const int32_t* ids_device;  /* optional DEVICE [N] ids (e.g. the previous step's argmax); checked on the
                                   device: an id outside the vocabulary sets DEC_DEV_BAD_ID and reads row 0 */
    const int32_t* positions;   /* [N] absolute positions; within a sequence they must be p_s, p_s+1, ... */
    const int32_t* seq_start;   /* [S+1] offsets of each sequence's tokens; seq_start[0]=0, seq_start[S]=N */
    const int32_t* block_table; /* [S * max_blocks] pool block ids; position j of sequence s lives in block
                                   block_table[s*max_blocks + j/B], slot j % B */
    int32_t max_blocks;         /* row stride of block_table */
} dec_batch;

/* ---- errors --------------------------------------------------------------- */
const char* dec_last_error(void);

/* Device error word bits (dec_device_status). */
#define DEC_DEV_BAD_ID   1u /* a device-side token id was outside the vocabulary */
#define DEC_DEV_TIMEOUT  2u /* a bounded wait in a kernel gave up */
#define DEC_DEV_CAPACITY 4u /* a kernel's fixed-size work list overflowed */
#define DEC_DEV_BOUNDS   8u /* DEC_DEBUG builds only: a kernel met a block-table column or pool
                               block id outside its range; it used block 0 instead */

/* ---- model ---------------------------------------------------------------- */
/* Check a config; DEC_OK if the decoder can run it. */
int dec_config_check(const dec_config* cfg);

/* Bytes of the packed-weight buffer dec_create needs for cfg (device). */
int dec_weights_bytes(const dec_config* cfg, size_t* bytes);

/* Bytes of the per-model workspace for steps of up to max_tokens new tokens,
 * max_seqs sequences and max_rows logits rows (device). */
int dec_workspace_bytes(const dec_config* cfg, int32_t max_tokens, int32_t max_seqs, size_t* bytes);

/* Build a model: validates cfg, packs the raw fp32 weights into packed_buf
 * (fused [Wq;Wk;Wv] and gate/up layouts; bf16 round-to-nearest-even in
 * DEC_BF16_F16KV mode) and fills the RoPE cos/sin table, computed on the host
 * in double precision and rounded once to fp32.  packed_buf (>= dec_weights_bytes)
 * and workspace (>= dec_workspace_bytes for max_tokens/max_seqs) are caller-owned
 * device buffers that must outlive the model, 256-byte aligned.  Synchronises
 * `stream` before returning. */
int dec_create(const dec_config* cfg, const dec_weights* w, void* packed_buf, size_t packed_bytes,
               void* workspace, size_t workspace_bytes, int32_t max_tokens, int32_t max_seqs,
               void* stream, dec_model** out);
void dec_destroy(dec_model* m);

/* Read and clear the device error word (synchronises the model's last stream). */
int dec_device_status(dec_model* m, uint32_t* flags);

/* Debug: when dump is non-NULL, every later dec_prefill/dec_decode copies the
 * fp32 residual stream x [N, d_model] after the embedding and after every layer
 * into dump[(i * N + t) * d_model + c], i = 0 .. n_layers (needs
 * (n_layers+1)*N*d_model floats; the caller sizes it for its largest step).
 * Layer-by-layer comparison against the oracle (1bit-MONSTER "Byte-identical",
 * "The validation loop closes"). NULL turns it off. */
int dec_set_dump(dec_model* m, float* dump, size_t dump_floats);

/* ---- paged KV pool (tinyllm L10.1 section 2.2, KvPool in section 4) -------- */
/* Layout: pool block b of layer l holds a K slab and a V slab, each
 * [n_kv_heads][block_tokens][head_dim] elements (f32 in DEC_FP32, f16 in
 * DEC_BF16_F16KV).  Slab (l, b, is_v) starts at element
 * ((l * n_blocks + b) * 2 + is_v) * n_kv_heads * block_tokens * head_dim of
 * the caller's slab buffer; K of KV head h, slot s starts at element
 * (h * block_tokens + s) * head_dim of its slab (section 3, "Where a key lands"). */
int dec_pool_bytes(const dec_config* cfg, int32_t n_blocks, size_t* bytes);
/* n_blocks == 0 is refused (DEC_EINVAL, kv_pool_rejects_zero_capacity).  The
 * slab memory is caller-owned device memory of >= dec_pool_bytes. */
int dec_pool_create(const dec_config* cfg, int32_t n_blocks, void* slabs, size_t bytes, dec_pool** out);
void dec_pool_destroy(dec_pool* p);
/* All-or-nothing: n blocks with refcount 1 and fill 0 into ids[0..n), or
 * DEC_ECAPACITY and nothing taken.  Free blocks go first; when they run short,
 * cached prefix blocks are evicted (their keys dropped), oldest release first
 * (kv_pool_evicts_the_oldest_cached_block). */
int dec_pool_alloc(dec_pool* p, int32_t n, int32_t* ids);
int dec_pool_retain(dec_pool* p, int32_t id);  /* refcount + 1; DEC_EBLOCK if not allocated */
/* refcount - 1; at 0 a registered block is cached (its K/V and key kept, in
 * release order) and any other block is free again.  DEC_EBLOCK if not allocated. */
int dec_pool_release(dec_pool* p, int32_t id);
int dec_pool_free_blocks(const dec_pool* p, int32_t* n);   /* free, not counting cached blocks */
int dec_pool_refcount(const dec_pool* p, int32_t id, int32_t* refs);

/* ---- prefix cache in the pool (KvPool's hash index and LRU, tinyllm L10.1
 * sections 1 and 4; its boundary tests kv_pool_bounds_and_cache_lifecycle) ---
 * The pages name no hash: a block's key is the caller's.  dec_prefix_key gives
 * a chained one: key_i = dec_prefix_key(key_{i-1}, tokens of block i,
 * block_tokens), key_{-1} = 0, so equal keys mean equal whole prefixes (up to
 * 64-bit collisions).  Definition: FNV-1a 64 (offset basis
 * 0xcbf29ce484222325, prime 0x100000001b3) over the 8 bytes of prev, then the
 * 4 bytes of every token, both little-endian. */
uint64_t dec_prefix_key(uint64_t prev, const int32_t* tokens, int32_t n);
/* Slots of an allocated block that hold K/V (0 .. block_tokens); a new block
 * starts at 0.  DEC_EBLOCK if not allocated, DEC_EINVAL if n is out of range. */
int dec_pool_set_fill(dec_pool* p, int32_t id, int32_t n);
/* Index a full allocated block under key: *registered = 1 if the key now
 * names this block (0: the key already names another block, which keeps it).
 * A block carries one key (a new key replaces its old one).  DEC_EINVAL if
 * the block is not full, DEC_EBLOCK if not allocated. */
int dec_pool_register(dec_pool* p, int32_t id, uint64_t key, int32_t* registered);
/* The block indexed under key, reacquired (refcount + 1; a cached block
 * leaves the cache), or *id = -1 if none.  DEC_OK either way. */
int dec_pool_lookup(dec_pool* p, uint64_t key, int32_t* id);
int dec_pool_cached_blocks(const dec_pool* p, int32_t* n);
/* Element offset (within the slab buffer) of K (is_v=0) or V of KV head h at
 * position pos of a sequence with the given block table; the same function the
 * kernels use.  DEC_ERANGE if the table is too short, DEC_EBLOCK on a bad id. */
int dec_kv_offset(const dec_pool* p, const int32_t* table, int32_t n_table, int32_t pos, int32_t layer,
                  int32_t kv_head, int32_t is_v, int64_t* offset);

/* ---- the step ------------------------------------------------------------- */
/* The checks dec_prefill / dec_decode make before launching anything, on
 * host data only (no GPU needed): sequence layout, consecutive positions
 * below max_positions, ids in the vocabulary (host ids), block tables long
 * enough and naming allocated blocks, and every block the step writes (those
 * holding positions p_s .. the last new position of each sequence) owned by
 * that sequence alone: refcount 1, not registered in the prefix cache, and
 * written for no other position of the batch (tinyllm L10.1 section 4,
 * forward_refuses_bad_batches).  decode != 0 also requires one token per
 * sequence.  DEC_OK, or the code and dec_last_error text the step would
 * return (DEC_EINVAL, DEC_ERANGE, DEC_EVOCAB, DEC_EBLOCK). */
int dec_batch_check(const dec_pool* pool, const dec_batch* b, int32_t decode);

/* Prefill (or any mixed step): run the batch's new tokens, write their K/V into
 * the blocks their tables name, and produce fp32 logits [R, vocab] and greedy ids
 * [R] (int32, device), R = N for DEC_ROWS_ALL or S for DEC_ROWS_LAST; rows are in
 * token / sequence order.  logits may be NULL (ids only).  Every block a sequence
 * reads (positions 0 .. its last new position) must be allocated in `pool`. */
int dec_prefill(dec_model* m, dec_pool* pool, const dec_batch* b, int32_t rows, float* logits,
                int32_t* argmax, void* stream);

/* Decode: exactly one new token per sequence (N == S).  Logits [S, vocab] and
 * ids [S] as for dec_prefill with DEC_ROWS_LAST.  Uses the split-K attention.
 * In the serving mode, a step of at most 8 sequences runs as one persistent
 * kernel (see dec_set_megakernel) when the shape and the device allow it. */
int dec_decode(dec_model* m, dec_pool* pool, const dec_batch* b, float* logits, int32_t* argmax,
               void* stream);

/* ---- profiling ------------------------------------------------------------
 * Kernel classes of one step, in launch order. */
#define DEC_K_EMBED       0 /* embedding gather */
#define DEC_K_QKV         1 /* RMSNorm + [Wq;Wk;Wv] product */
#define DEC_K_QKV_POST    2 /* QK-norm + RoPE + KV-cache write (parity mode; serving prefill steps of
                               17-32 tokens; serving decode steps fuse it into DEC_K_ATTN) */
#define DEC_K_ATTN        3 /* attention: split-K decode (serving: with QK-norm, RoPE and the
                               cache append of the step's token fused in) or tiled prefill */
#define DEC_K_ATTN_MERGE  4 /* reserved (the split-K merge is fused into DEC_K_ATTN) */
#define DEC_K_OPROJ       5 /* O projection + residual */
#define DEC_K_GATEUP      6 /* RMSNorm + gate/up + SiLU*mul */
#define DEC_K_DOWN        7 /* down projection + residual */
#define DEC_K_LMHEAD      8 /* final RMSNorm + LM head + argmax keys */
#define DEC_K_ARGMAX      9 /* argmax keys -> ids */
#define DEC_K_STEP       10 /* a whole decode step in one persistent kernel */
#define DEC_K_COUNT      11
/* Record CUDA events around every later launch of one kernel class (on the
 * step's stream) while on != 0. */
int dec_profile_enable(dec_model* m, int32_t kernel_class, int32_t on);
/* Synchronise, then return the summed event time and launch count of a class
 * since the last read, and reset them. */
int dec_profile_read(dec_model* m, int32_t kernel_class, double* total_ms, int64_t* launches);
/* Serving mode: the weight products run on the tcgen05 tensor cores (on by
 * default); off routes them to the CUDA-core kernels. */
int dec_set_tensor_cores(dec_model* m, int32_t on);
/* Decode steps replay CUDA graphs (on by default): the first step of a given
 * (batch size, logits, argmax, pool and its size; in the parity mode also the
 * decode attention grid, which grows every 256 positions) runs eagerly, the second is captured on
 * a private stream, later ones replay it on the caller's stream.  Off: every
 * step launches its kernels one by one.  Graphs are bypassed while a dump is
 * active.  Profiled kernel classes (dec_profile_enable) stay timed inside
 * graphs: their events become event-record nodes that each replay points at
 * fresh events; a step captured with one set of profiled classes replays only
 * while the same set is enabled. */
int dec_set_graphs(dec_model* m, int32_t on);
/* Serving-mode decode steps of at most 8 sequences run as one persistent
 * cooperative kernel, one CTA per SM (on by default): a loader warp streams
 * the CTA's weight rows and cached keys into a shared-memory ring while the
 * compute warps run the stages; between dependent stages each CTA counts its
 * outputs in on a step-wide counter and waits for every CTA's (attention
 * records: per sequence and KV head).  Off: the per-operation kernels above,
 * one launch each.  The per-layer dump and CUDA graphs do not apply to the
 * one-kernel step.  Same tolerances as the other paths. */
int dec_set_megakernel(dec_model* m, int32_t on);
/* Profiling aid for the one-kernel step: while `stamps` is set (DEVICE
 * memory, uint64 [n], n >= number of SMs x 320), every such step writes, per
 * CTA b, the global timer (ns) at stamps[b*320 + k]: k = 0 at the start; for
 * stage s (5 per layer: QKV, attention, O projection, gate/up, down; then the
 * LM head at s = 5 * n_layers) k = 1 + 2s once the stage's inputs are in
 * shared memory and k = 2 + 2s once its outputs are counted in; k = 284..308
 * points inside layer 1's stages (5 per stage); k = 310..315 when the loader
 * issued the first tile of layer 1's stages and of layer 2's QKV; k = 319
 * when the loader issued its last tile.  NULL turns it off.  DEC_EINVAL if n
 * is too small. */
int dec_set_step_trace(dec_model* m, uint64_t* stamps, size_t n);
/* Test hook for the bounded waits of the one-kernel step (no counterpart on
 * the pages): with extra > 0, every later one-kernel step's CTA hand-off
 * waits for `extra` more arrivals than will ever come and gives up after
 * limit_ns (1 us .. 1 s): the step then ends early with DEC_DEV_TIMEOUT in
 * the device error word (dec_device_status) and its logits and ids are not
 * valid; the GPU stays usable.  extra = 0 restores the normal waits (limit
 * 1 s).  DEC_EINVAL for a limit outside the range. */
int dec_debug_wait_timeout(dec_model* m, uint32_t extra, uint64_t limit_ns);
/* *available = 1 when this model's shape and device can run the one-kernel
 * decode step (serving mode, two query heads per KV head, head_dim 32, 64 or
 * 128, d_model <= 1024, cooperative launch), else 0. */
int dec_megakernel_available(const dec_model* m, int32_t* available);
/* Kernels this model launched since the last call (then reset); a replayed
 * graph counts every kernel it contains. */
int dec_launch_count(dec_model* m, int64_t* launches);

/* ---- decode attention on its own ---------------------------------------------
 * The split-K kernel dec_decode runs, callable alone: for each of n_seqs
 * sequences, the query of its newest token (position ctx[s]-1) attends over
 * keys 0 .. ctx[s]-1 of `layer` in the pool,
 *   o = sum_j softmax_j(q . k_j / sqrt(D)) v_j,  query head h reading KV head
 *   floor(h * Hkv / H)   (tinyllm L10.1 section 2.4).
 *   q            DEVICE fp32 [n_seqs, n_heads, head_dim], after QK-norm and RoPE
 *   ctx          HOST [n_seqs] context lengths, 1 .. max_positions
 *   block_table  HOST [n_seqs * max_blocks] (as in dec_batch); every block a
 *                sequence reads must be allocated in the pool (DEC_EBLOCK)
 *   out          DEVICE [n_seqs, n_heads * head_dim], fp32 (DEC_FP32) or bf16
 *   scratch      DEVICE, 256-byte aligned, >= dec_attend_scratch_bytes(...);
 *                holds the call's metadata, split-K records and merge
 *                counters; needs no initialisation and is overwritten.  Its
 *                first 32-bit word is the call's device error word
 *                (DEC_DEV_TIMEOUT if a bounded wait gave up).
 * Asynchronous on `stream`; the host arrays may be reused on return. */
int dec_attend_scratch_bytes(const dec_config* cfg, int32_t n_seqs, int32_t max_ctx, int32_t max_blocks,
                             size_t* bytes);
int dec_attend(const dec_pool* pool, int32_t layer, int32_t n_seqs, const float* q, const int32_t* ctx,
               const int32_t* block_table, int32_t max_blocks, void* out, void* scratch, size_t scratch_bytes,
               void* stream);

/* dec_attend without caller scratch (no counterpart on the pages: a service
 * of this library).  For callers that cannot allocate device memory at the
 * moment they need attention - code inside a host framework that owns every
 * device allocation, plug-ins with a memory budget fixed at load time, or
 * latency-critical loops that must not pay for the allocator, whose calls can
 * synchronise the device.  Same arguments and results as dec_attend minus the
 * scratch, which lives in a 4 MiB array inside the library that every GPU
 * loading the library holds until the process exits.  The call allocates
 * nothing.  Limits: at most 256 sequences, and the dec_attend_scratch_bytes
 * of the request must not exceed 4 MiB (e.g. 8 sequences of 2,048 keys at the
 * Qwen3-0.6B shape); larger requests return DEC_ERANGE with a message.
 * The array's device address on a device is looked up once: by dec_create
 * on that device, else by the first call there.  That first lookup loads the
 * library's module holding the array (with CUDA's lazy module loading, this
 * is when the array is allocated, and it may synchronise), so a caller that
 * never creates a model should make one call, or dec_attend_noalloc_status,
 * before any stream capture and before the loop that must not allocate.  The
 * looked-up address does not survive cudaDeviceReset.  Every call on a device
 * shares the one array and each call overwrites it (its counters and error
 * word are cleared at the start of every call), so calls that may overlap on
 * the GPU - on different streams, or from different threads - race: order
 * them on one stream.  The kernel's error word (DEC_DEV_TIMEOUT if a bounded
 * wait gave up) is read with dec_attend_noalloc_status after the call and
 * before the next one. */
int dec_attend_noalloc(const dec_pool* pool, int32_t layer, int32_t n_seqs, const float* q, const int32_t* ctx,
                       const int32_t* block_table, int32_t max_blocks, void* out, void* stream);
/* Synchronise `stream`, then read and clear the device error word that the
 * last dec_attend_noalloc call on the current device left in the library's
 * array (0: no bounded wait gave up).  Allocates nothing. */
int dec_attend_noalloc_status(void* stream, uint32_t* flags);

/* Quantize one f32 matrix to int4 as DEC_INT4_F16KV does at load (tinyllm L10.1
 * section 2.5): W device [rows, K] f32, K a multiple of 32; codes device
 * [rows, K/2] bytes (16-byte aligned), scales device [rows, K/32] f16 bits.
 * Asynchronous on `stream`. */
int dec_quantize_int4(const float* W, int32_t rows, int32_t K, void* codes, void* scales, void* stream);

/* Test hook: the device conversion the f16 KV store uses (f32 -> f16 round to
 * nearest even, tinyllm L10.1 section 2.3), applied to n device floats. */
int dec_f32_to_f16(const float* in, uint16_t* out, int64_t n, void* stream);

/* Test hook: one raw weight product Y[t, r] = sum_k X[t, k] W[r, k] with a
 * packed matrix of the model: which = 0 [Wq;Wk;Wv], 1 Wo, 2 gate/up (rows
 * interleaved in groups of 8), 3 Wd, 4 the embedding; layer ignored for 4.
 * X: device [T, K], fp32 in DEC_FP32, bf16 in DEC_BF16_F16KV; Y: device fp32
 * [T, rows].  path 0 runs the CUDA-core kernels, path 1 the tcgen05 kernel
 * for many tokens (serving mode, T > 32), path 2 the tcgen05 kernel for
 * decode steps (serving mode, T <= 32); otherwise DEC_EINVAL. */
int dec_debug_product(dec_model* m, int32_t which, int32_t layer, const void* X, int32_t T, float* Y, int32_t path,
                      void* stream);

/* ---- the sampler (tinyllm L10.1 section 2.6 "The sampler and PCG32") ------
 *
 * One sampling step per sequence after the LM head, on the device, in f64:
 * widen the logits; repetition penalty r over the distinct ids of prompt and
 * output (l /= r if l > 0, else l *= r); presence a_p and frequency a_f over
 * the output only (l -= a_f * count + a_p for ids the output holds); the
 * returned logprob is the log-softmax at that point; temperature 0 returns
 * the argmax (ties to the lowest id) and draws nothing; otherwise l /= T,
 * keep the top_k ids in (l desc, id asc) order, keep the nucleus up to and
 * including the id whose running probability reaches top_p, keep ids whose
 * probability is at least min_p times the largest, renormalise over the kept
 * ids, draw one uniform u and return the first id, in ascending id order,
 * whose cumulative probability exceeds u.  Off values: top_k = 0 (or >=
 * vocab), top_p = 1, min_p = 0, repetition_penalty = 1, presence and
 * frequency 0.  Sums run in fixed trees (the result is the same bits alone or
 * in a batch); they round differently from plain left-to-right loops, so a
 * token can differ from the loop form only where u or a filter threshold lies
 * within rounding (about 1e-12) of a cumulative sum. */

#define DEC_PURPOSE_SAMPLE 4 /* the stream purpose of sampling (child_seed(seed, 4)) */

typedef struct dec_sampling {
    double temperature;        /* >= 0; 0 = greedy */
    int32_t top_k;             /* >= 0; 0 or >= vocab = off */
    double top_p;              /* in [0, 1]; 1 = off */
    double min_p;              /* in [0, 1]; 0 = off */
    double repetition_penalty; /* > 0; 1 = off */
    double presence_penalty;   /* finite */
    double frequency_penalty;  /* finite */
} dec_sampling;

/* PCG32 state (M. E. O'Neill's XSH RR 64/32): a 64-bit LCG state and its odd
 * increment.  One uniform takes two 32-bit outputs a, b:
 * u = ((a >> 5) * 2^26 + (b >> 6)) * 2^-53. */
typedef struct dec_rng {
    uint64_t state, inc;
} dec_rng;

/* child_seed(seed, purpose) = mix64(seed + purpose * 0x9E3779B97F4A7C15),
 * mix64 being SplitMix64's finaliser (read so from the pages' worked example:
 * child_seed(0, 4) = 0xF88BB8A8724C81EC). */
uint64_t dec_child_seed(uint64_t seed, uint64_t purpose);
/* The stream of one request and purpose: PCG32 seeded (pcg32_srandom_r) with
 * child_seed(seed, purpose) on sequence `purpose`.  Host only. */
void dec_rng_stream(uint64_t seed, uint64_t purpose, dec_rng* out);
uint32_t dec_rng_next_u32(dec_rng* r); /* host: one 32-bit output */
double dec_rng_uniform(dec_rng* r);    /* host: one uniform in [0, 1), on the 2^-53 grid */

typedef struct dec_sampler dec_sampler;

/* Device workspace of a sampler for `vocab` ids and up to `max_seqs`
 * sequences a call (about 22 bytes per id per sequence).  vocab in
 * [1, 2^20]; DEC_EINVAL otherwise. */
int dec_sampler_workspace_bytes(int32_t vocab, int32_t max_seqs, size_t* bytes);
/* workspace: caller-owned device memory, 256-byte aligned, at least
 * dec_sampler_workspace_bytes; it is cleared here (synchronously) and must
 * not be touched while the sampler lives.  The sampler owns only host
 * bookkeeping (a small pinned staging ring). */
int dec_sampler_create(int32_t vocab, int32_t max_seqs, void* workspace, size_t bytes, dec_sampler** out);
void dec_sampler_destroy(dec_sampler* s);

/* Device error word bits of the sampler (dec_sampler_status). */
#define DEC_SAMPLE_BAD_ID    1u /* a history id outside [0, vocab): ignored */
#define DEC_SAMPLE_BAD_LOGIT 2u /* a NaN or +inf logit: read as -inf */
#define DEC_SAMPLE_NO_FINITE 4u /* every logit of a sequence is -inf: token -1 */
#define DEC_SAMPLE_OVERFLOW  8u /* internal: a candidate list outgrew shared memory */
/* Read (synchronously) the OR of the error bits every call so far raised. */
int dec_sampler_status(dec_sampler* s, uint32_t* flags);

/* Sample one token for each of n_seqs sequences.
 *   logits           device f32 [n_seqs, ld], ld >= vocab (the LM head's output)
 *   params           host [n_seqs], checked on the host (DEC_EINVAL)
 *   history          device int32: each sequence's prompt ids then its output
 *                    ids, sequence after sequence; NULL if all are empty
 *   history_offsets  host int32 [n_seqs + 1]: sequence i owns
 *                    history[offsets[i] .. offsets[i+1]); NULL = no history
 *   n_prompt         host int32 [n_seqs]: how many of those are prompt ids;
 *                    NULL = none
 *   rng              device dec_rng [n_seqs]: read, and advanced by exactly
 *                    one uniform for each sequence with temperature > 0
 *   tokens           device int32 [n_seqs]   logprobs  device f64 [n_seqs]
 * Asynchronous on `stream`; calls on one sampler must not overlap. */
int dec_sample(dec_sampler* s, const float* logits, int64_t ld, int32_t n_seqs, const dec_sampling* params,
               const int32_t* history, const int32_t* history_offsets, const int32_t* n_prompt, dec_rng* rng,
               int32_t* tokens, double* logprobs, void* stream);

/* Test hook: the sampler's double-f32 exponential (float head + tail; Tang's
 * table-driven method, accurate to about 2^-46 relative down to e^-60, 0 below
 * e^-87) on n device doubles x <= 0, written as doubles (head + tail). */
int dec_debug_df_exp(const double* x, double* y, int64_t n, void* stream);

/* Library version string. */
const char* dec_version(void);

/* ---- debug build ------------------------------------------------------------
 * Building with DEC_DEBUG defined (python -m decoder_qwen3_step_gb300.build
 * --debug writes libdec_debug.so beside libdec.so) adds device-side bounds
 * checks to every kernel that reads a block table: a column past the row or a
 * pool block id outside the pool sets DEC_DEV_BOUNDS in the model's device
 * error word (dec_device_status) and the access goes to block 0 instead, so
 * nothing outside the pool is read or written.  No check traps.  The release
 * build compiles the checks out; the host validates every step's batch
 * (dec_batch_check) in both builds. */
#define DEC_BUILD_DEBUG 1u
/* Bit mask of the build's options (DEC_BUILD_DEBUG). */
uint32_t dec_build_flags(void);

/* Debug builds only (DEC_EINVAL otherwise): the next step's device copy of
 * the block table gets `value` in column `col` of sequence `seq`'s row, after
 * the host has validated and used the real table; one step only.  Lets a test
 * reach the device bounds checks with an id the host would refuse. */
int dec_debug_poison_table(dec_model* m, int32_t seq, int32_t col, int32_t value);

#ifdef __cplusplus
}
#endif
#endif /* DEC_H */
