// prefix.cu - the prefix cache of the paged KV pool (host bookkeeping only).
//
// tinyllm L10.1 "Candle model runner ...", section 1 ("KvPool owns fixed-size
// f16 K and V slabs, block references, the prefix hash index, and LRU
// eviction") and the pool's boundary tests: capacity is all-or-nothing,
// references balance, full blocks register, release caches, lookup
// reacquires, and an exhausted allocation evicts the oldest cached block.
// The pages name no hash: a block's key is the caller's, and dec_prefix_key
// gives one chained over the block contents (see include/dec.h).
#include <cstdio>

#include "../../include/dec.h"
#include "internal.h"

namespace {

int fail_msg(int code, const char* fmt, int v) {
  char buf[160];
  snprintf(buf, sizeof buf, fmt, v);
  return dec::set_error(code, buf);
}

bool allocated(const dec_pool* p, int32_t id) { return id >= 0 && id < p->n_blocks && p->refs[id] > 0; }

}  // namespace

extern "C" {

int dec_pool_set_fill(dec_pool* p, int32_t id, int32_t n) {
  if (!p) return dec::set_error(DEC_EINVAL, "pool is NULL");
  if (!allocated(p, id)) return fail_msg(DEC_EBLOCK, "block %d is not allocated", id);
  if (n < 0 || n > p->cfg.block_tokens) return fail_msg(DEC_EINVAL, "fill %d outside 0 .. block_tokens", n);
  p->fill[id] = n;
  return DEC_OK;
}

int dec_pool_register(dec_pool* p, int32_t id, uint64_t key, int32_t* registered) {
  if (!p || !registered) return dec::set_error(DEC_EINVAL, "NULL argument");
  if (!allocated(p, id)) return fail_msg(DEC_EBLOCK, "block %d is not allocated", id);
  if (p->fill[id] != p->cfg.block_tokens) return fail_msg(DEC_EINVAL, "block %d is not full", id);
  *registered = 0;
  auto it = p->index.find(key);
  if (it != p->index.end()) {
    *registered = it->second == id;  // the key keeps its first block
    return DEC_OK;
  }
  if (p->registered[id]) p->index.erase(p->key[id]);  // a block is indexed under one key
  p->index.emplace(key, id);
  p->key[id] = key;
  p->registered[id] = 1;
  *registered = 1;
  return DEC_OK;
}

int dec_pool_lookup(dec_pool* p, uint64_t key, int32_t* id) {
  if (!p || !id) return dec::set_error(DEC_EINVAL, "NULL argument");
  *id = -1;
  auto it = p->index.find(key);
  if (it == p->index.end()) return DEC_OK;
  const int32_t b = it->second;
  if (p->refs[b] == 0) {  // cached: out of the eviction order, back in use
    p->lru.erase(p->lru_pos[b]);
    p->lru_pos[b] = p->lru.end();
  }
  ++p->refs[b];
  *id = b;
  return DEC_OK;
}

int dec_pool_cached_blocks(const dec_pool* p, int32_t* n) {
  if (!p || !n) return dec::set_error(DEC_EINVAL, "NULL argument");
  *n = (int32_t)p->lru.size();
  return DEC_OK;
}

uint64_t dec_prefix_key(uint64_t prev, const int32_t* tokens, int32_t n) {
  // FNV-1a, 64-bit: the 8 bytes of prev, then the 4 bytes of every token, little-endian
  uint64_t h = 0xcbf29ce484222325ull;
  auto mix = [&h](uint32_t byte) {
    h ^= byte;
    h *= 0x100000001b3ull;
  };
  for (int i = 0; i < 8; ++i) mix((uint32_t)(prev >> (8 * i)) & 0xFFu);
  for (int t = 0; t < n; ++t)
    for (int i = 0; i < 4; ++i) mix(((uint32_t)tokens[t] >> (8 * i)) & 0xFFu);
  return h;
}

}  // extern "C"
