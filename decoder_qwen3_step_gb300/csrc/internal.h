// internal.h - host-side definitions shared by the C-ABI translation units.
#pragma once

#include <stdint.h>

#include <list>
#include <unordered_map>
#include <vector>

#include "../../include/dec.h"

// The paged KV pool: caller-owned slabs plus host bookkeeping: refcounts, a
// free-list stack whose top is the next id handed out, and the prefix cache
// (filled slots per block, the key each registered full block is indexed
// under, and the released registered blocks in release order, oldest first).
struct dec_pool {
  dec_config cfg;
  int n_blocks;
  void* slabs;
  std::vector<int32_t> refs;
  std::vector<int32_t> free_list;
  std::vector<int32_t> fill;
  std::vector<uint8_t> registered;
  std::vector<uint64_t> key;
  std::unordered_map<uint64_t, int32_t> index;
  std::list<int32_t> lru;
  std::vector<std::list<int32_t>::iterator> lru_pos;
};

namespace dec {
// Record `msg` as the thread's last error and return `code`.
int set_error(int code, const char* msg);
// Look up the device address of dec_attend_noalloc's array on the current
// device (attend.cu); DEC_OK or an error code.
int noalloc_prepare();
}  // namespace dec
