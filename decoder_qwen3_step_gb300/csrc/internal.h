// internal.h - host-side definitions shared by the C-ABI translation units.
#pragma once

#include <stdint.h>

#include <vector>

#include "../../include/dec.h"

// The paged KV pool: caller-owned slabs plus host bookkeeping (refcounts and
// a free-list stack whose top is the next id handed out).
struct dec_pool {
  dec_config cfg;
  int n_blocks;
  void* slabs;
  std::vector<int32_t> refs;
  std::vector<int32_t> free_list;
};

namespace dec {
// Record `msg` as the thread's last error and return `code`.
int set_error(int code, const char* msg);
}  // namespace dec
