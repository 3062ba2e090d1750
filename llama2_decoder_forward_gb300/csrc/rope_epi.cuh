// Per-token part of the Q/K/V projection's RoPE + cache-append epilogue,
// shared by both GEMM kernels.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace llgb {

// Per-token part of the Q/K/V epilogue, computed once per tile token before
// the accumulator is ready: the RoPE position (-1 when outside the table; Q
// then keeps the angles of position 0) and the cache slot of the token for KV
// head 0 (head g adds g * capacity, or g * page_size when paged; -1: no cache
// write). Out-of-range positions and page ids are flagged here.
struct TokInfo {
  long long kv;
  int pos;
  int pad;
};

__device__ __forceinline__ TokInfo rope_token(const RopeAppendArgs& a, int r) {
  TokInfo t{-1, -1, 0};
  const int pos = a.positions ? a.positions[r] : r % a.rows_per_seq;
  if (pos < 0 || pos >= a.max_seq) {
    flag(a.status, LLAMA_FLAG_POS_RANGE);
    return t;
  }
  t.pos = pos;
  const int b = r / a.rows_per_seq;
  if (a.page_size == 0) {
    if (pos >= a.capacity) {
      flag(a.status, LLAMA_FLAG_POS_RANGE);
      return t;
    }
    t.kv = ((long long)a.layer * a.batch_cap + b) * a.n_kv * a.capacity + pos;
  } else {
    const int pi = pos / a.page_size;
    if (pi >= a.max_pages) {
      flag(a.status, LLAMA_FLAG_POS_RANGE);
      return t;
    }
    const int page = a.page_table[(size_t)b * a.max_pages + pi];
    if (page < 0 || page >= a.n_pages) {
      flag(a.status, LLAMA_FLAG_PAGE_RANGE);
      return t;
    }
    t.kv = ((long long)a.layer * a.n_pages + page) * a.n_kv * a.page_size + pos % a.page_size;
  }
  return t;
}

}  // namespace llgb
