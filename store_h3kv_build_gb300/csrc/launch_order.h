// launch_order.h -- the order in which an attention call over a device-resident
// store launches its query chunks (and heads).
#pragma once

#include <stdint.h>

#include "../../include/h3kv.h"
#include "kernels.h"

namespace h3kv {

// The launches of one attention call over a device-resident store.  For long
// key sequences (at least kHeadMajorKeys keys, a head's kvi8r store 34 MB or
// more) with more than one head and at least kHeadMajorCtas CTAs per head and
// query chunk, every query chunk of head 0 is launched, then every chunk of
// head 1, and so on: the CTAs in flight then read one or two heads' stores,
// and the L2 keeps much of a head's store for its later chunks (half the DRAM
// reads of a 32 x 217088 call in a serialised capture, in the same time).
// Otherwise each query chunk is one launch over all heads: shorter sequences'
// stores gain little from the reuse and their calls lose 1-7 % to the extra
// launches (measured).  Every launch after the first follows the one before it
// with programmatic dependent launch.  A query row's arithmetic is the same in
// every launch, so results do not depend on the order.
inline bool launch_head_major(int64_t q_seq, int64_t kv_seq, int64_t q_chunk, int32_t heads) {
  constexpr int64_t kHeadMajorCtas = 16;
  constexpr int64_t kHeadMajorKeys = 131072;
  const int64_t chunk_rows = q_chunk < q_seq ? q_chunk : q_seq;
  return heads > 1 && kv_seq >= kHeadMajorKeys &&
         (chunk_rows + kAttnRowsPerCta - 1) / kAttnRowsPerCta >= kHeadMajorCtas;
}

// Number of launches launch_query_chunks makes for one call.
inline int64_t launch_count(int64_t q_seq, int64_t kv_seq, int64_t q_chunk, int32_t heads) {
  if (q_seq <= 0 || q_chunk <= 0 || heads <= 0) return 0;
  const int64_t chunks = (q_seq + q_chunk - 1) / q_chunk;
  return launch_head_major(q_seq, kv_seq, q_chunk, heads) ? chunks * heads : chunks;
}

template <class Args, class Launch>
inline h3kv_status launch_query_chunks(Args a, int64_t q_seq, int64_t kv_seq, int64_t q_chunk, int32_t heads,
                                       Launch launch) {
  const bool head_major = launch_head_major(q_seq, kv_seq, q_chunk, heads);
  a.heads = head_major ? 1 : heads;
  bool first = true;
  for (int32_t hh = 0; hh < (head_major ? heads : 1); ++hh) {
    a.head_base = hh;
    for (int64_t c0 = 0; c0 < q_seq; c0 += q_chunk) {
      a.q_begin = c0;
      a.q_end = c0 + q_chunk < q_seq ? c0 + q_chunk : q_seq;
      if (launch(a, !first) != cudaSuccess) return H3KV_ERR_CUDA;
      first = false;
    }
  }
  return H3KV_OK;
}

}  // namespace h3kv
