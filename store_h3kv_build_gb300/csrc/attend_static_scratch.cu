// attend_static_scratch.cu -- h3kv_attend_staged_static: the staged kvi8r
// attention (h3kv_attend_staged) with its scratch -- the HBM staging block and
// the per-row combine state -- in a fixed device array that this library
// owns, for callers that may not allocate device memory themselves.
#include <cuda_runtime.h>
#include <mutex>

#include "../../include/h3kv.h"

namespace {

// Scratch of h3kv_attend_staged_static: the staging block first, then the
// per-row state (256-byte aligned).  Every GPU that loads the library holds
// this array until the process exits.  In host code the name is only a
// host-side stand-in; kernels get the device address from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_staged_scratch[H3KV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of the array on the current device, looked up once per
// device with that device current.
h3kv_status scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return H3KV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_staged_scratch) != cudaSuccess || !p) return H3KV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return H3KV_OK;
}

}  // namespace

extern "C" h3kv_status h3kv_attend_staged_static(const uint16_t *Q, int64_t q_seq, const h3kv_store *store,
                                                 int32_t q_chunk, int32_t kv_block, float softmax_scale, float *O,
                                                 void *stream) {
  // the argument checks h3kv_attend_staged makes first, in its order, so that
  // a store it does not take gets the same status here at every size
  if (!store || q_seq < 0 || store->heads < 0 || store->seq < 0) return H3KV_ERR_INVALID_ARG;
  if (store->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  if (q_chunk < 1 || kv_block < 0 || kv_block % H3KV_KV_TILE != 0) return H3KV_ERR_INVALID_ARG;
  if (store->scale_group == 32) return H3KV_ERR_UNSUPPORTED;
  if (store->scale_group != 0 && store->scale_group != 128) return H3KV_ERR_INVALID_ARG;
  if (store->heads == 0 || q_seq == 0) return H3KV_OK;
  // then the fixed scratch: the staging block (rounded up to 256 bytes), then
  // 8 bytes of row state per (head, query row).  q_seq is bounded before any
  // product that could wrap; nothing is touched on the device for a call
  // that does not fit.
  const size_t staging = h3kv_staging_bytes(store->heads, kv_block);
  const size_t staging_aligned = (staging + 255) & ~static_cast<size_t>(255);
  if (staging == 0 || staging_aligned > H3KV_STATIC_SCRATCH_BYTES) return H3KV_ERR_INVALID_ARG;
  const size_t row_state_bytes = 2 * sizeof(float) * static_cast<size_t>(store->heads);
  if (static_cast<uint64_t>(q_seq) > (H3KV_STATIC_SCRATCH_BYTES - staging_aligned) / row_state_bytes)
    return H3KV_ERR_INVALID_ARG;
  void *base = nullptr;
  const h3kv_status st = scratch_address(&base);
  if (st != H3KV_OK) return st;
  // Neither part needs clearing: each call writes a staging block before its
  // launches read it, and the first block's launches write the state before
  // any later launch reads it.
  float *state_ptr = reinterpret_cast<float *>(static_cast<unsigned char *>(base) + staging_aligned);
  return h3kv_attend_staged(Q, q_seq, store, q_chunk, kv_block, softmax_scale, O, base, staging_aligned, state_ptr,
                            stream);
}
