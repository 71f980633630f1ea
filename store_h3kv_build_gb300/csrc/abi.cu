// abi.cu -- the C ABI of libh3kv (declared in include/h3kv.h): host-side
// argument checks, TMA tensor-map encoding, per-chunk launches and the device
// error word.
#include <cudaTypedefs.h>
#include <math.h>
#include <atomic>
#include <mutex>

#include "../../include/h3kv.h"
#include "kernels.h"
#include "ptx.cuh"
#include "launch_order.h"

namespace {

// Device error word written by the kernels' bounded waits.  Host code must
// not take its address directly (that is a host shadow); the device address is
// fetched per device with cudaGetSymbolAddress.
__device__ uint32_t g_h3kv_error;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s per bounded wait
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int32_t> g_withhold_p_tile1{0};  // diagnostic, see h3kv_debug_withhold_p

// One CTA waits on an mbarrier that nothing ever arrives on: the bounded wait
// runs out, records the timeout in the device error word and the kernel
// returns.  No fault, no trap; the context stays usable.
__global__ void wait_selftest_kernel(uint32_t *err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    h3kv::mbar_init(h3kv::smem_u32(&bar), 1);
    abort_flag = 0;
    h3kv::fence_mbar_init();
  }
  __syncthreads();
  const h3kv::WaitCtx w{err, &abort_flag, timeout_ns};
  h3kv::mbar_wait(h3kv::smem_u32(&bar), 0, w);
  __syncthreads();
}

// Checks the reducing TMEM load of the attention kernels (tmem_ld128_max):
// one CTA of 128 threads allocates 128 TMEM columns, each thread stores
// known fp32 values (both signs, the group maxima at row-dependent columns)
// into the 128 columns of its lane, reloads them, and counts each 32-column
// group whose reduced maximum differs from the maximum of what it stored,
// and each loaded value that differs from the stored one.
__device__ int32_t g_tmem_selftest_mismatches;
__global__ void tmem_ld_max_selftest_kernel() {
  __shared__ uint32_t slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    h3kv::tmem_alloc(h3kv::smem_u32(&slot), 128);
    h3kv::tmem_relinquish();
  }
  h3kv::tc_fence_before();
  __syncthreads();
  h3kv::tc_fence_after();
  const uint32_t taddr = slot + (static_cast<uint32_t>(warp * 32) << 16);
  uint32_t v[128];
  float want[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < 128; ++c) {
    float x = static_cast<float>(((tid * 37 + c * 101) % 257) - 128) * 0.37f;
    if ((c & 31) == (tid * 7 + (c >> 5)) % 32) x = 50.0f + 0.25f * tid + (c >> 5);
    v[c] = __float_as_uint(x);
    want[c >> 5] = fmaxf(want[c >> 5], x);
  }
#pragma unroll
  for (int g = 0; g < 4; ++g) h3kv::tmem_st32(taddr + 32 * g, *reinterpret_cast<const uint32_t(*)[32]>(v + 32 * g));
  h3kv::tmem_wait_st();
  uint32_t r[128];
  float m[4];
  h3kv::tmem_ld128_max(taddr, r, m);
  int bad = 0;
#pragma unroll
  for (int c = 0; c < 128; ++c) bad += r[c] != v[c];
#pragma unroll
  for (int g = 0; g < 4; ++g) bad += m[g] != want[g];
  if (bad) atomicAdd(&g_tmem_selftest_mismatches, bad);
  h3kv::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    h3kv::tc_fence_after();
    h3kv::tmem_dealloc(slot, 128);
  }
}

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  uint32_t *err = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

h3kv_status device_info(DeviceInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return H3KV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return H3KV_ERR_CUDA;
    d.supported = (prop.major == 10 && prop.minor == 3);
    d.num_sms = prop.multiProcessorCount;
    if (d.supported) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_h3kv_error) != cudaSuccess) return H3KV_ERR_CUDA;
      d.err = static_cast<uint32_t *>(p);
      if (cudaMemset(d.err, 0, sizeof(uint32_t)) != cudaSuccess) return H3KV_ERR_CUDA;
      if (cudaDeviceSynchronize() != cudaSuccess) return H3KV_ERR_CUDA;
    }
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void *fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return H3KV_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  if (!d.supported) return H3KV_ERR_UNSUPPORTED;
  *out = &d;
  return H3KV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D map over a row-major [rows, 128] matrix of 1- or 2-byte elements.
bool encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t rows, uint32_t elem_bytes,
               uint32_t box_inner) {
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128ull * elem_bytes};
  const cuuint32_t box[2] = {box_inner, 128};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over bf16 [heads, seq, 128]: box 64 x 128 rows x 1 head; rows past
// `seq` read as zero.
bool encode_3d_bf16(CUtensorMap *m, const void *base, uint64_t seq, uint64_t heads) {
  const cuuint64_t dims[3] = {128, seq, heads};
  const cuuint64_t strides[2] = {256, seq * 256};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over 8-bit codes with 128-byte rows of 128 elements along the
// inner axis: dims {inner, mid, heads} with byte strides {mid_stride,
// head_stride}; box 128 x 128 x 1 with the 128-byte swizzle; elements past
// `inner` or `mid` read as zero.
bool encode_3d_u8(CUtensorMap *m, const void *base, uint64_t inner, uint64_t mid, uint64_t heads,
                  uint64_t mid_stride, uint64_t head_stride) {
  const cuuint64_t dims[3] = {inner, mid, heads};
  const cuuint64_t strides[2] = {mid_stride, head_stride};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA coordinates are signed 32-bit; keep every row index below 2^31.
constexpr int64_t kMaxRows = (1ll << 31) - 256;

// The attention kernels run one grid row per head (grid.y <= 65535).
constexpr int32_t kMaxHeads = 65535;

// hostio scratch: the two chunk buffers' ready words, padded to keep the
// region a multiple of 256 bytes.
constexpr size_t kHostioReadyBytes = 256;

h3kv_status check_chunks(int32_t q_chunk, int32_t kv_block) {
  if (q_chunk < 1) return H3KV_ERR_INVALID_ARG;
  if (kv_block < 0 || kv_block % H3KV_KV_TILE != 0) return H3KV_ERR_INVALID_ARG;
  return H3KV_OK;
}

// Scales per row of a store: 1 (scale_group 0 or 128) or 4 (scale_group 32);
// 0 for an invalid scale_group.
int scale_groups_of(const h3kv_store *st) {
  if (st->scale_group == 0 || st->scale_group == 128) return 1;
  if (st->scale_group == 32) return 4;
  return 0;
}

// Whether copies from `p` run in stream order: device, managed or pinned
// host memory.  Pageable host memory is not (its copies read it when they
// are issued).
bool copy_engine_ordered(const void *p) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error the query may leave
    return false;
  }
  return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged || attr.type == cudaMemoryTypeHost;
}

float scale_log2_of(float softmax_scale) {
  const float s = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(128.0f);
  return s * 1.4426950408889634f;
}

}  // namespace

extern "C" {

uint32_t h3kv_abi_version(void) { return H3KV_ABI_VERSION; }

size_t h3kv_store_bytes(int32_t heads, int64_t seq, int32_t head_dim) {
  if (heads < 0 || seq < 0 || head_dim != H3KV_HEAD_DIM) return 0;
  return static_cast<size_t>(2) * static_cast<size_t>(heads) * static_cast<size_t>(seq) *
         static_cast<size_t>(head_dim + 2);
}

const char *h3kv_strerror(h3kv_status status) {
  switch (status) {
    case H3KV_OK: return "ok";
    case H3KV_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size, q_chunk or kv_block)";
    case H3KV_ERR_UNSUPPORTED: return "unsupported (head_dim must be 128; device must be sm_103)";
    case H3KV_ERR_CUDA: return "CUDA runtime error";
    case H3KV_ERR_DEVICE_TIMEOUT: return "a bounded in-kernel wait ran out";
  }
  return "unknown status";
}

h3kv_status h3kv_build_store(const uint16_t *K, const uint16_t *V, int32_t heads, int64_t seq, int32_t head_dim,
                             const h3kv_store *out, void *stream) {
  if (heads < 0 || seq < 0 || !out) return H3KV_ERR_INVALID_ARG;
  if (head_dim != H3KV_HEAD_DIM || out->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  if (out->heads != heads || out->seq != seq) return H3KV_ERR_INVALID_ARG;
  const int groups = scale_groups_of(out);
  if (groups == 0) return H3KV_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(heads) * seq;
  if (rows == 0) return H3KV_OK;
  if (rows > kMaxRows) return H3KV_ERR_INVALID_ARG;
  if (!K || !V || !out->k_codes || !out->v_codes || !out->k_scales || !out->v_scales) return H3KV_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(out->k_codes) || !aligned16(out->v_codes) ||
      !aligned16(out->k_scales) || !aligned16(out->v_scales))
    return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  h3kv_status st = device_info(&d);
  if (st != H3KV_OK) return st;
  CUtensorMap k_in, v_in;
  if (!encode_2d(&k_in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, rows, 2, 64) ||
      !encode_2d(&v_in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, rows, 2, 64))
    return H3KV_ERR_CUDA;
  const cudaError_t e = h3kv::launch_store_build(k_in, v_in, out->k_codes, out->v_codes, out->k_scales, out->v_scales, rows,
                                                 d->num_sms, groups, d->err, g_timeout_ns.load(),
                                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? H3KV_OK : H3KV_ERR_CUDA;
}

h3kv_status h3kv_attend(const uint16_t *Q, int64_t q_seq, const h3kv_store *store, int32_t q_chunk,
                        int32_t kv_block, float softmax_scale, float *O, void *stream) {
  if (!store || q_seq < 0 || store->heads < 0 || store->seq < 0) return H3KV_ERR_INVALID_ARG;
  if (store->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  h3kv_status st = check_chunks(q_chunk, kv_block);
  if (st != H3KV_OK) return st;
  const int groups = scale_groups_of(store);
  if (groups == 0) return H3KV_ERR_INVALID_ARG;
  if (store->heads == 0 || q_seq == 0) return H3KV_OK;
  if (store->seq == 0 || store->heads > kMaxHeads) return H3KV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(store->heads) * q_seq > kMaxRows || static_cast<int64_t>(store->heads) * store->seq > kMaxRows)
    return H3KV_ERR_INVALID_ARG;
  if (!Q || !O || !store->k_codes || !store->v_codes || !store->k_scales || !store->v_scales)
    return H3KV_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(O) || !aligned16(store->k_codes) || !aligned16(store->v_codes) ||
      !aligned16(store->k_scales) || !aligned16(store->v_scales))
    return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != H3KV_OK) return st;
  const int32_t kvb = kv_block == 0 ? H3KV_DEFAULT_KV_BLOCK : kv_block;
  h3kv::AttnArgs a{};
  a.q = Q;
  a.k_codes = store->k_codes;
  a.v_codes = store->v_codes;
  a.k_scales = store->k_scales;
  a.v_scales = store->v_scales;
  a.o = O;
  a.q_seq = q_seq;
  a.kv_seq = store->seq;
  a.kv_stride = store->seq;
  a.scale_groups = groups;
  a.heads = store->heads;
  a.kv_block_tiles = kvb / H3KV_KV_TILE;
  a.scale_log2 = scale_log2_of(softmax_scale);
  a.err = d->err;
  a.timeout_ns = g_timeout_ns.load();
  a.withhold_p_tile1 = g_withhold_p_tile1.load();
  return h3kv::launch_query_chunks(a, q_seq, store->seq, q_chunk, store->heads, [&](const h3kv::AttnArgs &x, bool overlap) {
    return h3kv::launch_attend_kvi8r(x, overlap, static_cast<cudaStream_t>(stream));
  });
}

h3kv_status h3kv_attend_exact(const uint16_t *Q, int64_t q_seq, const uint16_t *K, const uint16_t *V,
                              int32_t heads, int64_t kv_seq, int32_t head_dim, int32_t q_chunk, int32_t kv_block,
                              float softmax_scale, float *O, void *stream) {
  if (q_seq < 0 || heads < 0 || kv_seq < 0) return H3KV_ERR_INVALID_ARG;
  if (head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  h3kv_status st = check_chunks(q_chunk, kv_block);
  if (st != H3KV_OK) return st;
  if (heads == 0 || q_seq == 0) return H3KV_OK;
  if (kv_seq == 0 || heads > kMaxHeads) return H3KV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(heads) * q_seq > kMaxRows || static_cast<int64_t>(heads) * kv_seq > kMaxRows)
    return H3KV_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O) return H3KV_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != H3KV_OK) return st;
  CUtensorMap tq, tk, tv;
  if (!encode_3d_bf16(&tq, Q, static_cast<uint64_t>(q_seq), static_cast<uint64_t>(heads)) ||
      !encode_3d_bf16(&tk, K, static_cast<uint64_t>(kv_seq), static_cast<uint64_t>(heads)) ||
      !encode_3d_bf16(&tv, V, static_cast<uint64_t>(kv_seq), static_cast<uint64_t>(heads)))
    return H3KV_ERR_CUDA;
  const int64_t n_tiles = (kv_seq + H3KV_KV_TILE - 1) / H3KV_KV_TILE;
  h3kv::AttnArgs a{};
  a.q = Q;
  a.o = O;
  a.q_seq = q_seq;
  a.kv_seq = kv_seq;
  a.kv_stride = kv_seq;
  a.scale_groups = 1;
  a.heads = heads;
  a.kv_block_tiles = kv_block == 0 ? static_cast<int32_t>(n_tiles) : kv_block / H3KV_KV_TILE;
  a.scale_log2 = scale_log2_of(softmax_scale);
  a.err = d->err;
  a.timeout_ns = g_timeout_ns.load();
  a.withhold_p_tile1 = g_withhold_p_tile1.load();
  return h3kv::launch_query_chunks(a, q_seq, kv_seq, q_chunk, heads, [&](const h3kv::AttnArgs &x, bool overlap) {
    return h3kv::launch_attend_exact(tq, tk, tv, x, overlap, static_cast<cudaStream_t>(stream));
  });
}

size_t h3kv_staging_bytes(int32_t heads, int32_t kv_block) {
  if (heads < 0 || kv_block < 0 || kv_block % H3KV_KV_TILE != 0) return 0;
  const size_t kvb = static_cast<size_t>(kv_block == 0 ? H3KV_DEFAULT_KV_BLOCK : kv_block);
  return 2 * static_cast<size_t>(heads) * kvb * (H3KV_HEAD_DIM + 2);
}

h3kv_status h3kv_attend_staged(const uint16_t *Q, int64_t q_seq, const h3kv_store *store, int32_t q_chunk,
                               int32_t kv_block, float softmax_scale, float *O, void *staging,
                               size_t staging_bytes, float *state, void *stream) {
  if (!store || q_seq < 0 || store->heads < 0 || store->seq < 0) return H3KV_ERR_INVALID_ARG;
  if (store->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  h3kv_status st = check_chunks(q_chunk, kv_block);
  if (st != H3KV_OK) return st;
  if (scale_groups_of(store) == 0) return H3KV_ERR_INVALID_ARG;
  if (scale_groups_of(store) != 1) return H3KV_ERR_UNSUPPORTED;
  if (store->heads == 0 || q_seq == 0) return H3KV_OK;
  if (store->seq == 0 || store->heads > kMaxHeads) return H3KV_ERR_INVALID_ARG;
  const int64_t H = store->heads;
  if (H * q_seq > kMaxRows || H * store->seq > kMaxRows) return H3KV_ERR_INVALID_ARG;
  if (!Q || !O || !staging || !state || !store->k_codes || !store->v_codes || !store->k_scales ||
      !store->v_scales)
    return H3KV_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(O) || !aligned16(staging) || !aligned16(state)) return H3KV_ERR_INVALID_ARG;
  const int64_t kvb = kv_block == 0 ? H3KV_DEFAULT_KV_BLOCK : kv_block;
  if (staging_bytes < h3kv_staging_bytes(store->heads, static_cast<int32_t>(kvb))) return H3KV_ERR_INVALID_ARG;
  // the block copies are stream-ordered only from device, managed or pinned
  // memory: from pageable memory the driver takes the bytes when the copy is
  // issued, before earlier work in the stream (a store build, say) has run
  for (const void *p : {static_cast<const void *>(store->k_codes), static_cast<const void *>(store->v_codes),
                        static_cast<const void *>(store->k_scales), static_cast<const void *>(store->v_scales)})
    if (!copy_engine_ordered(p)) return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != H3KV_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // staging: one or two blocks, each k codes [H, kvb, 128], v codes, k
  // scales [H, kvb], v scales; the second (if the scratch holds two) starts
  // at the first block's size rounded up to 256 bytes
  const size_t need = h3kv_staging_bytes(store->heads, static_cast<int32_t>(kvb));
  const size_t need_aligned = (need + 255) & ~static_cast<size_t>(255);
  const int nbuf = staging_bytes >= need_aligned + need ? 2 : 1;
  struct StageBuf {
    int8_t *kc, *vc;
    uint16_t *ks, *vs;
  } buf[2];
  for (int p = 0; p < nbuf; ++p) {
    buf[p].kc = static_cast<int8_t *>(staging) + p * need_aligned;
    buf[p].vc = buf[p].kc + H * kvb * 128;
    buf[p].ks = reinterpret_cast<uint16_t *>(buf[p].vc + H * kvb * 128);
    buf[p].vs = buf[p].ks + H * kvb;
  }
  h3kv::AttnArgs a{};
  a.q = Q;
  a.o = O;
  a.q_seq = q_seq;
  a.kv_stride = kvb;
  a.heads = store->heads;
  a.scale_log2 = scale_log2_of(softmax_scale);
  a.err = d->err;
  a.timeout_ns = g_timeout_ns.load();
  a.withhold_p_tile1 = g_withhold_p_tile1.load();
  a.state = reinterpret_cast<float2 *>(state);
  a.scale_groups = 1;
  const int64_t n_blocks = (store->seq + kvb - 1) / kvb;
  auto len_of = [&](int64_t b) { return store->seq - b * kvb < kvb ? store->seq - b * kvb : kvb; };
  // one block of every head into staging buffer p, on stream cs
  auto copy_block = [&](int64_t b, int p, cudaStream_t cs) {
    const int64_t b0 = b * kvb, len = len_of(b);
    return cudaMemcpy2DAsync(buf[p].kc, kvb * 128, store->k_codes + b0 * 128, store->seq * 128, len * 128, H,
                             cudaMemcpyDefault, cs) == cudaSuccess &&
           cudaMemcpy2DAsync(buf[p].vc, kvb * 128, store->v_codes + b0 * 128, store->seq * 128, len * 128, H,
                             cudaMemcpyDefault, cs) == cudaSuccess &&
           cudaMemcpy2DAsync(buf[p].ks, kvb * 2, store->k_scales + b0, store->seq * 2, len * 2, H,
                             cudaMemcpyDefault, cs) == cudaSuccess &&
           cudaMemcpy2DAsync(buf[p].vs, kvb * 2, store->v_scales + b0, store->seq * 2, len * 2, H,
                             cudaMemcpyDefault, cs) == cudaSuccess;
  };
  // Every query chunk of block b over buffer p.  Launches after a block's
  // first follow the previous one with programmatic dependent launch: they
  // touch other query rows and only read the staged block.  A block's first
  // launch is a plain one, after everything before it in the stream, so the
  // state and O rows that the previous block's launches carry are complete
  // (each launch completes only after the one before it).
  auto attend_block = [&](int64_t b, int p) {
    const int64_t len = len_of(b);
    a.k_codes = buf[p].kc;
    a.v_codes = buf[p].vc;
    a.k_scales = buf[p].ks;
    a.v_scales = buf[p].vs;
    a.kv_seq = len;
    a.kv_block_tiles = static_cast<int32_t>((len + H3KV_KV_TILE - 1) / H3KV_KV_TILE);
    a.stage_flags = (b == 0 ? 1 : 0) | (b == n_blocks - 1 ? 2 : 0);
    for (int64_t c0 = 0; c0 < q_seq; c0 += q_chunk) {
      a.q_begin = c0;
      a.q_end = c0 + q_chunk < q_seq ? c0 + q_chunk : q_seq;
      if (h3kv::launch_attend_kvi8r(a, c0 > 0, s) != cudaSuccess) return false;
    }
    return true;
  };
  if (nbuf == 1) {
    // each block's copy is stream-ordered after the previous block's
    // launches, which read the same buffer
    for (int64_t b = 0; b < n_blocks; ++b)
      if (!copy_block(b, 0, s) || !attend_block(b, 0)) return H3KV_ERR_CUDA;
    return H3KV_OK;
  }
  // Two buffers: block b + 1 is copied on a second stream while block b is
  // attended; the copy into buffer p waits for the launches of block b - 2,
  // the last ones to read it, and block b's launches wait for its copy.
  cudaStream_t cs = nullptr;
  cudaEvent_t entry = nullptr, copied[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr};
  h3kv_status result = H3KV_OK;
  const unsigned ef = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&entry, ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&copied[0], ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&copied[1], ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&done[0], ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&done[1], ef) == cudaSuccess;
  // the copies start after everything queued on the caller's stream (which
  // may have written the store)
  ok = ok && cudaEventRecord(entry, s) == cudaSuccess && cudaStreamWaitEvent(cs, entry, 0) == cudaSuccess;
  for (int64_t b = 0; ok && b < n_blocks; ++b) {
    const int p = static_cast<int>(b & 1);
    ok = (b < 2 || cudaStreamWaitEvent(cs, done[p], 0) == cudaSuccess) && copy_block(b, p, cs) &&
         cudaEventRecord(copied[p], cs) == cudaSuccess && cudaStreamWaitEvent(s, copied[p], 0) == cudaSuccess &&
         attend_block(b, p) && cudaEventRecord(done[p], s) == cudaSuccess;
  }
  if (!ok) result = H3KV_ERR_CUDA;
  // (every copy on cs is waited on by a launch on s, so later work on s is
  // ordered after all of them)
  for (cudaEvent_t e : {entry, copied[0], copied[1], done[0], done[1]})
    if (e) cudaEventDestroy(e);
  if (cs) cudaStreamDestroy(cs);
  return result;
}

size_t h3kv_hostio_scratch_bytes(int32_t heads, int32_t q_chunk) {
  if (heads < 0 || q_chunk < 1) return 0;
  return 2 * static_cast<size_t>(heads) * static_cast<size_t>(q_chunk) * H3KV_HEAD_DIM * (2 + 4) + kHostioReadyBytes;
}

namespace {

// Values the copy engine writes into hostio's ready words: entries 0 and 1
// are zero (the reset), entry v holds v.  Pinned host memory, so that the
// 4-byte copies run on the copy engine; allocated once, kept until exit.
constexpr int kReadyValues = 1024;
std::mutex g_ready_mu;
uint32_t *g_ready_table = nullptr;

const uint32_t *ready_table() {
  std::lock_guard<std::mutex> lock(g_ready_mu);
  if (!g_ready_table) {
    void *p = nullptr;
    if (cudaHostAlloc(&p, kReadyValues * sizeof(uint32_t), cudaHostAllocPortable) != cudaSuccess) return nullptr;
    uint32_t *t = static_cast<uint32_t *>(p);
    t[0] = t[1] = 0;
    for (int v = 2; v < kReadyValues; ++v) t[v] = static_cast<uint32_t>(v);
    g_ready_table = t;
  }
  return g_ready_table;
}

}  // namespace

h3kv_status h3kv_attend_hostio(const uint16_t *Q_host, int64_t q_seq, const h3kv_store *store, int32_t q_chunk,
                               int32_t kv_block, float softmax_scale, float *O_host, void *scratch,
                               size_t scratch_bytes, void *stream) {
  if (!store || q_seq < 0 || store->heads < 0 || store->seq < 0) return H3KV_ERR_INVALID_ARG;
  if (store->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  h3kv_status st = check_chunks(q_chunk, kv_block);
  if (st != H3KV_OK) return st;
  const int groups = scale_groups_of(store);
  if (groups == 0) return H3KV_ERR_INVALID_ARG;
  if (store->heads == 0 || q_seq == 0) return H3KV_OK;
  if (store->seq == 0 || store->heads > kMaxHeads) return H3KV_ERR_INVALID_ARG;
  const int64_t H = store->heads;
  if (H * q_seq > kMaxRows || H * store->seq > kMaxRows) return H3KV_ERR_INVALID_ARG;
  if (!Q_host || !O_host || !scratch || !store->k_codes || !store->v_codes || !store->k_scales ||
      !store->v_scales)
    return H3KV_ERR_INVALID_ARG;
  if (!aligned16(scratch) || !aligned16(store->k_codes) || !aligned16(store->v_codes) ||
      !aligned16(store->k_scales) || !aligned16(store->v_scales))
    return H3KV_ERR_INVALID_ARG;
  if (scratch_bytes < h3kv_hostio_scratch_bytes(store->heads, q_chunk)) return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != H3KV_OK) return st;
  const uint32_t *table = ready_table();
  if (!table) return H3KV_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // scratch: Q chunks [2][H, q_chunk, 128] bf16, O chunks [2][H, q_chunk, 128]
  // fp32, then the two buffers' ready words
  const int64_t qc = q_chunk;
  uint16_t *qbuf[2];
  float *obuf[2];
  qbuf[0] = static_cast<uint16_t *>(scratch);
  qbuf[1] = qbuf[0] + H * qc * 128;
  obuf[0] = reinterpret_cast<float *>(qbuf[1] + H * qc * 128);
  obuf[1] = obuf[0] + H * qc * 128;
  uint32_t *ready = reinterpret_cast<uint32_t *>(obuf[1] + H * qc * 128);
  const int32_t kvb = kv_block == 0 ? H3KV_DEFAULT_KV_BLOCK : kv_block;
  h3kv::AttnArgs a{};
  a.k_codes = store->k_codes;
  a.v_codes = store->v_codes;
  a.k_scales = store->k_scales;
  a.v_scales = store->v_scales;
  a.q_seq = qc;  // row stride of a chunk buffer
  a.kv_seq = store->seq;
  a.kv_stride = store->seq;
  a.scale_groups = groups;
  a.heads = store->heads;
  a.kv_block_tiles = kvb / H3KV_KV_TILE;
  a.scale_log2 = scale_log2_of(softmax_scale);
  a.err = d->err;
  a.timeout_ns = g_timeout_ns.load();
  a.withhold_p_tile1 = g_withhold_p_tile1.load();
  a.q_begin = 0;

  // Schedule.  Copy stream cs: reset both ready words, Q chunks 0 and 1 in;
  // then, per chunk c, once its attention is done: O chunk c out, Q chunk
  // c + 2 into the freed buffer, and that buffer's ready word set to the
  // value of chunk c + 2.  Caller's stream s: chunk 0's launch waits for its
  // Q copy (an event); launches 1 .. n-1 follow each other with programmatic
  // dependent launch and wait for their ready word inside the kernel, so no
  // stream wait sits between them (one would end the overlap of a launch's
  // tail with the next launch).  Progress: the word of chunk c needs chunk
  // c - 2 complete, and every CTA of chunk c - 2 is running or done before
  // chunk c can launch (c - 1 launches only after all of c - 2's CTAs have
  // started, c only after all of c - 1's), so a waiting CTA always sees its
  // word arrive.
  cudaStream_t cs = nullptr;
  cudaEvent_t entry = nullptr, fin = nullptr, q0_ready = nullptr, att_done[2] = {nullptr, nullptr};
  h3kv_status result = H3KV_OK;
  auto fail = [&](cudaError_t e) {
    if (e != cudaSuccess && result == H3KV_OK) result = H3KV_ERR_CUDA;
    return e != cudaSuccess;
  };
  const unsigned ef = cudaEventDisableTiming;
  if (!fail(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) && !fail(cudaEventCreateWithFlags(&entry, ef)) &&
      !fail(cudaEventCreateWithFlags(&fin, ef)) && !fail(cudaEventCreateWithFlags(&q0_ready, ef)) &&
      !fail(cudaEventCreateWithFlags(&att_done[0], ef)) && !fail(cudaEventCreateWithFlags(&att_done[1], ef))) {
    const int64_t n = (q_seq + qc - 1) / qc;
    auto rows_of = [&](int64_t c) { return (c + 1) * qc <= q_seq ? qc : q_seq - c * qc; };
    // ready value of chunk c >= 1: never 0 (the reset) and different from
    // chunk c - 2's, the previous value of the same word
    auto value_of = [](int64_t c) { return static_cast<uint32_t>(2 + c % (kReadyValues - 2)); };
    // Q rows [c qc, c qc + rows) of every head -> chunk buffer b
    auto copy_in = [&](int64_t c, int b) {
      return cudaMemcpy2DAsync(qbuf[b], qc * 256, Q_host + c * qc * 128, q_seq * 256, rows_of(c) * 256, H,
                               cudaMemcpyHostToDevice, cs);
    };
    auto copy_out = [&](int64_t c, int b) {
      return cudaMemcpy2DAsync(O_host + c * qc * 128, q_seq * 512, obuf[b], qc * 512, rows_of(c) * 512, H,
                               cudaMemcpyDeviceToHost, cs);
    };
    auto set_ready = [&](int64_t c) {
      return cudaMemcpyAsync(&ready[c & 1], &table[value_of(c)], sizeof(uint32_t), cudaMemcpyHostToDevice, cs);
    };
    // the copies start after everything queued on the caller's stream
    bool ok = !fail(cudaEventRecord(entry, s)) && !fail(cudaStreamWaitEvent(cs, entry, 0)) &&
              !fail(cudaMemcpyAsync(ready, table, 2 * sizeof(uint32_t), cudaMemcpyHostToDevice, cs)) &&
              !fail(copy_in(0, 0)) && !fail(cudaEventRecord(q0_ready, cs));
    if (ok && n > 1) ok = !fail(copy_in(1, 1)) && !fail(set_ready(1));
    for (int64_t c = 0; ok && c < n; ++c) {
      const int b = static_cast<int>(c & 1);
      a.q = qbuf[b];
      a.o = obuf[b];
      a.q_end = rows_of(c);
      a.q_ready = c > 0 ? &ready[b] : nullptr;
      a.q_ready_value = c > 0 ? value_of(c) : 0u;
      if (c == 0) ok = !fail(cudaStreamWaitEvent(s, q0_ready, 0));
      ok = ok && !fail(h3kv::launch_attend_kvi8r(a, c > 0, s)) && !fail(cudaEventRecord(att_done[b], s)) &&
           !fail(cudaStreamWaitEvent(cs, att_done[b], 0)) && !fail(copy_out(c, b));
      // buffer b is free again for chunk c + 2 once its O rows are out
      if (ok && c + 2 < n) ok = !fail(copy_in(c + 2, b)) && !fail(set_ready(c + 2));
    }
    // later work on the caller's stream sees every O row in host memory
    if (ok) ok = !fail(cudaEventRecord(fin, cs)) && !fail(cudaStreamWaitEvent(s, fin, 0));
    (void)ok;
  }
  for (cudaEvent_t e : {entry, fin, q0_ready, att_done[0], att_done[1]})
    if (e) cudaEventDestroy(e);
  if (cs) cudaStreamDestroy(cs);
  return result;
}

int64_t h3kv_f8_v_stride(int64_t seq) { return seq < 0 ? 0 : (seq + 15) / 16 * 16; }

size_t h3kv_store_f8_bytes(int32_t heads, int64_t seq, int32_t head_dim) {
  if (heads < 0 || seq < 0 || head_dim != H3KV_HEAD_DIM) return 0;
  const size_t H = static_cast<size_t>(heads);
  const size_t nblk = static_cast<size_t>((seq + H3KV_F8_K_BLOCK - 1) / H3KV_F8_K_BLOCK);
  return H * static_cast<size_t>(seq) * 128 + H * 128 * static_cast<size_t>(h3kv_f8_v_stride(seq)) +
         H * nblk * 4 + 2 * H * 128 * 4;
}

h3kv_status h3kv_build_store_f8(const uint16_t *K, const uint16_t *V, int32_t heads, int64_t seq,
                                int32_t head_dim, const h3kv_store_f8 *out, void *stream) {
  if (heads < 0 || seq < 0 || !out) return H3KV_ERR_INVALID_ARG;
  if (head_dim != H3KV_HEAD_DIM || out->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  if (out->heads != heads || out->seq != seq) return H3KV_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(heads) * seq;
  if (rows == 0) return H3KV_OK;
  if (rows > kMaxRows || heads > 65535) return H3KV_ERR_INVALID_ARG;
  if (!K || !V || !out->k_codes || !out->v_codes_t || !out->k_scales || !out->v_scales || !out->k_mean)
    return H3KV_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(out->k_codes) || !aligned16(out->v_codes_t) ||
      !aligned16(out->k_scales) || !aligned16(out->v_scales) || !aligned16(out->k_mean))
    return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  h3kv_status st = device_info(&d);
  if (st != H3KV_OK) return st;
  CUtensorMap k_in, v_in;
  if (!encode_3d_bf16(&k_in, K, static_cast<uint64_t>(seq), static_cast<uint64_t>(heads)) ||
      !encode_3d_bf16(&v_in, V, static_cast<uint64_t>(seq), static_cast<uint64_t>(heads)))
    return H3KV_ERR_CUDA;
  const cudaError_t e = h3kv::launch_store_build_f8(
      k_in, v_in, K, V, heads, seq, h3kv_f8_v_stride(seq), out->k_codes, out->v_codes_t, out->k_scales,
      out->v_scales, out->k_mean, d->num_sms, d->err, g_timeout_ns.load(), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? H3KV_OK : H3KV_ERR_CUDA;
}

h3kv_status h3kv_attend_f8(const uint16_t *Q, int64_t q_seq, const h3kv_store_f8 *store, int32_t q_chunk,
                           int32_t kv_block, float softmax_scale, float *O, void *stream) {
  if (!store || q_seq < 0 || store->heads < 0 || store->seq < 0) return H3KV_ERR_INVALID_ARG;
  if (store->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  h3kv_status st = check_chunks(q_chunk, kv_block);
  if (st != H3KV_OK) return st;
  if (store->heads == 0 || q_seq == 0) return H3KV_OK;
  if (store->seq == 0 || store->heads > kMaxHeads) return H3KV_ERR_INVALID_ARG;
  const int64_t H = store->heads;
  if (H * q_seq > kMaxRows || H * store->seq > kMaxRows) return H3KV_ERR_INVALID_ARG;
  if (!Q || !O || !store->k_codes || !store->v_codes_t || !store->k_scales || !store->v_scales)
    return H3KV_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(O) || !aligned16(store->k_codes) || !aligned16(store->v_codes_t) ||
      !aligned16(store->k_scales) || !aligned16(store->v_scales))
    return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != H3KV_OK) return st;
  const uint64_t L = static_cast<uint64_t>(store->seq);
  const uint64_t vs = static_cast<uint64_t>(h3kv_f8_v_stride(store->seq));
  CUtensorMap tk, tv;
  if (!encode_3d_u8(&tk, store->k_codes, 128, L, static_cast<uint64_t>(H), 128, L * 128) ||
      !encode_3d_u8(&tv, store->v_codes_t, L, 128, static_cast<uint64_t>(H), vs, 128 * vs))
    return H3KV_ERR_CUDA;
  const int32_t kvb = kv_block == 0 ? H3KV_DEFAULT_KV_BLOCK : kv_block;
  h3kv::F8Args a{};
  a.q = Q;
  a.o = O;
  a.k_scales = store->k_scales;
  a.v_scales = store->v_scales;
  a.q_seq = q_seq;
  a.kv_seq = store->seq;
  a.heads = store->heads;
  a.kv_block_tiles = kvb / H3KV_KV_TILE;
  a.k_blocks = static_cast<int32_t>((store->seq + H3KV_F8_K_BLOCK - 1) / H3KV_F8_K_BLOCK);
  a.scale_log2 = scale_log2_of(softmax_scale);
  a.err = d->err;
  a.timeout_ns = g_timeout_ns.load();
  a.withhold_p_tile1 = g_withhold_p_tile1.load();
  return h3kv::launch_query_chunks(a, q_seq, store->seq, q_chunk, store->heads, [&](const h3kv::F8Args &x, bool overlap) {
    return h3kv::launch_attend_f8(tk, tv, x, overlap, static_cast<cudaStream_t>(stream));
  });
}

size_t h3kv_store_fp4_bytes(int32_t heads, int64_t seq, int32_t head_dim) {
  if (heads < 0 || seq < 0 || head_dim != H3KV_HEAD_DIM) return 0;
  return 2 * static_cast<size_t>(heads) * static_cast<size_t>(seq) * (64 + 8);
}

h3kv_status h3kv_build_store_fp4(const uint16_t *K, const uint16_t *V, int32_t heads, int64_t seq,
                                 int32_t head_dim, const h3kv_store_fp4 *out, void *stream) {
  if (heads < 0 || seq < 0 || !out) return H3KV_ERR_INVALID_ARG;
  if (head_dim != H3KV_HEAD_DIM || out->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  if (out->heads != heads || out->seq != seq) return H3KV_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(heads) * seq;
  if (rows == 0) return H3KV_OK;
  if (rows > kMaxRows) return H3KV_ERR_INVALID_ARG;
  if (!K || !V || !out->k_codes || !out->v_codes || !out->k_scales || !out->v_scales) return H3KV_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(out->k_codes) || !aligned16(out->v_codes) ||
      !aligned16(out->k_scales) || !aligned16(out->v_scales))
    return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  h3kv_status st = device_info(&d);
  if (st != H3KV_OK) return st;
  CUtensorMap k_in, v_in;
  if (!encode_2d(&k_in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, rows, 2, 64) ||
      !encode_2d(&v_in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, rows, 2, 64))
    return H3KV_ERR_CUDA;
  const cudaError_t e = h3kv::launch_store_build_fp4(k_in, v_in, out->k_codes, out->v_codes, out->k_scales,
                                                     out->v_scales, rows,
                                                     d->num_sms, d->err, g_timeout_ns.load(),
                                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? H3KV_OK : H3KV_ERR_CUDA;
}

h3kv_status h3kv_attend_fp4(const uint16_t *Q, int64_t q_seq, const h3kv_store_fp4 *store, int32_t q_chunk,
                            int32_t kv_block, float softmax_scale, float *O, void *stream) {
  if (!store || q_seq < 0 || store->heads < 0 || store->seq < 0) return H3KV_ERR_INVALID_ARG;
  if (store->head_dim != H3KV_HEAD_DIM) return H3KV_ERR_UNSUPPORTED;
  h3kv_status st = check_chunks(q_chunk, kv_block);
  if (st != H3KV_OK) return st;
  if (store->heads == 0 || q_seq == 0) return H3KV_OK;
  if (store->seq == 0 || store->heads > kMaxHeads) return H3KV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(store->heads) * q_seq > kMaxRows || static_cast<int64_t>(store->heads) * store->seq > kMaxRows)
    return H3KV_ERR_INVALID_ARG;
  if (!Q || !O || !store->k_codes || !store->v_codes || !store->k_scales || !store->v_scales)
    return H3KV_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(O) || !aligned16(store->k_codes) || !aligned16(store->v_codes) ||
      !aligned16(store->k_scales) || !aligned16(store->v_scales))
    return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != H3KV_OK) return st;
  const int32_t kvb = kv_block == 0 ? H3KV_DEFAULT_KV_BLOCK : kv_block;
  h3kv::AttnArgs a{};
  a.q = Q;
  a.k_codes = reinterpret_cast<const int8_t *>(store->k_codes);
  a.v_codes = reinterpret_cast<const int8_t *>(store->v_codes);
  a.k_fp4_scales = store->k_scales;
  a.v_fp4_scales = store->v_scales;
  a.o = O;
  a.q_seq = q_seq;
  a.kv_seq = store->seq;
  a.kv_stride = store->seq;
  a.scale_groups = 1;
  a.heads = store->heads;
  a.kv_block_tiles = kvb / H3KV_KV_TILE;
  a.scale_log2 = scale_log2_of(softmax_scale);
  a.err = d->err;
  a.timeout_ns = g_timeout_ns.load();
  a.withhold_p_tile1 = g_withhold_p_tile1.load();
  return h3kv::launch_query_chunks(a, q_seq, store->seq, q_chunk, store->heads, [&](const h3kv::AttnArgs &x, bool overlap) {
    return h3kv::launch_attend_fp4(x, overlap, static_cast<cudaStream_t>(stream));
  });
}

int64_t h3kv_attend_launch_count(int64_t q_seq, int64_t kv_seq, int32_t heads, int32_t q_chunk) {
  return h3kv::launch_count(q_seq, kv_seq, q_chunk, heads);
}

h3kv_status h3kv_set_wait_timeout_ns(uint64_t timeout_ns) {
  g_timeout_ns.store(timeout_ns == 0 ? kDefaultTimeoutNs : timeout_ns);
  return H3KV_OK;
}

h3kv_status h3kv_debug_withhold_p(int32_t tile) {
  if (tile < -1) return H3KV_ERR_INVALID_ARG;
  g_withhold_p_tile1.store(tile + 1);
  return H3KV_OK;
}

h3kv_status h3kv_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
  DeviceInfo *d = nullptr;
  h3kv_status st = device_info(&d);
  if (st != H3KV_OK) return st;
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      d->err, timeout_ns == 0 ? kDefaultTimeoutNs : timeout_ns);
  return cudaGetLastError() == cudaSuccess ? H3KV_OK : H3KV_ERR_CUDA;
}

h3kv_status h3kv_selftest_tmem_ld_max(int32_t *mismatches, void *stream) {
  if (!mismatches) return H3KV_ERR_INVALID_ARG;
  DeviceInfo *d = nullptr;
  h3kv_status st = device_info(&d);
  if (st != H3KV_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t zero = 0;
  if (cudaMemcpyToSymbolAsync(g_tmem_selftest_mismatches, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return H3KV_ERR_CUDA;
  tmem_ld_max_selftest_kernel<<<1, 128, 0, s>>>();
  if (cudaGetLastError() != cudaSuccess) return H3KV_ERR_CUDA;
  if (cudaMemcpyFromSymbolAsync(mismatches, g_tmem_selftest_mismatches, sizeof(int32_t), 0, cudaMemcpyDeviceToHost,
                                s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return H3KV_ERR_CUDA;
  return H3KV_OK;
}

h3kv_status h3kv_sync_status(void *stream) {
  DeviceInfo *d = nullptr;
  h3kv_status st = device_info(&d);
  if (st != H3KV_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return H3KV_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, d->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return H3KV_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(d->err, 0, sizeof(uint32_t)) != cudaSuccess) return H3KV_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return H3KV_ERR_CUDA;
    // bit 0: a bounded wait ran out; bit 1: the shared-memory base could not
    // be aligned within the requested slack (the kernel returned at entry)
    return (word & h3kv::kErrTimeout) ? H3KV_ERR_DEVICE_TIMEOUT : H3KV_ERR_CUDA;
  }
  return H3KV_OK;
}

}  // extern "C"
