// store_f8.cu -- the kvf8s store build: K and V as fp8 e4m3 in the kvi8s
// layout ("The K/V store options" table of the Low VRAM write-up, kvi8s row;
// kv_store row of the H3 Streamed Blocks Inputs table), with fp8 K in place
// of int8 so that both products run on the fp8 tensor path.
//
//   K: k' = k H (the 128-wide Hadamard basis), smoothed by mu = the mean of
//      k' over all tokens of the head, one fp32 scale per 64-token block
//      s = absmax / 448, codes e4m3(x * fp32(1/s)).
//   V: not rotated; one fp32 scale per (head, channel) s = absmax over all
//      tokens / 448, codes e4m3(v * fp32(1/s)), stored channel-major [heads,
//      128, v_stride] (V transposed) so that P.V reads it K-major.
//
// Two passes: a statistics pass (the K mean and the V channel absmax of
// every head) and an encode pass.  Both are HBM streams; every sum is taken
// in a fixed order, so the store is the same on every run.
#include <cooperative_groups.h>

#include "kernels.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace h3kv {
namespace f8store {

constexpr int kStatCtas = 16;     // one cluster of CTAs per head (8 where 16 cannot launch)
constexpr int kStatThreads = 512;
constexpr int kBlockTok = 64;     // tokens per K scale block
constexpr int kEncThreads = 128;  // 4 warps x 16 tokens = one block
constexpr float kE4m3Max = 448.0f;

__device__ __forceinline__ void bf16x4(const uint2 w, float (&x)[4]) {
  x[0] = bf16lo_to_f32(w.x);
  x[1] = bf16hi_to_f32(w.x);
  x[2] = bf16lo_to_f32(w.y);
  x[3] = bf16hi_to_f32(w.y);
}

constexpr int kStatChunk = 64;    // rows per bulk copy
constexpr int kStatStages = 3;    // copies in flight per CTA

struct StatSmem {
  uint8_t k[kStatStages][kStatChunk * 256];  // bf16 rows of K
  uint8_t v[kStatStages][kStatChunk * 256];  // and of V
  float cta_sum[128];
  float cta_max[128];
  uint64_t full[kStatStages];
  int abort;
};
constexpr size_t kStatSmemBytes = sizeof(StatSmem) + 128;
static_assert(kStatChunk * 256 >= (kStatThreads / 16) * 128 * 4, "partials reuse a stage buffer");

// Pass 1, grid (cluster size, heads), one cluster per head.  CTA r of n
// covers the tokens [r * per, (r + 1) * per), per = ceil(seq / n), in chunks
// of 64 rows that bulk copies bring into a 3-stage shared-memory ring.
// Thread t sums channels 8 (t mod 16) .. +7 of rows t/16 and t/16 + 32 of
// every chunk.  Partials are then combined over the row groups, then CTA by
// CTA through distributed shared memory, always in index order, so the
// result does not depend on timing.
__global__ void __launch_bounds__(kStatThreads)
    stats_kernel(const uint16_t *K, const uint16_t *V, int64_t seq, float *k_mean, float *v_scales, uint32_t *err,
                 uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  StatSmem &sm = *reinterpret_cast<StatSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int nc = static_cast<int>(cluster.num_blocks());
  const int h = blockIdx.y;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int g = t & 15, rg = t >> 4;
  const int64_t per = (seq + nc - 1) / nc;
  const int64_t r0 = rank * per;
  const int64_t r1 = r0 + per < seq ? r0 + per : seq;
  const int n_chunks = r1 > r0 ? static_cast<int>((r1 - r0 + kStatChunk - 1) / kStatChunk) : 0;
  const int64_t hrow = static_cast<int64_t>(h) * seq;

  if (t == 0) {
    for (int st = 0; st < kStatStages; ++st) mbar_init(smem_u32(&sm.full[st]), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int c) {
    const int st = c % kStatStages;
    const int64_t row = r0 + static_cast<int64_t>(c) * kStatChunk;
    const uint32_t bytes = static_cast<uint32_t>((r1 - row < kStatChunk ? r1 - row : kStatChunk) * 256);
    const uint32_t bar = smem_u32(&sm.full[st]);
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_g2s(smem_u32(sm.k[st]), K + (hrow + row) * 128, bytes, bar);
    bulk_g2s(smem_u32(sm.v[st]), V + (hrow + row) * 128, bytes, bar);
  };
  int issued = 0;
  if (t == 0)
    for (; issued < kStatStages && issued < n_chunks; ++issued) issue(issued);

  const WaitCtx wctx{err, &sm.abort, timeout_ns};
  float s[8], m[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) s[c] = m[c] = 0.f;
  int c = 0;
  bool ok = true;
  for (; c < n_chunks; ++c) {
    const int st = c % kStatStages;
    ok = __syncthreads_and(mbar_wait(smem_u32(&sm.full[st]), (c / kStatStages) & 1, wctx));
    if (!ok) break;
    const int64_t row = r0 + static_cast<int64_t>(c) * kStatChunk;
    const int valid = static_cast<int>(r1 - row < kStatChunk ? r1 - row : kStatChunk);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int lr = rg + 32 * hr;
      if (lr < valid) {
        const uint4 kw = *reinterpret_cast<const uint4 *>(sm.k[st] + lr * 256 + g * 16);
        const uint4 vw = *reinterpret_cast<const uint4 *>(sm.v[st] + lr * 256 + g * 16);
        const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w};
        const uint32_t vv[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          s[2 * p] += bf16lo_to_f32(kk[p]);
          s[2 * p + 1] += bf16hi_to_f32(kk[p]);
          m[2 * p] = fmaxf(m[2 * p], fabsf(bf16lo_to_f32(vv[p])));
          m[2 * p + 1] = fmaxf(m[2 * p + 1], fabsf(bf16hi_to_f32(vv[p])));
        }
      }
    }
    __syncthreads();  // the stage is free again
    if (t == 0 && issued < n_chunks) issue(issued++);
  }
  if (!ok) {
    // copies still in flight must land before the CTA exits
    if (t == 0)
      for (int k = c; k < issued; ++k)
        mbar_wait_drain(smem_u32(&sm.full[k % kStatStages]), (k / kStatStages) & 1, kDrainNs);
    __syncthreads();
  }
  // row-group partials over the (now idle) first stage, summed in order
  float *part_sum = reinterpret_cast<float *>(sm.k[0]);
  float *part_max = reinterpret_cast<float *>(sm.v[0]);
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    part_sum[rg * 128 + 8 * g + cc] = s[cc];
    part_max[rg * 128 + 8 * g + cc] = m[cc];
  }
  __syncthreads();
  if (t < 128) {
    float a = 0.f, b = 0.f;
    for (int r = 0; r < kStatThreads / 16; ++r) {
      a += part_sum[r * 128 + t];
      b = fmaxf(b, part_max[r * 128 + t]);
    }
    sm.cta_sum[t] = a;
    sm.cta_max[t] = b;
  }
  cluster.sync();
  if (rank == 0 && warp == 0) {
    float x[4] = {0.f, 0.f, 0.f, 0.f}, mx[4] = {0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < nc; ++q) {
      const float *ps = cluster.map_shared_rank(sm.cta_sum, q);
      const float *pm = cluster.map_shared_rank(sm.cta_max, q);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        x[cc] += ps[4 * lane + cc];
        mx[cc] = fmaxf(mx[cc], pm[4 * lane + cc]);
      }
    }
    // mean of the raw channels, then rotated: mean(k) H = mean(k H)
    const float n = static_cast<float>(seq);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) x[cc] = __fdiv_rn(x[cc], n);
    fwht128_warp(x, lane);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      k_mean[static_cast<int64_t>(h) * 128 + 4 * lane + cc] = x[cc] * kInvSqrt128;
      v_scales[static_cast<int64_t>(h) * 128 + 4 * lane + cc] = __fdiv_rn(mx[cc], kE4m3Max);
    }
  }
  // the peers' shared memory must outlive rank 0's reads
  cluster.sync();
}

// e4m3 codes of x * r for four values, r = fp32(1/s) (all zero when s == 0).
__device__ __forceinline__ uint32_t encode4(const float (&x)[4], float s, float r) {
  if (!(s > 0.f)) return 0u;
  return pack_e4m3x4(__fmul_rn(x[0], r), __fmul_rn(x[1], r), __fmul_rn(x[2], r), __fmul_rn(x[3], r));
}

// Bytes c of words a, b, e, d (one per token) -> one word per channel c:
// in-lane 4 x 4 byte transpose.
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t e, uint32_t d, uint32_t (&out)[4]) {
  const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
  const uint32_t t2 = __byte_perm(e, d, 0x5140), t3 = __byte_perm(e, d, 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

struct EncSmem {
  uint8_t k[kBlockTok * 256];  // the block's bf16 K rows
  uint8_t v[kBlockTok * 256];  // and V rows
  uint64_t full;
  float warp_amax[kEncThreads / 32];
  int abort;
};

// Pass 2, grid (blocks of 64 tokens, heads), 4 warps.  One bulk copy each
// brings the block's K and V rows (contiguous within the head) into shared
// memory; warp w then takes tokens 16w .. 16w+15, one token at a time across
// the warp (lane l: channels 4l .. 4l+3).
__global__ void __launch_bounds__(kEncThreads)
    encode_kernel(const uint16_t *K, const uint16_t *V, int64_t seq, int64_t v_stride, const float *k_mean,
                  const float *v_scales, uint8_t *k_codes, float *k_scales, uint8_t *v_codes_t, uint32_t *err,
                  uint64_t timeout_ns) {
  __shared__ __align__(128) EncSmem sm;
  const int h = blockIdx.y;
  const int64_t blk = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t blk0 = blk * kBlockTok;
  const int64_t tok0 = blk0 + warp * 16;
  const int64_t nblk = (seq + kBlockTok - 1) / kBlockTok;
  const int64_t base = static_cast<int64_t>(h) * seq;
  const int valid = static_cast<int>(seq - blk0 < kBlockTok ? seq - blk0 : kBlockTok);
  const uint32_t bar = smem_u32(&sm.full);

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    sm.abort = 0;
    fence_mbar_init();
    const uint32_t bytes = static_cast<uint32_t>(valid) * 256u;
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_g2s(smem_u32(sm.k), K + (base + blk0) * 128, bytes, bar);
    bulk_g2s(smem_u32(sm.v), V + (base + blk0) * 128, bytes, bar);
  }
  // per-head constants load while the copies are in flight
  float mu[4], rv[4];
  uint32_t keep = 0u;  // byte mask of the V channels with a nonzero scale
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    mu[c] = k_mean[static_cast<int64_t>(h) * 128 + 4 * lane + c];
    const float sv = v_scales[static_cast<int64_t>(h) * 128 + 4 * lane + c];
    rv[c] = sv > 0.f ? __frcp_rn(sv) : 0.f;
    keep |= (sv > 0.f ? 0xFFu : 0u) << (8 * c);
  }
  __syncthreads();
  const WaitCtx wctx{err, &sm.abort, timeout_ns};
  if (!__syncthreads_and(mbar_wait(bar, 0, wctx))) {
    // the copies must land before the CTA exits
    if (threadIdx.x == 0) mbar_wait_drain(bar, 0, kDrainNs);
    return;
  }

  // ---- K: rotate, smooth, block absmax, encode
  float x[16][4];
  float amax = 0.f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int lr = warp * 16 + t;
    if (lr < valid) {
      bf16x4(*reinterpret_cast<const uint2 *>(sm.k + lr * 256 + 8 * lane), x[t]);
      fwht128_warp(x[t], lane);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        // k' rounded to fp32 before the mean is taken off (no fused rounding)
        x[t][c] = __fsub_rn(__fmul_rn(x[t][c], kInvSqrt128), mu[c]);
        amax = fmaxf(amax, fabsf(x[t][c]));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) sm.warp_amax[warp] = amax;
  __syncthreads();
  const float bmax = fmaxf(fmaxf(sm.warp_amax[0], sm.warp_amax[1]), fmaxf(sm.warp_amax[2], sm.warp_amax[3]));
  const float s = __fdiv_rn(bmax, kE4m3Max);
  const float rs = s > 0.f ? __frcp_rn(s) : 0.f;
  if (threadIdx.x == 0) k_scales[static_cast<int64_t>(h) * nblk + blk] = s;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int64_t tok = tok0 + t;
    if (tok < seq) *reinterpret_cast<uint32_t *>(k_codes + (base + tok) * 128 + 4 * lane) = encode4(x[t], s, rs);
  }

  // ---- V: per-channel scales, encode, write transposed
  uint32_t w[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int lr = warp * 16 + t;
    w[t] = 0u;
    if (lr < valid) {
      float v[4];
      bf16x4(*reinterpret_cast<const uint2 *>(sm.v + lr * 256 + 8 * lane), v);
      w[t] = pack_e4m3x4(__fmul_rn(v[0], rv[0]), __fmul_rn(v[1], rv[1]), __fmul_rn(v[2], rv[2]),
                         __fmul_rn(v[3], rv[3])) & keep;
    }
  }
  // 16 tokens x 4 channels -> 4 channel rows of 16 bytes; padding tokens
  // (past seq, inside v_stride) are written as zero codes
  if (tok0 < v_stride) {
    uint32_t col[4][4];  // [channel][token group of 4]
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t o[4];
      transpose4x4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3], o);
#pragma unroll
      for (int c = 0; c < 4; ++c) col[c][g] = o[c];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint8_t *dst = v_codes_t + (static_cast<int64_t>(h) * 128 + 4 * lane + c) * v_stride + tok0;
      *reinterpret_cast<uint4 *>(dst) = make_uint4(col[c][0], col[c][1], col[c][2], col[c][3]);
    }
  }
}

}  // namespace f8store

cudaError_t launch_store_build_f8(const uint16_t *K, const uint16_t *V, int32_t heads, int64_t seq, int64_t v_stride,
                                  uint8_t *k_codes, uint8_t *v_codes_t, float *k_scales, float *v_scales,
                                  float *k_mean, uint32_t *err, uint64_t timeout_ns, cudaStream_t stream) {
  if (heads <= 0 || seq <= 0) return cudaSuccess;
  // statistics: one 16-CTA cluster per head (a non-portable size), else 8
  cudaError_t e = cudaFuncSetAttribute(f8store::stats_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(f8store::stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(f8store::kStatSmemBytes));
  if (e != cudaSuccess) return e;
  for (int nc = f8store::kStatCtas; nc >= 8; nc /= 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nc), static_cast<unsigned>(heads));
    cfg.blockDim = dim3(f8store::kStatThreads);
    cfg.dynamicSmemBytes = f8store::kStatSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(nc);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (nc > 8 && (cudaOccupancyMaxActiveClusters(&clusters, f8store::stats_kernel, &cfg) != cudaSuccess ||
                   clusters < 1)) {
      cudaGetLastError();  // clear: fall back to the portable size
      continue;
    }
    e = cudaLaunchKernelEx(&cfg, f8store::stats_kernel, K, V, seq, k_mean, v_scales, err, timeout_ns);
    break;
  }
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nblk = (seq + f8store::kBlockTok - 1) / f8store::kBlockTok;
  f8store::encode_kernel<<<dim3(static_cast<unsigned>(nblk), static_cast<unsigned>(heads)), f8store::kEncThreads, 0,
                           stream>>>(K, V, seq, v_stride, k_mean, v_scales, k_codes, k_scales, v_codes_t, err,
                                     timeout_ns);
  return cudaGetLastError();
}

}  // namespace h3kv
