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
constexpr int kStatUnroll = 4;    // row pairs per warp in flight
constexpr int kStatWarps = kStatThreads / 32;
constexpr int kBlockTok = 64;     // tokens per K scale block
constexpr int kEncThreads = 128;  // 4 warps x 16 tokens = one block
constexpr float kE4m3Max = 448.0f;

__device__ __forceinline__ void bf16x4(const uint2 w, float (&x)[4]) {
  x[0] = bf16lo_to_f32(w.x);
  x[1] = bf16hi_to_f32(w.x);
  x[2] = bf16lo_to_f32(w.y);
  x[3] = bf16hi_to_f32(w.y);
}

// Pass 1, grid (cluster size, heads), one cluster per head.  CTA r of n sums
// the tokens [r * per, (r + 1) * per), per = ceil(seq / n).  Each warp reads two rows per load
// (half-warp = row, lane = 8 channels, 16-byte loads), kStatUnroll pairs at
// a time, stepping over the range by the CTA's warps.  Partials are combined
// half-warp, warp, then CTA by CTA through distributed shared memory, always
// in index order, so the result does not depend on timing.
__global__ void __launch_bounds__(kStatThreads)
    stats_kernel(const uint16_t *K, const uint16_t *V, int64_t seq, float *k_mean, float *v_scales) {
  __shared__ float part_sum[kStatWarps][128];
  __shared__ float part_max[kStatWarps][128];
  __shared__ float cta_sum[128];
  __shared__ float cta_max[128];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int nc = static_cast<int>(cluster.num_blocks());
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const int64_t per = (seq + nc - 1) / nc;
  const int64_t r0 = rank * per;
  const int64_t r1 = r0 + per < seq ? r0 + per : seq;
  const uint16_t *kh = K + static_cast<int64_t>(h) * seq * 128 + 8 * l16;
  const uint16_t *vh = V + static_cast<int64_t>(h) * seq * 128 + 8 * l16;
  float s[8], m[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) s[c] = m[c] = 0.f;
  constexpr int64_t kStep = 2 * kStatWarps;  // rows per sweep of the CTA
  for (int64_t base = r0 + 2 * warp + half; base < r1; base += kStep * kStatUnroll) {
    uint4 kw[kStatUnroll], vw[kStatUnroll];
#pragma unroll
    for (int u = 0; u < kStatUnroll; ++u) {
      const int64_t r = base + u * kStep;
      kw[u] = r < r1 ? *reinterpret_cast<const uint4 *>(kh + r * 128) : make_uint4(0u, 0u, 0u, 0u);
      vw[u] = r < r1 ? *reinterpret_cast<const uint4 *>(vh + r * 128) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kStatUnroll; ++u) {
      const uint32_t kk[4] = {kw[u].x, kw[u].y, kw[u].z, kw[u].w};
      const uint32_t vv[4] = {vw[u].x, vw[u].y, vw[u].z, vw[u].w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        s[2 * p] += bf16lo_to_f32(kk[p]);
        s[2 * p + 1] += bf16hi_to_f32(kk[p]);
        m[2 * p] = fmaxf(m[2 * p], fabsf(bf16lo_to_f32(vv[p])));
        m[2 * p + 1] = fmaxf(m[2 * p + 1], fabsf(bf16hi_to_f32(vv[p])));
      }
    }
  }
  // the two half-warps hold the same channels: add the upper into the lower
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float os = __shfl_down_sync(0xffffffffu, s[c], 16);
    const float om = __shfl_down_sync(0xffffffffu, m[c], 16);
    s[c] += os;
    m[c] = fmaxf(m[c], om);
  }
  if (half == 0) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      part_sum[warp][8 * l16 + c] = s[c];
      part_max[warp][8 * l16 + c] = m[c];
    }
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    float a = 0.f, b = 0.f;
    for (int w = 0; w < kStatWarps; ++w) {
      a += part_sum[w][threadIdx.x];
      b = fmaxf(b, part_max[w][threadIdx.x]);
    }
    cta_sum[threadIdx.x] = a;
    cta_max[threadIdx.x] = b;
  }
  cluster.sync();
  if (rank == 0 && warp == 0) {
    float x[4] = {0.f, 0.f, 0.f, 0.f}, mx[4] = {0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < nc; ++q) {
      const float *ps = cluster.map_shared_rank(cta_sum, q);
      const float *pm = cluster.map_shared_rank(cta_max, q);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        x[c] += ps[4 * lane + c];
        mx[c] = fmaxf(mx[c], pm[4 * lane + c]);
      }
    }
    // mean of the raw channels, then rotated: mean(k) H = mean(k H)
    const float n = static_cast<float>(seq);
#pragma unroll
    for (int c = 0; c < 4; ++c) x[c] = __fdiv_rn(x[c], n);
    fwht128_warp(x, lane);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      k_mean[static_cast<int64_t>(h) * 128 + 4 * lane + c] = x[c] * kInvSqrt128;
      v_scales[static_cast<int64_t>(h) * 128 + 4 * lane + c] = __fdiv_rn(mx[c], kE4m3Max);
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
  for (int nc = f8store::kStatCtas; nc >= 8; nc /= 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nc), static_cast<unsigned>(heads));
    cfg.blockDim = dim3(f8store::kStatThreads);
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
    e = cudaLaunchKernelEx(&cfg, f8store::stats_kernel, K, V, seq, k_mean, v_scales);
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
