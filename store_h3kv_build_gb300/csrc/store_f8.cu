// store_f8.cu -- the kvf8s store build: K and V as fp8 e4m3 in the kvi8s
// layout ("The K/V store options" table of the Low VRAM write-up, kvi8s row;
// kv_store row of the H3 Streamed Blocks Inputs table), with fp8 K in place
// of int8 so that both products run on the fp8 tensor path.
//
//   K: k' = k H (the 128-wide Hadamard basis), smoothed by mu = the mean of
//      k' over all tokens of the head, one fp32 scale per 64-token block
//      s = absmax / 448, codes e4m3(x / s), formed as x * fp32(1/s).
//   V: not rotated; one fp32 scale per (head, channel) s = absmax over all
//      tokens / 448, codes e4m3(v / s) with the quotient rounded once,
//      exactly (e4m3_quotient2 below), stored channel-major [heads, 128,
//      v_stride] (V transposed) so that P.V reads it K-major.
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

// The fp32 value whose e4m3 rounding (cvt.rn.satfinite) is the code of the
// quotient v / s rounded once, exactly, to the nearest e4m3 value (ties to
// the even code), given r = fp32(1/s) and r16 = r * 2^16, for two values at
// once (packed products and fmas; the bit tests per value).  t = fp32(v * r).
// t lies within two fp32 ulps of the quotient, so the two round differently
// only when an e4m3 rounding boundary -- the midpoint m of two neighbouring
// e4m3 values -- lies that close to t.  bf16 values over an fp32 scale land
// there often (about 1e-3 of N(0, 1) codes), so every such case is decided
// by the sign of |v| - m s: m has at most five significant bits and s 24, so
// the fma's single rounding keeps the sign of the exact difference.
//  - |t| >= 2^-6 (e4m3 normal range): the boundary inside t's cell is |t|
//    with its 20 low mantissa bits set to 0x80000.
//  - |t| < 2^-6 (e4m3 subnormals, spacing 2^-9): u = |t| + 2^-6 lies in the
//    binade [2^-6, 2^-5), whose e4m3 cells are 2^-9 wide as well, so the
//    same bits of u give the boundary m + 2^-6.
// Near a boundary the returned magnitude m + (|v| - m s) r16 sits on the
// quotient's side of m, at least one fp32 ulp and at most a quarter of the
// e4m3 spacing away -- or is m itself on an exact tie, which the conversion
// rounds to the even code; signs are carried through (m takes t's sign).  No
// branch: every value takes the same steps (branches measured 40 % slower).
// The procedure was checked against exact rational rounding of the quotient
// on 5e7 bf16 values before it ran on a GPU.
__device__ __forceinline__ float2 e4m3_quotient2(float2 v, float2 s, float2 r, float2 r16) {
  const float2 t = __fmul2_rn(v, r);
  float2 m;
  bool near[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float tk = k ? t.y : t.x;
    const float at = fabsf(tk);
    const bool sub = at < 0x1p-6f;
    const uint32_t ub = __float_as_uint(sub ? at + 0x1p-6f : at);
    const float mu = __uint_as_float((ub & 0xFFF00000u) | 0x00080000u);
    const float mk = copysignf(sub ? mu - 0x1p-6f : mu, tk);
    near[k] = ((ub & 0xFFFFFu) - 0x7FFFDu) < 7u;
    if (k) m.y = mk;
    else m.x = mk;
  }
  const float2 tn = __ffma2_rn(__ffma2_rn(make_float2(-m.x, -m.y), s, v), r16, m);
  return make_float2(near[0] ? tn.x : t.x, near[1] ? tn.y : t.y);
}

constexpr int kEncRows = 128;                  // tokens per tile = compute threads
constexpr int kEncStages = 3;                  // input ring depth (2 CTAs per SM)
constexpr int kEncTileBytes = kEncRows * 256;  // bf16 [128 tokens x 128 channels]
constexpr int kEncThreads = kEncRows + 32;     // 4 compute warps + 1 producer warp

struct EncSmem {
  uint8_t in[kEncStages][kEncTileBytes];  // 1024-byte aligned (128-byte swizzle)
  float neg_mu[128];   // -mean(k') of the current head
  float rv[128];       // fp32(1 / s_v) per V channel, 0 where s_v = 0
  float sv[128];       // s_v per V channel
  float rv16[128];     // fp32(1 / s_v) * 2^16
  uint32_t keep[32];   // byte mask of the V channels with s_v > 0
  float warp_amax[4];  // K: per-warp absmax (warps 0-1: first 64 tokens of the tile)
  uint64_t full[kEncStages];
  uint64_t empty[kEncStages];
  int abort;
};
constexpr size_t kEncSmemBytes = sizeof(EncSmem) + 1024;

// Byte offset, inside a V tile's code staging area (the first 16 KB of the
// drained input stage), of 16-byte granule g (channels 16g .. 16g+15) of
// token row r.  The XOR pattern keeps the row writes (8 consecutive rows
// per quarter-warp) and the column reads below (one 4-byte word of 32
// rows r = 32 tq + k, k fixed per instruction) free of bank conflicts.
__device__ __forceinline__ uint32_t vstage_off(uint32_t r, uint32_t g) {
  return r * 128u + ((g ^ (r & 7u) ^ (2u * ((r >> 5) & 3u))) << 4);
}

// Pass 2, a persistent grid (two CTAs per SM) over tiles of 128 tokens of
// one head, K and V tiles of the same tokens interleaved (tile u: token
// chunk u / 2, V when u is odd); CTA b takes the contiguous tile range
// [b n / grid, (b + 1) n / grid), so its head (and the per-head constants
// held in shared memory) changes at most a few times.  One producer warp
// fills a 3-stage ring with TMA (two 64-channel boxes per tile); the four
// compute warps hold one token row per thread.
//   K tile: the 128-point FWHT in registers (stage order stride 1 .. 64),
//     k' = fp32(x / sqrt 128) - mu rounded to fp32, the absmax of each
//     64-token block by a warp reduction and one 128-thread barrier, then
//     the row's codes straight to global memory.
//   V tile: the row's codes e4m3(v / s_v) are written back into the
//     drained stage, then each thread reads four channels of 32 tokens,
//     transposes them in registers and stores 32-token pieces of four
//     channel rows of the transposed V.
// Tokens past seq arrive as zero rows (the 3-D map fills them): they give
// zero V codes, which is what the transposed rows up to v_stride hold, and
// are left out of the K absmax and stores.  kWide: 32-byte code stores.
template <bool kWide>
__global__ void __launch_bounds__(kEncThreads, 2)
    encode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, int32_t heads,
                  int64_t seq, int64_t v_stride, const float *__restrict__ k_mean,
                  const float *__restrict__ v_scales, uint8_t *__restrict__ k_codes, float *__restrict__ k_scales,
                  uint8_t *__restrict__ v_codes_t, uint32_t *err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  EncSmem &sm = *reinterpret_cast<EncSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nch = (seq + kEncRows - 1) / kEncRows;    // token chunks per head
  const int64_t nblk = (seq + kBlockTok - 1) / kBlockTok;  // K scale blocks per head
  const int64_t n_tiles = 2 * static_cast<int64_t>(heads) * nch;
  const int64_t u_begin = n_tiles * blockIdx.x / gridDim.x;
  const int64_t u_end = n_tiles * (blockIdx.x + 1) / gridDim.x;

  if (tid == 0) {
    for (int st = 0; st < kEncStages; ++st) {
      mbar_init(smem_u32(&sm.full[st]), 1);
      mbar_init(smem_u32(&sm.empty[st]), kEncRows);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wctx{err, &sm.abort, timeout_ns};

  if (warp == 4) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      int it = 0, issued = 0;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int st = it % kEncStages;
        if (!mbar_wait(smem_u32(&sm.empty[st]), ((it / kEncStages) & 1) ^ 1, wctx)) break;
        const int64_t idx = u >> 1;
        const int32_t h = static_cast<int32_t>(idx / nch);
        const int32_t tok0 = static_cast<int32_t>((idx - static_cast<int64_t>(h) * nch) * kEncRows);
        const CUtensorMap *map = (u & 1) ? &tm_v : &tm_k;
        const uint32_t bar = smem_u32(&sm.full[st]);
        mbar_arrive_expect_tx(bar, kEncTileBytes);
        tma_load_3d(smem_u32(sm.in[st]), map, 0, tok0, h, bar);
        tma_load_3d(smem_u32(sm.in[st] + kEncTileBytes / 2), map, 64, tok0, h, bar);
        ++issued;
      }
      if (sm.abort) {
        // drain: every issued load must land before the CTA may exit
        for (int k = (issued > kEncStages ? issued - kEncStages : 0); k < issued; ++k)
          mbar_wait_drain(smem_u32(&sm.full[k % kEncStages]), (k / kEncStages) & 1, kDrainNs);
      }
    }
  } else {
    // ----------------------------------------------------------- compute
    const uint32_t r = static_cast<uint32_t>(tid);  // token row within the tile
    // transposed V read-back: channels 4 cg .. 4 cg + 3 of tokens 32 tq .. 32 tq + 31
    const uint32_t cg = r >> 2, tq = r & 3;
    const uint32_t rd_base = tq * 32u * 128u + (cg & 3u) * 4u;
    const uint32_t rd_gx = (cg >> 2) ^ (2u * tq);
    int64_t cur_h = -1;
    int it = 0;
    for (int64_t u = u_begin; u < u_end; ++u, ++it) {
      const int st = it % kEncStages;
      const bool is_v = (u & 1) != 0;
      const int64_t idx = u >> 1;
      const int64_t h = idx / nch;
      const int64_t c = idx - h * nch;
      const int64_t tok0 = c * kEncRows;
      const int valid = static_cast<int>(seq - tok0 < kEncRows ? seq - tok0 : kEncRows);
      if (h != cur_h) {
        // the head's constants, once every thread is done with the last head's
        const float mu = k_mean[h * 128 + r];
        const float sv = v_scales[h * 128 + r];
        named_bar_sync(1, kEncRows);
        sm.neg_mu[r] = -mu;
        sm.rv[r] = sv > 0.f ? __frcp_rn(sv) : 0.f;
        sm.sv[r] = sv;
        sm.rv16[r] = sm.rv[r] * 65536.f;
        reinterpret_cast<uint8_t *>(sm.keep)[r] = sv > 0.f ? 0xFFu : 0u;
        named_bar_sync(1, kEncRows);
        cur_h = h;
      }
      // every compute thread takes the same decision (a wait that gave up on
      // one thread stops all of them together)
      const bool ok = mbar_wait(smem_u32(&sm.full[st]), (it / kEncStages) & 1, wctx);
      if (!named_bar_and(1, kEncRows, ok)) break;
      uint8_t *tile = sm.in[st];

      if (!is_v) {
        float x[128];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 w = *reinterpret_cast<const uint4 *>(tile + hc * (kEncTileBytes / 2) + sw128_off(r, g));
            const int e = hc * 64 + g * 8;
            x[e + 0] = bf16lo_to_f32(w.x);
            x[e + 1] = bf16hi_to_f32(w.x);
            x[e + 2] = bf16lo_to_f32(w.y);
            x[e + 3] = bf16hi_to_f32(w.y);
            x[e + 4] = bf16lo_to_f32(w.z);
            x[e + 5] = bf16hi_to_f32(w.z);
            x[e + 6] = bf16lo_to_f32(w.w);
            x[e + 7] = bf16hi_to_f32(w.w);
          }
        }
        mbar_arrive(smem_u32(&sm.empty[st]));
        fwht128_packed(x);  // x = sqrt(128) * (row H)
        // k' = x / sqrt(128) rounded to fp32, then the mean taken off: two
        // scalar roundings (__fmul_rn / __fadd_rn are never contracted into
        // an fma; a packed multiply followed by a packed add was, which left
        // the product's rounding error in k' - mu)
        float am[2] = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 128; e += 4) {
          const float4 nm = *reinterpret_cast<const float4 *>(&sm.neg_mu[e]);
          x[e] = __fadd_rn(__fmul_rn(x[e], kInvSqrt128), nm.x);
          x[e + 1] = __fadd_rn(__fmul_rn(x[e + 1], kInvSqrt128), nm.y);
          x[e + 2] = __fadd_rn(__fmul_rn(x[e + 2], kInvSqrt128), nm.z);
          x[e + 3] = __fadd_rn(__fmul_rn(x[e + 3], kInvSqrt128), nm.w);
          am[0] = fmax3(am[0], fabsf(x[e]), fabsf(x[e + 1]));
          am[1] = fmax3(am[1], fabsf(x[e + 2]), fabsf(x[e + 3]));
        }
        float amax = static_cast<int>(r) < valid ? fmaxf(am[0], am[1]) : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) sm.warp_amax[warp] = amax;
        named_bar_sync(1, kEncRows);
        // block of 64 tokens: warps 0-1 or 2-3 (a warp never straddles two)
        const float bmax = fmaxf(sm.warp_amax[warp & ~1], sm.warp_amax[warp | 1]);
        const float s = __fdiv_rn(bmax, kE4m3Max);
        const float rs = s > 0.f ? __frcp_rn(s) : 0.f;
        if (static_cast<int>(r) < valid) {
          if ((r & 63u) == 0u) k_scales[h * nblk + 2 * c + (r >> 6)] = s;
          uint8_t *dst = k_codes + (h * seq + tok0 + r) * 128;
          const float2 rs2 = make_float2(rs, rs);
          uint32_t wp[8];  // granules g - 1 and g, stored together when kWide
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = g * 16 + k * 4;
              const float2 a = __fmul2_rn(make_float2(x[e], x[e + 1]), rs2);
              const float2 b = __fmul2_rn(make_float2(x[e + 2], x[e + 3]), rs2);
              // a block whose scale is 0 (or not a number) gets zero codes
              w[k] = s > 0.f ? pack_e4m3x4(a.x, a.y, b.x, b.y) : 0u;
            }
            if constexpr (kWide) {
#pragma unroll
              for (int k = 0; k < 4; ++k) wp[(g & 1) * 4 + k] = w[k];
              if (g & 1) st_global_v8(dst + (g - 1) * 16, wp);
            } else {
              *reinterpret_cast<uint4 *>(dst + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else {
        // codes of the row, 16 channels (one input granule pair) at a time
        uint32_t w[32];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int gi = 2 * g + hf;  // input granule: channels 8 gi .. 8 gi + 7
            const uint4 in =
                *reinterpret_cast<const uint4 *>(tile + (gi >> 3) * (kEncTileBytes / 2) + sw128_off(r, gi & 7));
            const float4 r0 = *reinterpret_cast<const float4 *>(&sm.rv[8 * gi]);
            const float4 r1 = *reinterpret_cast<const float4 *>(&sm.rv[8 * gi + 4]);
            const float4 s0 = *reinterpret_cast<const float4 *>(&sm.sv[8 * gi]);
            const float4 s1 = *reinterpret_cast<const float4 *>(&sm.sv[8 * gi + 4]);
            const float4 q0 = *reinterpret_cast<const float4 *>(&sm.rv16[8 * gi]);
            const float4 q1 = *reinterpret_cast<const float4 *>(&sm.rv16[8 * gi + 4]);
            const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
            const float r16[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            float v[8], t[8];
            bf16x4(make_uint2(in.x, in.y), *reinterpret_cast<float(*)[4]>(v));
            bf16x4(make_uint2(in.z, in.w), *reinterpret_cast<float(*)[4]>(v + 4));
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
              const float2 q = e4m3_quotient2(make_float2(v[k], v[k + 1]), make_float2(ss[k], ss[k + 1]),
                                              make_float2(rr[k], rr[k + 1]), make_float2(r16[k], r16[k + 1]));
              t[k] = q.x;
              t[k + 1] = q.y;
            }
            w[2 * gi] = pack_e4m3x4(t[0], t[1], t[2], t[3]);
            w[2 * gi + 1] = pack_e4m3x4(t[4], t[5], t[6], t[7]);
          }
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 kp = *reinterpret_cast<const uint4 *>(&sm.keep[4 * g]);
          w[4 * g] &= kp.x;
          w[4 * g + 1] &= kp.y;
          w[4 * g + 2] &= kp.z;
          w[4 * g + 3] &= kp.w;
        }
        named_bar_sync(1, kEncRows);  // every row of the stage has been read
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<uint4 *>(tile + vstage_off(r, g)) =
              make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
        named_bar_sync(1, kEncRows);  // the staged codes are complete
        uint32_t col[4][8];  // [channel][group of 4 tokens]
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t t4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t k = 4u * j + i;  // token 32 tq + k; (32 tq + k) & 7 = k & 7
            t4[i] = *reinterpret_cast<const uint32_t *>(tile + rd_base + k * 128u + ((rd_gx ^ (k & 7u)) << 4));
          }
          uint32_t o[4];
          transpose4x4(t4[0], t4[1], t4[2], t4[3], o);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) col[cc][j] = o[cc];
        }
        // the stage goes back to the TMA (async proxy) after these generic writes
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&sm.empty[st]));
        // tokens tok0 + 32 tq .. + 31; v_stride is a multiple of 16, so a
        // piece is whole, half (the last 16 tokens of the padded row) or past it
        const int64_t t_first = tok0 + 32 * static_cast<int64_t>(tq);
        const int64_t rem = v_stride - t_first;
        if (rem > 0) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint8_t *dst = v_codes_t + (h * 128 + 4 * cg + cc) * v_stride + t_first;
            if (rem >= 32) {
              if constexpr (kWide) {
                st_global_v8(dst, col[cc]);
              } else {
                *reinterpret_cast<uint4 *>(dst) = make_uint4(col[cc][0], col[cc][1], col[cc][2], col[cc][3]);
                *reinterpret_cast<uint4 *>(dst + 16) = make_uint4(col[cc][4], col[cc][5], col[cc][6], col[cc][7]);
              }
            } else {
              *reinterpret_cast<uint4 *>(dst) = make_uint4(col[cc][0], col[cc][1], col[cc][2], col[cc][3]);
            }
          }
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace f8store

cudaError_t launch_store_build_f8(const CUtensorMap &k_in, const CUtensorMap &v_in, const uint16_t *K,
                                  const uint16_t *V, int32_t heads, int64_t seq, int64_t v_stride, uint8_t *k_codes,
                                  uint8_t *v_codes_t, float *k_scales, float *v_scales, float *k_mean, int num_sms,
                                  uint32_t *err, uint64_t timeout_ns, cudaStream_t stream) {
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
  // whole-sector stores: device code buffers aligned to 32 bytes and V rows
  // of a multiple of 32 bytes
  const bool wide = wide_store_ok(k_codes, v_codes_t) && v_stride % 32 == 0;
  auto kernel = wide ? f8store::encode_kernel<true> : f8store::encode_kernel<false>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(f8store::kEncSmemBytes));
  if (e != cudaSuccess) return e;
  const int64_t n_tiles = 2 * static_cast<int64_t>(heads) * ((seq + f8store::kEncRows - 1) / f8store::kEncRows);
  int64_t grid = 2 * static_cast<int64_t>(num_sms);
  if (grid > n_tiles) grid = n_tiles;
  kernel<<<static_cast<unsigned>(grid), f8store::kEncThreads, f8store::kEncSmemBytes, stream>>>(
      k_in, v_in, heads, seq, v_stride, k_mean, v_scales, k_codes, k_scales, v_codes_t, err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace h3kv
