// store_fp4.cu -- the kvfp4 store build (kv_store row of the H3 Streamed
// Blocks Inputs table, kvfp4s: K/V as NVFP4 -- e2m1 values with one e4m3
// scale per 16 elements -- with Q and K Hadamard-rotated): every (token,
// head) row of K is rotated by the fixed orthonormal 128-wide Hadamard basis,
// V is not; each 16-value block of a row gets s = e4m3(max|x| / 6) and the
// codes e2m1(x / s), all zero where s == 0.
//
// GB300 design: the HBM-bound stream of the kvi8r build.  A persistent grid
// (two CTAs per SM) walks 128-row tiles (K tiles, then V tiles); one producer
// warp streams bf16 tiles into a 3-stage ring with TMA (128-byte swizzle), and
// eight compute warps give every row two threads, one per 64-value half (four
// 16-value blocks).  Each thread stores its half row's 32 code bytes (one
// 32-byte store when the code buffers are 32-byte aligned, else two 16-byte
// ones) and 4 scale bytes straight from registers.
#include "kernels.h"
#include "ptx.cuh"
#include "store_fwht.cuh"

namespace h3kv {
namespace {

constexpr int kRows = 128;                  // rows per tile
constexpr int kCompute = 2 * kRows;         // two compute threads per row
constexpr int kStages = 3;                  // input ring depth (2 CTAs per SM)
constexpr int kInTileBytes = kRows * 256;   // bf16 [128 x 128]
constexpr int kThreads = kCompute + 32;     // 8 compute warps + 1 producer warp
constexpr int kProducerWarp = kCompute / 32;

struct Fp4BuildSmem {
  uint8_t in[kStages][kInTileBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
};

constexpr size_t kFp4BuildSmemBytes = sizeof(Fp4BuildSmem) + 1024;

// x / d given r ~ 1/d (within 2 ulp): q0 = x r corrected once by its exact
// residual (Markstein's division step: e = q0 d - x by one fma, then
// q0 - e r).  For an exactly representable quotient t, q0 is within a few
// ulp of t, the residual e is exact, and q0 - e r = t - (q0 - t)(r d - 1)
// rounds to t; such quotients -- the only kind that can sit on a rounding
// midpoint of e2m1 or e4m3 here -- come out exact, so the nearest-even
// decision that follows is the one for x / d itself.  A zero keeps its sign.
__device__ __forceinline__ float div_step(float x, float d, float r) {
  const float q0 = x * r;
  const float e = fmaf(q0, d, -x);
  return fmaf(e, -r, q0);
}

// Reciprocal to within one ulp (the hardware approximation); s here is a
// normal fp32 number (an e4m3 scale, at least 2^-9).
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Codes of one 16-value block x[0..15] with scale s > 0 (r ~ 1/s): e2m1 of
// x / s.  Returns the 16 nibbles in two words, element 0 lowest.
__device__ __forceinline__ uint2 encode_block(const float *x, float s, float r) {
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = div_step(x[i], s, r);
  uint2 w;
  w.x = pack_e2m1x4(q[0], q[1], q[2], q[3]) | (pack_e2m1x4(q[4], q[5], q[6], q[7]) << 16);
  w.y = pack_e2m1x4(q[8], q[9], q[10], q[11]) | (pack_e2m1x4(q[12], q[13], q[14], q[15]) << 16);
  return w;
}

template <bool kWide>
__global__ void __launch_bounds__(kThreads, 2)
    store_fp4_kernel(const __grid_constant__ CUtensorMap tm_k_in, const __grid_constant__ CUtensorMap tm_v_in,
                     uint8_t *__restrict__ k_codes, uint8_t *__restrict__ v_codes,
                     uint8_t *__restrict__ k_scales, uint8_t *__restrict__ v_scales, int64_t rows,
                     int64_t tiles_per_tensor, uint32_t *err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  Fp4BuildSmem &sm =
      *reinterpret_cast<Fp4BuildSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t total_tiles = 2 * tiles_per_tensor;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kCompute);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtx wctx{err, &sm.abort, timeout_ns};

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_k_in);
      prefetch_tmap(&tm_v_in);
      int it = 0;
      int issued = 0;
      for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1, wctx)) break;
        const bool is_v = t >= tiles_per_tensor;
        const int32_t row0 = static_cast<int32_t>((is_v ? t - tiles_per_tensor : t) * kRows);
        const CUtensorMap *map = is_v ? &tm_v_in : &tm_k_in;
        const uint32_t bar = smem_u32(&sm.full[s]);
        mbar_arrive_expect_tx(bar, kInTileBytes);
        tma_load_2d(smem_u32(&sm.in[s][0]), map, 0, row0, bar);
        tma_load_2d(smem_u32(&sm.in[s][kInTileBytes / 2]), map, 64, row0, bar);
        ++issued;
      }
      if (sm.abort) {
        for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
          mbar_wait_drain(smem_u32(&sm.full[k % kStages]), (k / kStages) & 1, kDrainNs);
      }
    }
  } else {
    // ----------------------------------------------------------- compute
    // Threads 2r and 2r + 1 share row r: thread h takes values 64h .. 64h + 63
    // (blocks 4h .. 4h + 3).  For K, H128 = [[H64, H64], [H64, -H64]], so
    // half h of the rotated row is H64 applied to x_lo + x_hi (h = 0) or
    // x_lo - x_hi (h = 1); V is taken as it is.
    const uint32_t r = static_cast<uint32_t>(tid) >> 1;  // row within tile
    const int h = tid & 1;
    const float sg = h ? -1.f : 1.f;
    int it = 0;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      const int s = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      // each warp decides for itself (a warp whose wait gave up leaves; the
      // others see the abort flag at their next wait, and the producer's wait
      // for the stage's release runs out)
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.full[s]), ph, wctx))) break;

      const bool is_v = t >= tiles_per_tensor;
      float x[64];
      const uint8_t *tile = sm.in[s];
      if (!is_v) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 a = *reinterpret_cast<const uint4 *>(tile + sw128_off(r, g));
          const uint4 b = *reinterpret_cast<const uint4 *>(tile + kInTileBytes / 2 + sw128_off(r, g));
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 lo = make_float2(bf16lo_to_f32(aw[k]), bf16hi_to_f32(aw[k]));
            const float2 hi = make_float2(bf16lo_to_f32(bw[k]), bf16hi_to_f32(bw[k]));
            const float2 u = __ffma2_rn(hi, make_float2(sg, sg), lo);
            x[g * 8 + 2 * k] = u.x;
            x[g * 8 + 2 * k + 1] = u.y;
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 v = *reinterpret_cast<const uint4 *>(tile + h * (kInTileBytes / 2) + sw128_off(r, g));
          x[g * 8 + 0] = bf16lo_to_f32(v.x);
          x[g * 8 + 1] = bf16hi_to_f32(v.x);
          x[g * 8 + 2] = bf16lo_to_f32(v.y);
          x[g * 8 + 3] = bf16hi_to_f32(v.y);
          x[g * 8 + 4] = bf16lo_to_f32(v.z);
          x[g * 8 + 5] = bf16hi_to_f32(v.z);
          x[g * 8 + 6] = bf16lo_to_f32(v.w);
          x[g * 8 + 7] = bf16hi_to_f32(v.w);
        }
      }
      mbar_arrive(smem_u32(&sm.empty[s]));

      if (!is_v) {
        // k' = k H: the unnormalised transform, then 2^-3.5
        fwht64_packed(x);
        const float2 inv = make_float2(kInvSqrt128, kInvSqrt128);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float2 p = __fmul2_rn(make_float2(x[e], x[e + 1]), inv);
          x[e] = p.x;
          x[e + 1] = p.y;
        }
      }

      const int64_t row0 = (is_v ? t - tiles_per_tensor : t) * kRows;
      const bool row_ok = row0 + r < rows;
      uint8_t *oc = (is_v ? v_codes : k_codes) + (row_ok ? row0 + r : 0) * 64 + 32 * h;
      uint32_t sw = 0u;
      uint32_t wp[8];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        // local blocks 2c and 2c + 1 fill 16-byte chunk c of this half's 32 code bytes
        uint2 w[2];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int blk = 2 * c + hb;
          const float *xb = x + blk * 16;
          float am[2] = {0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            am[0] = fmax3(am[0], fabsf(xb[i]), fabsf(xb[i + 1]));
            am[1] = fmax3(am[1], fabsf(xb[i + 2]), fabsf(xb[i + 3]));
          }
          constexpr float kRcp6 = 0.16666667163372040f;  // 1/6 rounded to fp32
          const uint32_t sb = f32_to_e4m3(div_step(fmaxf(am[0], am[1]), 6.0f, kRcp6));
          const float sf = __half2float(__ushort_as_half(static_cast<uint16_t>(e4m3_to_f16x2_dup(sb))));
          sw |= sb << (blk * 8);
          w[hb] = encode_block(xb, sf, sf > 0.f ? rcp_approx(sf) : 0.f);
          if (!(sf > 0.f)) w[hb] = make_uint2(0u, 0u);
        }
        wp[c * 4 + 0] = w[0].x;
        wp[c * 4 + 1] = w[0].y;
        wp[c * 4 + 2] = w[1].x;
        wp[c * 4 + 3] = w[1].y;
      }
      if (row_ok) {
        if constexpr (kWide) {
          st_global_v8(oc, wp);
        } else {
          *reinterpret_cast<uint4 *>(oc) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
          *reinterpret_cast<uint4 *>(oc + 16) = make_uint4(wp[4], wp[5], wp[6], wp[7]);
        }
        uint8_t *scales = is_v ? v_scales : k_scales;
        *reinterpret_cast<uint32_t *>(scales + (row0 + r) * 8 + 4 * h) = sw;
      }
    }
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_store_build_fp4(const CUtensorMap &k_in, const CUtensorMap &v_in, uint8_t *k_out,
                                   uint8_t *v_out, uint8_t *k_scales, uint8_t *v_scales, int64_t rows,
                                   int num_sms, uint32_t *err, uint64_t timeout_ns, cudaStream_t stream) {
  const int64_t tiles = (rows + kRows - 1) / kRows;
  if (tiles == 0) return cudaSuccess;
  // whole-sector stores: device code buffers aligned to 32 bytes (rows are
  // multiples of 32 bytes, so every row's pairs of 16-byte pieces are too)
  const bool wide = wide_store_ok(k_out, v_out);
  auto kernel = wide ? store_fp4_kernel<true> : store_fp4_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kFp4BuildSmemBytes));
  if (e != cudaSuccess) return e;
  int64_t grid = static_cast<int64_t>(num_sms) * 2;
  if (grid > 2 * tiles) grid = 2 * tiles;
  kernel<<<static_cast<unsigned>(grid), kThreads, kFp4BuildSmemBytes, stream>>>(
      k_in, v_in, k_out, v_out, k_scales, v_scales, rows, tiles, err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace h3kv
