// store_build.cu -- the kvi8r store build (kv_store row of the H3 Streamed
// Blocks Inputs table; kvi8r row of "The K/V store options" table in the Low
// VRAM write-up): every (token, head) row of K and V is rotated by the fixed
// orthonormal 128-wide Hadamard basis, given one fp16 absmax scale and
// quantised to int8.
//
// GB300 design: HBM-bound stream.  Rows are flattened over heads (each row is
// independent).  A persistent grid of CTAs (two per SM) walks 128-row tiles;
// one producer warp streams bf16 tiles into a 3-stage shared-memory ring with
// TMA (128-byte swizzle), and eight compute warps give every row two threads
// (the swizzle makes the per-row shared-memory reads bank-conflict free).
// H128 = [[H64, H64], [H64, -H64]], so each thread forms the sums (or the
// differences) of the row's two 64-value halves and runs a 64-point FWHT in
// registers: 88 registers, 18 warps per SM instead of 10 with one row per
// thread.  Each thread stores its half row's codes (two 32-byte stores when
// the code buffers are 32-byte aligned, else four 16-byte ones); the pair
// shares its absmax with one shuffle.
#include "kernels.h"
#include "ptx.cuh"
#include "store_fwht.cuh"

namespace h3kv {
namespace {

constexpr int kRows = 128;                  // rows per tile
constexpr int kCompute = 2 * kRows;         // two compute threads per row
constexpr int kStages = 3;                  // input ring depth (2 CTAs per SM, 97 KB each)
constexpr int kInTileBytes = kRows * 256;   // bf16 [128 x 128]
constexpr int kThreads = kCompute + 32;     // 8 compute warps + 1 producer warp
constexpr int kProducerWarp = kCompute / 32;

struct BuildSmem {
  // 1024-byte aligned tiles first
  uint8_t in[kStages][kInTileBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
};

constexpr size_t kBuildSmemBytes = sizeof(BuildSmem) + 1024;

// Scale, clamp need and code multiplier of one row (or group of a row) from
// the absmax of its unnormalised FWHT values: s = fp16(absmax(x H) / 127),
// saturated at the largest finite fp16; codes are rne(x' / s) = rne(x * m)
// with m = 1 / (sqrt(128) s).
struct RowScale {
  __half sh;
  bool clamp;
  float m;
};

// x / 127 rounded to nearest: x * RN(1/127) corrected once by its exact
// residual (Markstein's division step).  Checked on the host against IEEE
// division for every non-negative finite fp32 x; infinities and NaN take
// x * RN(1/127), which is what division gives them.  About a third of the
// instructions of the library's correctly rounded division.
__device__ __forceinline__ float div127(float x) {
  constexpr float kRcp127 = 0.007874015718698502f;  // RN(1/127), 0x3C010204
  const float q0 = __fmul_rn(x, kRcp127);
  if (!(x < INFINITY)) return q0;
  const float r = __fmaf_rn(-q0, 127.0f, x);
  return __fmaf_rn(r, kRcp127, q0);
}

// 1 / p rounded to nearest for p = RN(s * sqrt(128)), s a positive finite
// fp16 scale: the hardware's approximate reciprocal refined by one fma step.
// Checked on the host for every such p and every starting value within two
// ulp of 1 / p.
__device__ __forceinline__ float rcp_scale(float p) {
  float y0;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(p));
  const float e = __fmaf_rn(-p, y0, 1.0f);
  return __fmaf_rn(e, y0, y0);
}

__device__ __forceinline__ RowScale row_scale(float amax) {
  RowScale rs;
  const float a = amax * kInvSqrt128;
  rs.sh = __float2half_rn(div127(a));
  rs.clamp = false;
  if (__hisinf(rs.sh)) {
    rs.sh = __ushort_as_half(0x7BFFu);  // 65504
    rs.clamp = true;
  }
  const float sf = __half2float(rs.sh);
  rs.clamp = rs.clamp || (sf < 6.103515625e-05f);  // fp16 subnormal scale: x'/s may exceed 127.5
  rs.m = sf > 0.f ? rcp_scale(sf * 11.313708498984761f) : 0.f;
  return rs;
}

// kGroups = 1: one scale per row; kGroups = 4: one per 32 consecutive
// rotated values (the per-32-value variant).  kWide: codes go out as 32-byte
// stores (whole L2 sectors), for code buffers aligned to 32 bytes.
template <int kGroups, bool kWide>
__global__ void __launch_bounds__(kThreads, 2)
    store_build_kernel(const __grid_constant__ CUtensorMap tm_k_in, const __grid_constant__ CUtensorMap tm_v_in,
                       int8_t *__restrict__ k_codes, int8_t *__restrict__ v_codes,
                       uint16_t *__restrict__ k_scales, uint16_t *__restrict__ v_scales, int64_t rows,
                       int64_t tiles_per_tensor, uint32_t *err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  BuildSmem &sm = *reinterpret_cast<BuildSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

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
        // drain: every issued load must land before the CTA may exit
        for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
          mbar_wait_drain(smem_u32(&sm.full[k % kStages]), (k / kStages) & 1, kDrainNs);
      }
    }
  } else {
    // ----------------------------------------------------------- compute
    // Threads 2r and 2r + 1 share row r.  With H128 = [[H64, H64], [H64, -H64]]
    // (Sylvester order), half h of (x H128) is H64 applied to x_lo + x_hi
    // (h = 0) or x_lo - x_hi (h = 1): each thread reads the whole row, forms
    // its 64 sums or differences and runs a 64-point FWHT in registers.
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

      // x[i] = row[i] +- row[i + 64]; element e of the row sits in 64-column
      // chunk e/64, granule (e%64)/8, swizzled
      float x[64];
      const uint8_t *tile = sm.in[s];
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
      mbar_arrive(smem_u32(&sm.empty[s]));

      fwht64_packed(x);  // x now holds sqrt(128) * (row H), elements 64h .. 64h + 63

      constexpr int kMine = kGroups == 1 ? 1 : kGroups / 2;  // scale groups within this half
      RowScale rs[kMine];
      if constexpr (kGroups == 1) {
        float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 64; e += 8) {
#pragma unroll
          for (int u = 0; u < 4; ++u) am[u] = fmax3(am[u], fabsf(x[e + 2 * u]), fabsf(x[e + 2 * u + 1]));
        }
        float a = fmax3(am[0], am[1], fmaxf(am[2], am[3]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        rs[0] = row_scale(a);
      } else {
#pragma unroll
        for (int gi = 0; gi < kMine; ++gi) {
          constexpr int kW = 128 / kGroups;
          float am[2] = {0.f, 0.f};
#pragma unroll
          for (int e = gi * kW; e < (gi + 1) * kW; e += 4) {
            am[0] = fmax3(am[0], fabsf(x[e]), fabsf(x[e + 1]));
            am[1] = fmax3(am[1], fabsf(x[e + 2]), fabsf(x[e + 3]));
          }
          rs[gi] = row_scale(fmaxf(am[0], am[1]));
        }
      }

      // code = rne(x' / s) = rne(x * m) with m = 1 / (sqrt(128) s): adding
      // 1.5 * 2^23 rounds to an integer held in the low mantissa bits, whose
      // low byte is the two's-complement int8 code.
      constexpr float kMagic = 12582912.0f;
      const bool is_v = t >= tiles_per_tensor;
      const int64_t row0 = (is_v ? t - tiles_per_tensor : t) * kRows;
      const bool row_ok = row0 + r < rows;
      int8_t *oc = (is_v ? v_codes : k_codes) + (row_ok ? row0 + r : 0) * 128 + 64 * h;
      uint32_t wp[8];  // granules g - 1 and g, stored together when kWide
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t q[4];
          const int e = g * 16 + k * 4;
          const RowScale &gs = rs[kGroups == 1 ? 0 : (e * kGroups) >> 7];
          const float m = gs.m;
          if (!gs.clamp) {
            const float2 mm = make_float2(m, m), mg = make_float2(kMagic, kMagic);
            const float2 lo = __ffma2_rn(make_float2(x[e], x[e + 1]), mm, mg);
            const float2 hi = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), mm, mg);
            q[0] = __float_as_uint(lo.x);
            q[1] = __float_as_uint(lo.y);
            q[2] = __float_as_uint(hi.x);
            q[3] = __float_as_uint(hi.y);
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              q[u] = __float_as_uint(fminf(fmaxf(x[e + u] * m, -127.f), 127.f) + kMagic);
          }
          const uint32_t lo = __byte_perm(q[0], q[1], 0x0040);
          const uint32_t hi = __byte_perm(q[2], q[3], 0x0040);
          w[k] = __byte_perm(lo, hi, 0x5410);
        }
        if constexpr (kWide) {
#pragma unroll
          for (int k = 0; k < 4; ++k) wp[(g & 1) * 4 + k] = w[k];
          if ((g & 1) && row_ok) st_global_v8(oc + (g - 1) * 16, wp);
        } else {
          if (row_ok) *reinterpret_cast<uint4 *>(oc + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      uint16_t *scales = is_v ? v_scales : k_scales;
      if (row_ok) {
        if constexpr (kGroups == 1) {
          if (h == 0) scales[row0 + r] = __half_as_ushort(rs[0].sh);
        } else {
#pragma unroll
          for (int gi = 0; gi < kMine; ++gi)
            scales[(row0 + r) * kGroups + kMine * h + gi] = __half_as_ushort(rs[gi].sh);
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_store_build(const CUtensorMap &k_in, const CUtensorMap &v_in, int8_t *k_out,
                               int8_t *v_out, uint16_t *k_scales, uint16_t *v_scales, int64_t rows,
                               int num_sms, int scale_groups, uint32_t *err, uint64_t timeout_ns,
                               cudaStream_t stream) {
  const int64_t tiles = (rows + kRows - 1) / kRows;
  if (tiles == 0) return cudaSuccess;
  // whole-sector stores: device code buffers aligned to 32 bytes (rows are
  // multiples of 32 bytes, so every row's pairs of 16-byte pieces are too)
  const bool wide = wide_store_ok(k_out, v_out);
  auto kernel = scale_groups == 4 ? (wide ? store_build_kernel<4, true> : store_build_kernel<4, false>)
                                  : (wide ? store_build_kernel<1, true> : store_build_kernel<1, false>);
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kBuildSmemBytes));
  if (e != cudaSuccess) return e;
  int64_t grid = static_cast<int64_t>(num_sms) * 2;
  if (grid > 2 * tiles) grid = 2 * tiles;
  kernel<<<static_cast<unsigned>(grid), kThreads, kBuildSmemBytes, stream>>>(k_in, v_in, k_out, v_out, k_scales,
                                                                              v_scales, rows, tiles, err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace h3kv
