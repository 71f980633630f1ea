// attend.cuh -- query-chunked attention over a whole-sequence K/V store on
// sm_103a tensor cores (tcgen05 + TMEM), shared by the kvi8r and the exact
// (bf16) store.
//
// kvi8r (kv_store row of the H3 Streamed Blocks Inputs table; kvi8r row and
// the rotation paragraph of "The K/V store options" in the Low VRAM
// write-up): the query chunk is rotated into the Hadamard basis (q' = q H,
// fp16), each K/V block is dequantised as int8 -> fp16 cast times the row
// scale, scores and P.V run in fp16 with fp32 accumulation, blocks of
// kv_block keys are combined by their log-sum-exp, and the output is
// un-rotated once (O = O' H^T).  The exact store runs the same pipeline on
// bf16 K/V without rotation or dequantisation.  The kvfp4 store (kvfp4s in
// the same kv_store row: NVFP4 K/V, e2m1 values with one e4m3 scale per 16,
// Q and K rotated) runs the kvi8r pipeline with each block dequantised as
// e2m1 -> fp16 times its e4m3 scale -- exact in fp16 -- and no un-rotation,
// V not being rotated.
//
// One CTA owns 256 query rows of one head (two 128-row tiles, so that the
// softmax of one tile overlaps the tensor-core work of the other) and walks
// every 128-key tile of that head in a fixed order, so a query row's
// arithmetic never depends on q_chunk or on which CTA holds it.
//
// Warp roles (512 threads):
//   warps 0-3   softmax / correction / epilogue of query tile 0 (thread = row)
//   warps 4-7   the same for query tile 1
//   warps 8-11  kvi8r / kvfp4: in-place int8 (e2m1) -> fp16 dequantisation
//               of K and V tiles
//   warp 12     producer: TMA / bulk copies of Q (exact) and K/V tiles
//   warp 13     TMEM allocation and tcgen05.mma issue (one elected lane)
//   warps 14-15 idle
// TMEM (512 columns x 128 lanes, fp32): S0 [0,128), S1 [128,256) with P0/P1
// (fp16/bf16 pairs) written over the first 64 columns of S0/S1, O0
// [256,384), O1 [384,512).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace h3kv {
namespace attn {

constexpr int kBM = 128;                    // query rows per tile (MMA M)
constexpr int kNQ = 2;                      // query tiles per CTA
constexpr int kBN = 128;                    // keys per tile
constexpr int kNK = 3;                      // K tile ring depth
constexpr int kNV = 2;                      // V tile ring depth
constexpr int kTileBytes = 128 * 128 * 2;   // one 16-bit [128 x 128] tile
constexpr int kChunkBytes = kTileBytes / 2; // 64-column half (one swizzle atom wide)
constexpr int kThreads = 512;
constexpr int kWarpsPerGroup = 4;           // arrivals on a barrier released by a warpgroup
constexpr float kLazyRescaleLog2 = 8.0f;    // rescale O only when the max grows by > 2^8

// Register split per warpgroup (setmaxnreg).  The launch gives every thread
// 128 (512 threads x 128 = the 64K register file); each split below sums to
// the same total: 128 x (2 x softmax + dequant + issue) = 65536.
constexpr uint32_t kRegSoftmaxKvi8r = 184, kRegDequantKvi8r = 72, kRegIssueKvi8r = 72;
constexpr uint32_t kRegSoftmaxExact = 184, kRegDequantExact = 56, kRegIssueExact = 88;
static_assert(2 * kRegSoftmaxKvi8r + kRegDequantKvi8r + kRegIssueKvi8r == 512, "register split");
static_assert(2 * kRegSoftmaxExact + kRegDequantExact + kRegIssueExact == 512, "register split");

struct Smem {
  uint8_t q[kNQ][kTileBytes];
  uint8_t k[kNK][kTileBytes];
  uint8_t v[kNV][kTileBytes];
  uint64_t q_full;
  uint64_t k_load[kNK], k_ready[kNK], k_free[kNK];
  uint64_t v_load[kNV], v_ready[kNV], v_free[kNV];
  uint64_t s_full[kNQ], p_full[kNQ];
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx &w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

// 16 int8 codes (one 16-byte granule) -> 16 fp16 values code * scale.  The
// code is biased to an unsigned byte u = c + 128, placed in the mantissa of
// the fp16 value 1024 + u by a byte permute, and 1152 is subtracted exactly,
// giving fp16(c) exactly; the multiply by the fp16 scale rounds once.
__device__ __forceinline__ void dequant16(const uint4 raw, const __half2 s2, uint32_t (&out)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t u = w[k] ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 ha = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&a), bias), s2);
    const __half2 hb = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&b), bias), s2);
    out[2 * k] = *reinterpret_cast<const uint32_t *>(&ha);
    out[2 * k + 1] = *reinterpret_cast<const uint32_t *>(&hb);
  }
}

// Row and 16-byte code granule handled by `lane` in iteration `it` of dequant
// warp `dw`: each instruction covers 4 rows; a quarter-warp takes 4 granules
// of an even row and the other-half 4 granules of the next (odd) row, so its
// 16-byte loads (linear codes) and its 16-byte stores (swizzled fp16) each
// touch 8 distinct bank groups.
__device__ __forceinline__ uint32_t dq_row(int dw, int it, int lane) {
  const int q4 = lane >> 3, hf = (lane >> 2) & 1;
  return dw * 32 + it * 4 + 2 * (q4 >> 1) + hf;
}
__device__ __forceinline__ uint32_t dq_granule(int lane) {
  const int q4 = lane >> 3, hf = (lane >> 2) & 1;
  return (lane & 3) + 4 * (hf ^ (q4 & 1));
}

// Shared-memory byte offsets of one lane's dequantisation work inside a K/V
// tile, computed once per kernel.  The lane's row in iteration `it` is
// dw*32 + 4*it + rr (rr = 2*(q4/2) + hf, below 4), so every address is a
// per-lane base plus it*512 bytes (a compile-time immediate once the loop is
// unrolled); in the 128-byte swizzle the row's low three bits alternate
// between rr and rr + 4, which flips bit 6 of the granule offset on odd
// iterations.
struct DqOffsets {
  uint32_t ld8;       // int8 codes of iteration 0 (second half of the tile); + it*512
  uint32_t ld4;       // kvfp4 codes of iteration 0 (start of the tile); + it*256
  uint32_t st[2][2];  // fp16 granules G0, G0 + 1 for even / odd iterations; + it*512
};
__device__ __forceinline__ DqOffsets dq_offsets(int dw, int lane) {
  const uint32_t g = dq_granule(lane);
  const uint32_t rr = 2u * (static_cast<uint32_t>(lane) >> 4) + ((static_cast<uint32_t>(lane) >> 2) & 1u);
  const uint32_t row0 = static_cast<uint32_t>(dw) * 32u + rr;
  const uint32_t base = (g >> 2) * kChunkBytes + row0 * 128u;
  const uint32_t G0 = (g & 3u) * 2u;
  const uint32_t a0 = (G0 ^ rr) << 4, a1 = ((G0 + 1u) ^ rr) << 4;
  DqOffsets o;
  o.ld8 = kChunkBytes + row0 * 128u + g * 16u;
  o.ld4 = row0 * 64u + g * 8u;
  o.st[0][0] = base + a0;
  o.st[0][1] = base + a1;
  o.st[1][0] = base + (a0 ^ 64u);
  o.st[1][1] = base + (a1 ^ 64u);
  return o;
}

// Scales of the rows this lane dequantises (rows past `valid` get 0).  With
// kGroups = 4 a row has one scale per 32 values and the lane's 16-value
// granule g takes scale g / 2 of its row.  Loaded through L2 (ld.global.cg):
// a CTA reads each scale once, so keeping it in L1 only displaces other lines
// (measured 0.3-0.6 % faster over the whole kvi8r kernel).
template <int kGroups>
__device__ __forceinline__ void dequant_scales(const uint16_t *scales, int valid, int dw, int lane,
                                               uint16_t (&sc)[8]) {
  // row of iteration it: dw*32 + rr + 4*it (dq_row); one base pointer, the
  // iterations at immediate offsets; bounds checks only on a ragged tile
  const int rr = 2 * (lane >> 4) + ((lane >> 2) & 1);
  const int grp = kGroups == 1 ? 0 : static_cast<int>(dq_granule(lane) >> 1);
  const uint16_t *p = scales + (dw * 32 + rr) * kGroups + grp;
  if (valid >= kBN) {
#pragma unroll
    for (int it = 0; it < 8; ++it) sc[it] = __ldcg(p + it * 4 * kGroups);
  } else {
#pragma unroll
    for (int it = 0; it < 8; ++it) sc[it] = dw * 32 + rr + 4 * it < valid ? __ldcg(p + it * 4 * kGroups) : 0;
  }
}

// In-place dequantisation of one K or V tile by the 128 dequant threads.
// On entry the int8 codes of the tile's rows sit linearly (128 bytes per row)
// in the second half of the tile buffer; on exit the whole buffer holds the
// fp16 tile in the 128B-swizzled layout the MMA descriptors expect (two
// 64-column halves of [128 rows x 128 bytes]).  Row r's codes share their
// 128-byte slot with row r's fp16 columns 64-127, and every row is read by
// one load instruction of its warp before any lane writes it, so in place is
// safe.
__device__ __forceinline__ void dequant_tile(uint8_t *tile, const uint16_t (&sc)[8], const DqOffsets &off) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(tile + off.ld8 + it * 512);
    const __half s = __ushort_as_half(sc[it]);
    uint32_t o[8];
    dequant16(raw, __halves2half2(s, s), o);
    uint8_t *row = tile + it * 512;
    *reinterpret_cast<uint4 *>(row + off.st[it & 1][0]) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(row + off.st[it & 1][1]) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// kvfp4: one 16-value block (8 code bytes, element 2i in the low nibble of
// byte i) -> 16 fp16 values code * scale.  Both conversions are exact, and so
// is the product: a 2-bit times a 4-bit significand, at most 2688 in size.
__device__ __forceinline__ void dequant16_fp4(const uint2 raw, uint32_t s2, uint32_t (&out)[8]) {
  uint32_t a[4], b[4];
  e2m1x8_to_f16x2(raw.x, a);
  e2m1x8_to_f16x2(raw.y, b);
  const __half2 s = *reinterpret_cast<const __half2 *>(&s2);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 ha = __hmul2(*reinterpret_cast<const __half2 *>(&a[k]), s);
    const __half2 hb = __hmul2(*reinterpret_cast<const __half2 *>(&b[k]), s);
    out[k] = *reinterpret_cast<const uint32_t *>(&ha);
    out[4 + k] = *reinterpret_cast<const uint32_t *>(&hb);
  }
}

// kvfp4: e4m3 scales of the blocks this lane dequantises (the lane's
// granule index is its block within the row), byte `it` of the pair of
// words for iteration `it`; rows past `valid` get 0.
__device__ __forceinline__ void dequant_scales_fp4(const uint8_t *scales, int valid, int dw, int lane,
                                                   uint32_t (&sc)[2]) {
  const int rr = 2 * (lane >> 4) + ((lane >> 2) & 1);
  const uint8_t *p = scales + (dw * 32 + rr) * 8 + static_cast<int>(dq_granule(lane));
  sc[0] = sc[1] = 0u;
  if (valid >= kBN) {
#pragma unroll
    for (int it = 0; it < 8; ++it) sc[it >> 2] |= static_cast<uint32_t>(__ldcg(p + it * 32)) << ((it & 3) * 8);
  } else {
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const uint32_t b = dw * 32 + rr + 4 * it < valid ? __ldcg(p + it * 32) : 0u;
      sc[it >> 2] |= b << ((it & 3) * 8);
    }
  }
}

// kvfp4 dequantisation of one K or V tile by the 128 dequant threads.  The
// packed codes sit linearly (64 bytes per row) at the start of the buffer,
// under fp16 output rows of other warps, so every thread first loads its
// codes, the four warps meet at named barrier 1 (which also ANDs the load
// waits' outcomes: every warp reaches it whether or not its wait succeeded),
// and only then does any thread write.  Returns false, having written
// nothing, when some warp's wait ran out.  Output layout as dequant_tile.
__device__ __forceinline__ bool dequant_tile_fp4(uint8_t *tile, bool loaded, const uint32_t (&sc)[2],
                                                 const DqOffsets &off) {
  uint2 raw[8];
#pragma unroll
  for (int it = 0; it < 8; ++it)
    raw[it] = loaded ? *reinterpret_cast<const uint2 *>(tile + off.ld4 + it * 256) : make_uint2(0u, 0u);
  if (!named_bar_and(1, 128, loaded)) return false;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    uint32_t o[8];
    // the iteration's scale byte twice: the fp16 pair (s, s)
    dequant16_fp4(raw[it], e4m3x2_to_f16x2(__byte_perm(sc[it >> 2], 0u, (it & 3) * 0x11u)), o);
    uint8_t *row = tile + it * 512;
    *reinterpret_cast<uint4 *>(row + off.st[it & 1][0]) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(row + off.st[it & 1][1]) = make_uint4(o[4], o[5], o[6], o[7]);
  }
  return true;
}

// Log-sum-exp merge of a finished block (m_b, l_b) into the running (M, Lam)
// (max in raw score units, c2 = softmax scale * log2 e): returns the weights
// of the running and the block output and updates (M, Lam).  Written with
// explicit fused operations so every merge -- inside one launch or across the
// launches of the staged path -- rounds identically.
__device__ __forceinline__ void lse_merge(float &M, float &Lam, float m_b, float l_b, float c2, float &al,
                                          float &be) {
  const float Mn = fmaxf(M, m_b);
  al = ex2(__fmul_rn(__fsub_rn(M, Mn), c2));
  be = ex2(__fmul_rn(__fsub_rn(m_b, Mn), c2));
  Lam = __fmaf_rn(Lam, al, __fmul_rn(l_b, be));
  M = Mn;
}

template <bool kKvi8r>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kKvi8r) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

template <bool kKvi8r, int kGroups, bool kFp4 = false>
__global__ void __launch_bounds__(kThreads, 1)
    attend_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = a.head_base + static_cast<int>(blockIdx.y);
  const int64_t row0 = a.q_begin + static_cast<int64_t>(blockIdx.x) * (kNQ * kBM);
  const int n_tiles = static_cast<int>((a.kv_seq + kBN - 1) / kBN);
  const int blk = a.kv_block_tiles;

  if (a.q_ready != nullptr) {
    // a query chunk streamed from host memory: its Q rows and O buffer are
    // ready once the copy engine has written the launch's value (before any
    // TMEM is taken, so a waiting CTA holds nothing the previous launch needs)
    if (tid == 0) sm.abort = wait_word_equal(a.q_ready, a.q_ready_value, a.err, a.timeout_ns) ? 0 : 1;
    __syncthreads();
    if (sm.abort) {
      if (tid == 0) pdl_wait_prerequisites();
      return;
    }
  }

  if (tid == 0) {
    mbar_init(smem_u32(&sm.q_full), kKvi8r ? kNQ * kBM : 1);
    for (int s = 0; s < kNK; ++s) {
      mbar_init(smem_u32(&sm.k_load[s]), 1);
      mbar_init(smem_u32(&sm.k_ready[s]), kWarpsPerGroup);
      mbar_init(smem_u32(&sm.k_free[s]), 1);
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(smem_u32(&sm.v_load[s]), 1);
      mbar_init(smem_u32(&sm.v_ready[s]), kWarpsPerGroup);
      mbar_init(smem_u32(&sm.v_free[s]), 1);
    }
    for (int q = 0; q < kNQ; ++q) {
      mbar_init(smem_u32(&sm.s_full[q]), 1);
      mbar_init(smem_u32(&sm.p_full[q]), kWarpsPerGroup);
    }
    mbar_init(smem_u32(&sm.o_full), 1);
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the next query chunk's launch may fill SMs that this grid's tail frees
  if (tid == 0) pdl_launch_dependents();
  const uint32_t tmem = sm.tmem_base;
  const WaitCtx wctx{a.err, &sm.abort, a.timeout_ns};

  if (warp < 8) {
    // =================================================== softmax warpgroups
    reg_alloc<kKvi8r ? kRegSoftmaxKvi8r : kRegSoftmaxExact>();
    const int q = warp >> 2;
    const uint32_t i = tid & 127;  // row in the query tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + q * 128;
    const uint32_t tO = tmem + lane_base + 256 + q * 128;
    const int64_t row = row0 + q * kBM + i;
    const bool row_ok = row < a.q_end;
    float *orow = a.o + (static_cast<int64_t>(h) * a.q_seq + (row_ok ? row : 0)) * 128;
    const float c2 = a.scale_log2;

    if constexpr (kKvi8r) {
      // q' = fp16(q H): each warp rotates its 32 rows of the query tile, one
      // row at a time across the warp (lane l holds elements 4l..4l+3), and
      // writes them in the 128B-swizzled K-major layout of the MMA's A operand.
      const int wq = warp & 3;
      uint2 buf[32];
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) {
        const int64_t r = row0 + q * kBM + wq * 32 + rr;
        // through L2 (ld.global.cg): a streamed chunk's buffer is rewritten
        // by the copy engine between launches that may share an SM
        buf[rr] = r < a.q_end ? __ldcg(reinterpret_cast<const uint2 *>(a.q + (static_cast<int64_t>(h) * a.q_seq + r) *
                                                                                   128 +
                                                                       4 * lane))
                              : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) {
        const uint32_t ti = wq * 32 + rr;
        float x[4] = {bf16lo_to_f32(buf[rr].x), bf16hi_to_f32(buf[rr].x), bf16lo_to_f32(buf[rr].y),
                      bf16hi_to_f32(buf[rr].y)};
        fwht128_warp(x, lane);
        const uint2 w = make_uint2(pack_f16x2(x[0] * kInvSqrt128, x[1] * kInvSqrt128),
                                   pack_f16x2(x[2] * kInvSqrt128, x[3] * kInvSqrt128));
        *reinterpret_cast<uint2 *>(sm.q[q] + (lane >> 4) * kChunkBytes + sw128_off(ti, (lane & 15) >> 1) +
                                   (lane & 1) * 8) = w;
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&sm.q_full));
    }

    float m_b = 0.f, l_b = 0.f;  // current block: running max (raw score units) and sum
    float M = 0.f, Lam = 0.f;    // blocks merged so far
    bool ok = true;
    int jb = 0;                  // position of tile j in its kv_block (j % blk, by a counter)
    for (int j = 0; j < n_tiles; ++j) {
      if (!warp_wait(smem_u32(&sm.s_full[q]), j & 1, wctx)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
      const int64_t valid = a.kv_seq - static_cast<int64_t>(j) * kBN;
      // The row max of a full tile comes with the S loads (the reducing
      // TMEM load returns each 32-column group's maximum: 3.5 % faster on
      // kvi8r, outputs bit-identical); the tile past the last key masks its
      // columns beyond `valid` and takes the max in software.  The two
      // arrangements of the loads below are the ones that compile without
      // spills for the quantised and the exact stores.
      float mt;
      float m4[4];
      if constexpr (kKvi8r) tmem_ld128_max(tS, *reinterpret_cast<uint32_t(*)[128]>(s), m4);
      if (valid >= kBN) {
        if constexpr (!kKvi8r) tmem_ld128_max(tS, *reinterpret_cast<uint32_t(*)[128]>(s), m4);
        mt = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      } else {
        if constexpr (!kKvi8r) tmem_ld128(tS, *reinterpret_cast<uint32_t(*)[128]>(s));
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < valid) ? s[c] : -INFINITY;
        // eight independent chains of 16 columns (0.3 % faster than four)
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = fmax3(s[u], s[u + 8], s[u + 16]);
#pragma unroll
        for (int c = 24; c < 120; c += 16) {
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = fmax3(m8[u], s[c + u], s[c + 8 + u]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = fmaxf(m8[u], s[120 + u]);
        mt = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      }

      if (jb == 0) {
        if (j > 0) {
          // merge the finished block (O_q, m_b, l_b) into (M, Lam, O row in
          // global memory, rotated basis, un-normalised)
          const bool first = j == blk;
          float al = 0.f, be = 1.f;
          if (!first) {
            lse_merge(M, Lam, m_b, l_b, c2, al, be);
          } else {
            M = m_b;
            Lam = l_b;
          }
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float o[16];
            tmem_ld16(tO + c * 16, *reinterpret_cast<uint32_t(*)[16]>(o));
            if (row_ok) {
              float4 *dst = reinterpret_cast<float4 *>(orow + c * 16);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float4 v = make_float4(o[4 * k] * be, o[4 * k + 1] * be, o[4 * k + 2] * be, o[4 * k + 3] * be);
                if (!first) {
                  const float4 g = dst[k];
                  v.x = fmaf(g.x, al, v.x);
                  v.y = fmaf(g.y, al, v.y);
                  v.z = fmaf(g.z, al, v.z);
                  v.w = fmaf(g.w, al, v.w);
                }
                dst[k] = v;
              }
            }
          }
        }
        m_b = mt;
        l_b = 0.f;
      } else {
        const bool need = (mt - m_b) * c2 > kLazyRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2((m_b - mt) * c2) : 1.f;
          if (need) {
            l_b *= alpha;
            m_b = mt;
          }
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
#pragma unroll
            for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st16(tO + c * 16, o);
          }
        }
      }

      // p = 2^(s c - m c) in packed pairs, written as fp16 (bf16) pairs over
      // the first 64 columns of S
      const float2 cc = make_float2(c2, c2);
      const float2 nm = make_float2(-m_b * c2, -m_b * c2);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int c = hlf * 64 + 2 * k;
          float2 e = __ffma2_rn(make_float2(s[c], s[c + 1]), cc, nm);
          e.x = ex2(e.x);
          e.y = ex2(e.y);
          if (k & 1) acc1 = __fadd2_rn(acc1, e);
          else acc0 = __fadd2_rn(acc0, e);
          pk[k] = pack2<kKvi8r>(e.x, e.y);
        }
        tmem_st32(tS + hlf * 32, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      // (a diagnostic may withhold one tile's arrival: see withhold_p_tile1)
      if (lane == 0 && j + 1 != a.withhold_p_tile1) mbar_arrive(smem_u32(&sm.p_full[q]));
      const float2 acc = __fadd2_rn(acc0, acc1);
      l_b += acc.x + acc.y;
      jb = jb + 1 == blk ? 0 : jb + 1;
    }

    if (ok && warp_wait(smem_u32(&sm.o_full), 0, wctx)) {
      // epilogue, phase 1: each thread finishes its own row (final block
      // merge, 1/Lambda) and stages it in shared memory, fp32, with 16-byte
      // granule gi of row i at position gi ^ (i mod 32).  The K/V rings are
      // free now: every MMA has completed and no copy is outstanding.
      tc_fence_after();
      const int n_blocks = (n_tiles + blk - 1) / blk;
      // staged attention: this launch is one block of a sequence of launches
      const bool staged = a.state != nullptr;
      const bool first_launch = !staged || (a.stage_flags & 1);
      const bool last_launch = !staged || (a.stage_flags & 2);
      float2 *st = staged ? a.state + (static_cast<int64_t>(h) * a.q_seq + (row_ok ? row : 0)) : nullptr;
      if (staged && !first_launch) {
        // blocks of earlier launches: (M, Lam) from the state, their
        // un-normalised output in the O row (n_blocks == 1 per staged launch)
        const float2 m_l = row_ok ? *st : make_float2(0.f, 1.f);
        M = m_l.x;
        Lam = m_l.y;
      }
      const bool has_prev = n_blocks > 1 || !first_launch;
      if (!last_launch) {
        // not the last block: merge into the running output and state only
        float al = 0.f, be = 1.f;
        if (has_prev) {
          lse_merge(M, Lam, m_b, l_b, c2, al, be);
        } else {
          M = m_b;
          Lam = l_b;
        }
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float o[16];
          tmem_ld16(tO + c * 16, *reinterpret_cast<uint32_t(*)[16]>(o));
          if (row_ok) {
            float4 *dst = reinterpret_cast<float4 *>(orow + c * 16);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float4 v = make_float4(o[4 * k] * be, o[4 * k + 1] * be, o[4 * k + 2] * be, o[4 * k + 3] * be);
              if (has_prev) {
                const float4 g = dst[k];
                v.x = fmaf(g.x, al, v.x);
                v.y = fmaf(g.y, al, v.y);
                v.z = fmaf(g.z, al, v.z);
                v.w = fmaf(g.w, al, v.w);
              }
              dst[k] = v;
            }
          }
        }
        if (row_ok) *st = make_float2(M, Lam);
      } else {
      uint8_t *stage = sm.k[0] + q * (kNQ * kTileBytes);
      float ga, gb;
      if (!has_prev) {
        ga = 0.f;
        gb = 1.f / l_b;
      } else {
        float al, be;
        lse_merge(M, Lam, m_b, l_b, c2, al, be);
        const float inv = 1.f / Lam;
        ga = al * inv;
        gb = be * inv;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(tO + c * 32, *reinterpret_cast<uint32_t(*)[32]>(o));
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] *= gb;
        if (has_prev && row_ok) {
          const float4 *src = reinterpret_cast<const float4 *>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 g = src[k];
            o[4 * k + 0] = fmaf(g.x, ga, o[4 * k + 0]);
            o[4 * k + 1] = fmaf(g.y, ga, o[4 * k + 1]);
            o[4 * k + 2] = fmaf(g.z, ga, o[4 * k + 2]);
            o[4 * k + 3] = fmaf(g.w, ga, o[4 * k + 3]);
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t gi = c * 8 + k;
          *reinterpret_cast<float4 *>(stage + i * 512 + ((gi ^ (i & 31)) << 4)) =
              make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
      }
      __syncwarp();
      // phase 2: each warp takes its 32 rows one at a time across the warp:
      // un-rotate (kvi8r: O = O' H^T, H symmetric) and store coalesced.
      const int wq = warp & 3;
#pragma unroll 4
      for (int rr = 0; rr < 32; ++rr) {
        const uint32_t ti = wq * 32 + rr;
        const float4 v = *reinterpret_cast<const float4 *>(stage + ti * 512 + ((lane ^ (ti & 31)) << 4));
        float x[4] = {v.x, v.y, v.z, v.w};
        if constexpr (kKvi8r && !kFp4) {
          fwht128_warp(x, lane);
#pragma unroll
          for (int t = 0; t < 4; ++t) x[t] *= kInvSqrt128;
        }
        const int64_t r = row0 + q * kBM + ti;
        if (r < a.q_end)
          *reinterpret_cast<float4 *>(a.o + (static_cast<int64_t>(h) * a.q_seq + r) * 128 + 4 * lane) =
              make_float4(x[0], x[1], x[2], x[3]);
      }
      }
    }
  } else if (warp < 12) {
    // ======================================================= dequantisers
    reg_dealloc<kKvi8r ? kRegDequantKvi8r : kRegDequantExact>();
    if constexpr (kFp4) {
      const int dw = warp - 8;
      const uint8_t *ksc = a.k_fp4_scales + static_cast<int64_t>(h) * a.kv_stride * 8;
      const uint8_t *vsc = a.v_fp4_scales + static_cast<int64_t>(h) * a.kv_stride * 8;
      uint32_t sck[2], scv[2];
      const DqOffsets off = dq_offsets(dw, lane);
      // ring slots and phases, and the scales of tile j, advanced by counters
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      const uint8_t *kst = ksc, *vst = vsc;
      int64_t left = a.kv_seq;
      for (int j = 0; j < n_tiles; ++j) {
        const int valid = static_cast<int>(left < kBN ? left : kBN);
        dequant_scales_fp4(kst, valid, dw, lane, sck);
        dequant_scales_fp4(vst, valid, dw, lane, scv);
        if (!dequant_tile_fp4(sm.k[ks], warp_wait(smem_u32(&sm.k_load[ks]), kph, wctx), sck, off)) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.k_ready[ks]));
        if (!dequant_tile_fp4(sm.v[vs], warp_wait(smem_u32(&sm.v_load[vs]), vph, wctx), scv, off)) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.v_ready[vs]));
        kst += kBN * 8;
        vst += kBN * 8;
        left -= kBN;
        if (++ks == kNK) {
          ks = 0;
          kph ^= 1u;
        }
        if (++vs == kNV) {
          vs = 0;
          vph ^= 1u;
        }
      }
    } else if constexpr (kKvi8r) {
      const int dw = warp - 8;
      const uint16_t *ksc = a.k_scales + static_cast<int64_t>(h) * a.kv_stride * kGroups;
      const uint16_t *vsc = a.v_scales + static_cast<int64_t>(h) * a.kv_stride * kGroups;
      uint16_t sck[8], scv[8];
      const DqOffsets off = dq_offsets(dw, lane);
      // ring slots and phases, and the scales of tile j, advanced by counters
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      const uint16_t *kst = ksc, *vst = vsc;
      int64_t left = a.kv_seq;
      for (int j = 0; j < n_tiles; ++j) {
        const int valid = static_cast<int>(left < kBN ? left : kBN);
        // scale loads go out before the waits so their latency hides there
        dequant_scales<kGroups>(kst, valid, dw, lane, sck);
        dequant_scales<kGroups>(vst, valid, dw, lane, scv);
        if (!warp_wait(smem_u32(&sm.k_load[ks]), kph, wctx)) break;
        dequant_tile(sm.k[ks], sck, off);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.k_ready[ks]));
        if (!warp_wait(smem_u32(&sm.v_load[vs]), vph, wctx)) break;
        dequant_tile(sm.v[vs], scv, off);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.v_ready[vs]));
        kst += kBN * kGroups;
        vst += kBN * kGroups;
        left -= kBN;
        if (++ks == kNK) {
          ks = 0;
          kph ^= 1u;
        }
        if (++vs == kNV) {
          vs = 0;
          vph ^= 1u;
        }
      }
    }
  } else {
    reg_dealloc<kKvi8r ? kRegIssueKvi8r : kRegIssueExact>();
    if (warp == 12) {
      // ========================================================== producer
      // the whole warp waits; one elected lane issues the copies
      const uint32_t go = elect_one();
      int k_issued[kNK] = {0, 0, 0};
      int v_issued[kNV] = {0, 0};
      if constexpr (!kKvi8r) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        const uint32_t bar = smem_u32(&sm.q_full);
        if (go) mbar_arrive_expect_tx(bar, kNQ * kTileBytes);
        if (go) for (int q = 0; q < kNQ; ++q)
          for (int c = 0; c < 2; ++c)
            tma_load_3d(smem_u32(sm.q[q] + c * kChunkBytes), &tm_q, c * 64, static_cast<int32_t>(row0 + q * kBM),
                        h, bar);
      }
      for (int j = 0; j < n_tiles; ++j) {
        const int64_t tok0 = static_cast<int64_t>(j) * kBN;
        const int ks = j % kNK, vs = j % kNV;
        if (!warp_wait(smem_u32(&sm.k_free[ks]), ((j / kNK) & 1) ^ 1, wctx)) break;
        if (go) {
          const uint32_t bar = smem_u32(&sm.k_load[ks]);
          if constexpr (kFp4) {
            const uint32_t bytes = static_cast<uint32_t>((a.kv_seq - tok0 < kBN ? a.kv_seq - tok0 : kBN) * 64);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(smem_u32(sm.k[ks]), a.k_codes + (static_cast<int64_t>(h) * a.kv_stride + tok0) * 64, bytes, bar);
          } else if constexpr (kKvi8r) {
            const uint32_t bytes = static_cast<uint32_t>((a.kv_seq - tok0 < kBN ? a.kv_seq - tok0 : kBN) * 128);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(smem_u32(sm.k[ks] + kChunkBytes), a.k_codes + (static_cast<int64_t>(h) * a.kv_stride + tok0) * 128,
                     bytes, bar);
          } else {
            mbar_arrive_expect_tx(bar, kTileBytes);
            tma_load_3d(smem_u32(sm.k[ks]), &tm_k, 0, static_cast<int32_t>(tok0), h, bar);
            tma_load_3d(smem_u32(sm.k[ks] + kChunkBytes), &tm_k, 64, static_cast<int32_t>(tok0), h, bar);
          }
        }
        ++k_issued[ks];
        if (!warp_wait(smem_u32(&sm.v_free[vs]), ((j / kNV) & 1) ^ 1, wctx)) break;
        if (go) {
          const uint32_t bar = smem_u32(&sm.v_load[vs]);
          if constexpr (kFp4) {
            const uint32_t bytes = static_cast<uint32_t>((a.kv_seq - tok0 < kBN ? a.kv_seq - tok0 : kBN) * 64);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(smem_u32(sm.v[vs]), a.v_codes + (static_cast<int64_t>(h) * a.kv_stride + tok0) * 64, bytes, bar);
          } else if constexpr (kKvi8r) {
            const uint32_t bytes = static_cast<uint32_t>((a.kv_seq - tok0 < kBN ? a.kv_seq - tok0 : kBN) * 128);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(smem_u32(sm.v[vs] + kChunkBytes), a.v_codes + (static_cast<int64_t>(h) * a.kv_stride + tok0) * 128,
                     bytes, bar);
          } else {
            mbar_arrive_expect_tx(bar, kTileBytes);
            tma_load_3d(smem_u32(sm.v[vs]), &tm_v, 0, static_cast<int32_t>(tok0), h, bar);
            tma_load_3d(smem_u32(sm.v[vs] + kChunkBytes), &tm_v, 64, static_cast<int32_t>(tok0), h, bar);
          }
        }
        ++v_issued[vs];
      }
      if (sm.abort) {
        // every copy this thread issued must land before the CTA exits
        for (int s = 0; s < kNK; ++s)
          if (k_issued[s]) mbar_wait_drain(smem_u32(&sm.k_load[s]), (k_issued[s] - 1) & 1, kDrainNs);
        for (int s = 0; s < kNV; ++s)
          if (v_issued[s]) mbar_wait_drain(smem_u32(&sm.v_load[s]), (v_issued[s] - 1) & 1, kDrainNs);
        if constexpr (!kKvi8r) mbar_wait_drain(smem_u32(&sm.q_full), 0, kDrainNs);
      }
    } else if (warp == 13) {
      // ====================================================== MMA issuer
      // The whole warp runs the loop and waits; one elected lane issues each
      // MMA and commit.  With the warp converged the descriptor arithmetic
      // stays warp-uniform: 7 % faster on kvi8r and 4-6 % on the exact path
      // than a loop run by lane 0 alone.
      const uint32_t go = elect_one();
      constexpr uint32_t idesc_qk = idesc_f16(!kKvi8r, false, kBM, kBN);
      constexpr uint32_t idesc_pv = idesc_f16(!kKvi8r, true, kBM, 128);
      uint64_t *k_rdy = kKvi8r ? sm.k_ready : sm.k_load;
      uint64_t *v_rdy = kKvi8r ? sm.v_ready : sm.v_load;
      // Descriptor start addresses advance by adding (byte offset >> 4) to
      // the low word; every tile lies below 256 KB so the field never wraps.
      // Q, K and V descriptors share the high word (stride 1024 bytes).
      const uint64_t dq0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint32_t dhi = static_cast<uint32_t>(dq0 >> 32);
      const uint32_t lq0 = static_cast<uint32_t>(dq0);
      const uint32_t lk0 = static_cast<uint32_t>(sdesc_sw128(smem_u32(sm.k[0]), 16, 1024));
      const uint32_t lv0 = static_cast<uint32_t>(sdesc_sw128(smem_u32(sm.v[0]), kChunkBytes, 1024));
      auto issue_qk = [&](int q, int ks) {
        const uint32_t lq = lq0 + q * (kTileBytes >> 4);
        const uint32_t lk = lk0 + ks * (kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss(go, tmem + q * 128, lq + off, lk + off, dhi, idesc_qk, kk > 0);
        }
      };
      auto issue_pv = [&](int q, int vs, bool acc) {
        const uint32_t lv = lv0 + vs * (kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(go, tmem + 256 + q * 128, tmem + q * 128 + kk * 8, lv + (kk * 2048 >> 4), dhi, idesc_pv,
                 (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = warp_wait(smem_u32(&sm.q_full), 0, wctx) && warp_wait(smem_u32(&k_rdy[0]), 0, wctx);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        mma_commit(go, smem_u32(&sm.s_full[0]));
        issue_qk(1, 0);
        mma_commit(go, smem_u32(&sm.s_full[1]));
        mma_commit(go, smem_u32(&sm.k_free[0]));
        int jb = 0;  // position of tile j in its kv_block (j % blk, by a counter)
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int vs = j % kNV;
          const bool acc = jb != 0;
          const bool more = j + 1 < n_tiles;
          const int ks1 = (j + 1) % kNK;
          ok = warp_wait(smem_u32(&v_rdy[vs]), (j / kNV) & 1, wctx) &&
               warp_wait(smem_u32(&sm.p_full[0]), j & 1, wctx);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, vs, acc);
          if (more) {
            if (!(ok = warp_wait(smem_u32(&k_rdy[ks1]), ((j + 1) / kNK) & 1, wctx))) break;
            tc_fence_after();
            issue_qk(0, ks1);
            mma_commit(go, smem_u32(&sm.s_full[0]));
          }
          if (!(ok = warp_wait(smem_u32(&sm.p_full[1]), j & 1, wctx))) break;
          tc_fence_after();
          issue_pv(1, vs, acc);
          mma_commit(go, smem_u32(&sm.v_free[vs]));
          if (more) {
            issue_qk(1, ks1);
            mma_commit(go, smem_u32(&sm.s_full[1]));
            mma_commit(go, smem_u32(&sm.k_free[ks1]));
          }
          jb = jb + 1 == blk ? 0 : jb + 1;
        }
        if (ok) mma_commit(go, smem_u32(&sm.o_full));
      }
      // every MMA issued must finish before TMEM is released
      mma_commit(go, smem_u32(&sm.drain));
      mbar_wait_drain(smem_u32(&sm.drain), 0, kDrainNs);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // complete only after the launch this one overlapped
  if (tid == 0) pdl_wait_prerequisites();
}

}  // namespace attn
}  // namespace h3kv
