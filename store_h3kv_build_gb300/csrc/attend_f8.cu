// attend_f8.cu -- attention over the kvf8s store (fp8 e4m3 K and V in the
// kvi8s layout; "The K/V store options" table of the Low VRAM write-up,
// kvi8s row: attended on fp8 tensor cores straight from the store, no
// dequantisation).
//
// Both products are tcgen05.mma kind::f8f6f4 (e4m3 x e4m3, fp32 in TMEM):
//   S = Qc Kc^T   with Qc the e4m3 codes of q' = q H (one fp32 scale per query
//                 row) and Kc the stored codes (one scale per 64-token block);
//   O = Pc Vc     with Pc the e4m3 encoding of the un-normalised softmax
//                 weights and Vc the stored channel-major V codes.
// The scales never touch the tiles: s_q * s_k * softmax_scale becomes the
// per-column-half multiplier of the exponent (a 128-key tile spans two K
// blocks), and the per-channel V scale multiplies O once in the epilogue.
// V is not rotated, so the output needs no un-rotation.
//
// Layout and schedule follow the bf16/kvi8r kernel (attend.cuh): one CTA =
// 256 query rows of one head as two 128-row tiles ping-ponging between
// softmax and the tensor core; warps 0-7 softmax, warp 12 TMA producer,
// warp 13 MMA issuer.  There is no dequantisation warpgroup.
#include "attend.cuh"

namespace h3kv {
namespace attn_f8 {

using attn::kBM;
using attn::kBN;
using attn::kNQ;
using attn::kThreads;
using attn::kWarpsPerGroup;

constexpr int kTile8 = 128 * 128;  // one [128 x 128] tile of 8-bit codes
constexpr int kNK = 6;             // K ring depth
constexpr int kNV = 4;             // V ring depth
// Lazy rescale threshold (log2 units): O and the running sum are rescaled
// only when a row's max grows by more than 2^3, so the un-normalised weights
// stay below 2^3; with p' = p * 448 / 2^3 the largest weight is e4m3's 448
// and smaller ones keep the format's normal range down to ~2.8e-4.
constexpr float kLazyLog2 = 3.0f;
constexpr float kLog2PScale = 5.807354922057604f;  // log2(448 / 8)
constexpr uint32_t kRegSoftmax = 200, kRegIdle = 24, kRegIssue = 88;
static_assert(2 * kRegSoftmax + kRegIdle + kRegIssue == 512, "register split");

struct Smem {
  uint8_t q[kNQ][kTile8];
  uint8_t k[kNK][kTile8];
  uint8_t v[kNV][kTile8];
  uint64_t q_full;
  uint64_t k_full[kNK], k_free[kNK];
  uint64_t v_full[kNV], v_free[kNV];
  uint64_t s_full[kNQ], p_full[kNQ];
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
// the epilogue stages kNQ x [128 rows x 512 bytes] of fp32 over q and k
static_assert(sizeof(Smem::q) + sizeof(Smem::k) >= kNQ * 128 * 512, "epilogue staging");

__global__ void __launch_bounds__(kThreads, 1)
    attend_f8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const F8Args a) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = a.head_base + static_cast<int>(blockIdx.y);
  const int64_t row0 = a.q_begin + static_cast<int64_t>(blockIdx.x) * (kNQ * kBM);
  const int n_tiles = static_cast<int>((a.kv_seq + kBN - 1) / kBN);
  const int blk = a.kv_block_tiles;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.q_full), 2 * kWarpsPerGroup);
    for (int s = 0; s < kNK; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_free[s]), 1);
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(smem_u32(&sm.v_full[s]), 1);
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
    reg_alloc<kRegSoftmax>();
    const int q = warp >> 2;
    const uint32_t i = tid & 127;  // row in the query tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + q * 128;
    const uint32_t tO = tmem + lane_base + 256 + q * 128;
    const int64_t row = row0 + q * kBM + i;
    const bool row_ok = row < a.q_end;
    float *orow = a.o + (static_cast<int64_t>(h) * a.q_seq + (row_ok ? row : 0)) * 128;

    // Query rows: q' = q H, one fp32 scale s = absmax/448 per row, e4m3
    // codes of q' * fp32(1/s) written K-major (128 bytes per row, 128B swizzle).  Warp
    // w encodes its own 32 rows one at a time across the warp; lane rr keeps
    // the scale of row rr, which is its own TMEM lane.
    float my_sq = 0.f;
    {
      const int wq = warp & 3;
      uint2 buf[32];
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) {
        const int64_t r = row0 + q * kBM + wq * 32 + rr;
        buf[rr] = r < a.q_end ? *reinterpret_cast<const uint2 *>(a.q + (static_cast<int64_t>(h) * a.q_seq + r) * 128 +
                                                                  4 * lane)
                              : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) {
        const uint32_t ti = wq * 32 + rr;
        float x[4] = {bf16lo_to_f32(buf[rr].x), bf16hi_to_f32(buf[rr].x), bf16lo_to_f32(buf[rr].y),
                      bf16hi_to_f32(buf[rr].y)};
        fwht128_warp(x, lane);
        float amax = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          x[t] *= kInvSqrt128;
          amax = fmaxf(amax, fabsf(x[t]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(amax, 448.0f);
        const float rs = s > 0.f ? __frcp_rn(s) : 0.f;
        const uint32_t w = s > 0.f ? pack_e4m3x4(__fmul_rn(x[0], rs), __fmul_rn(x[1], rs), __fmul_rn(x[2], rs),
                                                 __fmul_rn(x[3], rs))
                                   : 0u;
        *reinterpret_cast<uint32_t *>(sm.q[q] + sw128_off(ti, lane >> 2) + (lane & 3) * 4) = w;
        if (lane == rr) my_sq = s;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.q_full));
    }

    // Every quantity below is in log2 units of the scaled score ("x"):
    // x = S * s_q * s_k * softmax_scale * log2(e).
    const float cq = a.scale_log2 * my_sq;
    const float *ksc = a.k_scales + static_cast<int64_t>(h) * a.k_blocks;
    float m_b = 0.f, l_b = 0.f;  // current kv_block: running max and sum of the (scaled) weights
    float M = 0.f, Lam = 0.f;    // blocks merged so far
    bool ok = true;
    int jb = 0;                  // position of tile j in its kv_block (j % blk, by a counter)
    for (int j = 0; j < n_tiles; ++j) {
      // the tile's two K block scales (loaded before the wait hides their latency)
      const int b0 = 2 * j;
      const float sk0 = ksc[b0];
      const float sk1 = b0 + 1 < a.k_blocks ? ksc[b0 + 1] : 0.f;
      if (!attn::warp_wait(smem_u32(&sm.s_full[q]), j & 1, wctx)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
      float m4[4];  // raw maxima of the four 32-key groups, from the loads
      tmem_ld128_max(tS, *reinterpret_cast<uint32_t(*)[128]>(s), m4);
      float mult0 = cq * sk0, mult1 = cq * sk1;
      const int64_t valid = a.kv_seq - static_cast<int64_t>(j) * kBN;
      if (valid < kBN) {
        // tail tile: scale explicitly and mask the keys past the sequence
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < valid) ? s[c] * (c < 64 ? mult0 : mult1) : -INFINITY;
        mult0 = mult1 = 1.f;
      }
      float mt;
      if (valid >= kBN) {
        // raw maxima of each 64-key half, then scaled (multipliers >= 0)
        mt = fmaxf(fmaxf(m4[0], m4[1]) * mult0, fmaxf(m4[2], m4[3]) * mult1);
      } else {
        // the tail tile, scaled and masked above
        // elements 2 .. 63 of each half: 31 pairs over two accumulators
        float h0[2] = {s[0], s[1]}, h1[2] = {s[64], s[65]};
#pragma unroll
        for (int p = 0; p < 31; ++p) {
          const int c = 2 + 2 * p;
          h0[p & 1] = fmax3(h0[p & 1], s[c], s[c + 1]);
          h1[p & 1] = fmax3(h1[p & 1], s[64 + c], s[64 + c + 1]);
        }
        mt = fmaxf(fmaxf(h0[0], h0[1]) * mult0, fmaxf(h1[0], h1[1]) * mult1);
      }

      if (jb == 0) {
        if (j > 0) {
          // merge the finished kv_block (O_q, m_b, l_b) into (M, Lam, O row
          // in global memory, un-normalised)
          const bool first = j == blk;
          float al = 0.f, be = 1.f;
          if (!first) {
            attn::lse_merge(M, Lam, m_b, l_b, 1.0f, al, be);
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
        const bool need = mt - m_b > kLazyLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m_b - mt) : 1.f;
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

      // p' = 2^(x - m_b) * 448 / 2^3, four per 32-bit column as e4m3, over
      // the first 32 columns of S
      const float2 nm = make_float2(kLog2PScale - m_b, kLog2PScale - m_b);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const float2 mm = hlf ? make_float2(mult1, mult1) : make_float2(mult0, mult0);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int c = hlf * 64 + 4 * k;
          float2 e0 = __ffma2_rn(make_float2(s[c], s[c + 1]), mm, nm);
          float2 e1 = __ffma2_rn(make_float2(s[c + 2], s[c + 3]), mm, nm);
          e0.x = ex2(e0.x);
          e0.y = ex2(e0.y);
          e1.x = ex2(e1.x);
          e1.y = ex2(e1.y);
          acc0 = __fadd2_rn(acc0, e0);
          acc1 = __fadd2_rn(acc1, e1);
          pk[hlf * 16 + k] = pack_e4m3x4(e0.x, e0.y, e1.x, e1.y);
        }
      }
      tmem_st32(tS, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      // (a diagnostic may withhold one tile's arrival: see withhold_p_tile1)
      if (lane == 0 && j + 1 != a.withhold_p_tile1) mbar_arrive(smem_u32(&sm.p_full[q]));
      const float2 acc = __fadd2_rn(acc0, acc1);
      l_b += acc.x + acc.y;
      jb = jb + 1 == blk ? 0 : jb + 1;
    }

    if (ok && attn::warp_wait(smem_u32(&sm.o_full), 0, wctx)) {
      // epilogue, phase 1: each thread finishes its own row (final block
      // merge, 1/Lambda) and stages it in shared memory, fp32, with 16-byte
      // granule gi of row i at position gi ^ (i mod 32).  The operand rings
      // are free now: every MMA has completed and no copy is outstanding.
      tc_fence_after();
      const int n_blocks = (n_tiles + blk - 1) / blk;
      uint8_t *stage = sm.q[0] + q * (128 * 512);
      float ga, gb;
      if (n_blocks == 1) {
        ga = 0.f;
        gb = 1.f / l_b;
      } else {
        float al, be;
        attn::lse_merge(M, Lam, m_b, l_b, 1.0f, al, be);
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
        if (n_blocks > 1 && row_ok) {
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
      // phase 2: each warp takes its 32 rows one at a time across the warp,
      // applies the per-channel V scales and stores coalesced
      const int wq = warp & 3;
      const float4 sv = *reinterpret_cast<const float4 *>(a.v_scales + static_cast<int64_t>(h) * 128 + 4 * lane);
#pragma unroll 4
      for (int rr = 0; rr < 32; ++rr) {
        const uint32_t ti = wq * 32 + rr;
        const float4 v = *reinterpret_cast<const float4 *>(stage + ti * 512 + ((lane ^ (ti & 31)) << 4));
        const int64_t r = row0 + q * kBM + ti;
        if (r < a.q_end)
          *reinterpret_cast<float4 *>(a.o + (static_cast<int64_t>(h) * a.q_seq + r) * 128 + 4 * lane) =
              make_float4(v.x * sv.x, v.y * sv.y, v.z * sv.z, v.w * sv.w);
      }
    }
  } else if (warp < 12) {
    reg_dealloc<kRegIdle>();
  } else {
    reg_dealloc<kRegIssue>();
    if (warp == 12) {
      // ========================================================== producer
      // the whole warp waits; one elected lane issues the copies
      const uint32_t go = elect_one();
      int k_issued[kNK] = {};
      int v_issued[kNV] = {};
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      for (int j = 0; j < n_tiles; ++j) {
        const int32_t tok0 = j * kBN;
        const int ks = j % kNK, vs = j % kNV;
        if (!attn::warp_wait(smem_u32(&sm.k_free[ks]), ((j / kNK) & 1) ^ 1, wctx)) break;
        if (go) {
          const uint32_t bar = smem_u32(&sm.k_full[ks]);
          mbar_arrive_expect_tx(bar, kTile8);
          tma_load_3d(smem_u32(sm.k[ks]), &tm_k, 0, tok0, h, bar);
        }
        ++k_issued[ks];
        if (!attn::warp_wait(smem_u32(&sm.v_free[vs]), ((j / kNV) & 1) ^ 1, wctx)) break;
        if (go) {
          const uint32_t bar = smem_u32(&sm.v_full[vs]);
          mbar_arrive_expect_tx(bar, kTile8);
          tma_load_3d(smem_u32(sm.v[vs]), &tm_v, tok0, 0, h, bar);
        }
        ++v_issued[vs];
      }
      if (sm.abort) {
        // every copy this thread issued must land before the CTA exits
        for (int s = 0; s < kNK; ++s)
          if (k_issued[s]) mbar_wait_drain(smem_u32(&sm.k_full[s]), (k_issued[s] - 1) & 1, kDrainNs);
        for (int s = 0; s < kNV; ++s)
          if (v_issued[s]) mbar_wait_drain(smem_u32(&sm.v_full[s]), (v_issued[s] - 1) & 1, kDrainNs);
      }
    } else if (warp == 13) {
      // ====================================================== MMA issuer
      // the whole warp runs the loop and waits (warp-uniform operands); one
      // elected lane issues each MMA and commit
      const uint32_t go = elect_one();
      constexpr uint32_t idesc = idesc_e4m3(kBM, 128);
      // K-major 128-byte-swizzled operands; one K step (32 codes = 32 bytes)
      // advances the start address by 32 bytes (2 in the >>4 field of the
      // low word); the three descriptors share the high word
      const uint64_t dq0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint32_t dhi = static_cast<uint32_t>(dq0 >> 32);
      const uint32_t lq0 = static_cast<uint32_t>(dq0);
      const uint32_t lk0 = static_cast<uint32_t>(sdesc_sw128(smem_u32(sm.k[0]), 16, 1024));
      const uint32_t lv0 = static_cast<uint32_t>(sdesc_sw128(smem_u32(sm.v[0]), 16, 1024));
      auto issue_qk = [&](int q, int ks) {
        const uint32_t lq = lq0 + q * (kTile8 >> 4);
        const uint32_t lk = lk0 + ks * (kTile8 >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ss_f8(go, tmem + q * 128, lq + 2 * kk, lk + 2 * kk, dhi, idesc, kk > 0);
      };
      auto issue_pv = [&](int q, int vs, bool acc) {
        const uint32_t lv = lv0 + vs * (kTile8 >> 4);
        // P: 32 keys per step = 8 TMEM columns of four e4m3 values
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_f8(go, tmem + 256 + q * 128, tmem + q * 128 + kk * 8, lv + 2 * kk, dhi, idesc,
                    (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = attn::warp_wait(smem_u32(&sm.q_full), 0, wctx) && attn::warp_wait(smem_u32(&sm.k_full[0]), 0, wctx);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        mma_commit(go, smem_u32(&sm.s_full[0]));
        issue_qk(1, 0);
        mma_commit(go, smem_u32(&sm.s_full[1]));
        mma_commit(go, smem_u32(&sm.k_free[0]));
        int jb = 0;  // j mod kv_block_tiles, kept by a counter (no division in the issue loop)
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int vs = j % kNV;
          const bool acc = jb != 0;
          const bool more = j + 1 < n_tiles;
          const int ks1 = (j + 1) % kNK;
          ok = attn::warp_wait(smem_u32(&sm.v_full[vs]), (j / kNV) & 1, wctx) &&
               attn::warp_wait(smem_u32(&sm.p_full[0]), j & 1, wctx);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, vs, acc);
          if (more) {
            if (!(ok = attn::warp_wait(smem_u32(&sm.k_full[ks1]), ((j + 1) / kNK) & 1, wctx))) break;
            tc_fence_after();
            issue_qk(0, ks1);
            mma_commit(go, smem_u32(&sm.s_full[0]));
          }
          if (!(ok = attn::warp_wait(smem_u32(&sm.p_full[1]), j & 1, wctx))) break;
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

}  // namespace attn_f8

cudaError_t launch_attend_f8(const CUtensorMap &k_codes, const CUtensorMap &v_codes_t, const F8Args &args,
                             bool overlap_previous, cudaStream_t stream) {
  const int64_t rows = args.q_end - args.q_begin;
  if (rows <= 0 || args.heads <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_f8::attend_f8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(attn_f8::kSmemBytes));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((rows + kAttnRowsPerCta - 1) / kAttnRowsPerCta),
                  static_cast<unsigned>(args.heads));
  return launch_maybe_overlapped(attn_f8::attend_f8_kernel, grid, attn_f8::kSmemBytes, overlap_previous, stream,
                                 k_codes, v_codes_t, args);
}

}  // namespace h3kv
