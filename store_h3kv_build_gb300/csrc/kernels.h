// kernels.h -- internal launchers behind the C ABI (not part of the public
// header).  Every launcher validates nothing: the C-ABI layer has checked the
// arguments before calling.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <initializer_list>
#include <utility>

namespace h3kv {

// True when both pointers are device memory aligned to 32 bytes: the store
// builds then write codes with 32-byte stores (host-mapped buffers keep the
// 16-byte stores).
inline bool wide_store_ok(const void *a, const void *b) {
  if (((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 31u) != 0) return false;
  for (const void *p : {a, b}) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
      cudaGetLastError();  // clear the error the query may leave
      return false;
    }
    if (attr.type != cudaMemoryTypeDevice) return false;
  }
  return true;
}

// Store build over `rows` = heads * seq rows of K and V.  Tensor maps: bf16
// [rows, 128] inputs (box 64 x 128, 128B swizzle); int8 codes [rows, 128] and
// fp16 scales are written through plain pointers.
cudaError_t launch_store_build(const CUtensorMap &k_in, const CUtensorMap &v_in, int8_t *k_out,
                               int8_t *v_out, uint16_t *k_scales, uint16_t *v_scales, int64_t rows,
                               int num_sms, int scale_groups, uint32_t *err, uint64_t timeout_ns,
                               cudaStream_t stream);

struct AttnArgs {
  const uint16_t *q;        // bf16 [heads, q_seq, 128]
  const int8_t *k_codes;    // kvi8r store (unused by the exact path); kvfp4:
  const int8_t *v_codes;    //   packed e2m1 pairs, 64 bytes per row
  const uint16_t *k_scales;
  const uint16_t *v_scales;
  const uint8_t *k_fp4_scales;  // kvfp4: e4m3, 8 per row (one per 16 values)
  const uint8_t *v_fp4_scales;
  float *o;                 // fp32 [heads, q_seq, 128]
  int64_t q_seq;
  int64_t kv_seq;           // keys attended by this launch
  int64_t kv_stride;        // rows between heads in the K/V store arrays (kv_seq unless staged)
  int64_t q_begin;          // this launch's query chunk [q_begin, q_end)
  int64_t q_end;
  int32_t heads;            // heads of this launch (grid rows)
  int32_t head_base;        // the head of grid row 0
  int32_t kv_block_tiles;   // 128-key tiles per kv_block
  float scale_log2;         // softmax_scale * log2(e)
  uint32_t *err;
  uint64_t timeout_ns;
  // Staged attention (one kv_block per launch, blocks in order): running
  // (max, sum) per query row [heads, q_seq], carried between launches with O
  // as the running un-normalised output; nullptr for a single launch over all
  // keys.  stage_flags: bit 0 = first block, bit 1 = last block.
  float2 *state;
  int32_t stage_flags;
  int32_t scale_groups;     // kvi8r scales per row: 1, or 4 (one per 32 values)
  // Query chunks streamed from host memory: when q_ready is set, every CTA
  // first waits (bounded) until the word equals q_ready_value, which the copy
  // engine writes once this launch's Q rows are in place and its O buffer is
  // free; nullptr: no wait.
  const uint32_t *q_ready;
  uint32_t q_ready_value;
  // Failure-path diagnostic: 1 + the 128-key tile of each launch whose P-ready
  // arrival the softmax warps withhold, so that the MMA warp's wait for it
  // runs out; 0 (the default) withholds nothing.
  int32_t withhold_p_tile1;
};

constexpr int kAttnRowsPerCta = 256;  // two 128-row query tiles per CTA

// One launch over the query chunk [args.q_begin, args.q_end) of heads
// args.head_base .. args.head_base + args.heads - 1 (one grid row each).
// The exact path reads Q, K, V through 3-D tensor maps ({128, seq, heads},
// box 64 x 128 x 1, 128B swizzle); the kvi8r path reads Q with plain loads
// and the store with bulk copies (the maps are unused).
// overlap_previous: launch with programmatic stream serialization, so that
// this grid's CTAs may start on SMs the previous launch's tail frees.  Only
// for a launch that touches nothing the previous kernel writes (another
// query chunk or head of the same call); the kernels keep completion in
// stream order.
cudaError_t launch_attend_kvi8r(const AttnArgs &args, bool overlap_previous, cudaStream_t stream);

// kvfp4 store build: K rotated, V not; per 16-value block an e4m3 scale and
// e2m1 codes.  Tensor maps: bf16 [rows, 128] inputs (box 64 x 128, 128B
// swizzle); codes [rows, 64] and scales [rows, 8] through plain pointers.
cudaError_t launch_store_build_fp4(const CUtensorMap &k_in, const CUtensorMap &v_in, uint8_t *k_out,
                                   uint8_t *v_out, uint8_t *k_scales, uint8_t *v_scales, int64_t rows,
                                   int num_sms, uint32_t *err, uint64_t timeout_ns, cudaStream_t stream);

// kvfp4 attention over [q_begin, q_end): the kvi8r kernel with the store's
// K/V blocks dequantised from e2m1 x e4m3 (exact in fp16) and no output
// un-rotation (V is not rotated).
cudaError_t launch_attend_fp4(const AttnArgs &args, bool overlap_previous, cudaStream_t stream);

// kvf8s store build: statistics pass (K mean, V channel absmax) then the
// encode pass.  Tensor maps: bf16 [heads, seq, 128] inputs ({128, seq,
// heads}, box 64 x 128 x 1, 128B swizzle; the statistics pass reads K and V
// through the plain pointers).  V codes are written channel-major with row
// stride v_stride (a multiple of 16, >= seq).
cudaError_t launch_store_build_f8(const CUtensorMap &k_in, const CUtensorMap &v_in, const uint16_t *K,
                                  const uint16_t *V, int32_t heads, int64_t seq, int64_t v_stride, uint8_t *k_codes,
                                  uint8_t *v_codes_t, float *k_scales, float *v_scales, float *k_mean, int num_sms,
                                  uint32_t *err, uint64_t timeout_ns, cudaStream_t stream);

struct F8Args {
  const uint16_t *q;        // bf16 [heads, q_seq, 128]
  float *o;                 // fp32 [heads, q_seq, 128]
  const float *k_scales;    // [heads, k_blocks], one per 64 keys
  const float *v_scales;    // [heads, 128], one per channel
  int64_t q_seq;
  int64_t kv_seq;
  int64_t q_begin;          // this launch's query chunk [q_begin, q_end)
  int64_t q_end;
  int32_t heads;            // heads of this launch (grid rows)
  int32_t head_base;        // the head of grid row 0
  int32_t kv_block_tiles;   // 128-key tiles per kv_block
  int32_t k_blocks;         // ceil(kv_seq / 64)
  float scale_log2;         // softmax_scale * log2(e)
  uint32_t *err;
  uint64_t timeout_ns;
  int32_t withhold_p_tile1;  // as AttnArgs::withhold_p_tile1
};

// kvf8s attention over [q_begin, q_end): K codes through a 3-D map {128,
// seq, heads} and channel-major V codes through {seq, 128, heads}, both u8,
// box 128 x 128 x 1, 128B swizzle.
cudaError_t launch_attend_f8(const CUtensorMap &k_codes, const CUtensorMap &v_codes_t, const F8Args &args,
                             bool overlap_previous, cudaStream_t stream);
cudaError_t launch_attend_exact(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const AttnArgs &args, bool overlap_previous, cudaStream_t stream);

// Launch `kernel` (512 threads) normally, or with programmatic stream
// serialization when `overlap` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_overlapped(void (*kernel)(KArgs...), dim3 grid, size_t smem, bool overlap,
                                    cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(512);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace h3kv
