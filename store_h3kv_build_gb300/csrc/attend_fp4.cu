// attend_fp4.cu -- kvfp4 attention launcher (NVFP4 store dequantised to fp16).
#include "attend.cuh"

namespace h3kv {

cudaError_t launch_attend_fp4(const AttnArgs &args, bool overlap_previous, cudaStream_t stream) {
  const int64_t rows = args.q_end - args.q_begin;
  if (rows <= 0 || args.heads <= 0) return cudaSuccess;
  auto kernel = attn::attend_kernel<true, 1, true>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(attn::kSmemBytes));
  if (e != cudaSuccess) return e;
  CUtensorMap unused;
  memset(&unused, 0, sizeof(unused));
  const dim3 grid(static_cast<unsigned>((rows + kAttnRowsPerCta - 1) / kAttnRowsPerCta),
                  static_cast<unsigned>(args.heads));
  return launch_maybe_overlapped(kernel, grid, attn::kSmemBytes, overlap_previous, stream, unused, unused, unused,
                                 args);
}

}  // namespace h3kv
