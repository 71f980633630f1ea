// attend_exact.cu -- exact-store attention launcher (bf16 K/V).
#include "attend.cuh"

namespace h3kv {

cudaError_t launch_attend_exact(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const AttnArgs &args, bool overlap_previous, cudaStream_t stream) {
  const int64_t rows = args.q_end - args.q_begin;
  if (rows <= 0 || args.heads <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn::attend_kernel<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(attn::kSmemBytes));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((rows + kAttnRowsPerCta - 1) / kAttnRowsPerCta),
                  static_cast<unsigned>(args.heads));
  return launch_maybe_overlapped(attn::attend_kernel<false, 1>, grid, attn::kSmemBytes, overlap_previous, stream, q,
                                 k, v, args);
}

}  // namespace h3kv
