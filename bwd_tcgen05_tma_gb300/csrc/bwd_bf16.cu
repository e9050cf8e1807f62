// The 64-row dK/dV pass and the 192-wide dQ pass for bf16 elements.
#include "bwd_passes.cuh"

namespace attn {
template cudaError_t launch_bwd_dkdv_t<ElemBf16>(const KernelArgs&, bool, int, cudaStream_t);
template cudaError_t launch_bwd_dq_t<ElemBf16>(const KernelArgs&, int, cudaStream_t);
}  // namespace attn

#ifdef ATTN_TIMELINE
// Debug builds only: timeline of this translation unit's kernels.
extern "C" int attn_debug_timeline_b64(unsigned long long* out, int cap) {
  cudaDeviceSynchronize();
  const int n = cap < attn::kTimelineCap ? cap : attn::kTimelineCap;
  cudaMemcpyFromSymbol(out, attn::g_timeline, sizeof(unsigned long long) * n);
  static unsigned long long zeros[attn::kTimelineCap];
  cudaMemcpyToSymbol(attn::g_timeline, zeros, sizeof(zeros));
  return n;
}
#endif
