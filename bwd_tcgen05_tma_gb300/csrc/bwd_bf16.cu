// The 64-row dK/dV pass and the 192-wide dQ pass for bf16 elements.
#include "bwd_passes.cuh"

namespace attn {
template cudaError_t launch_bwd_dkdv_t<ElemBf16>(const KernelArgs&, bool, int, cudaStream_t);
template cudaError_t launch_bwd_dq_t<ElemBf16>(const KernelArgs&, int, cudaStream_t);
}  // namespace attn
