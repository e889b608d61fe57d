// Decode-path expert kernels with int4 group-128 (AutoRound / GPTQ layout)
// routed experts (one instance per shared expert format); the kernels
// themselves are in decode_impl.cuh.
#include "decode_impl.cuh"

namespace qmoe {

cudaError_t launch_expert_int4g128(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s) {
  return dec::launch_expert_pair<MOE_FMT_INT4_G128>(sfmt, down, a, smem, s);
}

}  // namespace qmoe
