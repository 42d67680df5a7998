// pi_tc_bf16_down.cu -- tensor-core batch >= 16 kernels, bf16 weights, down products (see pi_tc.cuh).
#include "pi_tc.cuh"

namespace pi {
template cudaError_t launch_tc_mode<1, 4>(int, int, const TcArgs &, int, size_t, cudaStream_t, bool);
}  // namespace pi
