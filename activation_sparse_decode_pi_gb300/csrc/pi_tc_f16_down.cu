// pi_tc_f16_down.cu -- tensor-core batch >= 16 kernels, f16 weights, down products (see pi_tc.cuh).
#include "pi_tc.cuh"

namespace pi {
template cudaError_t launch_tc_mode<2, 4>(int, int, const TcArgs &, int, size_t, cudaStream_t, bool);
}  // namespace pi
