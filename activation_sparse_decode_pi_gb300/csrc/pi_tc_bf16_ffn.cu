// pi_tc_bf16_ffn.cu -- tensor-core batch >= 16 kernels, bf16 weights, ffn products (see pi_tc.cuh).
#include "pi_tc.cuh"

namespace pi {
template cudaError_t launch_tc_mode<1, 2>(int, int, const TcArgs &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_tc_mode<1, 3>(int, int, const TcArgs &, int, size_t, cudaStream_t, bool);
}  // namespace pi
