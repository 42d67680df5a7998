// pi_tc_f16_pred.cu -- tensor-core batch >= 16 kernels, f16 weights, pred products (see pi_tc.cuh).
#include "pi_tc.cuh"

namespace pi {
template cudaError_t launch_tc_mode<2, 0>(int, int, const TcArgs &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_tc_mode<2, 1>(int, int, const TcArgs &, int, size_t, cudaStream_t, bool);
template cudaError_t launch_tc_split_wt<2>(const float *, int, int, int, int, int, float, uint16_t *, uint16_t *,
                                           cudaStream_t, bool);
}  // namespace pi
