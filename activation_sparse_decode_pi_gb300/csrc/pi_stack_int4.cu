// pi_stack_int4.cu -- persistent decode-step kernel, int4 FFN weights (see pi_stack.cuh).
#include "pi_stack.cuh"

namespace pi {
template cudaError_t launch_stack_wt<3>(int, int, const StackArgs &, int, size_t, cudaStream_t);
}  // namespace pi
