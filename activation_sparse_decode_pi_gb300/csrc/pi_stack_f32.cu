// pi_stack_f32.cu -- persistent decode-step kernel, f32 FFN weights (see pi_stack.cuh).
#include "pi_stack.cuh"

namespace pi {
template cudaError_t launch_stack_wt<0>(int, int, const StackArgs &, int, size_t, cudaStream_t);
}  // namespace pi
