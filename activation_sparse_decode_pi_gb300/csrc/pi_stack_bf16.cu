// pi_stack_bf16.cu -- persistent decode-step kernel, bf16 FFN weights (see pi_stack.cuh).
#include "pi_stack.cuh"

namespace pi {
template cudaError_t launch_stack_wt<1>(int, int, const StackArgs &, int, size_t, cudaStream_t);
}  // namespace pi
