// Kernel instances and launches for bfloat16 inputs.
#include "h3qk_launch.cuh"

cudaError_t h3qk_internal_launch_bf16(int P, int mode, const h3qk::Params& p, cudaStream_t st)
{
    return h3qk_launch::launch_m<true>(P, mode, p, st);
}
