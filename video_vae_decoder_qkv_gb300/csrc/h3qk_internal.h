// Library-internal helpers shared by the translation units of libh3qk (not
// part of the C-ABI; hidden from the exported symbols).
#pragma once

#include <cuda_runtime.h>

#include "h3qk.h"

__attribute__((visibility("hidden"))) int h3qk_internal_sm_count();
__attribute__((visibility("hidden"))) void h3qk_internal_count_launch();
__attribute__((visibility("hidden"))) h3qk_status h3qk_internal_fail_cuda(cudaError_t e);

namespace h3qk {
struct Params;
}
// Launch the fused kernel of `mode` for P chunk slots per head row on bf16 /
// binary16 inputs (h3qk_launch_bf16.cu, h3qk_launch_fp16.cu).
__attribute__((visibility("hidden"))) cudaError_t h3qk_internal_launch_bf16(int P, int mode, const h3qk::Params& p,
                                                                             cudaStream_t st);
__attribute__((visibility("hidden"))) cudaError_t h3qk_internal_launch_fp16(int P, int mode, const h3qk::Params& p,
                                                                             cudaStream_t st);
