// Library-internal helpers shared by the translation units of libh3qk (not
// part of the C-ABI; hidden from the exported symbols).
#pragma once

#include <cuda_runtime.h>

#include "h3qk.h"

__attribute__((visibility("hidden"))) int h3qk_internal_sm_count();
__attribute__((visibility("hidden"))) void h3qk_internal_count_launch();
__attribute__((visibility("hidden"))) h3qk_status h3qk_internal_fail_cuda(cudaError_t e);
