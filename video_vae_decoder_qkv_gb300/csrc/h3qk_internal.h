// Library-internal helpers shared by the translation units of libh3qk (not
// part of the C-ABI; hidden from the exported symbols).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "h3qk.h"
#include "h3qk_kernels.cuh"

#define H3QK_HIDDEN __attribute__((visibility("hidden")))

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

// Pieces of the device entry points that the host-buffer entry point
// (h3qk_host.cu) reuses; defined in h3qk_api.cu.
namespace h3qk_detail {

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

// One checked call: the kernel parameters, the launch geometry and the byte
// ranges of the inputs (for the aliasing checks of the outputs).
struct Plan {
    h3qk::Params p;
    bool bf16 = false;
    int P = 1;
    cudaStream_t st = nullptr;
    Range ins[5];  // qkv, norm_wq, norm_wk, positions, valid_lens
    int64_t HD = 0;
};

H3QK_HIDDEN bool aligned(const void* p, uintptr_t a);
H3QK_HIDDEN Range range_of(const void* p, int64_t bytes);
H3QK_HIDDEN bool overlap(Range a, Range b);
// Checks of everything that describes the input rows (sizes, options, input
// pointers and their alignment) and the launch plan; `parts` input tensors
// per row (3 packed, 1 single tensor).
H3QK_HIDDEN h3qk_status plan_inputs(const void* qkv, const float* norm_wq, const float* norm_wk,
                                    const int32_t* positions, int64_t tokens, int32_t heads, int32_t head_dim,
                                    int32_t rotary_dim, int64_t valid_len, int default_in, const h3qk_opts& o,
                                    h3qk_stream_t stream, Plan* plan, int parts = 3);
H3QK_HIDDEN bool overlaps_inputs(const Plan& pl, Range r);
// True when the workspace or the counters of extra = {static table, workspace,
// counters} overlap an input, the static table or each other.
H3QK_HIDDEN bool scratch_overlaps(const Plan& pl, const Range (&extra)[3]);
// Zero the amax words, then run the amax pass.
H3QK_HIDDEN h3qk_status run_amax(const Plan& pl);
// The fused kernel of `mode` on the plan's input type.
H3QK_HIDDEN cudaError_t launch(bool bf16, int P, int mode, const h3qk::Params& p, cudaStream_t st);
// Zero three amax words on a stream (no validation).
H3QK_HIDDEN cudaError_t launch_amax_init(unsigned int* words, cudaStream_t st);

}  // namespace h3qk_detail
