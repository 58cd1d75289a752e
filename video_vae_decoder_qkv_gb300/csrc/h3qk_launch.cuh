// Kernel launches of one input type (BF16 true or false): the mode's lane
// layout, the plain or head-sliced kernel, and the grid.  Included by
// h3qk_launch_bf16.cu and h3qk_launch_fp16.cu, one instance set each.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "h3qk_internal.h"
#include "h3qk_kernels.cuh"

// Grid size per mode: 0 = up to 8 blocks per SM (the kernel grid-strides over
// the rest); k > 0 = k whole waves of the blocks that fit on an SM at once.
#ifndef H3QK_BLOCKS_PER_SM
#define H3QK_BLOCKS_PER_SM 8
#endif
#ifndef H3QK_WAVES_OUT16
#define H3QK_WAVES_OUT16 0
#endif
#ifndef H3QK_WAVES_AMAX
#define H3QK_WAVES_AMAX 1
#endif
#ifndef H3QK_WAVES_CAST
#define H3QK_WAVES_CAST 4
#endif
#ifndef H3QK_WAVES_SAGE
#define H3QK_WAVES_SAGE 0
#endif

namespace h3qk_launch {
// Internal linkage on purpose: function-local statics of templates with
// external linkage become process-wide unique symbols, which the dynamic
// linker would share with any other copy of this library in the process
// (one copy would then skip raising the shared memory limit of its own
// kernels).
namespace {

constexpr int kMaxDevices = 64;

template <int MODE>
constexpr int waves()
{
    return MODE == h3qk::kOut16 ? H3QK_WAVES_OUT16
                                : (MODE == h3qk::kAmax ? H3QK_WAVES_AMAX
                                                       : (MODE == h3qk::kCast || MODE == h3qk::kCastCount
                                                              ? H3QK_WAVES_CAST
                                                              : H3QK_WAVES_SAGE));
}

// One launch of a mode.  The grid covers the call's row groups (32/LPR
// token rows per warp, Shape<MODE, LPR>::W warps per block), capped at 8
// blocks per SM or at whole waves (waves() above); the kernel grid-strides
// over the rest.  Modes with a shared-memory pipeline
// take dynamic shared memory; the kernel's dynamic limit is raised to that
// size once per device (static and dynamic together may exceed the 48 KB
// default).
template <bool BF16, int LPR, int CH, int MODE, bool SLICED, int RM>
cudaError_t launch_sliced(const h3qk::Params& p, cudaStream_t st)
{
    constexpr size_t smem = h3qk::stage_bytes<LPR, CH, MODE>();
    static_assert(smem <= 227 * 1024, "a block's pipeline stages exceed the 227 KB of shared memory per block");
    constexpr int W = h3qk::Shape<MODE, LPR>::W;
    constexpr int NT = h3qk::Shape<MODE, LPR>::NT;
    auto* kernel = h3qk::qkprep_kernel<BF16, LPR, CH, MODE, SLICED, RM>;
    if constexpr (smem > 0) {
        static std::mutex mu;
        static bool raised[kMaxDevices] = {false};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
        std::lock_guard<std::mutex> lock(mu);
        if (!raised[dev]) {
            const cudaError_t e =
                cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            raised[dev] = true;
        }
    }
    constexpr int64_t tpw = h3qk::rows_per_item<MODE, LPR>();
    const int64_t groups = ((p.rows + tpw - 1) / tpw) << (SLICED ? p.hs_shift : 0);
    const int64_t want = (groups + W - 1) / W;
    int64_t cap = static_cast<int64_t>(h3qk_internal_sm_count()) * H3QK_BLOCKS_PER_SM;
    if constexpr (waves<MODE>() > 0) {
        // A whole number of waves of the blocks that fit on an SM at once.
        static int occ[kMaxDevices] = {0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
        if (occ[dev] == 0) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, NT, smem) != cudaSuccess || n < 1)
                n = 1;
            occ[dev] = n;
        }
        cap = static_cast<int64_t>(h3qk_internal_sm_count()) * occ[dev] * waves<MODE>();
    }
    const int blocks = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
    if (p.chained) {
        // A programmatic dependent of the previous kernel on the stream: it
        // may be scheduled before that kernel completes and waits for it
        // (griddepcontrol.wait) before touching what it writes.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(NT);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
        h3qk_internal_count_launch();
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    kernel<<<blocks, NT, smem, st>>>(p);
    h3qk_internal_count_launch();
    return cudaGetLastError();
}

// A call whose row groups would fill fewer than about 16 warps per SM splits
// each group's heads into 2^shift slices of at least 2 heads (no slice
// empty: the copy pipeline walks one batch sequence per slice and part) and
// runs the sliced kernel; every other call runs the plain kernel.
// The instance for the call's rotation mode: the e4m3 modes on pairs of
// chunks have one per RotMode (rotation choices fixed at compile time), the
// other modes only the general one.
template <bool BF16, int LPR, int CH, int MODE, bool SLICED>
cudaError_t launch_rm(const h3qk::Params& p, cudaStream_t st)
{
    constexpr bool pairs = (MODE == h3qk::kAmax || MODE == h3qk::kCast || MODE == h3qk::kCastCount) && CH >= 2;
    if constexpr (pairs) {
        switch (h3qk::rot_mode_of(p.rotary_dim, p.head_dim, LPR, CH)) {
        case h3qk::kRotAll: return launch_sliced<BF16, LPR, CH, MODE, SLICED, h3qk::kRotAll>(p, st);
        case h3qk::kRotFirst:
            if constexpr (CH == 2) return launch_sliced<BF16, LPR, CH, MODE, SLICED, h3qk::kRotFirst>(p, st);
            break;
        default: break;
        }
    }
    return launch_sliced<BF16, LPR, CH, MODE, SLICED, h3qk::kRotAny>(p, st);
}

template <bool BF16, int LPR, int CH, int MODE>
cudaError_t launch_one(const h3qk::Params& p0, cudaStream_t st)
{
    constexpr int64_t tpw = h3qk::rows_per_item<MODE, LPR>();
    const int64_t groups = (p0.rows + tpw - 1) / tpw;
    const int64_t target = static_cast<int64_t>(h3qk_internal_sm_count()) * 16;
    const int heads = p0.heads;
    int shift = 0;
    while (shift < 4 && (groups << shift) < target && (heads + (2 << shift) - 1) / (2 << shift) >= 2) ++shift;
    int per = (heads + (1 << shift) - 1) >> shift;
    while (shift > 0 && ((1 << shift) - 1) * per >= heads) {
        --shift;
        per = (heads + (1 << shift) - 1) >> shift;
    }
    if (shift == 0) return launch_rm<BF16, LPR, CH, MODE, false>(p0, st);
    h3qk::Params p = p0;
    p.hs_shift = shift;
    p.hs_heads = per;
    return launch_rm<BF16, LPR, CH, MODE, true>(p, st);
}

// P = next_pow2(D/8) chunk slots per head row: the mode's CH per lane on
// P/CH lanes (fewer per lane when P < CH).
template <bool BF16, int MODE>
cudaError_t launch_p(int P, const h3qk::Params& p, cudaStream_t st)
{
    constexpr int CH = h3qk::Tune<MODE>::CH;
    static_assert(CH == 1 || CH == 2 || CH == 4, "1, 2 or 4 chunks per lane");
    if (P < CH) {
        if (P == 1) return launch_one<BF16, 1, 1, MODE>(p, st);
        return launch_one<BF16, 1, 2, MODE>(p, st);  // P == 2 < CH == 4
    }
    switch (P / CH) {
    case 1: return launch_one<BF16, 1, CH, MODE>(p, st);
    case 2: return launch_one<BF16, 2, CH, MODE>(p, st);
    case 4: return launch_one<BF16, 4, CH, MODE>(p, st);
    case 8: return launch_one<BF16, 8, CH, MODE>(p, st);
    case 16: return launch_one<BF16, 16, CH, MODE>(p, st);
    default: return launch_one<BF16, 32 / CH, CH, MODE>(p, st);
    }
}

template <bool BF16>
cudaError_t launch_m(int P, int mode, const h3qk::Params& p, cudaStream_t st)
{
    switch (mode) {
    case h3qk::kOut16: return launch_p<BF16, h3qk::kOut16>(P, p, st);
    case h3qk::kAmax: return launch_p<BF16, h3qk::kAmax>(P, p, st);
    case h3qk::kSage: return launch_p<BF16, h3qk::kSage>(P, p, st);
    case h3qk::kCastCount: return launch_p<BF16, h3qk::kCastCount>(P, p, st);
    default: return launch_p<BF16, h3qk::kCast>(P, p, st);
    }
}


}  // namespace
}  // namespace h3qk_launch
