// Adjacent VAE-block operations of the MiniMax-H3 decoder block, as in the
// vllm-omni MiniMax-H3 VAE decoder operators page ("Operations" table):
//  - SwiGLU: SiLU(gate) * up after the 16-bit w1 projection;
//  - scaled residual: FP32 residual + 16-bit branch * FP32 scale, with
//    multiply-add contraction disabled.
// Both are streaming elementwise kernels bound by HBM bandwidth: each thread
// moves 8 elements per step with 128-bit loads and stores, grid-stride over
// a grid of at most 8 blocks per SM.  Every rounding point is an explicit
// correctly rounded intrinsic, so results match the CPU oracle bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "h3qk.h"
#include "h3qk_internal.h"

namespace {

constexpr int kThreads = 256;

template <bool BF16>
__device__ __forceinline__ float2 widen2v(uint32_t w)
{
    if constexpr (BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        return __half22float2(h);
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t round2v(float lo, float hi)
{
    if constexpr (BF16) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&b);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// e^x: the library's own routine.  Cody & Waite reduction x = k ln2 + r with
// ln2 split in two binary32 parts (each step one fused multiply-add), the
// Taylor series of e^r to r^8 in Horner form, then one rounded product with
// 2^k (k = 128 as 2^127 then 2).  NaN stays NaN, x > 89 gives +inf, results
// below 2^-126 give 0 (there 1 + e^x already rounds to 1).  Constants:
// log2(e), ln2 and its tail, 1/n!, each rounded to binary32.
__device__ __forceinline__ float exp_h3(float x)
{
    constexpr float kLog2e = 0x1.715476p+0f;
    constexpr float kLn2Hi = 0x1.62e430p-1f;
    constexpr float kLn2Lo = -0x1.05c610p-29f;
    constexpr float kE2 = 0x1.000000p-1f, kE3 = 0x1.555556p-3f, kE4 = 0x1.555556p-5f;
    constexpr float kE5 = 0x1.111112p-7f, kE6 = 0x1.6c16c2p-10f, kE7 = 0x1.a01a02p-13f;
    constexpr float kE8 = 0x1.a01a02p-16f;
    if (x != x) return x;
    if (x > 89.0f) return __int_as_float(0x7f800000);
    if (x < -104.0f) return 0.0f;
    const float k = rintf(__fmul_rn(x, kLog2e));
    float r = __fmaf_rn(-k, kLn2Hi, x);
    r = __fmaf_rn(-k, kLn2Lo, r);
    float p = __fmaf_rn(kE8, r, kE7);
    p = __fmaf_rn(p, r, kE6);
    p = __fmaf_rn(p, r, kE5);
    p = __fmaf_rn(p, r, kE4);
    p = __fmaf_rn(p, r, kE3);
    p = __fmaf_rn(p, r, kE2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ki = static_cast<int>(k);
    if (ki < -126) return 0.0f;
    // k = 128: 2^128 is not a binary32; scale by 2^127, then by 2 (both exact
    // until overflow).
    const int k1 = ki > 127 ? 127 : ki;
    const float y = __fmul_rn(p, __int_as_float((k1 + 127) << 23));
    return ki > 127 ? __fmul_rn(y, 2.0f) : y;
}

// SiLU(g) = g / (1 + e^-g): one rounded sum, one correctly rounded division.
__device__ __forceinline__ float silu_h3(float g)
{
    return __fdiv_rn(g, __fadd_rn(1.0f, exp_h3(-g)));
}

// out[r, j] = round16(silu(x[r, j]) * x[r, f + j]) for j < f, eight j per step.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) silu_and_mul_kernel(const uint16_t* __restrict__ x,
                                                                uint16_t* __restrict__ out, int64_t rows,
                                                                int f, int64_t row_stride)
{
    const int64_t per_row = f / 8;
    const int64_t n = rows * per_row;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; v < n;
         v += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t r = v / per_row;
        const int64_t j = (v - r * per_row) * 8;
        const uint4 gw = __ldg(reinterpret_cast<const uint4*>(x + r * row_stride + j));
        const uint4 uw = __ldg(reinterpret_cast<const uint4*>(x + r * row_stride + f + j));
        const uint32_t g4[4] = {gw.x, gw.y, gw.z, gw.w};
        const uint32_t u4[4] = {uw.x, uw.y, uw.z, uw.w};
        uint32_t o4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 g = widen2v<BF16>(g4[i]);
            const float2 u = widen2v<BF16>(u4[i]);
            o4[i] = round2v<BF16>(__fmul_rn(silu_h3(g.x), u.x), __fmul_rn(silu_h3(g.y), u.y));
        }
        *reinterpret_cast<uint4*>(out + r * f + j) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
}

// out[i] = residual[i] + branch[i] * scale[c]: the product rounded on its own
// (__fmul_rn is never merged into a multiply-add), then the sum.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) scaled_residual_kernel(const float* residual,
                                                                   const uint16_t* __restrict__ branch,
                                                                   const float* __restrict__ scale,
                                                                   float* out, int64_t n, int channels,
                                                                   int scale_len)
{
    for (int64_t v = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; v * 8 < n;
         v += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t i = v * 8;
        const int c = static_cast<int>(i % channels);
        const float4 r0 = reinterpret_cast<const float4*>(residual + i)[0];
        const float4 r1 = reinterpret_cast<const float4*>(residual + i)[1];
        const uint4 bw = __ldg(reinterpret_cast<const uint4*>(branch + i));
        float sc[8];
        if (scale_len == 1) {
            const float s0 = __ldg(scale);
#pragma unroll
            for (int k = 0; k < 8; ++k) sc[k] = s0;
        } else {
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(scale + c));
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(scale + c) + 1);
            sc[0] = s0.x; sc[1] = s0.y; sc[2] = s0.z; sc[3] = s0.w;
            sc[4] = s1.x; sc[5] = s1.y; sc[6] = s1.z; sc[7] = s1.w;
        }
        const float res[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const uint32_t b4[4] = {bw.x, bw.y, bw.z, bw.w};
        float o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 b = widen2v<BF16>(b4[k]);
            o[2 * k] = __fadd_rn(res[2 * k], __fmul_rn(b.x, sc[2 * k]));
            o[2 * k + 1] = __fadd_rn(res[2 * k + 1], __fmul_rn(b.y, sc[2 * k + 1]));
        }
        reinterpret_cast<float4*>(out + i)[0] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(out + i)[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
}

int grid_for(int64_t vectors)
{
    const int64_t want = (vectors + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(h3qk_internal_sm_count()) * 8;
    return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

}  // namespace

extern "C" h3qk_status h3qk_silu_and_mul(const void* x, h3qk_dtype dtype, int64_t rows, int32_t f,
                                         int64_t row_stride, void* out, h3qk_stream_t stream)
{
    if (rows < 0 || f < 0 || f % 8) return H3QK_ERR_INVALID_ARG;
    if (dtype != H3QK_FP16 && dtype != H3QK_BF16) return H3QK_ERR_INVALID_ARG;
    if (row_stride == 0) row_stride = 2 * static_cast<int64_t>(f);
    if (row_stride < 2 * static_cast<int64_t>(f)) return H3QK_ERR_INVALID_ARG;
    if (rows > 0 && f > 0 && (!x || !out)) return H3QK_ERR_INVALID_ARG;
    if (row_stride % 8 || !aligned16(x) || !aligned16(out)) return H3QK_ERR_MISALIGNED;
    const int64_t in_bytes = rows > 0 ? ((rows - 1) * row_stride + 2 * static_cast<int64_t>(f)) * 2 : 0;
    if (overlaps(out, rows * f * 2, x, in_bytes)) return H3QK_ERR_ALIAS;
    if (rows == 0 || f == 0) return H3QK_OK;
    const int blocks = grid_for(rows * (f / 8));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == H3QK_BF16)
        silu_and_mul_kernel<true><<<blocks, kThreads, 0, st>>>(static_cast<const uint16_t*>(x),
                                                                static_cast<uint16_t*>(out), rows, f, row_stride);
    else
        silu_and_mul_kernel<false><<<blocks, kThreads, 0, st>>>(static_cast<const uint16_t*>(x),
                                                                 static_cast<uint16_t*>(out), rows, f, row_stride);
    h3qk_internal_count_launch();
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3QK_OK : h3qk_internal_fail_cuda(e);
}

extern "C" h3qk_status h3qk_scaled_residual(const float* residual, const void* branch, h3qk_dtype branch_dtype,
                                            const float* scale, int64_t rows, int32_t channels,
                                            int32_t scale_len, float* out, h3qk_stream_t stream)
{
    if (rows < 0 || channels < 0 || channels % 8) return H3QK_ERR_INVALID_ARG;
    if (branch_dtype != H3QK_FP16 && branch_dtype != H3QK_BF16) return H3QK_ERR_INVALID_ARG;
    if (scale_len != 1 && scale_len != channels) return H3QK_ERR_INVALID_ARG;
    const int64_t n = rows * channels;
    if (n > 0 && (!residual || !branch || !scale || !out)) return H3QK_ERR_INVALID_ARG;
    if (!aligned16(residual) || !aligned16(branch) || !aligned16(out)) return H3QK_ERR_MISALIGNED;
    if (scale_len != 1 && !aligned16(scale)) return H3QK_ERR_MISALIGNED;
    if (scale_len == 1 && (reinterpret_cast<uintptr_t>(scale) & 3u)) return H3QK_ERR_MISALIGNED;
    // out may be the residual itself (an in-place update), nothing else.
    if (out != residual && overlaps(out, n * 4, residual, n * 4)) return H3QK_ERR_ALIAS;
    if (overlaps(out, n * 4, branch, n * 2) || overlaps(out, n * 4, scale, scale_len * 4)) return H3QK_ERR_ALIAS;
    if (n == 0) return H3QK_OK;
    const int blocks = grid_for(n / 8);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (branch_dtype == H3QK_BF16)
        scaled_residual_kernel<true><<<blocks, kThreads, 0, st>>>(residual, static_cast<const uint16_t*>(branch),
                                                                   scale, out, n, channels, scale_len);
    else
        scaled_residual_kernel<false><<<blocks, kThreads, 0, st>>>(residual, static_cast<const uint16_t*>(branch),
                                                                    scale, out, n, channels, scale_len);
    h3qk_internal_count_launch();
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3QK_OK : h3qk_internal_fail_cuda(e);
}
